"""The C ABI used from plain C: tests/c/fa_c_consumer.c includes include/fa.h,
links libfa.so and the CUDA runtime, and calls fa_fwd / fa_bwd on buffers it
allocates itself.  On CPU: the header compiles as C11 and the program links.
On the GPU: its outputs match the fp64 oracle on the inputs it drew."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from flashattention_backward_preprocess_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "fa_c_consumer.c")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _compile(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = build.build()
    libdir = os.path.dirname(lib)
    cuda = _cuda_home()
    cudalib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                os.path.join(cuda, "targets", "sbsa-linux", "lib"))
                    if os.path.exists(os.path.join(p, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("libcudart.so not found")
    exe = tmp_path / "fa_c_consumer"
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lfa", "-L", cudalib, "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_header_compiles_as_c_and_program_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


def _bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 300, 128, 1), (2, 2, 2, 130, 257, 64, 0)])
def test_c_program_results_match_oracle(tmp_path, shape):
    exe = _compile(tmp_path)
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(out), *map(str, shape)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
    raw = out.read_bytes()
    B, H, H_kv, S_q, S_k, d, causal = np.frombuffer(raw[:28], dtype=np.int32)
    nq, nk, nr = B * H * S_q * d, B * H_kv * S_k * d, B * H * S_q
    arr = np.frombuffer(raw[28:28 + 2 * (4 * nq + 4 * nk)], dtype=np.uint16)
    lse = np.frombuffer(raw[28 + 2 * (4 * nq + 4 * nk):], dtype=np.float32).astype(np.float64)
    sizes = [nq, nk, nk, nq, nq, nq, nk, nk]
    parts, o = [], 0
    for n in sizes:
        parts.append(_bf16(arr[o:o + n]))
        o += n
    qs, ks = (B, H, S_q, d), (B, H_kv, S_k, d)
    Q, K, V, dO, O, dQ, dK, dV = (p.reshape(s) for p, s in zip(parts, [qs, ks, ks, qs, qs, qs, ks, ks]))
    LSE = lse.reshape(B, H, S_q)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    O64, L64 = oracle.ref_fwd(Q, K, V, scale, bool(causal))
    den = np.max(np.abs(O64))
    assert np.max(np.abs(O - O64)) / den <= 2e-2
    fin = np.isfinite(L64)
    assert np.max(np.abs(LSE[fin] - L64[fin])) <= 1e-4
    ref = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, bool(causal))
    for name, got, want in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref[:3]):
        assert np.max(np.abs(got - want)) / np.max(np.abs(want)) <= 2e-2, name
