"""Host-side checks of the C ABI (no GPU needed).

* the library builds and exports every function include/fa.h declares;
* argument validation rejects bad calls before anything is enqueued (the
  checks of boostr flash_bwd.rs flash_attention_bwd_impl and rustytorch
  backward.rs flash_attention_backward, restated for raw pointers), so these
  run without a device: the pointers below are never dereferenced;
* the workspace size formula.
"""
import ctypes
import os
import re

import pytest

import flashattention_backward_preprocess_gb300 as fa
from flashattention_backward_preprocess_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert set(_declared()) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert "sm_103a" in fa.fa_version()


# fake, 256-byte aligned device addresses: validation fails before any use
P = [0x10000 * (i + 1) for i in range(9)]


def _bwd(lib, **kw):
    a = dict(dO=P[0], Q=P[1], K=P[2], V=P[3], O=P[4], LSE=P[5], dQ=P[6], dK=P[7], dV=P[8],
             B=1, H=4, H_kv=2, S_q=128, S_k=128, d=64, scale=0.125, causal=0, dtype=fa.FA_BF16,
             stream=None)
    a.update(kw)
    return lib.fa_bwd(a["dO"], a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["dQ"], a["dK"], a["dV"],
                      a["B"], a["H"], a["H_kv"], a["S_q"], a["S_k"], a["d"], a["scale"], a["causal"],
                      a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status,arg", [
    (dict(H=5, H_kv=2), 1, "H_kv"),
    (dict(H_kv=0), 1, "H_kv"),
    (dict(B=0), 1, "B"),
    (dict(S_q=0), 1, "S_q"),
    (dict(S_k=-3), 1, "S_k"),
    (dict(dtype=7), 1, "dtype"),
    (dict(d=80), 2, "d"),
    (dict(d=512), 2, "d"),
    (dict(scale=0.0), 1, "scale"),
    (dict(scale=float("nan")), 1, "scale"),
    (dict(scale=-1.0), 1, "scale"),
    (dict(causal=2), 1, "causal"),
    (dict(dO=None), 1, "dO"),
    (dict(LSE=None), 1, "LSE"),
    (dict(dV=None), 1, "dV"),
    (dict(Q=P[1] + 8), 1, "Q"),       # not 16-byte aligned (TMA needs 16)
    (dict(dK=P[7] + 2), 1, "dK"),
    (dict(LSE=P[5] + 2), 1, "LSE"),   # float32 needs 4
])
def test_bwd_rejects_bad_arguments(lib, kw, status, arg):
    rc = _bwd(lib, **kw)
    assert rc == status
    assert fa.fa_last_error().startswith(arg + ":"), fa.fa_last_error()


def test_preprocess_and_fwd_validate(lib):
    assert lib.fa_bwd_preprocess(None, P[1], P[2], 1, 2, 16, 64, fa.FA_F16, None) == 1
    assert fa.fa_last_error().startswith("dO:")
    assert lib.fa_bwd_preprocess(P[0], P[1], P[2], 1, 2, 16, 80, fa.FA_F16, None) == 2
    assert lib.fa_fwd(P[0], P[1], P[2], P[3], P[4], 1, 6, 4, 8, 8, 64, 0.1, 0, fa.FA_BF16, None) == 1
    assert fa.fa_last_error().startswith("H_kv:")
    assert lib.fa_fwd(P[0], P[1], P[2], P[3], P[4], 1, 4, 4, 8, 8, 64, float("inf"), 0, fa.FA_BF16, None) == 1


def test_workspace_bytes(lib):
    # err words, padded LSE*log2e and D copies (rows padded to 128), fp32 dQ accumulator,
    # one turn counter per (query head, 128-row query tile) for the deterministic dQ mode and
    # its CTA ticket counter (rounded up to 256 bytes)
    B, H, S, d = 4, 32, 2048, 128
    rows = B * H * S
    sem = (B * H * (S // 128) * 4 + 4 + 255) // 256 * 256
    assert fa.fa_bwd_workspace_bytes(B, H, S, d) == 256 + 2 * rows * 4 + rows * d * 4 + sem
    B, H, S, d = 1, 2, 200, 64
    rows_pad = B * H * 256
    got = fa.fa_bwd_workspace_bytes(B, H, S, d)
    assert got >= 256 + 2 * rows_pad * 4 + B * H * S * d * 4 and got % 256 == 0
    assert fa.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0


def test_binding_rejects_host_tensors_for_device_entry_points():
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(fa.FaError, match="device pointers required"):
        fa.fa_bwd(q, q, q, q, q, lse)
    with pytest.raises(fa.FaError, match="4-D"):
        fa.fa_bwd(q, q[0], q, q, q, lse)


def test_selftest_rejects_bad_limit(lib):
    assert lib.fa_selftest_timeout(0, None) == 1
    assert fa.fa_last_error().startswith("limit_ns:")
    assert lib.fa_selftest_timeout(2_000_000_000, None) == 1


def test_ex_entry_points_validate(lib):
    a = [P[0], P[1], P[2], P[3], P[4], P[5], P[6], P[7], P[8], 1, 4, 2, 128, 128, 64, 0.125, 1]
    assert lib.fa_bwd_ex(*a, -1, 0, fa.FA_BF16, None) == 1
    assert fa.fa_last_error().startswith("window_size:")
    assert lib.fa_bwd_ex(*a, 0, 2, fa.FA_BF16, None) == 1
    assert fa.fa_last_error().startswith("deterministic:")
    assert lib.fa_bwd_ex(*a[:9], 1, 5, 2, 128, 128, 64, 0.125, 1, 64, 0, fa.FA_BF16, None) == 1
    assert fa.fa_last_error().startswith("H_kv:")
    f = [P[0], P[1], P[2], P[3], P[4], 1, 4, 4, 8, 8, 64, 0.1, 0]
    assert lib.fa_fwd_ex(*f, -5, fa.FA_BF16, None) == 1
    assert fa.fa_last_error().startswith("window_size:")
    assert lib.fa_fwd_ex(*f[:10], 80, 0.1, 0, 3, fa.FA_BF16, None) == 2
