"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some users run this library inside a framework whose allocator owns all GPU
memory, or in a host loop where the implicit device synchronization of
cudaMalloc / cudaFree is not acceptable; for them the library offers one entry
point that uses a fixed scratch array compiled into the library instead of a
workspace it allocates.  These tests call it through the C ABI and check its
results against fa_bwd (the allocating entry point) on two calls in a row,
since every call reuses the same scratch.  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import flashattention_backward_preprocess_gb300 as fa
from flashattention_backward_preprocess_gb300.inputs import Workload, make_inputs

TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 2e-2}
DT = {"f32": fa.FA_F32, "f16": fa.FA_F16, "bf16": fa.FA_BF16}


def _rel(a, b):
    a = a.detach().to("cpu", torch.float64)
    b = b.detach().to("cpu", torch.float64)
    den = float(b.abs().max())
    return float((a - b).abs().max()) / (den if den > 0 else 1.0)


def _call(lib, w, dO, Q, K, V, O, LSE, dQ, dK, dV):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.fa_bwd_noalloc(dO.data_ptr(), Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                              LSE.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), w.B, w.H,
                              w.H_kv, w.S_q, w.S_k, w.d, ctypes.c_float(w.scale), int(w.causal),
                              DT[w.dtype], stream)


@pytest.mark.gpu
@pytest.mark.parametrize("w", [
    Workload("noalloc_bf16", "bf16", 1, 4, 2, 300, 300, 128, True, seed=31),
    Workload("noalloc_f16", "f16", 2, 2, 1, 200, 333, 64, False, seed=32),
    # the other main kernels through the same scratch: fp32, and head dim 256
    Workload("noalloc_f32", "f32", 1, 4, 2, 200, 200, 128, True, seed=33),
    Workload("noalloc_bf16_d256", "bf16", 1, 2, 1, 300, 300, 256, True, seed=34),
], ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_on_two_calls(w):
    lib = fa.load_library()
    dev = torch.device("cuda", 0)
    Q, K, V, dO = (x.to(dev) for x in make_inputs(w))
    O, LSE = fa.fa_fwd(Q, K, V, scale=w.scale, causal=w.causal)
    ref = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    for _ in range(2):
        out = [torch.full_like(x, float("nan")) for x in (Q, K, V)]
        rc = _call(lib, w, dO, Q, K, V, O, LSE, *out)
        assert rc == 0, fa.fa_last_error()
        torch.cuda.synchronize()
        for name, got, r in zip(("dQ", "dK", "dV"), out, ref):
            assert bool(torch.isfinite(got).all()), name
            assert _rel(got, r) <= TOL[w.dtype], (name, _rel(got, r))
    fa.fa_check_device()  # no bounded wait of either entry point ran out


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = fa.load_library()
    w = Workload("too_big", "bf16", 4, 32, 8, 2048, 2048, 128, True)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = x.data_ptr()
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, w.B, w.H, w.H_kv, w.S_q, w.S_k, w.d,
                            ctypes.c_float(w.scale), 1, fa.FA_BF16, None)
    assert rc == 1  # FA_ERR_INVALID_ARG
    assert fa.fa_last_error().startswith("scratch:")
