"""Why the fp32 backward runs on the FMA pipe: the error of tensor-core tf32 operands,
measured on the CPU against the fp64 oracle.

The fp32 gate is max|err| / max|ref| <= 1e-4 per output tensor.  A tcgen05 kind::tf32
product reads each fp32 operand with a 10-bit mantissa.  This test emulates that in numpy:
each of the five products of the backward (S = Q K^T, dP = dO V^T, dV = P^T dO,
dK = dS^T Q, dQ = dS K) takes its operands rounded to tf32 (to nearest even, and
truncated), and the sums are formed in float64.  The same is done for the 3xtf32 split
a*b ~ hi(a)hi(b) + hi(a)lo(b) + lo(a)hi(b), with hi = tf32(a) and lo = tf32(a - hi).
The softmax pieces stay in float64, so only the operand precision is measured.  Plain
tf32 misses the gate: 5-8e-4 with rounded operands, 4-6e-3 with truncated ones.  3xtf32
meets it (2e-7 to 3e-6), at three products per product, with a second fp32 copy (the low
parts) of every operand tile.  fp32 operand
tiles are already twice the size of 16-bit ones.  The library therefore computes the fp32
backward with FFMA (csrc/bwd_simt.cu).
"""
import numpy as np
import pytest

import oracle
from flashattention_backward_preprocess_gb300.inputs import WORKLOADS, Workload, make_inputs


def tf32(x, mode):
    """fp32 -> the nearest (mode "rn") or truncated (mode "rz") value with a 10-bit mantissa."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    if mode == "rn":
        b = b + 0xFFF + ((b >> 13) & 1)
    b = (b & 0xFFFFE000) & 0xFFFFFFFF
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def product(a, b, kind, mode):
    """a @ b with operands as a kind::tf32 product would see them (kind "1x" or "3x"), or
    (kind "f32") computed in float32 arithmetic, as the FFMA path does."""
    a32, b32 = a.astype(np.float32), b.astype(np.float32)
    if kind == "f32":
        return (a32 @ b32).astype(np.float64)
    ah, bh = tf32(a32, mode), tf32(b32, mode)
    if kind == "1x":
        return ah @ bh
    al = tf32((a32.astype(np.float64) - ah).astype(np.float32), mode)
    bl = tf32((b32.astype(np.float64) - bh).astype(np.float32), mode)
    return ah @ bh + ah @ bl + al @ bh


def bwd_emulated(dO, Q, K, V, O, LSE, scale, causal, kind, mode):
    """The backward of one (batch, head) stack with every product in emulated tf32."""
    B, H, S_q, d = Q.shape
    S_k = K.shape[2]
    g = H // K.shape[1]
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    i = np.arange(S_q)[:, None] + (S_k - S_q)
    j = np.arange(S_k)[None, :]
    mask = (j <= i) if causal else np.ones((S_q, S_k), bool)
    for b in range(B):
        for h in range(H):
            hk = h // g
            q, k, v, do, o = Q[b, h], K[b, hk], V[b, hk], dO[b, h], O[b, h]
            s = product(q, k.T, kind, mode) * scale
            p = np.where(mask, np.exp(s - LSE[b, h][:, None]), 0.0)
            Dv = np.sum(do * o, axis=1)
            dp = product(do, v.T, kind, mode)
            ds = p * (dp - Dv[:, None])
            dV[b, hk] += product(p.T, do, kind, mode)
            dK[b, hk] += scale * product(ds.T, q, kind, mode)
            dQ[b, h] = scale * product(ds, k, kind, mode)
    return dQ, dK, dV


def rel_err(a, r):
    return float(np.max(np.abs(a - r)) / np.max(np.abs(r)))


CASES = [
    WORKLOADS["fp32_b1_h2_s128_d64"],
    Workload("f32_causal_gqa", "f32", 1, 4, 2, 256, 256, 128, True, seed=7),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tf32_operands_miss_the_fp32_gate_and_3xtf32_meets_it(w):
    Q, K, V, dO = (x.double().numpy() for x in make_inputs(w))
    O, LSE = oracle.ref_fwd(Q, K, V, w.scale, w.causal)
    ref = oracle.ref_bwd(dO, Q, K, V, O, LSE, w.scale, w.causal)[:3]
    errs = {}
    for kind in ("1x", "3x"):
        for mode in ("rn", "rz"):
            got = bwd_emulated(dO, Q, K, V, O, LSE, w.scale, w.causal, kind, mode)
            errs[(kind, mode)] = max(rel_err(a, r) for a, r in zip(got, ref))
    for mode in ("rn", "rz"):
        assert errs[("1x", mode)] > 1e-4, errs   # plain tf32: fails the fp32 tolerance
        assert errs[("3x", mode)] < 1e-5, errs   # 3xtf32: within it, with margin
    # the products in float32 arithmetic (the FFMA path): far inside the gate
    f32 = bwd_emulated(dO, Q, K, V, O, LSE, w.scale, w.causal, "f32", "rn")
    assert max(rel_err(a, r) for a, r in zip(f32, ref)) < 1e-5
