"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Gate (per output tensor X in dQ, dK, dV):  max|X_gpu - X_ref| / max|X_ref|
  <= 1e-4 (fp32), 5e-3 (fp16), 2e-2 (bf16).
The oracle gets exactly the buffers the GPU got (dO, Q, K, V, O, LSE upcast
to fp64), so the comparison isolates the backward.  O and LSE come from the
library forward for 16-bit inputs and from the oracle forward for fp32.

Every workload, edge shape and option is compared element by element over the
whole of dQ, dK and dV: the five workloads (the three large ones launched
exactly as the benchmark launches them) and the 16K-token windowed workload
run the full fp64 oracle backward on the host cores (seconds to about a
minute each).
"""
import math

import numpy as np
import pytest
import torch

import flashattention_backward_preprocess_gb300 as fa
import oracle
from flashattention_backward_preprocess_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 2e-2}


def rel_err(a, b):
    den = float(np.max(np.abs(b)))
    return float(np.max(np.abs(a - b))) / (den if den > 0 else 1.0)


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def prepare(w: Workload):
    Q, K, V, dO = make_inputs(w)
    dev = torch.device("cuda", 0)
    g = [x.to(dev) for x in (Q, K, V, dO)]
    if w.dtype == "f32":
        O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, w.causal, w.window)
        O = torch.from_numpy(O64).to(torch.float32).to(dev)
        LSE = torch.from_numpy(L64).to(torch.float32).to(dev)
    else:
        O, LSE = fa.fa_fwd(g[0], g[1], g[2], scale=w.scale, causal=w.causal, window_size=w.window)
    return g[0], g[1], g[2], g[3], O, LSE


def run_bwd(w, Q, K, V, dO, O, LSE):
    dQ, dK, dV = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=w.causal, window_size=w.window)
    torch.cuda.synchronize()
    fa.fa_check_device()
    return dQ, dK, dV


def check_full(w: Workload):
    Q, K, V, dO, O, LSE = prepare(w)
    dQ, dK, dV = run_bwd(w, Q, K, V, dO, O, LSE)
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, w.causal, w.window)
    tol = TOL[w.dtype]
    errs = {}
    for name, got, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref[:3]):
        g = f64(got)
        assert np.all(np.isfinite(g)), f"{name} has non-finite values"
        errs[name] = rel_err(g, r)
    assert all(e <= tol for e in errs.values()), (w, errs)
    return errs


@pytest.mark.parametrize("name", ["fp32_b1_h2_s128_d64", "bf16_b2_h8_s1024_d64_causal",
                                  "bf16_b4_h32_kv8_s2048_d128_causal", "fp16_b1_h16_s8192_d128",
                                  "bf16_b8_h16_kv2_sq512_sk4096_d64",
                                  "bf16_b1_h32_kv8_s16384_d128_causal_w4096",
                                  "bf16_b1_h16_kv4_s4096_d256_causal",
                                  "fp32_b2_h8_kv2_s2048_d128_causal"])
def test_workload_full(name):
    check_full(WORKLOADS[name])


EDGE = [
    # dtype, B, H, H_kv, S_q, S_k, d, causal
    ("bf16", 1, 2, 1, 200, 200, 128, True),     # ragged tail, GQA 2
    ("f16", 2, 4, 4, 77, 77, 64, False),        # one partial tile
    ("bf16", 1, 8, 1, 300, 300, 64, True),      # GQA 8
    ("bf16", 1, 2, 2, 1, 1, 128, False),        # S = 1
    ("f16", 1, 2, 2, 1, 1, 64, True),
    ("bf16", 1, 2, 1, 100, 300, 128, True),     # S_q < S_k, bottom-right causal
    ("bf16", 1, 2, 1, 300, 100, 64, True),      # S_q > S_k: rows that see no key
    ("f16", 1, 2, 1, 129, 257, 128, False),
    ("bf16", 3, 3, 1, 384, 384, 128, True),     # several full tiles, odd head count
    ("bf16", 1, 4, 2, 256, 513, 64, False),     # key tail of one row
    ("f32", 1, 4, 2, 200, 200, 128, True),
    ("f32", 2, 2, 1, 65, 33, 64, False),
    ("f32", 1, 2, 2, 33, 65, 64, True),
    # non-causal with 8 (batch, kv head) groups: the CTAs run in two blocks of 4 groups
    ("bf16", 2, 8, 4, 300, 300, 128, False),
    ("f16", 4, 4, 2, 200, 333, 64, False),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(map(str, c)))
def test_edge_shapes(case):
    dt, B, H, H_kv, S_q, S_k, d, causal = case
    check_full(Workload("edge", dt, B, H, H_kv, S_q, S_k, d, causal, seed=99))


def test_dk_dv_deterministic_and_outputs_bounded():
    w = Workload("det", "bf16", 2, 4, 2, 333, 333, 128, True, seed=5)
    Q, K, V, dO, O, LSE = prepare(w)
    canary = 12345.0

    def guarded(shape):
        n = int(np.prod(shape))
        buf = torch.full((n + 2048,), canary, dtype=torch.bfloat16, device="cuda")
        return buf, buf[1024:1024 + n].view(shape)

    outs = []
    for _ in range(2):
        bq, dQ = guarded(Q.shape)
        bk, dK = guarded(K.shape)
        bv, dV = guarded(V.shape)
        fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=True, dQ=dQ, dK=dK, dV=dV)
        torch.cuda.synchronize()
        for b in (bq, bk, bv):
            assert bool((b[:1024] == canary).all()) and bool((b[-1024:] == canary).all())
        outs.append((dQ.clone(), dK.clone(), dV.clone()))
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])
    assert rel_err(f64(outs[0][0]), f64(outs[1][0])) < 1e-2


SPLIT = [
    # shapes whose heaviest causal key tile outlasts an even share of the work over the SMs,
    # so each key tile runs as a cluster of two CTAs that split its query tiles and add their
    # dK / dV partials through distributed shared memory (at least one CTA per SM)
    ("bf16", 1, 10, 10, 2048, 2048, 128, True),   # 160 key tiles of 128, 16 query tiles deep
    ("f16", 1, 5, 5, 4096, 4096, 64, True),      # d = 64 instance: 160 key tiles, 32 query tiles deep
    ("bf16", 1, 4, 4, 4096, 4096, 256, True),    # d = 256: 256 key tiles of 64
    ("bf16", 1, 8, 4, 3000, 3000, 256, True),    # d = 256, GQA 2, ragged tails
]


@pytest.mark.parametrize("case", SPLIT, ids=lambda c: "-".join(map(str, c)))
def test_long_causal_key_tiles_split_over_a_cluster(case):
    dt, B, H, H_kv, S_q, S_k, d, causal = case
    check_full(Workload("split", dt, B, H, H_kv, S_q, S_k, d, causal, seed=95))


def test_accumulator_state_across_calls_and_paths():
    """The tensor-core kernel converts dQ itself and leaves the fp32 accumulator zero; the
    deterministic and CUDA-core paths leave it holding values and mark it, so the next
    call's preprocess zeroes it.  A sequence of calls on one stream that switches between
    the paths and between larger and smaller shapes must stay correct at every step."""
    seq = [
        ("bf16", 2, 4, 2, 640, 640, 128, True, False),   # fused
        ("bf16", 2, 4, 2, 640, 640, 128, True, False),   # fused again: starts from its own zeroes
        ("bf16", 1, 4, 2, 300, 300, 128, True, True),    # deterministic: leaves values
        ("bf16", 2, 4, 2, 640, 640, 128, True, False),   # fused after it: larger than the marked part
        ("f32", 1, 2, 1, 200, 200, 64, False, False),    # CUDA cores: leaves values
        ("f16", 1, 2, 2, 130, 260, 64, False, False),    # fused, smaller than the marked part
        ("bf16", 2, 4, 2, 640, 640, 128, True, False),   # fused, covers it again
        ("bf16", 1, 2, 1, 200, 200, 256, True, False),   # d = 256 kernel: separate finalisation
        ("bf16", 1, 4, 1, 260, 130, 64, True, False),    # fused; rows and tiles that see no key
    ]
    for k, (dt, B, H, H_kv, S_q, S_k, d, causal, det) in enumerate(seq):
        w = Workload("seq", dt, B, H, H_kv, S_q, S_k, d, causal, seed=80 + k)
        Q, K, V, dO, O, LSE = prepare(w)
        got = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=causal, deterministic=det)
        torch.cuda.synchronize()
        fa.fa_check_device()
        ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, causal)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref[:3]):
            assert rel_err(f64(g), r) <= TOL[dt], (k, name, rel_err(f64(g), r))


@pytest.mark.parametrize("dt,d,S", [("bf16", 128, 2048), ("f16", 64, 333), ("f32", 128, 77)])
def test_preprocess_entry_point(dt, d, S):
    w = Workload("pre", dt, 2, 3, 3, S, S, d, False, seed=3)
    Q, K, V, dO = make_inputs(w)
    O = make_inputs(w.with_(seed=4))[0]
    D = fa.fa_bwd_preprocess(dO.cuda(), O.cuda())
    torch.cuda.synchronize()
    ref = oracle.ref_preprocess(f64(dO), f64(O))
    scale = float(np.max(np.sum(np.abs(f64(dO) * f64(O)), axis=-1)))
    assert float(np.max(np.abs(f64(D) - ref))) <= 1e-5 * scale


@pytest.mark.parametrize("dt,causal,S_q,S_k,d", [
    ("bf16", True, 300, 300, 128), ("f16", False, 129, 200, 64), ("f32", True, 100, 160, 64),
    # tensor-core forward: one tile, several tiles with the diagonal, keys past the queries,
    # rows that see no key (S_q > S_k, causal), a single element
    ("bf16", False, 128, 128, 128), ("bf16", True, 1000, 1000, 128), ("f16", True, 130, 1030, 128),
    ("bf16", True, 260, 130, 128), ("bf16", False, 200, 700, 64), ("f16", False, 1, 1, 64),
    # d = 256: 64-key tiles, two S buffers (ragged tails of both kinds, rows with no key)
    ("bf16", True, 300, 300, 256), ("f16", False, 129, 1000, 256), ("bf16", True, 200, 70, 256)])
def test_forward_helper(dt, causal, S_q, S_k, d):
    w = Workload("fwd", dt, 1, 4, 2, S_q, S_k, d, causal, seed=8)
    Q, K, V, _ = make_inputs(w)
    O, LSE = fa.fa_fwd(Q.cuda(), K.cuda(), V.cuda(), scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    fa.fa_check_device()
    O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, causal)
    assert bool(torch.isfinite(O).all())
    assert rel_err(f64(O), O64) <= TOL[dt]
    lse, fin = f64(LSE), np.isfinite(L64)
    assert bool(np.all(np.isneginf(lse[~fin]))) and bool(np.all(np.isfinite(lse[fin])))
    if fin.any():
        assert float(np.max(np.abs(lse[fin] - L64[fin]))) <= 1e-4


@pytest.mark.parametrize("dt,B,H,H_kv,S_q,S_k,d,causal,win", [
    # more query tiles than SMs: the persistent forward (256-row items of two query tiles);
    # ragged last items (the second tile partly or wholly past S_q), rows that see no key
    # (S_q > S_k, causal), keys past the queries, sliding windows, both head dims
    ("bf16", 2, 16, 4, 2300, 2300, 128, True, 0),
    ("f16", 2, 32, 8, 1100, 1500, 64, True, 0),
    ("bf16", 1, 32, 8, 1500, 1100, 128, True, 0),
    ("bf16", 1, 32, 8, 2200, 2200, 128, True, 300),
    ("f16", 2, 16, 16, 1130, 1130, 64, True, 100),
    ("bf16", 1, 48, 16, 1200, 1200, 96, True, 0),
    ("bf16", 1, 32, 8, 2000, 2000, 128, False, 500)])
def test_forward_persistent_path(dt, B, H, H_kv, S_q, S_k, d, causal, win):
    w = Workload("fwd_persistent", dt, B, H, H_kv, S_q, S_k, d, causal, seed=S_q + 7 * S_k + win, window=win)
    Q, K, V, _ = make_inputs(w)
    O, LSE = fa.fa_fwd(Q.cuda(), K.cuda(), V.cuda(), scale=w.scale, causal=causal, window_size=win)
    torch.cuda.synchronize()
    fa.fa_check_device()
    O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, causal, win)
    assert bool(torch.isfinite(O).all())
    assert rel_err(f64(O), O64) <= TOL[dt]
    lse, fin = f64(LSE), np.isfinite(L64)
    assert bool(np.all(np.isneginf(lse[~fin]))) and bool(np.all(np.isfinite(lse[fin])))
    if fin.any():
        assert float(np.max(np.abs(lse[fin] - L64[fin]))) <= 1e-4


def test_host_buffer_entry_point_matches_device():
    w = Workload("host", "bf16", 1, 4, 2, 256, 256, 64, True, seed=6)
    Q, K, V, dO, O, LSE = prepare(w)
    dQ, dK, dV = run_bwd(w, Q, K, V, dO, O, LSE)
    host = [x.cpu().pin_memory() for x in (dO, Q, K, V, O, LSE)]
    hQ, hK, hV = fa.fa_bwd_host(*host, scale=w.scale, causal=True)
    assert torch.equal(hK, dK.cpu()) and torch.equal(hV, dV.cpu())
    assert rel_err(f64(hQ), f64(dQ)) < 1e-2


def test_host_buffer_entry_point_pipelined_chunks():
    # 73 MB of input: fa_bwd_host splits the 10 (batch, kv head) units into 4 chunks of
    # 2, 3, 2, 3 units, whose copies overlap the other chunks' compute.  The single device
    # call has enough CTAs to split its long causal key tiles over 2-CTA clusters (dK / dV
    # summed in two halves), the chunks do not, so the two agree to rounding, not bit for bit
    w = Workload("host_chunks", "bf16", 5, 8, 2, 2048, 2048, 128, True, seed=16)
    Q, K, V, dO, O, LSE = prepare(w)
    dQ, dK, dV = run_bwd(w, Q, K, V, dO, O, LSE)
    host = [x.cpu().pin_memory() for x in (dO, Q, K, V, O, LSE)]
    hQ, hK, hV = fa.fa_bwd_host(*host, scale=w.scale, causal=True)
    for got, ref in ((hQ, dQ), (hK, dK), (hV, dV)):
        assert rel_err(f64(got), f64(ref)) < 1e-2
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, True)
    for name, got, r in zip(("dQ", "dK", "dV"), (hQ, hK, hV), ref[:3]):
        assert rel_err(f64(got), r) <= TOL[w.dtype], name


def test_causal_scale_and_rows_without_keys_are_finite():
    # S_q > S_k causal: the first S_q - S_k query rows see no key (LSE = -inf); their dQ is 0
    w = Workload("masked", "bf16", 1, 2, 2, 260, 130, 128, True, seed=9)
    Q, K, V, dO, O, LSE = prepare(w)
    assert bool(torch.isinf(LSE[:, :, :130]).all())
    dQ, dK, dV = run_bwd(w, Q, K, V, dO, O, LSE)
    assert bool(torch.isfinite(dQ).all() and torch.isfinite(dK).all() and torch.isfinite(dV).all())
    assert bool((dQ[:, :, :130] == 0).all())


def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A device wait that nothing completes runs out after 1 ms, the kernel returns,
    fa_check_device reports FA_ERR_TIMEOUT once, and the next backward is correct."""
    fa.fa_selftest_timeout(1_000_000)
    with pytest.raises(fa.FaError) as ei:
        fa.fa_check_device()
    assert ei.value.status == 4
    fa.fa_check_device()  # the record was cleared
    check_full(Workload("after_timeout", "bf16", 1, 2, 1, 130, 130, 64, True, seed=10))


WINDOW = [
    # dtype, B, H, H_kv, S_q, S_k, d, causal, window
    ("bf16", 1, 4, 2, 700, 700, 128, True, 256),    # band over several tiles, skipped on both sides
    ("bf16", 1, 2, 1, 515, 515, 64, True, 100),     # band narrower than a tile
    ("f16", 1, 2, 2, 400, 400, 128, False, 150),    # non-causal: band on both sides of the diagonal
    ("bf16", 1, 2, 1, 300, 600, 128, True, 200),    # S_q < S_k
    ("bf16", 1, 2, 1, 600, 300, 64, False, 130),    # S_q > S_k: the first rows see no key
    ("f16", 1, 2, 1, 333, 333, 64, True, 1),        # diagonal only
    ("bf16", 1, 2, 2, 256, 256, 128, True, 128),    # band edge on tile boundaries
    ("bf16", 2, 4, 1, 1024, 1024, 64, True, 4096),  # wider than the problem: plain causal
    ("bf16", 2, 8, 4, 400, 400, 64, True, 100),     # 8 groups: two blocks of 4 in the CTA order
    ("f32", 1, 2, 1, 200, 200, 64, True, 37),
    ("f32", 1, 2, 2, 150, 90, 128, False, 20),
]


@pytest.mark.parametrize("case", WINDOW, ids=lambda c: "-".join(map(str, c)))
def test_sliding_window_backward(case):
    dt, B, H, H_kv, S_q, S_k, d, causal, win = case
    check_full(Workload("window", dt, B, H, H_kv, S_q, S_k, d, causal, seed=31, window=win))


@pytest.mark.parametrize("case", WINDOW, ids=lambda c: "-".join(map(str, c)))
def test_sliding_window_forward(case):
    dt, B, H, H_kv, S_q, S_k, d, causal, win = case
    w = Workload("window_fwd", dt, B, H, H_kv, S_q, S_k, d, causal, seed=32, window=win)
    Q, K, V, _ = make_inputs(w)
    O, LSE = fa.fa_fwd(Q.cuda(), K.cuda(), V.cuda(), scale=w.scale, causal=causal, window_size=win)
    torch.cuda.synchronize()
    fa.fa_check_device()
    O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, causal, win)
    assert bool(torch.isfinite(O).all())
    assert rel_err(f64(O), O64) <= TOL[dt]
    lse, fin = f64(LSE), np.isfinite(L64)
    assert bool(np.all(np.isneginf(lse[~fin]))) and bool(np.all(np.isfinite(lse[fin])))
    assert float(np.max(np.abs(lse[fin] - L64[fin]))) <= 1e-4


def test_window_wider_than_problem_equals_no_window():
    # the band then holds every causal pair: dK / dV bit-identical to the plain call
    w = Workload("wide", "bf16", 1, 4, 2, 640, 640, 128, True, seed=33)
    Q, K, V, dO, O, LSE = prepare(w)
    a = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=True)
    b = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=True, window_size=640)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert rel_err(f64(a[0]), f64(b[0])) < 1e-2


DET = [
    # dtype, B, H, H_kv, S_q, S_k, d, causal, window
    ("bf16", 2, 8, 2, 700, 700, 128, True, 0),      # causal, GQA 4, ragged tail
    ("f16", 1, 4, 4, 513, 300, 64, False, 0),       # S_q > S_k, d = 64
    ("bf16", 1, 4, 1, 300, 600, 128, True, 200),    # window: turns start past key tile 0
    ("bf16", 1, 2, 2, 600, 600, 64, False, 130),    # two-sided window
    ("bf16", 2, 8, 2, 300, 700, 64, False, 0),      # d = 64 GQA: 12 iterations per CTA, both dS tiles
    ("f16", 2, 8, 4, 300, 300, 128, False, 0),      # 8 groups, non-causal: order stays interleaved
    ("f32", 1, 4, 2, 200, 333, 128, True, 0),       # CUDA-core dQ kernel
    ("f32", 1, 2, 1, 150, 150, 64, False, 40),
]


@pytest.mark.parametrize("case", DET, ids=lambda c: "-".join(map(str, c)))
def test_deterministic_dq_matches_oracle_and_is_reproducible(case):
    dt, B, H, H_kv, S_q, S_k, d, causal, win = case
    w = Workload("det_dq", dt, B, H, H_kv, S_q, S_k, d, causal, seed=41, window=win)
    Q, K, V, dO, O, LSE = prepare(w)
    runs = []
    for _ in range(3):
        runs.append(fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=causal, window_size=win,
                              deterministic=True))
        torch.cuda.synchronize()
        fa.fa_check_device()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, causal, win)
    for name, got, r in zip(("dQ", "dK", "dV"), runs[0], ref[:3]):
        assert rel_err(f64(got), r) <= TOL[dt], name
    # dK / dV do not depend on how dQ is reduced
    nd = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=causal, window_size=win)
    torch.cuda.synchronize()
    assert torch.equal(nd[1], runs[0][1]) and torch.equal(nd[2], runs[0][2])


def test_deterministic_dq_bench_workload_bitwise():
    # full size, as the benchmark launches it: two deterministic calls give the same bits, and
    # the whole of dQ, dK and dV matches the oracle
    w = WORKLOADS["bf16_b4_h32_kv8_s2048_d128_causal"]
    Q, K, V, dO, O, LSE = prepare(w)
    a = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=True, deterministic=True)
    b = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=True, deterministic=True)
    torch.cuda.synchronize()
    fa.fa_check_device()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, True)
    for name, got, r in zip(("dQ", "dK", "dV"), a, ref[:3]):
        assert rel_err(f64(got), r) <= TOL[w.dtype], name


D256 = [
    # dtype, B, H, H_kv, S_q, S_k, causal, window: the d = 256 tensor-core backward (64-key CTAs,
    # 64-row query tiles, M = 64 products): one tile, ragged tails of both kinds, several query
    # and key tiles with the causal diagonal inside a tile, GQA 4 and 8, S_q != S_k either way
    # (rows that see no key), windows narrower than a tile and over several tiles
    ("bf16", 1, 2, 2, 64, 64, False, 0),
    ("f16", 1, 2, 1, 77, 77, True, 0),
    ("bf16", 2, 8, 2, 700, 700, True, 0),
    ("bf16", 1, 8, 1, 300, 513, False, 0),
    ("f16", 1, 4, 4, 513, 300, True, 0),
    ("bf16", 1, 4, 2, 129, 1000, True, 0),
    ("bf16", 1, 4, 1, 600, 600, True, 50),
    ("f16", 2, 2, 2, 400, 400, False, 150),
]


@pytest.mark.parametrize("case", D256, ids=lambda c: "-".join(map(str, c)))
def test_head_dim_256_tensor_core_backward(case):
    dt, B, H, H_kv, S_q, S_k, causal, win = case
    check_full(Workload("d256", dt, B, H, H_kv, S_q, S_k, 256, causal, seed=91, window=win))


HEAD_DIMS = [
    # dtype, B, H, H_kv, S_q, S_k, d, causal, window, deterministic
    ("bf16", 1, 4, 2, 300, 300, 96, True, 0, False),    # tensor cores, 128-wide kernel, 32 zero columns
    ("f16", 1, 4, 4, 257, 129, 96, False, 0, False),
    ("bf16", 1, 4, 1, 260, 260, 32, True, 0, False),    # tensor cores, 64-wide kernel
    ("f16", 2, 2, 2, 130, 390, 32, False, 100, False),  # + window
    ("bf16", 1, 4, 2, 333, 333, 96, True, 0, True),     # + deterministic dQ
    ("bf16", 1, 2, 1, 200, 200, 256, True, 0, False),   # d = 256: tensor cores both ways
    ("f16", 1, 2, 2, 130, 70, 256, False, 0, True),     # d = 256 deterministic: dQ on CUDA cores
    ("bf16", 2, 2, 1, 500, 500, 256, True, 130, False),  # + window
    ("f32", 1, 2, 1, 150, 150, 96, True, 0, False),
    ("f32", 1, 2, 2, 100, 160, 32, False, 30, True),
    ("f32", 1, 2, 1, 90, 90, 256, True, 0, False),
]


@pytest.mark.parametrize("case", HEAD_DIMS, ids=lambda c: "-".join(map(str, c)))
def test_head_dims_forward_and_backward(case):
    dt, B, H, H_kv, S_q, S_k, d, causal, win, det = case
    w = Workload("hd", dt, B, H, H_kv, S_q, S_k, d, causal, seed=61, window=win)
    Q, K, V, dO = (x.cuda() for x in make_inputs(w))
    O, LSE = fa.fa_fwd(Q, K, V, scale=w.scale, causal=causal, window_size=win)
    torch.cuda.synchronize()
    fa.fa_check_device()
    O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, causal, win)
    assert rel_err(f64(O), O64) <= TOL[dt]
    fin = np.isfinite(L64)
    assert float(np.max(np.abs(f64(LSE)[fin] - L64[fin]))) <= 1e-4
    if dt == "f32":  # the backward gate isolates the backward: fp32 O / LSE from the oracle
        O = torch.from_numpy(O64).float().cuda()
        LSE = torch.from_numpy(L64).float().cuda()
    dQ, dK, dV = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=causal, window_size=win,
                           deterministic=det)
    torch.cuda.synchronize()
    fa.fa_check_device()
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, causal, win)
    for name, got, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref[:3]):
        g = f64(got)
        assert np.all(np.isfinite(g)), name
        assert rel_err(g, r) <= TOL[dt], (name, rel_err(g, r))


@pytest.mark.parametrize("det", [False, True])
def test_backward_captures_into_a_cuda_graph(det):
    # after one call on a stream (which caches that stream's workspace) fa_bwd enqueues
    # kernels and, in deterministic mode, one memset, and nothing else: it can be captured
    # into a CUDA graph, and replays on new input values match direct calls
    w = Workload("graph", "bf16", 2, 8, 2, 700, 700, 128, True, seed=71)
    Q, K, V, dO, O, LSE = prepare(w)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fa_bwd(dO, Q, K, V, O, LSE, causal=True, dQ=dQ, dK=dK, dV=dV, deterministic=det)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fa.fa_bwd(dO, Q, K, V, O, LSE, causal=True, dQ=dQ, dK=dK, dV=dV, deterministic=det)
    for seed in (72, 73):
        Qn, Kn, Vn, dOn = make_inputs(w.with_(seed=seed))
        for dst, src in zip((Q, K, V, dO), (Qn, Kn, Vn, dOn)):
            dst.copy_(src)
        On, Ln = fa.fa_fwd(Q, K, V, causal=True)
        O.copy_(On)
        LSE.copy_(Ln)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        fa.fa_check_device()
        ref = fa.fa_bwd(dO, Q, K, V, O, LSE, causal=True, deterministic=det)
        torch.cuda.synchronize()
        assert torch.equal(dK, ref[1]) and torch.equal(dV, ref[2])
        if det:
            assert torch.equal(dQ, ref[0])
        else:
            assert rel_err(f64(dQ), f64(ref[0])) < 1e-2


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        dt = str(rng.choice(["bf16", "f16", "f32"], p=[0.45, 0.35, 0.2]))
        d = int(rng.choice([32, 64, 96, 128, 256], p=[0.15, 0.3, 0.15, 0.3, 0.1]))
        H_kv = int(rng.integers(1, 3))
        g = int(rng.choice([1, 2, 4]))
        S_q = int(rng.integers(1, 450))
        S_k = int(rng.integers(1, 450))
        causal = bool(rng.integers(0, 2))
        win = int(rng.choice([0, 0, int(rng.integers(1, 300))]))
        det = bool(rng.integers(0, 2))
        cases.append((dt, 1, g * H_kv, H_kv, S_q, S_k, d, causal, win, det))
    return cases


@pytest.mark.parametrize("case", _random_cases(30, 2026), ids=lambda c: "-".join(map(str, c)))
def test_random_configurations(case):
    """Seeded random draws over the whole option space (dtype, head dim, GQA ratio, ragged S_q
    and S_k in either order, causal, window, deterministic): forward and backward against the
    oracle."""
    dt, B, H, H_kv, S_q, S_k, d, causal, win, det = case
    w = Workload("rand", dt, B, H, H_kv, S_q, S_k, d, causal, seed=S_q * 1000 + S_k, window=win)
    Q, K, V, dO = (x.cuda() for x in make_inputs(w))
    O, LSE = fa.fa_fwd(Q, K, V, scale=w.scale, causal=causal, window_size=win)
    torch.cuda.synchronize()
    fa.fa_check_device()
    O64, L64 = oracle.ref_fwd(f64(Q), f64(K), f64(V), w.scale, causal, win)
    assert rel_err(f64(O), O64) <= TOL[dt]
    lse, fin = f64(LSE), np.isfinite(L64)
    assert bool(np.all(np.isneginf(lse[~fin])))
    if fin.any():
        assert float(np.max(np.abs(lse[fin] - L64[fin]))) <= 1e-4
    if dt == "f32":
        O = torch.from_numpy(O64).float().cuda()
        LSE = torch.from_numpy(L64).float().cuda()
    dQ, dK, dV = fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=causal, window_size=win,
                           deterministic=det)
    torch.cuda.synchronize()
    fa.fa_check_device()
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, causal, win)
    for name, got, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref[:3]):
        g_ = f64(got)
        assert np.all(np.isfinite(g_)), name
        assert rel_err(g_, r) <= TOL[dt], (name, rel_err(g_, r))
