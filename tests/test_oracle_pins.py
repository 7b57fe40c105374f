"""Pins for the fp64 oracle, against things other than the oracle itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped D term,
a wrong sign, a transposed operand, a wrong head-group mapping, a causal
off-by-one, a missing scale) breaks at least one of them; test_oracle_mutants
checks exactly that by planting such slips in a copy of the oracle source.

  * torch autograd through scaled_dot_product_attention in float64 (a library
    routine that reduces to the same mathematics),
  * central finite differences of L = sum(dO * O) through the oracle forward,
  * closed forms: S_k = 1, Q = 0 (uniform attention), causal row 0,
  * invariants: D_i = sum_j P_ij dP_ij, sum_j dS_ij = 0 (seen through a shift
    of every key by one vector), linearity in dO, GQA = sum over the group of
    per-head gradients with K, V repeated,
  * agreement of the sampled-row entry points with the full backward.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _mask(S_q, S_k, causal):
    i = np.arange(S_q)[:, None]
    j = np.arange(S_k)[None, :]
    if not causal:
        return np.ones((S_q, S_k), dtype=bool)
    return j <= i + (S_k - S_q)


def _sdpa_grads(Q, K, V, dO, scale, causal):
    """dQ, dK, dV and O by torch autograd through float64 SDPA (math backend)."""
    B, H, S_q, d = Q.shape
    H_kv, S_k = K.shape[1], K.shape[2]
    g = H // H_kv
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    kr = k.repeat_interleave(g, dim=1)
    vr = v.repeat_interleave(g, dim=1)
    m = torch.tensor(_mask(S_q, S_k, causal))
    o = F.scaled_dot_product_attention(q, kr, vr, attn_mask=m, scale=scale)
    o.backward(torch.tensor(dO))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy(), o.detach().numpy()


SHAPES = [
    # B, H, H_kv, S_q, S_k, d, causal
    (1, 1, 1, 1, 1, 4, False),
    (1, 2, 1, 3, 3, 4, True),
    (1, 4, 2, 5, 5, 8, True),
    (2, 4, 1, 17, 17, 8, False),
    (1, 2, 2, 17, 17, 8, True),
    (1, 2, 1, 3, 5, 4, True),     # S_q < S_k: bottom-right causal alignment
    (1, 2, 2, 6, 9, 8, False),
    (2, 8, 2, 33, 29, 16, False),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_torch_sdpa(shape):
    B, H, H_kv, S_q, S_k, d, causal = shape
    rng = np.random.default_rng(11)
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.ref_fwd(Q, K, V, scale, causal)
    g = H // H_kv
    s = scale * np.einsum("bhid,bhjd->bhij", Q, np.repeat(K, g, axis=1))
    s = np.where(_mask(S_q, S_k, causal), s, -np.inf)
    lse_t = torch.logsumexp(torch.tensor(s), dim=-1).numpy()
    np.testing.assert_allclose(LSE, lse_t, rtol=1e-13, atol=1e-13)
    _, _, _, O_t = _sdpa_grads(Q, K, V, np.zeros_like(Q), scale, causal)
    np.testing.assert_allclose(O, O_t, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_matches_torch_autograd(shape):
    B, H, H_kv, S_q, S_k, d, causal = shape
    rng = np.random.default_rng(12)
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.ref_fwd(Q, K, V, scale, causal)
    dQ, dK, dV, D = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, causal)
    tq, tk, tv, _ = _sdpa_grads(Q, K, V, dO, scale, causal)
    for name, a, b in (("dQ", dQ, tq), ("dK", dK, tk), ("dV", dV, tv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11, err_msg=name)


def _loss(Q, K, V, dO, scale, causal):
    O, _ = oracle.ref_fwd(Q, K, V, scale, causal)
    return float(np.sum(dO * O))


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, 1, 4, False),
    (1, 2, 1, 3, 3, 4, True),
    (1, 4, 2, 5, 5, 8, False),
    (1, 2, 2, 17, 17, 4, True),
    (1, 2, 1, 5, 3, 4, True),     # S_q > S_k: first rows see no key
    (1, 4, 1, 3, 17, 8, True),
])
def test_bwd_matches_finite_differences(shape):
    B, H, H_kv, S_q, S_k, d, causal = shape
    rng = np.random.default_rng(13)
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.ref_fwd(Q, K, V, scale, causal)
    grads = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, causal)[:3]
    eps = 1e-5
    for which, (X, G) in enumerate(zip((Q, K, V), grads)):
        fd = np.zeros_like(X)
        for idx in itertools.product(*map(range, X.shape)):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += eps
            lp = _loss(*args, dO, scale, causal)
            args[which][idx] -= 2 * eps
            lm = _loss(*args, dO, scale, causal)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(fd - G)) / max(np.max(np.abs(G)), 1e-30)
        assert err < 1e-7, (which, err)


def test_preprocess_equals_sum_p_dp():
    """D_i = sum_c dO_ic O_ic must equal sum_j P_ij dP_ij when O is the exact forward."""
    rng = np.random.default_rng(14)
    B, H, H_kv, S, d = 2, 4, 2, 19, 8
    Q, K, V = _rand(rng, B, H, S, d), _rand(rng, B, H_kv, S, d), _rand(rng, B, H_kv, S, d)
    dO = _rand(rng, B, H, S, d)
    scale = 0.3
    for causal in (False, True):
        O, LSE = oracle.ref_fwd(Q, K, V, scale, causal)
        D = oracle.ref_preprocess(dO, O)
        Kr, Vr = np.repeat(K, 2, axis=1), np.repeat(V, 2, axis=1)
        s = scale * np.einsum("bhid,bhjd->bhij", Q, Kr)
        s = np.where(_mask(S, S, causal), s, -np.inf)
        P = torch.softmax(torch.tensor(s), dim=-1).numpy()
        dP = np.einsum("bhid,bhjd->bhij", dO, Vr)
        np.testing.assert_allclose(D, np.sum(P * dP, axis=-1), rtol=1e-12, atol=1e-12)
        # the D the backward reports is the same preprocess value
        D2 = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, causal)[3]
        np.testing.assert_allclose(D2, D, rtol=0, atol=1e-14)


def test_key_shift_leaves_dq_unchanged():
    """sum_j dS_ij = 0: moving every key by one vector c shifts each score row by a
    constant, so P and dS are unchanged and dQ_i gains scale * c * sum_j dS_ij = 0."""
    rng = np.random.default_rng(15)
    B, H, H_kv, S, d = 1, 4, 2, 23, 8
    Q, K, V = _rand(rng, B, H, S, d), _rand(rng, B, H_kv, S, d), _rand(rng, B, H_kv, S, d)
    dO = _rand(rng, B, H, S, d)
    c = 3.0 * _rand(rng, d)
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        O, LSE = oracle.ref_fwd(Q, K, V, scale, causal)
        dQ = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, causal)[0]
        O2, LSE2 = oracle.ref_fwd(Q, K + c, V, scale, causal)
        dQ2 = oracle.ref_bwd(dO, Q, K + c, V, O2, LSE2, scale, causal)[0]
        np.testing.assert_allclose(dQ2, dQ, rtol=1e-10, atol=1e-10)
        # constant keys: P uniform over the visible keys, dQ = 0
        Kc = np.broadcast_to(c, K.shape).copy()
        O3, LSE3 = oracle.ref_fwd(Q, Kc, V, scale, causal)
        dQ3 = oracle.ref_bwd(dO, Q, Kc, V, O3, LSE3, scale, causal)[0]
        assert np.max(np.abs(dQ3)) < 1e-12


def test_closed_form_single_key():
    """S_k = 1: P = 1, dS = 0, so dQ = dK = 0 and dV = sum over group rows of dO."""
    rng = np.random.default_rng(16)
    B, H, H_kv, S_q, d = 2, 4, 2, 7, 8
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, 1, d), _rand(rng, B, H_kv, 1, d)
    dO = _rand(rng, B, H, S_q, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, False)
    np.testing.assert_allclose(O, np.broadcast_to(np.repeat(V, 2, axis=1), O.shape), atol=1e-15)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.5, False)
    assert np.max(np.abs(dQ)) < 1e-14 and np.max(np.abs(dK)) < 1e-14
    expect = dO.reshape(B, H_kv, 2 * S_q, d).sum(axis=2, keepdims=True)
    np.testing.assert_allclose(dV, expect, rtol=1e-13, atol=1e-13)


def test_closed_form_uniform_attention():
    """Q = 0, non-causal: P = 1/S_k, LSE = log S_k, O = mean_j V_j, dV_j = (1/S_k) sum_i dO_i."""
    rng = np.random.default_rng(17)
    B, H, H_kv, S_q, S_k, d = 1, 2, 1, 5, 9, 4
    Q = np.zeros((B, H, S_q, d))
    K, V = _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.7, False)
    np.testing.assert_allclose(LSE, math.log(S_k), rtol=1e-14)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=2, keepdims=True), O.shape), atol=1e-14)
    _, _, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.7, False)
    expect = np.broadcast_to(dO.sum(axis=(1, 2), keepdims=True)[:, :1] / S_k, dV.shape)
    np.testing.assert_allclose(dV, expect, rtol=1e-13, atol=1e-13)


def test_closed_form_causal_first_row():
    """Causal, S_q = S_k: query 0 sees only key 0, so P_00 = 1, O_0 = V_0 and dQ_0 = 0."""
    rng = np.random.default_rng(18)
    B, H, S, d = 1, 3, 8, 4
    Q, K, V, dO = (_rand(rng, B, H, S, d) for _ in range(4))
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, True)
    np.testing.assert_allclose(O[:, :, 0], V[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(LSE[:, :, 0], 0.5 * np.sum(Q[:, :, 0] * K[:, :, 0], -1), atol=1e-14)
    dQ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.5, True)[0]
    assert np.max(np.abs(dQ[:, :, 0])) < 1e-15


def test_fully_masked_rows_are_zero():
    """Causal with S_q > S_k: query rows i < S_q - S_k see no key: LSE = -inf, O = 0, dQ = 0."""
    rng = np.random.default_rng(19)
    B, H, S_q, S_k, d = 1, 2, 6, 3, 4
    Q, dO = _rand(rng, B, H, S_q, d), _rand(rng, B, H, S_q, d)
    K, V = _rand(rng, B, H, S_k, d), _rand(rng, B, H, S_k, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, True)
    assert np.all(np.isneginf(LSE[:, :, :3])) and np.all(O[:, :, :3] == 0)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.5, True)
    assert np.all(np.isfinite(dQ)) and np.all(np.isfinite(dK)) and np.all(np.isfinite(dV))
    assert np.all(dQ[:, :, :3] == 0)


def test_linear_in_dO():
    rng = np.random.default_rng(20)
    B, H, H_kv, S, d = 1, 4, 2, 13, 8
    Q, K, V = _rand(rng, B, H, S, d), _rand(rng, B, H_kv, S, d), _rand(rng, B, H_kv, S, d)
    a, b = _rand(rng, B, H, S, d), _rand(rng, B, H, S, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.4, True)
    ga = oracle.ref_bwd(a, Q, K, V, O, LSE, 0.4, True)
    gb = oracle.ref_bwd(b, Q, K, V, O, LSE, 0.4, True)
    gab = oracle.ref_bwd(2 * a - 3 * b, Q, K, V, O, LSE, 0.4, True)
    for x, y, z in zip(ga[:3], gb[:3], gab[:3]):
        np.testing.assert_allclose(z, 2 * x - 3 * y, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_is_sum_over_group(causal):
    rng = np.random.default_rng(21)
    B, H, H_kv, S, d = 2, 8, 2, 11, 8
    g = H // H_kv
    Q, K, V = _rand(rng, B, H, S, d), _rand(rng, B, H_kv, S, d), _rand(rng, B, H_kv, S, d)
    dO = _rand(rng, B, H, S, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.35, causal)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.35, causal)
    Kr, Vr = np.repeat(K, g, axis=1), np.repeat(V, g, axis=1)
    Or, LSEr = oracle.ref_fwd(Q, Kr, Vr, 0.35, causal)
    np.testing.assert_allclose(Or, O, atol=1e-14)
    dQm, dKm, dVm, _ = oracle.ref_bwd(dO, Q, Kr, Vr, Or, LSEr, 0.35, causal)
    np.testing.assert_allclose(dQ, dQm, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dK, dKm.reshape(B, H_kv, g, S, d).sum(2), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dV, dVm.reshape(B, H_kv, g, S, d).sum(2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_match_full_backward(causal):
    rng = np.random.default_rng(22)
    B, H, H_kv, S_q, S_k, d = 2, 4, 2, 21, 37 if not causal else 21, 8
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.3, causal)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.3, causal)
    qrows = np.array([0, 5, S_q - 1, S_q, B * H * S_q - 1])
    krows = np.array([0, 7, S_k - 1, S_k + 3, B * H_kv * S_k - 1])
    np.testing.assert_allclose(oracle.ref_dq_rows(dO, Q, K, V, O, LSE, qrows, 0.3, causal),
                               dQ.reshape(-1, d)[qrows], rtol=1e-13, atol=1e-14)
    dk, dv = oracle.ref_dkv_rows(dO, Q, K, V, O, LSE, krows, 0.3, causal)
    np.testing.assert_allclose(dk, dK.reshape(-1, d)[krows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv, dV.reshape(-1, d)[krows], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# Sliding window (window_size > 0).  Reading: query i sits at key position
# p_i = i + S_k - S_q; a causal query sees keys p_i - w < j <= p_i, a
# non-causal one keys with |j - p_i| < w.

def _band_torch(S_q, S_k, causal, window):
    """The visible set as a band of the all-ones matrix cut by torch.tril/triu
    (diagonal offsets instead of per-element index tests)."""
    off = S_k - S_q
    m = torch.ones(S_q, S_k, dtype=torch.bool)
    if causal:
        m = m.tril(diagonal=off)
    if window > 0:
        m = m.triu(diagonal=off - window + 1)
        if not causal:
            m = m.tril(diagonal=off + window - 1)
    return m


def _sdpa_band_grads(Q, K, V, dO, scale, mask):
    g = Q.shape[1] // K.shape[1]
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    o = F.scaled_dot_product_attention(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1),
                                       attn_mask=mask, scale=scale)
    o.backward(torch.tensor(dO))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy(), o.detach().numpy()


WSHAPES = [
    # B, H, H_kv, S_q, S_k, d, causal, window   (every row keeps at least one key)
    (1, 2, 1, 9, 9, 4, True, 3),
    (1, 2, 2, 9, 9, 4, False, 3),
    (1, 4, 2, 7, 12, 8, True, 4),     # S_q < S_k
    (1, 2, 1, 12, 7, 4, False, 6),    # S_q > S_k, non-causal band
    (2, 4, 1, 17, 17, 8, True, 1),
    (1, 2, 1, 20, 20, 8, False, 7),
    (1, 2, 2, 5, 5, 4, True, 5),      # window = S: same as plain causal
]


@pytest.mark.parametrize("shape", WSHAPES)
def test_window_matches_torch_sdpa_band(shape):
    B, H, H_kv, S_q, S_k, d, causal, w = shape
    rng = np.random.default_rng(23)
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.ref_fwd(Q, K, V, scale, causal, w)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, scale, causal, w)
    tq, tk, tv, to = _sdpa_band_grads(Q, K, V, dO, scale, _band_torch(S_q, S_k, causal, w))
    np.testing.assert_allclose(O, to, rtol=1e-12, atol=1e-12)
    for name, a, b in (("dQ", dQ, tq), ("dK", dK, tk), ("dV", dV, tv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_window_single_query_is_trailing_slice(causal):
    """S_q = 1 sits at the last key: a window w keeps exactly the last w keys, so
    the result is unmasked attention over K[S_k-w:], V[S_k-w:] and the other
    keys get zero gradient."""
    rng = np.random.default_rng(24)
    B, H, H_kv, S_k, d, w = 1, 2, 1, 13, 8, 5
    Q, dO = _rand(rng, B, H, 1, d), _rand(rng, B, H, 1, d)
    K, V = _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.4, causal, w)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.4, causal, w)
    tq, tk, tv, to = _sdpa_band_grads(Q, K[:, :, -w:], V[:, :, -w:], dO, 0.4, None)
    np.testing.assert_allclose(O, to, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dQ, tq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK[:, :, -w:], tk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV[:, :, -w:], tv, rtol=1e-10, atol=1e-12)
    assert np.all(dK[:, :, :-w] == 0) and np.all(dV[:, :, :-w] == 0)


def test_window_noncausal_first_row_is_leading_slice():
    """Non-causal, S_q = S_k: query 0 sees keys 0 .. w-1 and no others."""
    rng = np.random.default_rng(25)
    B, H, S, d, w = 1, 2, 11, 8, 4
    Q, K, V, dO = (_rand(rng, B, H, S, d) for _ in range(4))
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, False, w)
    _, _, _, to = _sdpa_band_grads(Q[:, :, :1], K[:, :, :w], V[:, :, :w], dO[:, :, :1], 0.5, None)
    np.testing.assert_allclose(O[:, :, :1], to, rtol=1e-12, atol=1e-13)
    rows = np.array([0, S])   # query 0 of heads 0 and 1
    tq = _sdpa_band_grads(Q[:, :, :1], K[:, :, :w], V[:, :, :w], dO[:, :, :1], 0.5, None)[0]
    np.testing.assert_allclose(oracle.ref_dq_rows(dO, Q, K, V, O, LSE, rows, 0.5, False, w),
                               tq.reshape(-1, d), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal,S_q,S_k", [(True, 6, 9), (False, 6, 9), (True, 9, 6), (False, 9, 6)])
def test_window_one_is_diagonal(causal, S_q, S_k):
    """w = 1: query i sees only key p_i = i + S_k - S_q (if it exists), so O_i = V_{p_i},
    LSE_i = scale <Q_i, K_{p_i}>, P = 1, dS = 0 (dQ = dK = 0) and dV_j sums dO_i over the
    group rows with p_i = j; rows with p_i < 0 see nothing."""
    rng = np.random.default_rng(26)
    B, H, H_kv, d = 1, 4, 2, 4
    g = H // H_kv
    Q, dO = _rand(rng, B, H, S_q, d), _rand(rng, B, H, S_q, d)
    K, V = _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, causal, 1)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.5, causal, 1)
    expect_dV = np.zeros_like(V)
    for h in range(H):
        for i in range(S_q):
            p = i + S_k - S_q
            if p < 0:
                assert np.isneginf(LSE[0, h, i]) and np.all(O[0, h, i] == 0)
                continue
            np.testing.assert_allclose(O[0, h, i], V[0, h // g, p], atol=1e-15)
            np.testing.assert_allclose(LSE[0, h, i], 0.5 * Q[0, h, i] @ K[0, h // g, p], atol=1e-14)
            expect_dV[0, h // g, p] += dO[0, h, i]
    assert np.max(np.abs(dQ)) < 1e-14 and np.max(np.abs(dK)) < 1e-14
    np.testing.assert_allclose(dV, expect_dV, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_window_wider_than_problem_is_no_window(causal):
    rng = np.random.default_rng(27)
    B, H, H_kv, S_q, S_k, d = 1, 2, 1, 7, 10, 4
    Q, dO = _rand(rng, B, H, S_q, d), _rand(rng, B, H, S_q, d)
    K, V = _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    O0, L0 = oracle.ref_fwd(Q, K, V, 0.5, causal)
    Ow, Lw = oracle.ref_fwd(Q, K, V, 0.5, causal, S_q + S_k)
    assert np.array_equal(O0, Ow) and np.array_equal(L0, Lw)
    for a, b in zip(oracle.ref_bwd(dO, Q, K, V, O0, L0, 0.5, causal),
                    oracle.ref_bwd(dO, Q, K, V, Ow, Lw, 0.5, causal, S_q + S_k)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [(1, 2, 1, 6, 6, 4, True, 2), (1, 2, 2, 5, 7, 4, False, 3)])
def test_window_matches_finite_differences(shape):
    B, H, H_kv, S_q, S_k, d, causal, w = shape
    rng = np.random.default_rng(28)
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.5, causal, w)
    grads = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.5, causal, w)[:3]
    eps = 1e-5
    for which, (X, G) in enumerate(zip((Q, K, V), grads)):
        fd = np.zeros_like(X)
        for idx in itertools.product(*map(range, X.shape)):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += eps
            lp = float(np.sum(dO * oracle.ref_fwd(*args, 0.5, causal, w)[0]))
            args[which][idx] -= 2 * eps
            lm = float(np.sum(dO * oracle.ref_fwd(*args, 0.5, causal, w)[0]))
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(fd - G)) / max(np.max(np.abs(G)), 1e-30)
        assert err < 1e-7, (which, err)


@pytest.mark.parametrize("causal", [False, True])
def test_window_sampled_rows_match_full_backward(causal):
    rng = np.random.default_rng(29)
    B, H, H_kv, S_q, S_k, d, w = 1, 4, 2, 19, 23, 8, 5
    Q, K, V = _rand(rng, B, H, S_q, d), _rand(rng, B, H_kv, S_k, d), _rand(rng, B, H_kv, S_k, d)
    dO = _rand(rng, B, H, S_q, d)
    O, LSE = oracle.ref_fwd(Q, K, V, 0.3, causal, w)
    dQ, dK, dV, _ = oracle.ref_bwd(dO, Q, K, V, O, LSE, 0.3, causal, w)
    qrows = np.array([0, 4, S_q - 1, S_q + 2, B * H * S_q - 1])
    krows = np.array([0, 3, 9, S_k - 1, S_k + 10, B * H_kv * S_k - 1])
    np.testing.assert_allclose(oracle.ref_dq_rows(dO, Q, K, V, O, LSE, qrows, 0.3, causal, w),
                               dQ.reshape(-1, d)[qrows], rtol=1e-13, atol=1e-14)
    dk, dv = oracle.ref_dkv_rows(dO, Q, K, V, O, LSE, krows, 0.3, causal, w)
    np.testing.assert_allclose(dk, dK.reshape(-1, d)[krows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv, dV.reshape(-1, d)[krows], rtol=1e-13, atol=1e-14)
