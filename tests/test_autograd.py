"""torch.autograd integration (autograd.py): the backward of flash_attention is the
library's backward, fed the q, k, v, O and LSE its forward saved (boostr
autograd_attention.rs, FlashAttentionBackward / var_flash_attention)."""
import math

import numpy as np
import pytest
import torch

import flashattention_backward_preprocess_gb300 as fa
import oracle
from flashattention_backward_preprocess_gb300.inputs import Workload, make_inputs

TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 2e-2}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(a, b):
    den = float(np.max(np.abs(b)))
    return float(np.max(np.abs(a - b))) / (den if den > 0 else 1.0)


def test_host_tensors_are_rejected_not_computed_on_cpu():
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, requires_grad=True)
    with pytest.raises(fa.FaError, match="device pointers required"):
        fa.flash_attention(q, q, q)


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    ("bf16", 2, 8, 2, 300, 300, 128, True, 0, False),
    ("f16", 1, 4, 4, 200, 333, 64, False, 0, False),
    ("bf16", 1, 4, 1, 400, 400, 128, True, 150, True),   # window + deterministic
    ("f32", 1, 2, 1, 130, 130, 64, True, 0, False),
])
def test_autograd_gradients_are_the_library_backward(case):
    dt, B, H, H_kv, S_q, S_k, d, causal, win, det = case
    w = Workload("ag", dt, B, H, H_kv, S_q, S_k, d, causal, seed=51, window=win)
    Q, K, V, dO = (x.cuda() for x in make_inputs(w))
    q, k, v = (x.clone().requires_grad_(True) for x in (Q, K, V))
    out = fa.flash_attention(q, k, v, causal=causal, window_size=win, deterministic=det)
    out.backward(dO)
    torch.cuda.synchronize()
    fa.fa_check_device()
    # the same O / LSE the wrapper saved (the forward is deterministic), then fa_bwd directly
    O, LSE = fa.fa_fwd(Q, K, V, causal=causal, window_size=win)
    assert torch.equal(O, out.detach())
    dQ, dK, dV = fa.fa_bwd(dO, Q, K, V, O, LSE, causal=causal, window_size=win, deterministic=det)
    torch.cuda.synchronize()
    assert torch.equal(k.grad, dK) and torch.equal(v.grad, dV)
    assert rel_err(f64(q.grad), f64(dQ)) <= (0 if det else 1e-2)
    ref = oracle.ref_bwd(f64(dO), f64(Q), f64(K), f64(V), f64(O), f64(LSE), w.scale, causal, win)
    for name, g, r in zip(("dQ", "dK", "dV"), (q.grad, k.grad, v.grad), ref[:3]):
        assert rel_err(f64(g), r) <= TOL[dt], name


@pytest.mark.gpu
def test_autograd_noncontiguous_inputs_and_no_grad():
    w = Workload("ag_nc", "bf16", 1, 4, 2, 256, 256, 64, True, seed=52)
    Q, K, V, dO = (x.cuda() for x in make_inputs(w))
    # q as a transposed view of a [B, S, H, d] buffer
    q_bshd = Q.transpose(1, 2).contiguous().requires_grad_(True)
    q = q_bshd.transpose(1, 2)
    assert not q.is_contiguous()
    out = fa.flash_attention(q, K, V, causal=True)
    out.backward(dO)
    torch.cuda.synchronize()
    O, LSE = fa.fa_fwd(Q, K, V, causal=True)
    dQ = fa.fa_bwd(dO, Q, K, V, O, LSE, causal=True)[0]
    assert rel_err(f64(q_bshd.grad.transpose(1, 2)), f64(dQ)) < 1e-2
    with torch.no_grad():
        o2 = fa.flash_attention(Q, K, V, causal=True)
    assert o2.grad_fn is None and torch.equal(o2, O)


@pytest.mark.gpu
def test_training_step_through_a_projection_matches_fp32_math_attention():
    """x -> Linear -> q, k, v -> attention -> loss: the projection's weight gradient through
    this library matches the one through PyTorch's fp32 math attention."""
    torch.manual_seed(0)
    B, S, E, H, d = 2, 256, 512, 4, 128
    x = torch.randn(B, S, E, device="cuda")
    proj = torch.nn.Linear(E, 3 * H * d, bias=False, device="cuda")
    target = torch.randn(B, H, S, d, device="cuda")

    def qkv(p):
        t = p(x).view(B, S, 3, H, d).permute(2, 0, 3, 1, 4)
        return t[0], t[1], t[2]

    def loss_of(o):
        return ((o.float() - target) ** 2).mean()

    proj.weight.grad = None
    q, k, v = qkv(proj)
    loss_of(fa.flash_attention(q.bfloat16(), k.bfloat16(), v.bfloat16(), causal=True)).backward()
    g_lib = proj.weight.grad.clone()

    proj.weight.grad = None
    q, k, v = qkv(proj)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=1.0 / math.sqrt(d))
    loss_of(ref).backward()
    g_ref = proj.weight.grad.clone()
    assert rel_err(f64(g_lib), f64(g_ref)) < 3e-2
