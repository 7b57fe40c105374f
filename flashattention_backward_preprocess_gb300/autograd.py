"""torch.autograd integration: attention whose backward is this library's backward.

Follows boostr autograd_attention.rs (FlashAttentionBackward and
var_flash_attention): the forward runs the attention forward, keeps q, k, v,
the output and the per-row log-sum-exp, and the backward hands those and the
incoming gradient to the FlashAttention-2 backward, returning dQ, dK, dV.
As on that page the backward is first order only (its result does not build a
graph of its own), and the log-sum-exp stays internal: the function returns
the output alone.

Both passes run in the C-ABI library (fa_fwd_ex / fa_bwd_ex through the ctypes
binding); nothing here computes attention.  Layouts are those of the library:
q [B, H, S_q, d], k and v [B, H_kv, S_k, d], contiguous, on one CUDA device.
"""
from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import binding


class FlashAttentionFunction(torch.autograd.Function):
    """O = softmax(scale * q k^T [masked]) v with the library's backward.

    Saved for backward (autograd_attention.rs, saved_tensors): q, k, v, O, LSE;
    the configuration (causal, window_size, scale, deterministic) rides on ctx,
    like FlashAttentionConfig.
    """

    @staticmethod
    def forward(ctx, q, k, v, causal: bool = False, window_size: int = 0, scale: float | None = None,
                deterministic: bool = False):
        q, k, v = (x.contiguous() for x in (q, k, v))
        o, lse = binding.fa_fwd(q, k, v, scale=scale, causal=causal, window_size=window_size)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal = bool(causal)
        ctx.window_size = int(window_size)
        ctx.scale = scale
        ctx.deterministic = bool(deterministic)
        return o

    @staticmethod
    @once_differentiable
    def backward(ctx, grad_out):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = binding.fa_bwd(grad_out.contiguous(), q, k, v, o, lse, scale=ctx.scale,
                                    causal=ctx.causal, window_size=ctx.window_size,
                                    deterministic=ctx.deterministic)
        # one gradient per forward input: q, k, v, then the four configuration arguments
        return dq, dk, dv, None, None, None, None


def flash_attention(q, k, v, causal: bool = False, window_size: int = 0, scale: float | None = None,
                    deterministic: bool = False):
    """Attention output with autograd support (the var_flash_attention of the pages).

    When none of q, k, v requires grad this is a plain forward: autograd records
    nothing, as var_flash_attention registers no backward then.
    """
    return FlashAttentionFunction.apply(q, k, v, causal, window_size, scale, deterministic)
