"""Seeded synthetic inputs for attention-backward workloads.

This module holds no attention arithmetic: it only draws Q, K, V and dO from
seeded normal distributions and rounds them to the working dtype.  Both the
CUDA path and the fp64 oracle are fed from here (O and LSE are produced by a
forward pass on the drawn inputs, by whichever side the caller chooses).

Workloads (shapes and value distributions of the attention-backward configs
this library is measured on):

  name                              dtype  B  H  H_kv  S_q   S_k   d   causal  dO std
  fp32_b1_h2_s128_d64               f32    1  2   2     128   128  64   no      1
  bf16_b2_h8_s1024_d64_causal       bf16   2  8   8    1024  1024  64   yes     1
  bf16_b4_h32_kv8_s2048_d128_causal bf16   4 32   8    2048  2048 128   yes     0.1
  fp16_b1_h16_s8192_d128            f16    1 16  16    8192  8192 128   no      1
  bf16_b8_h16_kv2_sq512_sk4096_d64  bf16   8 16   2     512  4096  64   no      1
  bf16_b1_h32_kv8_s16384_d128_causal_w4096
                                    bf16   1 32   8   16384 16384 128   yes     1
                                    (sliding window of 4096 keys)
  bf16_b1_h16_kv4_s4096_d256_causal bf16   1 16   4    4096  4096 256   yes     1
  fp32_b2_h8_kv2_s2048_d128_causal  f32    2  8   2    2048  2048 128   yes     1

scale = 1/sqrt(d) everywhere.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" | "f16" | "bf16"
    B: int
    H: int
    H_kv: int
    S_q: int
    S_k: int
    d: int
    causal: bool
    do_std: float = 1.0
    seed: int = 1234
    window: int = 0     # sliding-window size, 0 = none

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def pairs(self) -> float:
        """(query, key) pairs per head the flop counts use: S_q * S_k, halved if causal
        (the usual causal-adjusted count); with a sliding window, the pairs of the band
        (a causal query at key position p keeps keys p-w+1..p, a non-causal one
        p-w+1..p+w-1, clipped to the keys that exist)."""
        if self.window <= 0:
            n = float(self.S_q) * self.S_k
            return n * 0.5 if self.causal else n
        p = np.arange(self.S_q, dtype=np.int64) + (self.S_k - self.S_q)
        lo = np.maximum(p - self.window + 1, 0)
        hi = np.minimum(p + 1 if self.causal else p + self.window, self.S_k)
        return float(np.maximum(hi - lo, 0).sum())

    def flops(self) -> float:
        """Five S_q x S_k x d GEMMs of the backward (2 flops per MAC) over pairs()."""
        return 10.0 * self.B * self.H * self.pairs() * self.d

    def fwd_flops(self) -> float:
        """Two GEMMs of the forward (2 flops per MAC) over pairs()."""
        return 4.0 * self.B * self.H * self.pairs() * self.d

    def algorithmic_bytes(self) -> int:
        """Read Q, K, V, O, dO, LSE; D written and read once; write dQ, dK, dV."""
        nq = self.B * self.H * self.S_q * self.d
        nk = self.B * self.H_kv * self.S_k * self.d
        rows = self.B * self.H * self.S_q
        return self.elem_bytes * (4 * nq + 4 * nk) + 12 * rows

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("fp32_b1_h2_s128_d64", "f32", 1, 2, 2, 128, 128, 64, False, seed=1235),
        Workload("bf16_b2_h8_s1024_d64_causal", "bf16", 2, 8, 8, 1024, 1024, 64, True, seed=1236),
        Workload("bf16_b4_h32_kv8_s2048_d128_causal", "bf16", 4, 32, 8, 2048, 2048, 128, True,
                 do_std=0.1, seed=1237),
        Workload("fp16_b1_h16_s8192_d128", "f16", 1, 16, 16, 8192, 8192, 128, False, seed=1238),
        Workload("bf16_b8_h16_kv2_sq512_sk4096_d64", "bf16", 8, 16, 2, 512, 4096, 64, False,
                 seed=1239),
        Workload("bf16_b1_h32_kv8_s16384_d128_causal_w4096", "bf16", 1, 32, 8, 16384, 16384, 128, True,
                 seed=1240, window=4096),
        # head dim 256 (the tensor-core kernel with 64-key tiles)
        Workload("bf16_b1_h16_kv4_s4096_d256_causal", "bf16", 1, 16, 4, 4096, 4096, 256, True, seed=1241),
        # fp32 at a size where the CUDA-core backward is measured
        Workload("fp32_b2_h8_kv2_s2048_d128_causal", "f32", 2, 8, 2, 2048, 2048, 128, True, seed=1242),
    )
}

#: the workload the benchmark times
BENCH_WORKLOAD = "bf16_b4_h32_kv8_s2048_d128_causal"


def _normal(rng: np.random.Generator, shape, std: float) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x)


def make_inputs(w: Workload, seed: int | None = None):
    """Q, K, V, dO as CPU tensors of w's dtype (round-to-nearest-even from fp32 draws).

    Draw order: Q, K, V, dO from one PCG64 stream seeded with ``seed`` (default
    ``w.seed``).  Q, K, V ~ N(0, 1); dO ~ N(0, w.do_std^2).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    q_shape = (w.B, w.H, w.S_q, w.d)
    kv_shape = (w.B, w.H_kv, w.S_k, w.d)
    Q = _normal(rng, q_shape, 1.0)
    K = _normal(rng, kv_shape, 1.0)
    V = _normal(rng, kv_shape, 1.0)
    dO = _normal(rng, q_shape, w.do_std)
    dt = w.torch_dtype
    return Q.to(dt), K.to(dt), V.to(dt), dO.to(dt)
