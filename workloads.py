"""Seeded synthetic attention workloads, shared by the tests, the bench and the oracle checks.

This module only draws random numbers and names shapes; it holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from here
without sharing any of the method.

Recipe (the pages measure at the FlashAttention-4 paper's S = 4K / 8K / 16K shapes with
head_dim 128, BF16, dense and non-causal, and do not state batch or heads):

* a CPU ``torch.Generator`` seeded with the workload's seed draws Q, then K, then V as
  fp32 standard normals of shape ``[B, H, S, D]``;
* for the ragged long workload, Q and K are multiplied by 3 in fp32 (peaky softmax rows,
  score std about 9 after the 1/sqrt(128) scale, so the online-softmax rebase path runs);
* each tensor is rounded once, round-to-nearest-even, to BF16.

The oracle reads the very same BF16 values, widened exactly to fp64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int = 128
    qk_gain: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> int:
        """Two dense contractions, 2*S*S*D multiply-adds each, per (b, h): 4*B*H*S^2*D."""
        return 4 * self.B * self.H * self.S * self.S * self.D

    @property
    def rows(self) -> int:
        return self.B * self.H * self.S

    def label(self) -> str:
        g = f" QKx{self.qk_gain:g}" if self.qk_gain != 1.0 else ""
        return f"{self.name}: B={self.B} H={self.H} S={self.S} D={self.D}{g}"


# The five workloads: a small parity case and the pages' three sequence lengths, plus a
# long ragged one whose S is not a multiple of the 128-row tile.
TINY = Workload("tiny", B=1, H=1, S=256, seed=0)
S4K = Workload("s4k", B=4, H=16, S=4096, seed=1)
S8K = Workload("s8k", B=2, H=16, S=8192, seed=2)
S16K = Workload("s16k", B=1, H=16, S=16384, seed=3)
RAGGED = Workload("ragged", B=2, H=24, S=17550, qk_gain=3.0, seed=4)

ALL = {w.name: w for w in (TINY, S4K, S8K, S16K, RAGGED)}


def make_qkv(w: Workload, seed: int | None = None):
    """Return (q, k, v) as contiguous CPU BF16 tensors of shape [B, H, S, D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.H, w.S, w.D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.qk_gain != 1.0:
        q.mul_(w.qk_gain)
        k.mul_(w.qk_gain)
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_custom(B: int, H: int, S: int, D: int = 128, seed: int = 0, qk_gain: float = 1.0):
    """Same recipe for an arbitrary shape (edge-case parity tests)."""
    return make_qkv(Workload("custom", B=B, H=H, S=S, D=D, qk_gain=qk_gain, seed=seed))


def to_f64(t: torch.Tensor):
    """Exact widening of a BF16 (or any float) CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
