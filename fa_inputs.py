"""Seeded synthetic inputs for the attention forward workloads.

This module is shared by the CUDA path's tests and bench and by the fp64
oracle's callers.  It only draws random numbers and names workload shapes; it
holds none of the attention arithmetic, so neither side can lean on the other
through it.

Workloads (all tensors are contiguous [B, H, S, D]):

* ``tiny``            1 x 2 x 128 x 64, fp16, run with and without the causal mask
* ``batch1_causal``   1 x 16 x 1024 x 64, fp16, causal (batch-1 long-text decode
                      scene of "CUDA手写masked multi-head attention", section 1)
* ``wide_noncausal``  10 x 64 x 1024 x 64, fp16, no mask (the B=10, N_h=64,
                      S=1024, D=64 shape measured in "FlashAttention的Triton性能考古学")
* ``train_causal``    4 x 32 x 4096 x 128, bf16, causal
* ``stress_causal``   1 x 32 x 16384 x 128, bf16, causal; Q and K are 3*N(0,1),
                      and K gets a bias that rises linearly with the key index,
                      so the running row maximum keeps climbing and the lazy
                      rescale of "G6: Cluster 与 2CTA 探索", V41, has to fire.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; fp32 ``randn`` drawn in
the order Q, K, V with shape [B, H, S, D]; then cast to the workload dtype.
The stress workload scales Q and K by 3 and adds ``GAMMA * j / (S - 1)`` to
every element of key row j (GAMMA = 32) before the cast.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

GAMMA = 32.0  # slope of the stress workload's key bias over the whole sequence

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str        # "fp16" | "bf16"
    causal: bool
    kind: str = "randn"   # "randn" | "stress"

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)

    def flops(self) -> float:
        """Useful FLOPs: 4*B*H*S^2*D (QK^T and PV), halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.S * self.S * self.D
        return f / 2.0 if self.causal else f

    def io_bytes(self) -> int:
        """Q, K, V read once, O written once (dtype) plus the fp32 LSE."""
        n = self.B * self.H * self.S
        return 4 * n * self.D * 2 + 4 * n


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 64, "fp16", False),
    "tiny_causal": Workload("tiny_causal", 1, 2, 128, 64, "fp16", True),
    "batch1_causal": Workload("batch1_causal", 1, 16, 1024, 64, "fp16", True),
    "wide_noncausal": Workload("wide_noncausal", 10, 64, 1024, 64, "fp16", False),
    "train_causal": Workload("train_causal", 4, 32, 4096, 128, "bf16", True),
    "stress_causal": Workload("stress_causal", 1, 32, 16384, 128, "bf16", True, "stress"),
}


def make_qkv(B: int, H: int, S: int, D: int, dtype: str = "fp16", seed: int = 0,
             kind: str = "randn"):
    """Return CPU tensors (q, k, v) of shape [B, H, S, D] in ``dtype``."""
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    g = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, S, D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if kind == "stress":
        q.mul_(3.0)
        k.mul_(3.0)
        ramp = torch.arange(S, dtype=torch.float32) * (GAMMA / max(S - 1, 1))
        k.add_(ramp.view(1, 1, S, 1))
    elif kind != "randn":
        raise ValueError(f"unknown input kind {kind!r}")
    t = DTYPES[dtype]
    return q.to(t), k.to(t), v.to(t)


def make_workload(w: Workload, seed: int = 0):
    return make_qkv(w.B, w.H, w.S, w.D, w.dtype, seed, w.kind)


def to_f64(x) -> "numpy.ndarray":
    """Exact widening of a 16-bit CPU tensor to a contiguous float64 numpy array."""
    return x.to(torch.float64).contiguous().numpy()
