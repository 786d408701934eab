"""Seeded synthetic workloads (inputs only -- no attention arithmetic here).

Both the CUDA path and the fp64 oracle are fed from this module, so it holds
nothing but the workload shapes and the random draws: i.i.d. Gaussian Q, K, V
and dO, drawn in that order as float32 from a CPU ``torch.Generator`` seeded
with ``seed`` (default 0), with Q optionally scaled by ``q_std``, then rounded
to the 16-bit dtype (round-to-nearest-even). The pages measure on no dataset;
these tensors stand in for activations of the shapes below.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "workload_inputs", "HEADLINE"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "fp16" | "bf16"
    causal: bool
    q_std: float = 1.0

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    def fwd_flops(self) -> float:
        """4*B*H*N^2*d, halved under the causal mask (the usual convention)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


_W = [
    Workload("fp16_b1h1_n128_d64", 1, 1, 128, 64, "fp16", False),
    Workload("causal_bf16_b2h4_n1024_d64", 2, 4, 1024, 64, "bf16", True),
    Workload("bf16_b8h16_n2048_d128", 8, 16, 2048, 128, "bf16", False),
    Workload("causal_bf16_b8h16_n2048_d128", 8, 16, 2048, 128, "bf16", True),
    Workload("causal_bf16_b1h2_n16384_d128", 1, 2, 16384, 128, "bf16", True),
    Workload("causal_bf16_b4h32_n8192_d128_qstd3", 4, 32, 8192, 128, "bf16", True, 3.0),
]
# Same per-head shape as the headline with fewer heads: a profiling case whose
# inputs still exceed L2 but whose captures stay small.
_W.append(Workload("causal_bf16_b2h16_n8192_d128_qstd3", 2, 16, 8192, 128, "bf16", True, 3.0))
# The other head size and the other 16-bit type at the long-sequence shape.
_W.append(Workload("causal_bf16_b4h64_n8192_d64", 4, 64, 8192, 64, "bf16", True))
_W.append(Workload("causal_fp16_b4h32_n8192_d128", 4, 32, 8192, 128, "fp16", True))
WORKLOADS = {w.name: w for w in _W}

# Long-sequence, d=128 causal workload the throughput target is stated on.
HEADLINE = "causal_bf16_b4h32_n8192_d128_qstd3"


def make_inputs(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, q_std: float = 1.0,
                seed: int = 0):
    """(q, k, v, do): CPU tensors [B, H, N, d] of ``dtype``."""
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    if q_std != 1.0:
        q = q * q_std
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    return tuple(t.to(dtype) for t in (q, k, v, do))


def workload_inputs(w: Workload, seed: int = 0):
    return make_inputs(w.B, w.H, w.N, w.d, w.torch_dtype, w.q_std, seed)
