"""Helpers shared by the GPU parity tests: run the CUDA path and the fp64
oracle on the same seeded inputs and compare with the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances (fp16, bf16): max |dO| on O, max |dL| on L, relative Frobenius
# error on dQ, dK, dV.
TOL = {
    torch.float16: dict(o=1e-2, lse=1e-3, grad=5e-2),
    torch.bfloat16: dict(o=2e-2, lse=2e-3, grad=5e-2),
}


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_fwd(q, k, v, causal, scale, heads=None):
    """Oracle forward on CPU tensors; ``heads`` = list of (b, h) to restrict to."""
    if heads is None:
        return oracle.forward(to64(q), to64(k), to64(v), causal=causal, scale=scale)
    return [oracle.forward(to64(q[b:b + 1, h:h + 1]), to64(k[b:b + 1, h:h + 1]),
                           to64(v[b:b + 1, h:h + 1]), causal=causal, scale=scale)
            for b, h in heads]


def oracle_bwd(q, k, v, do, causal, scale, heads=None):
    if heads is None:
        return oracle.backward(to64(q), to64(k), to64(v), to64(do), causal=causal, scale=scale)
    return [oracle.backward(to64(q[b:b + 1, h:h + 1]), to64(k[b:b + 1, h:h + 1]),
                            to64(v[b:b + 1, h:h + 1]), to64(do[b:b + 1, h:h + 1]),
                            causal=causal, scale=scale) for b, h in heads]


def max_abs(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_fro(a: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(a - ref))
    return num / den if den > 0 else num


def seeded_heads(w, count: int, seed: int):
    """``count`` distinct (b, h) heads of workload ``w`` drawn by a seeded RNG."""
    flat = np.random.default_rng(seed).choice(w.B * w.H, size=count, replace=False)
    return sorted((int(x) // w.H, int(x) % w.H) for x in flat)
