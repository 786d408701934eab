"""Backward parity: the CUDA path (through the C ABI) against the fp64 oracle's
naive chain-rule backward."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from tests.parity import TOL, oracle_bwd, rel_fro, to64

pytestmark = pytest.mark.gpu


def _run(fa2, dev, q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa2.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa2.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2.device_status() == 0
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


def _check_grads(got, ref, tol):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g64 = to64(g)
        assert np.all(np.isfinite(g64)), name
        err = rel_fro(g64, r)
        assert err <= tol["grad"], (name, err)


EDGE = [
    (1, 1, 1, 64, torch.bfloat16, False),
    (1, 1, 1, 128, torch.float16, True),
    (1, 3, 2, 64, torch.bfloat16, True),
    (1, 1, 63, 128, torch.bfloat16, True),
    (1, 1, 127, 128, torch.bfloat16, False),
    (1, 1, 129, 64, torch.float16, True),
    (2, 1, 255, 128, torch.bfloat16, True),
    (1, 3, 256, 64, torch.bfloat16, False),
    (1, 2, 257, 128, torch.float16, False),
    (1, 1, 384, 128, torch.bfloat16, True),
    (1, 2, 1000, 64, torch.bfloat16, True),
    (1, 1, 1000, 128, torch.float16, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", EDGE)
def test_bwd_edge_shapes(cuda_device, fa2_lib, B, H, N, d, dtype, causal):
    q, k, v, do = make_inputs(B, H, N, d, dtype, seed=7 * N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, causal, scale)
    ref = oracle_bwd(q, k, v, do, causal, scale)
    _check_grads((dq, dk, dv), ref, TOL[dtype])


@pytest.mark.parametrize("name", ["fp16_b1h1_n128_d64", "causal_bf16_b2h4_n1024_d64"])
def test_bwd_small_workloads_full(cuda_device, fa2_lib, name):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    ref = oracle_bwd(q, k, v, do, w.causal, w.scale)
    _check_grads((dq, dk, dv), ref, TOL[w.torch_dtype])


@pytest.mark.parametrize("name", ["bf16_b8h16_n2048_d128", "causal_bf16_b8h16_n2048_d128",
                                  "causal_bf16_b1h2_n16384_d128",
                                  "causal_bf16_b4h32_n8192_d128_qstd3"])
def test_bwd_full_size_sampled_heads(cuda_device, fa2_lib, name):
    """Full-size launch; whole heads chosen by a seeded draw go through the oracle."""
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    rng = np.random.default_rng(2)
    nheads = 1 if w.N >= 8192 else 2
    heads = sorted({(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(nheads)})
    refs = oracle_bwd(q, k, v, do, w.causal, w.scale, heads=heads)
    tol = TOL[w.torch_dtype]
    for (b, h), (dq_r, dk_r, dv_r) in zip(heads, refs):
        _check_grads((dq[b:b + 1, h:h + 1], dk[b:b + 1, h:h + 1], dv[b:b + 1, h:h + 1]),
                     (dq_r, dk_r, dv_r), tol)


def test_bwd_invariants_full_size(cuda_device, fa2_lib):
    """Properties that hold at any size, on every head of a full-size run:
    rows of P sum to 1 => sum_j dV_j = sum_i dO_i; rows of dS sum to 0 =>
    sum_j dK_j = 0."""
    w = WORKLOADS["causal_bf16_b8h16_n2048_d128"]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    sdv = to64(dv).sum(axis=2)
    sdo = to64(do).sum(axis=2)
    assert np.max(np.abs(sdv - sdo)) / np.max(np.abs(sdo)) <= 2e-2
    sdk = to64(dk).sum(axis=2)
    assert np.max(np.abs(sdk)) <= 2e-2 * np.max(np.abs(to64(dk))) * math.sqrt(w.N)


def test_bwd_dq_is_deterministic(cuda_device, fa2_lib):
    """dQ has no atomics: two runs give bit-identical gradients."""
    q, k, v, do = make_inputs(1, 4, 1000, 128, torch.bfloat16, seed=13)
    r1 = _run(fa2_lib, cuda_device, q, k, v, do, True, 128 ** -0.5)
    r2 = _run(fa2_lib, cuda_device, q, k, v, do, True, 128 ** -0.5)
    for a, b in zip(r1[2:], r2[2:]):
        assert torch.equal(a, b)


def test_autograd_function(cuda_device, fa2_lib):
    q, k, v, do = make_inputs(1, 2, 300, 64, torch.bfloat16, seed=11)
    dev = cuda_device
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    out = fa2_lib.attention(qd, kd, vd, causal=True)
    out.backward(do.to(dev))
    ref = oracle_bwd(q, k, v, do, True, 0.125)
    _check_grads((qd.grad.cpu(), kd.grad.cpu(), vd.grad.cpu()), ref, TOL[torch.bfloat16])
