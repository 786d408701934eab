"""Backward parity: the CUDA path (through the C ABI) against the fp64 oracle's
naive chain-rule backward."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from tests.parity import TOL, oracle_bwd, rel_fro, seeded_heads, to64

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
                                  "causal_bf16_b1h2_n16384_d128"])
def test_bwd_full_size_every_head(cuda_device, fa2_lib, name):
    """Full-size launch; every head's dQ, dK, dV go through the oracle."""
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    tol = TOL[w.torch_dtype]
    for b in range(w.B):
        for h in range(w.H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            ref = oracle_bwd(q[sl], k[sl], v[sl], do[sl], w.causal, w.scale)
            _check_grads((dq[sl], dk[sl], dv[sl]), ref, tol)


def test_bwd_headline_eight_seeded_heads(cuda_device, fa2_lib):
    """The 128-head long-sequence workload at full size; eight whole heads
    drawn by a seeded RNG go through the oracle, and every head's gradients are
    finite."""
    w = WORKLOADS["causal_bf16_b4h32_n8192_d128_qstd3"]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    heads = seeded_heads(w, 8, 2)
    refs = oracle_bwd(q, k, v, do, w.causal, w.scale, heads=heads)
    tol = TOL[w.torch_dtype]
    for (b, h), (dq_r, dk_r, dv_r) in zip(heads, refs):
        _check_grads((dq[b:b + 1, h:h + 1], dk[b:b + 1, h:h + 1], dv[b:b + 1, h:h + 1]),
                     (dq_r, dk_r, dv_r), tol)


def test_bwd_column_sums_of_dv(cuda_device, fa2_lib):
    """Rows of P sum to 1, so sum_j dV_j = sum_i dO_i for every head (a property
    of the whole head that element parity checks only term by term)."""
    w = WORKLOADS["causal_bf16_b8h16_n2048_d128"]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = _run(fa2_lib, cuda_device, q, k, v, do, w.causal, w.scale)
    sdv = to64(dv).sum(axis=2)
    sdo = to64(do).sum(axis=2)
    assert np.max(np.abs(sdv - sdo)) / np.max(np.abs(sdo)) <= 2e-2


def test_bwd_dq_is_deterministic(cuda_device, fa2_lib):
    """dQ has no atomics: two runs give bit-identical gradients."""
    q, k, v, do = make_inputs(1, 4, 1000, 128, torch.bfloat16, seed=13)
    r1 = _run(fa2_lib, cuda_device, q, k, v, do, True, 128 ** -0.5)
    r2 = _run(fa2_lib, cuda_device, q, k, v, do, True, 128 ** -0.5)
    for a, b in zip(r1[2:], r2[2:]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["causal_bf16_b8h16_n2048_d128", "bf16_b8h16_n2048_d128"])
def test_bwd_repeats_bit_for_bit(cuda_device, fa2_lib, name):
    """Four backward calls on a full-size 128-head workload give the same bits
    for dQ, dK and dV, and every value is finite. The main launch hands its
    work items to CTAs through a counter, so which SM runs which key or query
    block, and what runs beside it, changes from call to call; the gradients
    must not."""
    w = WORKLOADS[name]
    q, k, v, do = (t.to(cuda_device) for t in workload_inputs(w))
    o, lse = fa2_lib.forward(q, k, v, causal=w.causal, scale=w.scale, num_splits=1)
    runs = [fa2_lib.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale) for _ in range(4)]
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    for g in runs[0]:
        assert bool(torch.isfinite(g).all())
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,N,d,dtype,causal", EDGE[::2] + [(2, 2, 640, 128, torch.bfloat16, True)])
def test_bwd_atomic_edge_shapes(cuda_device, fa2_lib, B, H, N, d, dtype, causal):
    """fa2_bwd_atomic (column workers, dQ by fp32 reduce-adds) against the oracle."""
    q, k, v, do = make_inputs(B, H, N, d, dtype, seed=7 * N + d + 1)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    o, lse = fa2_lib.forward(qd, kd, vd, causal=causal, scale=scale)
    grads = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, atomic=True)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    _check_grads([g.cpu() for g in grads], oracle_bwd(q, k, v, do, causal, scale), TOL[dtype])


def test_bwd_atomic_headline_two_seeded_heads(cuda_device, fa2_lib):
    """fa2_bwd_atomic on the 128-head long-sequence workload at full size; two
    seeded heads through the oracle; its dK and dV are bit-reproducible (only
    dQ goes through reduce-adds)."""
    w = WORKLOADS["causal_bf16_b4h32_n8192_d128_qstd3"]
    q, k, v, do = workload_inputs(w)
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    o, lse = fa2_lib.forward(qd, kd, vd, causal=True, scale=w.scale)
    g1 = [t.clone() for t in fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale,
                                              atomic=True)]
    g2 = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale, atomic=True)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    heads = seeded_heads(w, 2, 3)
    refs = oracle_bwd(q, k, v, do, True, w.scale, heads=heads)
    for (b, h), ref in zip(heads, refs):
        _check_grads([t[b:b + 1, h:h + 1].cpu() for t in g1], ref, TOL[w.torch_dtype])


def test_autograd_function(cuda_device, fa2_lib):
    q, k, v, do = make_inputs(1, 2, 300, 64, torch.bfloat16, seed=11)
    dev = cuda_device
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    out = fa2_lib.attention(qd, kd, vd, causal=True)
    out.backward(do.to(dev))
    ref = oracle_bwd(q, k, v, do, True, 0.125)
    _check_grads((qd.grad.cpu(), kd.grad.cpu(), vd.grad.cpu()), ref, TOL[torch.bfloat16])
