"""Failure path of every kernel kind, without faulting the GPU: a host-armed
fault (fa2_debug_arm_fault) makes one TMA producer skip one load, a consumer's
bounded wait runs out after a short limit, the kernel records
FA2_ERR_DEVICE_TIMEOUT and returns, and the next call is correct again."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, max_abs, oracle_bwd, oracle_fwd, rel_fro, to64

pytestmark = pytest.mark.gpu

FA2_ERR_DEVICE_TIMEOUT = 6


def _arm(fa2, kind, ms=20):
    assert fa2.load_library().fa2_debug_arm_fault(kind, ms) == 0


def _fresh_forward_is_correct(fa2, dev, q, k, v, causal, scale, num_splits=1):
    o, lse = fa2.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                         num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa2.device_status() == 0
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
    assert max_abs(to64(o.cpu()), o_ref) <= TOL[q.dtype]["o"]
    assert max_abs(to64(lse.cpu()), lse_ref) <= TOL[q.dtype]["lse"]


def test_split_forward_timeout_path(cuda_device, fa2_lib):
    """Kind 2: every part of a K/V-split forward misses its first V tile."""
    B, H, N, d = 1, 1, 640, 128
    q, k, v, _ = make_inputs(B, H, N, d, torch.bfloat16, seed=41)
    scale = 1.0 / math.sqrt(d)
    _arm(fa2_lib, 2)
    fa2_lib.forward(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), causal=True,
                    scale=scale, num_splits=3)
    assert fa2_lib.device_status() == FA2_ERR_DEVICE_TIMEOUT
    _fresh_forward_is_correct(fa2_lib, cuda_device, q, k, v, True, scale, num_splits=3)


@pytest.mark.parametrize("kind,atomic", [(3, False), (3, True), (4, False)])
def test_backward_timeout_paths(cuda_device, fa2_lib, kind, atomic):
    """Kind 3: the K/V column workers (of either backward) miss their first dO
    tile; kind 4: fa2_bwd's dQ workers miss their first V tile. Either wait
    runs out inside the backward's main launch; the status says so and a
    fresh backward is correct."""
    B, H, N, d = 1, 1, 384, 128
    q, k, v, do = make_inputs(B, H, N, d, torch.bfloat16, seed=40 + kind)
    dev = cuda_device
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa2_lib.forward(qd, kd, vd, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    _arm(fa2_lib, kind)
    fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale,
                     atomic=atomic)
    assert fa2_lib.device_status() == FA2_ERR_DEVICE_TIMEOUT
    dq, dk, dv = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale,
                                  atomic=atomic)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    ref = oracle_bwd(q, k, v, do, True, scale)
    for g, r in zip((dq, dk, dv), ref):
        assert rel_fro(to64(g.cpu()), r) <= TOL[torch.bfloat16]["grad"]


def test_armed_fault_waits_for_its_own_kind(cuda_device, fa2_lib):
    """A backward fault is not consumed by a forward call, a dQ-worker fault
    not by fa2_bwd_atomic, which has no dQ workers (and a disarmed fault by
    nothing)."""
    B, H, N, d = 1, 2, 256, 64
    q, k, v, do = make_inputs(B, H, N, d, torch.bfloat16, seed=45)
    scale = 1.0 / math.sqrt(d)
    _arm(fa2_lib, 4)
    _fresh_forward_is_correct(fa2_lib, cuda_device, q, k, v, False, scale)
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    o, lse = fa2_lib.forward(qd, kd, vd, causal=False, scale=scale)
    fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=False, scale=scale, atomic=True)
    assert fa2_lib.device_status() == 0
    assert fa2_lib.load_library().fa2_debug_arm_fault(0, 0) == 0
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    o, lse = fa2_lib.forward(qd, kd, vd, causal=False, scale=scale)
    fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=False, scale=scale)
    assert fa2_lib.device_status() == 0
    assert np.isfinite(to64(o.cpu())).all()
