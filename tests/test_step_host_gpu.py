"""fa2_step_host: forward + backward on host buffers, pipelined by head chunks
over internal streams. Every (batch, head) is independent, so each chunk runs
the same kernels on the same per-head data as a whole-tensor launch: the
results must be the same bits as fa2_fwd (unsplit) + fa2_bwd on device copies."""

import math

import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,dtype,causal,hpc", [
    (1, 1, 1, 64, torch.bfloat16, False, 0),
    (2, 3, 300, 128, torch.bfloat16, True, 1),      # 6 chunks of one head
    (2, 3, 300, 128, torch.float16, False, 4),      # a short last chunk
    (1, 5, 1000, 64, torch.bfloat16, True, 0),      # auto: 1 head per chunk
    (4, 8, 1024, 128, torch.bfloat16, True, 3),     # 11 chunks over 2 slots
])
def test_step_host_matches_the_device_path_bitwise(cuda_device, fa2_lib, B, H, N, d, dtype, causal,
                                                  hpc):
    q, k, v, do = make_inputs(B, H, N, d, dtype, seed=11 * N + H)
    scale = 1.0 / math.sqrt(d)
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    with torch.cuda.device(cuda_device):
        o, lse, dq, dk, dv = fa2_lib.step_host(hq, hk, hv, hdo, causal=causal, scale=scale,
                                               heads_per_chunk=hpc, device=cuda_device)
    qd, kd, vd, dod = (t.to(cuda_device) for t in (q, k, v, do))
    o2, lse2 = fa2_lib.forward(qd, kd, vd, causal=causal, scale=scale, num_splits=1)
    dq2, dk2, dv2 = fa2_lib.backward(qd, kd, vd, o2, lse2, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    for a, b, name in ((o, o2, "o"), (lse, lse2, "lse"), (dq, dq2, "dq"), (dk, dk2, "dk"),
                       (dv, dv2, "dv")):
        assert torch.equal(a, b.cpu()), name


def test_step_host_from_pageable_memory(cuda_device, fa2_lib):
    """Unpinned host buffers still give the same bits (the copies just do not overlap)."""
    B, H, N, d = 1, 4, 256, 64
    q, k, v, do = make_inputs(B, H, N, d, torch.bfloat16, seed=2)
    with torch.cuda.device(cuda_device):
        a = fa2_lib.step_host(q, k, v, do, causal=True, heads_per_chunk=1, device=cuda_device)
        b = fa2_lib.step_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), do.pin_memory(),
                              causal=True, heads_per_chunk=3, device=cuda_device)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("hpc", [4, 16])
def test_step_host_repeated_long_sequence_chunks(cuda_device, fa2_lib, hpc):
    """Repeated steps over 16 causal heads of 8192 rows in chunks of 1 to 16
    heads: consecutive chunks' backward launches overlap on the two slot
    streams, and every call ends with a clean device status and the same bits
    as the first."""
    q, k, v, do = make_inputs(1, 16, 8192, 128, torch.bfloat16, seed=5)
    scale = 128 ** -0.5
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    first = None
    for _ in range(4):
        with torch.cuda.device(cuda_device):
            out = fa2_lib.step_host(hq, hk, hv, hdo, causal=True, scale=scale,
                                    heads_per_chunk=hpc, device=cuda_device)
        assert fa2_lib.device_status() == 0
        if first is None:
            first = [t.clone() for t in out]
        else:
            for a, b in zip(first, out):
                assert torch.equal(a, b)
