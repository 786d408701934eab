"""The entry points are stream-ordered with no host synchronisation, so a
whole step can be captured in a CUDA graph and replayed: replays give the
bits of eager calls, also after the inputs are overwritten in place."""

import math

import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


def _eager(fa2, q, k, v, do, causal, splits):
    o, lse = fa2.forward(q, k, v, causal=causal, num_splits=splits)
    dq, dk, dv = fa2.backward(q, k, v, o, lse, do, causal=causal)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal,splits", [(True, 1), (False, 1), (True, 3)])
def test_step_replays_from_a_cuda_graph(cuda_device, fa2_lib, causal, splits):
    B, H, N, d = 2, 3, 700, 128
    dev = cuda_device
    q, k, v, do = (t.to(dev) for t in make_inputs(B, H, N, d, torch.bfloat16, seed=21))
    q2, k2, v2, do2 = (t.to(dev) for t in make_inputs(B, H, N, d, torch.bfloat16, seed=22))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):  # warm-up outside the capture (per-device set-up)
        _eager(fa2_lib, q, k, v, do, causal, splits)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = _eager(fa2_lib, q, k, v, do, causal, splits)
    for src in ((q, k, v, do), (q2, k2, v2, do2)):
        want = _eager(fa2_lib, *(t.clone() for t in src), causal, splits)
        for dst, s in zip((q, k, v, do), src):
            dst.copy_(s)
        g.replay()
        torch.cuda.synchronize()
        assert fa2_lib.device_status() == 0
        for a, b, name in zip(outs, want, ("o", "lse", "dq", "dk", "dv")):
            assert torch.equal(a, b), name


def test_host_buffer_step_replays_from_a_cuda_graph(cuda_device, fa2_lib):
    """fa2_step_host forks its internal streams from the capturing stream and
    joins them back, so the uploads, kernels and downloads are one graph."""
    B, H, N, d = 1, 6, 512, 64
    dev = cuda_device
    q, k, v, do = (t.pin_memory() for t in make_inputs(B, H, N, d, torch.bfloat16, seed=23))
    lib = fa2_lib.load_library()
    outs = tuple(torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    nbytes = lib.fa2_step_host_workspace_size(B, H, N, d, 2)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d)

    def call(stream):
        o, dq, dk, dv = outs
        code = lib.fa2_step_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, N, d, 1, scale, 1, 2, ws.data_ptr(), nbytes,
                                 stream.cuda_stream)
        assert code == 0

    with torch.cuda.device(dev):
        side = torch.cuda.Stream(dev)
        call(side)
        side.synchronize()
        want = tuple(t.clone() for t in outs) + (lse.clone(),)
        for t in outs + (lse,):
            t.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(torch.cuda.current_stream(dev))
        g.replay()
        torch.cuda.synchronize()
    for a, b in zip(outs + (lse,), want):
        assert torch.equal(a, b)
