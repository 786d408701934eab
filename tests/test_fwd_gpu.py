"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from tests.parity import TOL, max_abs, oracle_fwd, seeded_heads, to64

pytestmark = pytest.mark.gpu


def _run(fa2, dev, q, k, v, causal, scale):
    o, lse = fa2.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2.device_status() == 0
    return o.cpu(), lse.cpu()


# Small shapes spanning several tiles and ragged tails.
EDGE = [
    # (B, H, N, d, dtype, causal)
    (1, 1, 1, 64, torch.bfloat16, False),
    (1, 1, 1, 128, torch.float16, True),
    (1, 3, 2, 64, torch.bfloat16, True),
    (1, 1, 127, 128, torch.bfloat16, False),
    (1, 1, 129, 64, torch.float16, True),
    (2, 1, 255, 128, torch.bfloat16, True),
    (1, 3, 256, 64, torch.bfloat16, False),
    (1, 2, 257, 128, torch.float16, False),
    (1, 1, 384, 128, torch.bfloat16, True),
    (1, 2, 1000, 64, torch.bfloat16, True),
    (1, 1, 1000, 128, torch.float16, False),
    (2, 2, 640, 128, torch.bfloat16, True),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", EDGE)
def test_fwd_edge_shapes(cuda_device, fa2_lib, B, H, N, d, dtype, causal):
    q, k, v, _ = make_inputs(B, H, N, d, dtype, seed=N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa2_lib, cuda_device, q, k, v, causal, scale)
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
    tol = TOL[dtype]
    assert np.all(np.isfinite(to64(o)))
    assert max_abs(to64(o), o_ref) <= tol["o"]
    assert max_abs(to64(lse), lse_ref) <= tol["lse"]


@pytest.mark.parametrize("name", ["fp16_b1h1_n128_d64", "causal_bf16_b2h4_n1024_d64"])
def test_fwd_small_workloads_full(cuda_device, fa2_lib, name):
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w)
    o, lse = _run(fa2_lib, cuda_device, q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle_fwd(q, k, v, w.causal, w.scale)
    tol = TOL[w.torch_dtype]
    assert max_abs(to64(o), o_ref) <= tol["o"]
    assert max_abs(to64(lse), lse_ref) <= tol["lse"]


@pytest.mark.parametrize("name,num_splits", [("bf16_b8h16_n2048_d128", 1),
                                             ("causal_bf16_b8h16_n2048_d128", 1),
                                             ("causal_bf16_b1h2_n16384_d128", 1),
                                             ("causal_bf16_b1h2_n16384_d128", "auto")])
def test_fwd_full_size_every_head(cuda_device, fa2_lib, name, num_splits):
    """Full-size launch; every head goes through the oracle (the two-head long
    sequence both unsplit and with the library's own K/V split choice)."""
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w)
    o, lse = fa2_lib.forward(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                             causal=w.causal, scale=w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    o_ref, lse_ref = oracle_fwd(q, k, v, w.causal, w.scale)
    tol = TOL[w.torch_dtype]
    o64, l64 = to64(o.cpu()), to64(lse.cpu())
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(l64))
    for b in range(w.B):
        for h in range(w.H):
            assert max_abs(o64[b, h], o_ref[b, h]) <= tol["o"], (b, h)
            assert max_abs(l64[b, h], lse_ref[b, h]) <= tol["lse"], (b, h)


def test_fwd_headline_eight_seeded_heads(cuda_device, fa2_lib):
    """The 128-head long-sequence workload at full size; eight whole heads
    drawn by a seeded RNG go through the oracle, and every head's outputs are
    finite."""
    w = WORKLOADS["causal_bf16_b4h32_n8192_d128_qstd3"]
    q, k, v, _ = workload_inputs(w)
    o, lse = _run(fa2_lib, cuda_device, q, k, v, w.causal, w.scale)
    heads = seeded_heads(w, 8, 1)
    refs = oracle_fwd(q, k, v, w.causal, w.scale, heads=heads)
    tol = TOL[w.torch_dtype]
    o64, l64 = to64(o), to64(lse)
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(l64))
    for (b, h), (o_ref, lse_ref) in zip(heads, refs):
        assert max_abs(o64[b, h], o_ref[0, 0]) <= tol["o"], (b, h)
        assert max_abs(l64[b, h], lse_ref[0, 0]) <= tol["lse"], (b, h)


@pytest.mark.parametrize("B,H,N", [(1, 2, 1000), (4, 15, 1380)])
def test_fwd_causal_tiles_skipped(cuda_device, fa2_lib, B, H, N):
    """Each row block loads exactly the K/V tiles up to the diagonal, none past
    it. The second shape has 360 row blocks, so the persistent grid runs several
    per CTA (causal: pairs, and a last round of halves)."""
    d = 128
    q, k, v, _ = make_inputs(B, H, N, d, torch.bfloat16, seed=3)
    dev = cuda_device
    for causal in (False, True):
        _, _, counts = fa2_lib.forward_instrumented(q.to(dev), k.to(dev), v.to(dev), causal=causal)
        counts = counts.cpu().numpy()
        (gx, gy, gz), _ = fa2_lib.fwd_grid(B, H, N)
        for blk in range(gx * gy * gz):
            bx = blk % gx
            _, _, want = fa2_lib.fwd_block_work(bx, N, causal)
            assert counts[blk] == want, (causal, blk)


def test_fwd_device_timeout_path(cuda_device, fa2_lib):
    """An armed host-side fault makes one bounded wait run out; the kernel
    reports FA2_ERR_DEVICE_TIMEOUT and returns, and the context stays usable."""
    q, k, v, _ = make_inputs(1, 1, 256, 64, torch.bfloat16, seed=5)
    dev = cuda_device
    assert fa2_lib.load_library().fa2_debug_arm_fault(1, 20) == 0
    fa2_lib.forward(q.to(dev), k.to(dev), v.to(dev))
    assert fa2_lib.device_status() == 6
    # The next call is normal again.
    o, lse = _run(fa2_lib, dev, q, k, v, False, 0.125)
    o_ref, _ = oracle_fwd(q, k, v, False, 0.125)
    assert max_abs(to64(o), o_ref) <= 2e-2
