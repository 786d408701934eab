"""K/V-split forward ("大猿搬砖简记", thread-block section): each worker's K/V
range cut into parts run by separate CTAs and merged by the online-softmax rule.
The CUDA path (fa2_fwd_split through the C ABI) against the fp64 oracle, which
computes the unsplit definition."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from tests.parity import TOL, max_abs, oracle_fwd, to64

pytestmark = pytest.mark.gpu


def _run(fa2, dev, q, k, v, causal, scale, num_splits):
    o, lse = fa2.forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                         num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa2.device_status() == 0
    return o.cpu(), lse.cpu()


# Shapes with 1 to 8 K/V tiles of 128 keys and ragged tails; split counts
# below, at and above the number of tiles (parts left empty).
CASES = [
    # (B, H, N, d, dtype, causal, num_splits)
    (1, 1, 1, 64, torch.bfloat16, False, 2),
    (1, 2, 130, 128, torch.float16, True, 2),
    (1, 1, 300, 128, torch.bfloat16, True, 7),
    (2, 1, 511, 64, torch.bfloat16, False, 3),
    (1, 3, 640, 128, torch.bfloat16, True, 5),
    (1, 1, 1000, 128, torch.float16, False, 8),
    (1, 2, 1024, 64, torch.bfloat16, True, 128),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,S", CASES)
def test_fwd_split_matches_oracle(cuda_device, fa2_lib, B, H, N, d, dtype, causal, S):
    q, k, v, _ = make_inputs(B, H, N, d, dtype, seed=3 * N + d + S)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa2_lib, cuda_device, q, k, v, causal, scale, S)
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
    tol = TOL[dtype]
    assert np.all(np.isfinite(to64(o))) and np.all(np.isfinite(to64(lse)))
    assert max_abs(to64(o), o_ref) <= tol["o"]
    assert max_abs(to64(lse), lse_ref) <= tol["lse"]


@pytest.mark.parametrize("split", ["auto", 7])
def test_fwd_split_on_the_two_head_long_sequence(cuda_device, fa2_lib, split):
    """B=1 H=2 N=16384 causal launches only 128 forward CTAs; the library's rule
    splits it (4 parts on 152 SMs, the measured fastest launch). Full-size
    launch, one whole head through the oracle, and agreement with the unsplit
    kernel on every head."""
    w = WORKLOADS["causal_bf16_b1h2_n16384_d128"]
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    S = fa2_lib.num_splits(w.B, w.H, w.N, w.d, w.causal, sms)
    assert S > 1
    q, k, v, _ = workload_inputs(w)
    o, lse = _run(fa2_lib, cuda_device, q, k, v, w.causal, w.scale, split)
    o1, lse1 = _run(fa2_lib, cuda_device, q, k, v, w.causal, w.scale, 1)
    tol = TOL[w.torch_dtype]
    assert max_abs(to64(o), to64(o1)) <= tol["o"]
    assert max_abs(to64(lse), to64(lse1)) <= tol["lse"]
    h = int(np.random.default_rng(5).integers(w.H))
    (o_ref, lse_ref), = oracle_fwd(q, k, v, w.causal, w.scale, heads=[(0, h)])
    assert max_abs(to64(o[:, h:h + 1]), o_ref) <= tol["o"]
    assert max_abs(to64(lse[:, h:h + 1]), lse_ref) <= tol["lse"]


def test_fwd_split_rejects_bad_split_counts(cuda_device, fa2_lib):
    lib = fa2_lib.load_library()
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=cuda_device)
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 128, dtype=torch.float32, device=cuda_device)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_device)
    for S in (0, 129):
        assert lib.fa2_fwd_split(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 1, 1, 128, 64, 0, 0.125, 1, S, ws.data_ptr(),
                                 ws.numel(), None) == 1
    # Workspace too small for 4 parts.
    assert lib.fa2_fwd_split(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), 1, 1, 128, 64, 0, 0.125, 1, 4, ws.data_ptr(), 16,
                             None) == 7


def test_fwd_split_reuses_a_dirty_workspace(cuda_device, fa2_lib):
    """The workspace's contents are ignored on entry: a buffer full of garbage,
    then the same buffer again (arrival counters left at their final values),
    give the same bits as a fresh run."""
    B, H, N, d, S = 1, 2, 1000, 128, 5
    q, k, v, _ = make_inputs(B, H, N, d, torch.bfloat16, seed=77)
    qd, kd, vd = (t.to(cuda_device) for t in (q, k, v))
    lib = fa2_lib.load_library()
    nbytes = lib.fa2_fwd_split_workspace_size(B, H, N, d, S)
    ws = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device=cuda_device)
    outs = []
    for _ in range(2):
        o = torch.empty_like(qd)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
        code = lib.fa2_fwd_split(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, 1, 1.0 / math.sqrt(d), 1, S,
                                 ws.data_ptr(), nbytes, None)
        assert code == 0
        torch.cuda.synchronize()
        outs.append((o.cpu(), lse.cpu()))
    assert fa2_lib.device_status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    o_ref, lse_ref = oracle_fwd(q, k, v, True, 1.0 / math.sqrt(d))
    assert max_abs(to64(outs[0][0]), o_ref) <= TOL[torch.bfloat16]["o"]
    assert max_abs(to64(outs[0][1]), lse_ref) <= TOL[torch.bfloat16]["lse"]
