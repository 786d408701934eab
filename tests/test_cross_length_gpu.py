"""Different query and key lengths (fa2_fwd_qk / fa2_bwd_qk): the CUDA path
through the C ABI against the fp64 oracle. The causal mask is top-left: query
i sees keys 0 .. min(i, N_k - 1)."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, max_abs, oracle_bwd, oracle_fwd, rel_fro, to64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, Nq, Nk, d, dtype, causal)
    (1, 2, 128, 300, 128, torch.bfloat16, True),
    (1, 1, 300, 128, 64, torch.bfloat16, True),
    (2, 1, 1, 257, 128, torch.float16, False),
    (1, 2, 257, 1, 64, torch.bfloat16, True),
    (1, 1, 640, 200, 128, torch.bfloat16, True),
    (1, 1, 200, 640, 128, torch.bfloat16, True),
    (1, 3, 1000, 333, 64, torch.float16, False),
    (1, 1, 129, 1000, 128, torch.float16, False),
    # 80 heads x 4 row blocks: the persistent forward runs causal pairs (160 of
    # them on 152 CTAs, the last 8 as halves) with N_k < N_q.
    (4, 20, 1024, 600, 64, torch.bfloat16, True),
]


def _inputs(B, H, Nq, Nk, d, dtype, seed):
    q, _, _, do = make_inputs(B, H, Nq, d, dtype, seed=seed)
    _, k, v, _ = make_inputs(B, H, Nk, d, dtype, seed=seed + 1)
    return q, k, v, do


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal", CASES)
def test_cross_length_forward_and_backward(cuda_device, fa2_lib, B, H, Nq, Nk, d, dtype, causal):
    q, k, v, do = _inputs(B, H, Nq, Nk, d, dtype, seed=Nq * 7 + Nk)
    scale = 1.0 / math.sqrt(d)
    dev = cuda_device
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa2_lib.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
    tol = TOL[dtype]
    assert max_abs(to64(o.cpu()), o_ref) <= tol["o"]
    assert max_abs(to64(lse.cpu()), lse_ref) <= tol["lse"]
    dq_r, dk_r, dv_r = oracle_bwd(q, k, v, do, causal, scale)
    for got, ref, name in ((dq, dq_r, "dq"), (dk, dk_r, "dk"), (dv, dv_r, "dv")):
        g = to64(got.cpu())
        assert np.all(np.isfinite(g)), name
        assert rel_fro(g, ref) <= tol["grad"], name
    if causal and Nk > Nq:
        # Keys no query sees: zero gradients.
        assert np.all(to64(dk.cpu())[:, :, Nq:] == 0.0)
        assert np.all(to64(dv.cpu())[:, :, Nq:] == 0.0)


def test_cross_length_equal_lengths_match_self_attention(cuda_device, fa2_lib):
    """fa2_fwd_qk with N_q = N_k is the plain forward, bit for bit."""
    B, H, N, d = 1, 2, 300, 128
    q, k, v, _ = make_inputs(B, H, N, d, torch.bfloat16, seed=9)
    qd, kd, vd = (t.to(cuda_device) for t in (q, k, v))
    lib = fa2_lib.load_library()
    o1, lse1 = fa2_lib.forward(qd, kd, vd, causal=True, num_splits=1)
    o2 = torch.empty_like(qd)
    lse2 = torch.empty_like(lse1)
    code = lib.fa2_fwd_qk(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(),
                          lse2.data_ptr(), B, H, N, N, d, 1, 1.0 / math.sqrt(d), 1, None)
    assert code == 0
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
