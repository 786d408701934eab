"""Forward in the FlashAttention-1 loop order ("FlashAttention学习笔记(2)", the
FlashAttention-1 forward algorithm): K/V blocks outer, query blocks inner, the
running O, m, l of each query block kept in HBM. The CUDA path through the C
ABI against the fp64 oracle (the definition), and against fa2_fwd."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, max_abs, oracle_fwd, to64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, N, d, dtype, causal): 1 to 8 tiles of 128, ragged tails
    (1, 1, 1, 64, torch.bfloat16, False),
    (1, 2, 128, 128, torch.float16, True),
    (2, 1, 130, 64, torch.bfloat16, True),
    (1, 1, 300, 128, torch.bfloat16, False),
    (1, 3, 511, 128, torch.bfloat16, True),
    (2, 2, 1000, 64, torch.float16, True),
    (1, 1, 1024, 128, torch.float16, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", CASES)
def test_kv_outer_forward_matches_oracle(cuda_device, fa2_lib, B, H, N, d, dtype, causal):
    q, k, v, _ = make_inputs(B, H, N, d, dtype, seed=5 * N + d)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = (t.to(cuda_device) for t in (q, k, v))
    o, lse = fa2_lib.forward_kv_outer(qd, kd, vd, causal=causal, scale=scale)
    o2, lse2 = fa2_lib.forward(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
    tol = TOL[dtype]
    g, gl = to64(o.cpu()), to64(lse.cpu())
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(gl))
    assert max_abs(g, o_ref) <= tol["o"]
    assert max_abs(gl, lse_ref) <= tol["lse"]
    # Both loop orders compute the same numbers up to rounding.
    assert max_abs(g, to64(o2.cpu())) <= 2 * tol["o"]


def test_kv_outer_rejects_bad_arguments(cuda_device, fa2_lib):
    lib = fa2_lib.load_library()
    B, H, N, d = 1, 1, 256, 64
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=cuda_device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=cuda_device)
    need = lib.fa2_fwd_kv_outer_workspace_size(B, H, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 0,
            0.125, 1)
    assert lib.fa2_fwd_kv_outer(*args, ws.data_ptr(), need - 1, None) != 0   # workspace too small
    assert lib.fa2_fwd_kv_outer(*args, None, need, None) != 0                # no workspace
    assert lib.fa2_fwd_kv_outer(*args, q.data_ptr(), need, None) != 0        # overlaps the inputs
