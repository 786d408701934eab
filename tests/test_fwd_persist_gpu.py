"""The unsplit forward's persistent grid, branch by branch: row blocks dealt
round robin without a mask; causal pairs with a middle block alone (odd
row-block count); the last partial round run as halves, with a ragged last
block; several middle pairs reserved per head, two of them run whole. Each
shape reaches its branch on a 152-SM GB300 (checked through fa2_fwd_schedule).
Rows sampled from every row block of every head go through the oracle, so a
block skipped, run twice or written to the wrong rows fails."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, to64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, N, d, dtype, causal, split pairs expected on 152 SMs)
    (2, 41, 1000, 64, torch.bfloat16, False, None),  # 328 blocks round robin
    (3, 40, 640, 128, torch.bfloat16, True, 0),      # 3 blocks per head: pair + middle alone
    # 6 blocks per head, the last one 100 rows: 180 pairs = 152 + 28; the
    # middle pairs (blocks 2 and 3) of the last 28 heads run as halves.
    (4, 15, 1380, 128, torch.float16, True, 28),
    # 128 blocks per head: 192 pairs = 152 + 40; T = 14 middle pairs of each
    # of the 3 heads reserved (42), 2 run whole, 40 as halves.
    (1, 3, 32768, 64, torch.bfloat16, True, 40),
]


def _split_pairs(fa2, B, H, N, sms):
    """Causal pairs (blocks q and nm-1-q of a head) whose two blocks run on
    different CTAs."""
    _, cta, _ = fa2.fwd_schedule(B, H, N, True, sms)
    nm = fa2.fwd_grid(1, 1, N)[0][0]
    split = 0
    for hb in range(B * H):
        for q in range(nm // 2):
            if cta[hb * nm + q] != cta[hb * nm + nm - 1 - q]:
                split += 1
    return split


def _sample_rows(N):
    rows = set()
    for r0 in range(0, N, 256):
        rows |= {r0, r0 + 127, r0 + 128, r0 + 255}
    return sorted(r for r in rows if r < N)


@pytest.mark.parametrize("B,H,N,d,dtype,causal,split", CASES)
def test_fwd_persistent_schedule_branches(cuda_device, fa2_lib, B, H, N, d, dtype, causal, split):
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    G, _, _ = fa2_lib.fwd_schedule(B, H, N, causal, sms)
    nm = fa2_lib.fwd_grid(1, 1, N)[0][0]
    assert B * H * nm > G  # CTAs run more than one row block
    if causal and sms == 152:
        assert _split_pairs(fa2_lib, B, H, N, sms) == split
    q, k, v, _ = make_inputs(B, H, N, d, dtype, seed=17 * N + H)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa2_lib.forward(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), causal=causal,
                             scale=scale, num_splits=1)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rows = _sample_rows(N)
    if N > 8192:
        rows = [r for r in rows if r % 256 in (0, 255) or r == N - 1]
    o_got, l_got = to64(o[:, :, rows].cpu()), to64(lse[:, :, rows].cpu())
    q64, k64, v64 = to64(q), to64(k), to64(v)
    tol = TOL[dtype]
    for b in range(B):
        for h in range(H):
            if not causal:
                o_ref, l_ref = oracle.forward(q64[b, h][rows][None, None], k64[b, h][None, None],
                                              v64[b, h][None, None], causal=False, scale=scale)
                assert np.max(np.abs(o_got[b, h] - o_ref[0, 0])) <= tol["o"], (b, h)
                assert np.max(np.abs(l_got[b, h] - l_ref[0, 0])) <= tol["lse"], (b, h)
                continue
            for n, i in enumerate(rows):
                # Row i under the top-left causal mask sees exactly keys 0..i.
                o_ref, l_ref = oracle.forward(q64[b, h][i:i + 1][None, None], k64[b, h][: i + 1][None, None],
                                              v64[b, h][: i + 1][None, None], causal=False, scale=scale)
                assert np.max(np.abs(o_got[b, h, n] - o_ref[0, 0, 0])) <= tol["o"], (b, h, i)
                assert abs(l_got[b, h, n] - l_ref[0, 0, 0]) <= tol["lse"], (b, h, i)
