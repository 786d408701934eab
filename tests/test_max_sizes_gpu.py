"""Maximum sizes: a million-token sequence (the longest causal worker visits
8192 K/V tiles) and the largest batch the grid takes. Outputs the oracle can
compute one by one are checked against it in fp64; the rest by properties
that hold at any size."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
import oracle
from tests.parity import TOL, oracle_fwd, rel_fro, to64

pytestmark = pytest.mark.gpu


def _row_problem(t, i):
    """Query row i of a causal head as a one-row, non-causal problem over the
    key prefix 0..i: under the top-left causal mask row i sees exactly those
    keys, so the oracle's result for this problem is row i of the full one."""
    return t[i:i + 1][None, None]


def _prefix(t, i):
    """Rows 0..i of a [N, d] array as a one-head [1, 1, i+1, d] array."""
    return t[: i + 1][None, None]


def test_million_token_causal_head(cuda_device, fa2_lib):
    """N = 2^20 causal, d = 128. Sampled query rows (O, L, dQ) and the
    gradients of the last keys (dK, dV) are checked against the oracle, each
    computed from the rows that determine it; dV's column sums by the
    row-stochastic property of P."""
    N, d = 1 << 20, 128
    dt = torch.bfloat16
    q, k, v, do = make_inputs(1, 1, N, d, dt, seed=31)
    dev = cuda_device
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa2_lib.forward(qd, kd, vd, causal=True, scale=scale)
    dq, dk, dv = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    tol = TOL[dt]
    q64, k64, v64, do64 = (to64(t[0, 0]) for t in (q, k, v, do))
    # Query rows: O_i, L_i and dQ_i depend only on row i and the keys 0..i.
    rows = sorted({0, 1, 127, 128, 4095, 65537, N // 2, N - 129} |
                  set(np.random.default_rng(2).integers(0, N, 4).tolist()))
    o_got, l_got, dq_got = (to64(t[0, 0, rows].cpu()) for t in (o, lse, dq))
    for n, i in enumerate(rows):
        args = (_row_problem(q64, i), _prefix(k64, i), _prefix(v64, i))
        o_ref, l_ref = oracle.forward(*args, causal=False, scale=scale)
        assert np.max(np.abs(o_got[n] - o_ref[0, 0, 0])) <= tol["o"], i
        assert abs(l_got[n] - l_ref[0, 0, 0]) <= tol["lse"], i
        dq_ref, _, _ = oracle.backward(*args, _row_problem(do64, i), causal=False, scale=scale)
        assert rel_fro(dq_got[n], dq_ref[0, 0, 0]) <= tol["grad"], i
    # The last m keys: key j is seen only by the queries j..N-1, so dK_j and
    # dV_j are the sums of the one-row problems of those queries, restricted
    # to key j.
    m = 8
    dk_ref = np.zeros((m, d))
    dv_ref = np.zeros((m, d))
    for i in range(N - m, N):
        _, dki, dvi = oracle.backward(_row_problem(q64, i), _prefix(k64, i), _prefix(v64, i),
                                      _row_problem(do64, i), causal=False, scale=scale)
        # keys N-m .. i exist in row i's problem
        dk_ref[: i + 1 - (N - m)] += dki[0, 0, N - m:]
        dv_ref[: i + 1 - (N - m)] += dvi[0, 0, N - m:]
        del dki, dvi
    assert rel_fro(to64(dk[0, 0, N - m:].cpu()), dk_ref) <= tol["grad"]
    assert rel_fro(to64(dv[0, 0, N - m:].cpu()), dv_ref) <= tol["grad"]
    g = {n: to64(t[0, 0].cpu()) for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
    for n, t in g.items():
        assert np.all(np.isfinite(t)), n
    sum_do = do64.sum(0)
    assert np.max(np.abs(g["dv"].sum(0) - sum_do)) / np.max(np.abs(sum_do)) <= 2e-2
    # Causal row 0 sees only key 0, so P_00 = 1 and dS_00 = 0: dQ_0 = 0.
    assert np.max(np.abs(g["dq"][0])) <= 1e-6


def test_largest_batch_axis(cuda_device, fa2_lib):
    """B = 65535 (the grid's batch axis limit) with one-token heads: O = V,
    L = scale q.k, dV = dO, and dQ = dK = 0 up to rounding (dS = dP - D, where
    the tensor core forms dP = dO.v and the preprocessing pass D = dO.o, in
    different fp32 summation orders) for every head."""
    B, H, N, d = 65535, 1, 1, 64
    dt = torch.bfloat16
    q, k, v, do = make_inputs(B, H, N, d, dt, seed=32)
    dev = cuda_device
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa2_lib.forward(qd, kd, vd, causal=False, scale=scale)
    dq, dk, dv = fa2_lib.backward(qd, kd, vd, o, lse, dod, causal=False, scale=scale)
    torch.cuda.synchronize()
    assert fa2_lib.device_status() == 0
    assert torch.equal(o.cpu(), v)
    want_l = (q.double() * k.double()).sum(-1) * scale
    assert np.max(np.abs(to64(lse.cpu()) - want_l.numpy())) <= 1e-4
    assert dq.abs().max().item() <= 1e-4 and dk.abs().max().item() <= 1e-4
    assert torch.equal(dv.cpu(), do)
    # and a few whole heads against the oracle
    o_ref, l_ref = oracle_fwd(q[:4], k[:4], v[:4], False, scale)
    assert np.max(np.abs(to64(o[:4].cpu()) - o_ref)) <= TOL[dt]["o"]
