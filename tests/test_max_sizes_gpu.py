"""Maximum sizes: a million-token sequence (the longest causal worker visits
8192 K/V tiles) and the largest batch the grid takes. Outputs the oracle can
compute one by one are checked against the definition in fp64; the rest by
properties that hold at any size."""

import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, oracle_fwd, rel_fro, to64

pytestmark = pytest.mark.gpu


def _rows_reference(q, k, v, rows, causal, scale):
    """O and L of single query rows straight from the definition (fp64):
    L_i = logsumexp_j(scale q_i.k_j), O_i = sum_j exp(scale q_i.k_j - L_i) v_j."""
    k64, v64 = k.double().numpy(), v.double().numpy()
    out, lse = [], []
    for i in rows:
        s = (k64[: i + 1] if causal else k64) @ q[i].double().numpy() * scale
        m = s.max()
        w = np.exp(s - m)
        tot = w.sum()
        out.append((w / tot) @ (v64[: i + 1] if causal else v64))
        lse.append(m + math.log(tot))
    return np.stack(out), np.array(lse)


def test_million_token_causal_head(cuda_device, fa2_lib):
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
    rows = sorted({0, 1, 127, 128, 4095, 65537, N // 2, N - 129, N - 2, N - 1} |
                  set(np.random.default_rng(2).integers(0, N, 6).tolist()))
    o_ref, l_ref = _rows_reference(q[0, 0], k[0, 0], v[0, 0], rows, True, scale)
    o_got = to64(o[0, 0, rows].cpu())
    l_got = to64(lse[0, 0, rows].cpu())
    assert np.max(np.abs(o_got - o_ref)) <= TOL[dt]["o"]
    assert np.max(np.abs(l_got - l_ref)) <= TOL[dt]["lse"]
    # Backward: rows of P sum to 1, so sum_j dV_j = sum_i dO_i; rows of dS sum
    # to 0, so sum_j dK_j = 0; causal row 0 sees only key 0, so dQ_0 = 0.
    g = {n: to64(t[0, 0].cpu()) for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
    for n, t in g.items():
        assert np.all(np.isfinite(t)), n
    sum_do = to64(do[0, 0]).sum(0)
    assert np.max(np.abs(g["dv"].sum(0) - sum_do)) / np.max(np.abs(sum_do)) <= 2e-2
    assert np.max(np.abs(g["dk"].sum(0))) <= 2e-2 * np.max(np.abs(g["dk"])) * math.sqrt(N)
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
