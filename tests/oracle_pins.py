"""Pins of the fp64 oracle: checks against what the mathematics fixes, each a
function of the oracle module so that the same checks can be run on a copy of
the oracle with a mistake planted in it (tests/test_oracle_mutations.py).

Every pin raises AssertionError when it fails. None of them re-types the
oracle's own formula: they use closed forms, brute force in pure Python,
finite differences, invariants and a library routine
(torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU).
"""

from __future__ import annotations

import math

import numpy as np


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err} > {tol}"


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
def pin_zero_query(ora):
    """Q = 0 makes every visible score equal: P is uniform over the visible keys.
    Non-causal: O_i = column mean of V, L_i = ln N. Causal: O_i = mean of V_0..V_i,
    L_i = ln(i+1). dK = 0 exactly (dK = scale dS^T Q). dV_j = sum_i P_ij dO_i."""
    B, H, N, d = 1, 2, 7, 3
    r = _rng(1)
    k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(3))
    q = np.zeros((B, H, N, d))
    for causal in (False, True):
        for chunk in (1024, 2):
            o, lse = ora.forward(q, k, v, causal=causal, scale=0.7, row_chunk=chunk)
            dq, dk, dv = ora.backward(q, k, v, do, causal=causal, scale=0.7, row_chunk=chunk)
            for b in range(B):
                for h in range(H):
                    for i in range(N):
                        n_vis = (i + 1) if causal else N
                        _close(o[b, h, i], v[b, h, :n_vis].mean(axis=0), 1e-12, "O(Q=0)")
                        _close(lse[b, h, i], math.log(n_vis), 1e-12, "L(Q=0)")
                    for j in range(N):
                        want = np.zeros(d)
                        for i in range(N):
                            if causal and j > i:
                                continue
                            want += do[b, h, i] / ((i + 1) if causal else N)
                        _close(dv[b, h, j], want, 1e-12, "dV(Q=0)")
            assert np.all(dk == 0.0), "dK(Q=0) must be exactly zero"


def pin_causal_row_zero(ora):
    """Under the causal mask query 0 sees only key 0: O_0 = V_0,
    L_0 = scale * q_0 . k_0, and dQ_0 = 0 (a one-key softmax has zero gradient)."""
    B, H, N, d = 2, 1, 9, 4
    r = _rng(2)
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.37
    o, lse = ora.forward(q, k, v, causal=True, scale=scale)
    dq, _, _ = ora.backward(q, k, v, do, causal=True, scale=scale)
    for b in range(B):
        _close(o[b, 0, 0], v[b, 0, 0], 1e-12, "O_0")
        _close(lse[b, 0, 0], scale * float(np.dot(q[b, 0, 0], k[b, 0, 0])), 1e-12, "L_0")
        _close(dq[b, 0, 0], np.zeros(d), 1e-12, "dQ_0")


def pin_single_token(ora):
    """N = 1: O = V, L = scale q.k, dQ = dK = 0, dV = dO."""
    r = _rng(3)
    q, k, v, do = (r.standard_normal((2, 3, 1, 5)) for _ in range(4))
    for causal in (False, True):
        o, lse = ora.forward(q, k, v, causal=causal, scale=0.5)
        dq, dk, dv = ora.backward(q, k, v, do, causal=causal, scale=0.5)
        _close(o, v, 1e-12, "O(N=1)")
        _close(lse, 0.5 * np.sum(q * k, axis=-1), 1e-12, "L(N=1)")
        _close(dq, 0 * q, 1e-12, "dQ(N=1)")
        _close(dk, 0 * k, 1e-12, "dK(N=1)")
        _close(dv, do, 1e-12, "dV(N=1)")


def pin_single_query_cross_length(ora):
    """N_q = 1 against N_k > 1 keys. Causal (top-left): the query sees key 0
    only, so O = V_0, L = scale q.k_0, dV_0 = dO and every other dK, dV row is
    0. Not causal: L = ln sum_j exp(scale q.k_j), by hand."""
    r = _rng(11)
    q, do = (r.standard_normal((2, 2, 1, 4)) for _ in range(2))
    k, v = (r.standard_normal((2, 2, 6, 4)) for _ in range(2))
    o, lse = ora.forward(q, k, v, causal=True, scale=0.7)
    dq, dk, dv = ora.backward(q, k, v, do, causal=True, scale=0.7)
    _close(o, v[:, :, :1], 1e-12, "O(causal, N_q=1)")
    _close(lse, 0.7 * np.sum(q[:, :, 0] * k[:, :, 0], axis=-1)[..., None], 1e-12, "L(causal, N_q=1)")
    _close(dv[:, :, :1], do, 1e-12, "dV_0(causal, N_q=1)")
    _close(dv[:, :, 1:], 0 * dv[:, :, 1:], 1e-12, "dV of unseen keys")
    _close(dk, 0 * dk, 1e-12, "dK(causal, N_q=1)")
    _close(dq, 0 * dq, 1e-12, "dQ(causal, N_q=1)")
    _, lse = ora.forward(q, k, v, causal=False, scale=0.7)
    for b in range(2):
        for h in range(2):
            want = math.log(sum(math.exp(0.7 * float(np.dot(q[b, h, 0], k[b, h, j]))) for j in range(6)))
            _close(lse[b, h, 0], want, 1e-12, "L(N_q=1)")


def pin_constant_values(ora):
    """All V rows equal c: O_i = c whatever P is, and the output no longer
    depends on Q or K, so dQ = dK = 0."""
    B, H, N, d = 1, 2, 6, 3
    r = _rng(4)
    q, k, do = (r.standard_normal((B, H, N, d)) for _ in range(3))
    c = r.standard_normal((B, H, 1, d))
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    for causal in (False, True):
        o, _ = ora.forward(q, k, v, causal=causal)
        dq, dk, _ = ora.backward(q, k, v, do, causal=causal)
        _close(o, np.broadcast_to(c, o.shape), 1e-12, "O(V=c)")
        _close(dq, 0 * dq, 1e-12, "dQ(V=c)")
        _close(dk, 0 * dk, 1e-12, "dK(V=c)")


def pin_two_tokens_by_hand(ora):
    """N = 2, d = 1, worked by hand with the logistic function
    sigma(x) = 1/(1+e^-x): row i has weights (sigma(s_i0 - s_i1), sigma(s_i1 - s_i0)),
    O_i = v_0 sigma(s_i0 - s_i1) + v_1 sigma(s_i1 - s_i0),
    L_i = s_i0 + ln(1 + e^(s_i1 - s_i0)). Causal row 0 keeps only key 0."""
    qv, kv, vv = [1.0, 2.0], [0.5, -1.0], [3.0, -2.0]
    scale = 0.8
    q = np.array(qv).reshape(1, 1, 2, 1)
    k = np.array(kv).reshape(1, 1, 2, 1)
    v = np.array(vv).reshape(1, 1, 2, 1)

    def sig(x):
        return 1.0 / (1.0 + math.exp(-x))

    o, lse = ora.forward(q, k, v, causal=False, scale=scale)
    for i in range(2):
        s0, s1 = scale * qv[i] * kv[0], scale * qv[i] * kv[1]
        want_o = vv[0] * sig(s0 - s1) + vv[1] * sig(s1 - s0)
        want_l = s0 + math.log(1.0 + math.exp(s1 - s0))
        _close(o[0, 0, i, 0], want_o, 1e-14, "O two tokens")
        _close(lse[0, 0, i], want_l, 1e-14, "L two tokens")
    o, lse = ora.forward(q, k, v, causal=True, scale=scale)
    _close(o[0, 0, 0, 0], vv[0], 1e-14, "causal O_0")
    _close(lse[0, 0, 0], scale * qv[0] * kv[0], 1e-14, "causal L_0")
    s0, s1 = scale * qv[1] * kv[0], scale * qv[1] * kv[1]
    _close(o[0, 0, 1, 0], vv[0] * sig(s0 - s1) + vv[1] * sig(s1 - s0), 1e-14, "causal O_1")


# ---------------------------------------------------------------------------
# Brute force
# ---------------------------------------------------------------------------
def pin_lse_brute_force(ora):
    """L equals the row logsumexp computed by pure-Python loops, for equal and
    for different query and key lengths."""
    r = _rng(5)
    for (B, H, N, Nk, d) in ((1, 1, 5, 5, 3), (2, 2, 7, 7, 4), (1, 2, 4, 9, 3), (2, 1, 9, 4, 3)):
        q = r.standard_normal((B, H, N, d))
        k, v = (r.standard_normal((B, H, Nk, d)) for _ in range(2))
        for causal in (False, True):
            _, lse = ora.forward(q, k, v, causal=causal, scale=0.45, row_chunk=3)
            _close(lse, ora.lse_brute_force(q, k, causal=causal, scale=0.45), 1e-12, "L brute")


def pin_output_brute_force(ora):
    """O by explicit loops over keys with math.exp (no NumPy reductions)."""
    r = _rng(6)
    B, H, N, d = 1, 2, 6, 3
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    scale = 0.6
    for causal in (False, True):
        o, _ = ora.forward(q, k, v, causal=causal, scale=scale)
        for b in range(B):
            for h in range(H):
                for i in range(N):
                    keys = [j for j in range(N) if not (causal and j > i)]
                    sc = [scale * sum(q[b, h, i, c] * k[b, h, j, c] for c in range(d)) for j in keys]
                    m = max(sc)
                    w = [math.exp(x - m) for x in sc]
                    z = sum(w)
                    for c in range(d):
                        want = sum(wj * v[b, h, j, c] for wj, j in zip(w, keys)) / z
                        assert abs(o[b, h, i, c] - want) <= 1e-12, "O brute force"


# ---------------------------------------------------------------------------
# Finite differences
# ---------------------------------------------------------------------------
def pin_finite_differences(ora):
    """Central differences of f(Q,K,V) = sum(O o dO) match the backward,
    relative error <= 1e-6, on tiny fp64 inputs, both mask modes."""
    r = _rng(7)
    h = 1e-6
    for N in (1, 2, 3, 5):
        for d in (1, 2, 4):
            q, k, v, do = (r.standard_normal((1, 1, N, d)) for _ in range(4))
            for causal in (False, True):
                dq, dk, dv = ora.backward(q, k, v, do, causal=causal, scale=0.9)
                grads = {"q": dq, "k": dk, "v": dv}
                for name in ("q", "k", "v"):
                    base = {"q": q, "k": k, "v": v}
                    fd = np.zeros_like(base[name])
                    for idx in np.ndindex(base[name].shape):
                        args_p = {kk: vv.copy() for kk, vv in base.items()}
                        args_m = {kk: vv.copy() for kk, vv in base.items()}
                        args_p[name][idx] += h
                        args_m[name][idx] -= h
                        op, _ = ora.forward(args_p["q"], args_p["k"], args_p["v"], causal=causal, scale=0.9)
                        om, _ = ora.forward(args_m["q"], args_m["k"], args_m["v"], causal=causal, scale=0.9)
                        fd[idx] = (np.sum(op * do) - np.sum(om * do)) / (2 * h)
                    den = max(1.0, float(np.max(np.abs(fd))))
                    err = float(np.max(np.abs(fd - grads[name]))) / den
                    assert err <= 1e-6, f"FD d{name} N={N} d={d} causal={causal}: {err}"


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
def pin_invariants(ora):
    r = _rng(8)
    B, H, N, d = 2, 2, 11, 5
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.5
    for causal in (False, True):
        o, lse = ora.forward(q, k, v, causal=causal, scale=scale)
        dq, dk, dv = ora.backward(q, k, v, do, causal=causal, scale=scale, row_chunk=4)
        # rows of P sum to 1  =>  sum_j dV_j = sum_i dO_i
        _close(dv.sum(axis=2), do.sum(axis=2), 1e-12, "sum dV")
        # rows of dS sum to 0  =>  sum_j dK_j = 0
        _close(dk.sum(axis=2), 0 * dk.sum(axis=2), 1e-12, "sum dK")
        # shifting every key by u: P, O, dQ unchanged, L_i shifts by scale q_i.u
        u = r.standard_normal(d)
        o2, lse2 = ora.forward(q, k + u, v, causal=causal, scale=scale)
        dq2, _, _ = ora.backward(q, k + u, v, do, causal=causal, scale=scale)
        _close(o2, o, 1e-12, "key shift O")
        _close(lse2 - lse, scale * np.einsum("bhnd,d->bhn", q, u), 1e-12, "key shift L")
        _close(dq2, dq, 1e-12, "key shift dQ")
        # huge scores: finite, and O a convex combination of V rows
        o3, lse3 = ora.forward(100.0 * q, k, v, causal=causal, scale=scale)
        assert np.all(np.isfinite(o3)) and np.all(np.isfinite(lse3))
        vmin = v.min(axis=2, keepdims=True)
        vmax = v.max(axis=2, keepdims=True)
        assert np.all(o3 >= vmin - 1e-12) and np.all(o3 <= vmax + 1e-12)
    # non-causal: permuting the keys (K and V rows together) changes nothing
    perm = r.permutation(N)
    o, lse = ora.forward(q, k, v, causal=False, scale=scale)
    o4, lse4 = ora.forward(q, k[:, :, perm], v[:, :, perm], causal=False, scale=scale)
    _close(o4, o, 1e-12, "key permutation O")
    _close(lse4, lse, 1e-12, "key permutation L")
    # chunking of query rows does not change anything
    for causal in (False, True):
        a = ora.forward(q, k, v, causal=causal, scale=scale, row_chunk=3)
        b = ora.forward(q, k, v, causal=causal, scale=scale, row_chunk=1024)
        _close(a[0], b[0], 1e-13, "chunked O")
        _close(a[1], b[1], 1e-13, "chunked L")


def pin_combine_partials(ora):
    """Attention over disjoint key subsets, merged, equals attention over all keys."""
    r = _rng(9)
    B, H, Nq, N, d = 1, 2, 5, 12, 3
    q = r.standard_normal((B, H, Nq, d))
    k, v = r.standard_normal((B, H, N, d)), r.standard_normal((B, H, N, d))

    def attend(keys):
        # plain attention of the Nq queries over a key subset, written with explicit loops
        o = np.zeros((B, H, Nq, d))
        l = np.zeros((B, H, Nq))
        for b in range(B):
            for h in range(H):
                for i in range(Nq):
                    sc = [0.4 * float(np.dot(q[b, h, i], k[b, h, j])) for j in keys]
                    m = max(sc)
                    w = [math.exp(x - m) for x in sc]
                    z = sum(w)
                    l[b, h, i] = m + math.log(z)
                    o[b, h, i] = sum(wj * v[b, h, j] for wj, j in zip(w, keys)) / z
        return o, l

    parts = [list(range(0, 4)), list(range(4, 9)), list(range(9, 12))]
    po, pl = zip(*(attend(p) for p in parts))
    o_all, l_all = attend(list(range(N)))
    o_m, l_m = ora.combine_partials(np.stack(po), np.stack(pl))
    _close(o_m, o_all, 1e-12, "combine O")
    _close(l_m, l_all, 1e-12, "combine L")
    # an empty part (L = -inf) contributes nothing
    o_e, l_e = ora.combine_partials(np.stack([o_all, np.full_like(o_all, np.nan)]),
                                    np.stack([l_all, np.full_like(l_all, -np.inf)]))
    _close(o_e, o_all, 1e-12, "combine with empty part O")
    _close(l_e, l_all, 1e-12, "combine with empty part L")


# ---------------------------------------------------------------------------
# Library special case
# ---------------------------------------------------------------------------
def pin_sdpa_cross_check(ora):
    """torch's scaled_dot_product_attention in fp64 on the CPU, with autograd,
    as a second witness of the oracle."""
    import torch
    import torch.nn.functional as F

    r = _rng(10)
    B, H, d = 2, 3, 8
    # Equal lengths, and both orders of different query / key lengths (torch's
    # is_causal mask is top-left aligned for a non-square score matrix).
    for N, Nk in ((17, 17), (5, 13), (13, 5)):
        q, do = (r.standard_normal((B, H, N, d)) for _ in range(2))
        k, v = (r.standard_normal((B, H, Nk, d)) for _ in range(2))
        for causal in (False, True):
            tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
            out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.3)
            out.backward(torch.tensor(do, dtype=torch.float64))
            o, _ = ora.forward(q, k, v, causal=causal, scale=0.3)
            dq, dk, dv = ora.backward(q, k, v, do, causal=causal, scale=0.3)
            _close(o, out.detach().numpy(), 1e-12, "SDPA O")
            _close(dq, tq.grad.numpy(), 1e-12, "SDPA dQ")
            _close(dk, tk.grad.numpy(), 1e-12, "SDPA dK")
            _close(dv, tv.grad.numpy(), 1e-12, "SDPA dV")


ALL_PINS = [
    pin_zero_query,
    pin_causal_row_zero,
    pin_single_token,
    pin_single_query_cross_length,
    pin_constant_values,
    pin_two_tokens_by_hand,
    pin_lse_brute_force,
    pin_output_brute_force,
    pin_finite_differences,
    pin_invariants,
    pin_combine_partials,
    pin_sdpa_cross_check,
]
