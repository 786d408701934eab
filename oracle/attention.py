"""fp64 reference for exact multi-head attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports or calls this module.

What FlashAttention-2 computes
------------------------------
The pages agree that the tiled algorithm reaches *exactly* the result of
ordinary attention: once every K/V block has been visited, the running O equals
the global softmax(S) V ("大猿搬砖简记", walk-through of the V2 forward;
"flash-attention123和ring-attention", section 1). Rows are
independent because softmax is taken along each row ("FlashAttention学习笔记(2)",
opening paragraphs) and heads are independent ("大猿搬砖简记", thread-block
section, multi-head paragraph). So this oracle is the plain definition, written
per (batch, head), not the tiled loop:

    S = scale * Q K^T                       (the score block of the V2 forward)
    S_ij = -inf for j > i  when causal      (causal mask; key j visible to query i iff j <= i)
    L_i  = m_i + ln(sum_j exp(S_ij - m_i))  (only L = m + log l is kept:
                                             "FlashAttention学习笔记(2)", V2 forward)
    P    = exp(S - L)                       (backward recompute with L in place of m,
                                             "flash-attention123和ring-attention", 优化1)
    O    = P V                              (un-normalised O with a single diag(l)^-1
                                             at the end: 优化2 of the same page)

The backward is the naive chain rule through softmax, given dO:

    dV = P^T dO
    dP = dO V^T
    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)
    dQ = scale * dS K,   dK = scale * dS^T Q

It deliberately does NOT use the shortcut D_i = rowsum(dO o O) that the pages'
backward uses ("大猿搬砖简记", V2 backward, last paragraph), so that the GPU's
use of the shortcut is checked against an independent route.

Readings where the pages are silent (each listed in the design notes):
  * scale multiplies S before the mask; L is the logsumexp of the scaled S, in
    natural-log units;
  * causal alignment is top-left (key j visible to query i iff j <= i), also
    when the key length N_k differs from the query length N_q (the pages keep
    seqlen_q and seqlen_k distinct but say nothing about the mask then):
    query i sees keys 0..min(i, N_k - 1);
  * inputs arrive already rounded to the kernel dtype and are upcast to fp64.

Memory: rows are processed in chunks of at most ``row_chunk`` queries; each
chunk holds complete rows, so this is still the plain definition.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["forward", "backward", "lse_brute_force", "combine_partials"]


def _check(q, k, v):
    if (q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or k.shape[:2] != q.shape[:2]
            or k.shape[3] != q.shape[3]):
        raise ValueError("q must be [B, H, N_q, d] and k, v [B, H, N_k, d]")


def _scores(qc, k, row0, causal, scale):
    """Scaled scores of query rows [row0, row0+len(qc)) against all keys, with the
    causal mask applied as -inf."""
    s = scale * (qc @ k.T)
    if causal:
        rows = np.arange(row0, row0 + qc.shape[0])[:, None]
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def _row_logsumexp(s):
    """L_i = m_i + ln(sum_j exp(s_ij - m_i)) with m_i the row max (max-shifted
    so that no exp overflows)."""
    m = np.max(s, axis=1)
    return m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))


def forward(q, k, v, causal=False, scale=None, row_chunk=1024):
    """Exact attention forward.

    Args:
      q: array [B, H, N_q, d]; k, v: arrays [B, H, N_k, d] (any float type;
         computed in fp64). N_k may differ from N_q.
      causal: apply the top-left causal mask (key j visible to query i iff j <= i).
      scale: score scale; default 1/sqrt(d).
    Returns:
      (o, lse): o [B, H, N_q, d] fp64, lse [B, H, N_q] fp64 natural-log logsumexp
      of the scaled, masked scores.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    _check(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                r1 = min(N, r0 + row_chunk)
                s = _scores(q[b, h, r0:r1], k[b, h], r0, causal, scale)
                L = _row_logsumexp(s)
                p = np.exp(s - L[:, None])
                o[b, h, r0:r1] = p @ v[b, h]
                lse[b, h, r0:r1] = L
    return o, lse


def backward(q, k, v, do, causal=False, scale=None, row_chunk=1024):
    """Naive chain-rule backward of ``forward`` given the output gradient dO.

    Returns (dq, dk, dv): dq like q, dk and dv like k (fp64). A key that no
    query sees (causal, N_k > N_q) gets zero gradients.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    _check(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must have the shape of q")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            kb, vb = k[b, h], v[b, h]
            for r0 in range(0, N, row_chunk):
                r1 = min(N, r0 + row_chunk)
                qc, doc = q[b, h, r0:r1], do[b, h, r0:r1]
                s = _scores(qc, kb, r0, causal, scale)
                p = np.exp(s - _row_logsumexp(s)[:, None])
                dv[b, h] += p.T @ doc
                dp = doc @ vb.T
                ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
                dq[b, h, r0:r1] = scale * (ds @ kb)
                dk[b, h] += scale * (ds.T @ qc)
    return dq, dk, dv


def lse_brute_force(q, k, causal=False, scale=None):
    """Row logsumexp by pure-Python loops (no NumPy reductions): for tiny inputs
    only. L_i = ln(sum over visible j of exp(scale * q_i . k_j)), max-shifted."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, H, N, d = q.shape
    n_k = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                vals = []
                for j in range(n_k):
                    if causal and j > i:
                        continue
                    dot = 0.0
                    for c in range(d):
                        dot += float(q[b, h, i, c]) * float(k[b, h, j, c])
                    vals.append(scale * dot)
                m = max(vals)
                out[b, h, i] = m + math.log(sum(math.exp(x - m) for x in vals))
    return out


def combine_partials(o_parts, lse_parts):
    """Merge attention results computed over disjoint key subsets.

    Each part s holds O_s = softmax over its own keys applied to its V rows and
    L_s = logsumexp of its scores. The merged result rescales every part by
    exp(L_s - L) with L = logsumexp_s L_s -- the same running-max rescale the
    pages describe for visiting K/V blocks one after another
    ("flash-attention123和ring-attention", section 1; "大猿搬砖简记", V2 forward),
    applied here to whole parts (the KV-split the thread-block section mentions).
    A part with L_s = -inf (no visible key) contributes nothing.

    Args: o_parts [S, ..., d], lse_parts [S, ...] (fp64-convertible).
    Returns: (o, lse) merged over the leading axis.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe[None])
    tot = np.sum(w, axis=0)
    lse = m_safe + np.log(tot)
    contrib = np.where(w[..., None] > 0.0, w[..., None] * np.nan_to_num(o_parts), 0.0)
    o = np.sum(contrib, axis=0) / tot[..., None]
    return o, lse
