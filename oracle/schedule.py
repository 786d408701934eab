"""Integer work mapping of FlashAttention-2, as the pages describe it.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Forward ("FlashAttention学习笔记(2)" and "大猿搬砖简记", sections on the V2
thread-block layout): one worker per (Q row block, batch, head); the number of
row blocks is ceil(seqlen_q / kBlockM) and the grid is (num_m_block, batch,
heads), with the row-block index varying fastest so that the workers that read
the same K/V run close together (L2 reuse).

Backward ("Foward和backward中的thread block划分" section of the first page, and
the matching section of "大猿搬砖简记"): one worker per K/V column block, since
dK and dV accumulate along the query direction and only dQ accumulates along
the key direction.

KV split ("大猿搬砖简记", thread-block section; the num_splits_heuristic_fwd
paragraph): when the (row block, batch, head) workers cannot fill the SMs, the
K/V range of each worker may be cut into num_splits parts whose partial results
are merged afterwards. The split count is chosen by computing the SM
utilisation of each candidate, taking the best, and picking the smallest
candidate whose utilisation is at least 0.95 of it. Candidates run from 1 to
min(max_splits, num_sms, number of K/V tiles): more parts than K/V tiles leave
parts empty, more than the SM count add no wave. The page does not define the
utilisation. Two readings are kept here:
  * split_utilisation: the filled fraction of the waves, w / ceil(w) with
    w = workers * s / num_sms, which counts CTAs and treats them as equal;
  * split_utilisation_makespan (the library's rule): the fraction of the SMs'
    time spent on K/V tiles, useful tiles / (num_sms * makespan), when the
    launch's CTAs start in launch order, each on the SM that frees first, and
    a CTA takes its tiles plus a fixed cost, plus a further cost if its row
    block is split (its partial write and its share of the merge). Under the
    causal mask the workers are unequal and the waves reading cannot see the
    tail; this one can, and with equal workers and no costs it reduces to the
    waves reading.

Causal tile skipping ("flash-attention123和ring-attention", 优化3): key/query
tile pairs that the causal mask hides completely are dropped, not computed.
Reading (the first two pages say such tiles are still loaded; the third says
they are skipped): they are neither loaded nor computed. A tile pair is fully
masked iff every key index in it exceeds every query index in it.
"""

from __future__ import annotations

import heapq

__all__ = [
    "ceil_div",
    "fwd_grid",
    "fwd_work_order",
    "fwd_kv_tile_range",
    "bwd_grid",
    "bwd_q_tile_range",
    "split_utilisation",
    "num_splits_heuristic",
    "split_num_parts",
    "split_part_range",
    "split_launch",
    "greedy_makespan",
    "split_utilisation_makespan",
    "num_splits_makespan",
    "SPLIT_CTA_COST",
    "SPLIT_PART_COST",
]


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def fwd_grid(B: int, H: int, N: int, block_m: int):
    """(num_m_block, B, H): the forward grid of the pages."""
    return (ceil_div(N, block_m), B, H)


def fwd_work_order(B: int, H: int, N: int, block_m: int):
    """Linear order of forward workers: list of (m_block, b, h), m fastest."""
    nm, _, _ = fwd_grid(B, H, N, block_m)
    return [(m, b, h) for h in range(H) for b in range(B) for m in range(nm)]


def _tile_fully_masked(q0, q1, k0, k1):
    """Query rows [q0, q1) and key columns [k0, k1): fully hidden by the causal
    mask iff the smallest key index exceeds the largest query index."""
    return k0 > q1 - 1


def fwd_kv_tile_range(m_block: int, N: int, block_m: int, block_n: int, causal: bool,
                      n_k: int | None = None):
    """Half-open range [j_begin, j_end) of K/V tiles a forward worker visits.
    N is the query length and n_k the key length (default N).

    Derived by brute force over all tiles, dropping fully masked ones, so that
    it is independent of any closed-form bound.
    """
    n_k = N if n_k is None else n_k
    q0, q1 = m_block * block_m, min(N, (m_block + 1) * block_m)
    visited = []
    for j in range(ceil_div(n_k, block_n)):
        k0, k1 = j * block_n, min(n_k, (j + 1) * block_n)
        if causal and _tile_fully_masked(q0, q1, k0, k1):
            continue
        visited.append(j)
    if not visited:
        return (0, 0)
    assert visited == list(range(visited[0], visited[-1] + 1))
    return (visited[0], visited[-1] + 1)


def bwd_grid(B: int, H: int, N: int, block_n: int):
    """(num_n_block, B, H): one backward worker per K/V column block."""
    return (ceil_div(N, block_n), B, H)


def bwd_q_tile_range(n_block: int, N: int, block_m: int, block_n: int, causal: bool,
                     n_k: int | None = None):
    """Half-open range [i_begin, i_end) of Q tiles a backward column worker visits
    (brute force over all tiles, dropping fully masked ones). N is the query
    length and n_k the key length (default N); a worker whose keys no query
    sees gets the empty range."""
    n_k = N if n_k is None else n_k
    k0, k1 = n_block * block_n, min(n_k, (n_block + 1) * block_n)
    visited = []
    for i in range(ceil_div(N, block_m)):
        q0, q1 = i * block_m, min(N, (i + 1) * block_m)
        if causal and _tile_fully_masked(q0, q1, k0, k1):
            continue
        visited.append(i)
    if not visited:
        return (0, 0)
    assert visited == list(range(visited[0], visited[-1] + 1))
    return (visited[0], visited[-1] + 1)


def split_utilisation(workers: int, num_sms: int, s: int) -> float:
    """Filled fraction of the waves when `workers` workers are each cut into
    `s` parts on `num_sms` SMs (the reading of the page's "SM utilisation")."""
    waves = workers * s / num_sms
    return waves / ceil_div(workers * s, num_sms)


def num_splits_heuristic(workers: int, num_sms: int, num_n_blocks: int, max_splits: int) -> int:
    """The page's rule: best utilisation over the candidates, then the smallest
    candidate whose utilisation is >= 0.95 of the best."""
    top = max(1, min(max_splits, num_sms, num_n_blocks))
    eff = [split_utilisation(workers, num_sms, s) for s in range(1, top + 1)]
    best = max(eff)
    for s in range(1, top + 1):
        if eff[s - 1] >= 0.95 * best:
            return s
    return 1


def split_num_parts(n: int, num_splits: int, n_max: int) -> int:
    """Part count of a worker with n K/V tiles when the longest worker (n_max
    tiles) is cut into num_splits parts: proportionally fewer for a shorter
    range, min(n, ceil(n * num_splits / n_max)), never an empty part. Reading
    of the page's split paragraph, which gives the part count of a worker but
    not how unequal (causal) workers share it."""
    if n <= 0:
        return 0
    if num_splits <= 1:
        return 1
    return min(n, ceil_div(n * num_splits, n_max))


def split_part_range(j_begin: int, j_end: int, parts: int, part: int):
    """Part `part` of `parts` contiguous, balanced parts of the tile range
    [j_begin, j_end): lengths floor or ceil of len / parts, in order."""
    n = j_end - j_begin
    return (j_begin + part * n // parts, j_begin + (part + 1) * n // parts)


# Costs of the makespan reading, in K/V tiles of work (one tile = one 128-key
# step of a 256-row forward worker). Fitted to forward times measured on
# GB300 over split counts 1..16 of six long-sequence shapes (d = 128, causal
# and not): a CTA's fixed start and finish costs about one tile, and a part of
# a split row block about six more (its fp32 partial write and merge share).
SPLIT_CTA_COST = 1
SPLIT_PART_COST = 6


def split_launch(block_tiles, BH: int, s: int):
    """The CTAs of a forward launch with split count s, in launch order: the
    row blocks in the given order (longest first), each block's parts in
    order, each part repeated for the BH heads (heads fastest). Returns a list
    of (tiles, split) pairs, split being True when the block has more than one
    part (s = 1: one part per block)."""
    n_max = max(block_tiles)
    out = []
    for n in block_tiles:
        p = split_num_parts(n, s, n_max)
        for part in range(p):
            lo, hi = split_part_range(0, n, p, part)
            out.extend([(hi - lo, p > 1)] * BH)
    return out


def greedy_makespan(costs, num_sms: int):
    """Time at which the last SM finishes when every CTA, in launch order,
    starts on the SM that becomes free first (list scheduling; the SMs' free
    times kept in a heap)."""
    free = [0] * num_sms
    for c in costs:
        heapq.heappush(free, heapq.heappop(free) + c)
    return max(free)


def split_utilisation_makespan(block_tiles, BH: int, num_sms: int, s: int,
                               cta_cost=SPLIT_CTA_COST, part_cost=SPLIT_PART_COST) -> float:
    """Useful tiles / (num_sms * makespan) of the split-s launch."""
    ctas = split_launch(block_tiles, BH, s)
    useful = sum(t for t, _ in ctas)
    span = greedy_makespan([t + cta_cost + (part_cost if sp else 0) for t, sp in ctas], num_sms)
    return useful / (num_sms * span)


def num_splits_makespan(block_tiles, BH: int, num_sms: int, max_splits: int,
                        cta_cost=SPLIT_CTA_COST, part_cost=SPLIT_PART_COST) -> int:
    """The page's selection rule over the makespan utilisation: the best over
    the candidates 1 .. min(max_splits, num_sms, K/V tiles of the longest
    block), then the smallest candidate within 0.95 of it."""
    top = max(1, min(max_splits, num_sms, max(block_tiles)))
    eff = [split_utilisation_makespan(block_tiles, BH, num_sms, c, cta_cost, part_cost)
           for c in range(1, top + 1)]
    best = max(eff)
    for c in range(1, top + 1):
        if eff[c - 1] >= 0.95 * best:
            return c
    return 1
