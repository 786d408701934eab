"""Pins of the oracle's work mapping (CPU only)."""

import json
from pathlib import Path

import pytest

from oracle import schedule

GOLDEN = Path(__file__).resolve().parent / "golden" / "grid_example.json"


def test_worked_grid_example_from_the_pages():
    g = json.loads(GOLDEN.read_text())
    block_m = 128
    N = g["num_m_block"] * block_m
    grid = schedule.fwd_grid(g["batch_size"], g["num_heads"], N, block_m)
    assert grid == (g["num_m_block"], g["batch_size"], g["num_heads"])
    order = schedule.fwd_work_order(g["batch_size"], g["num_heads"], N, block_m)
    assert len(order) == g["blocks"]
    # m fastest: the first num_m_block workers are head 0's row blocks 0..3
    assert [w[0] for w in order[: g["num_m_block"]]] == list(range(g["num_m_block"]))
    assert all(w[2] == 0 for w in order[: g["num_m_block"]])


def test_num_m_block_is_ceil():
    for N, bm, want in ((1, 128, 1), (128, 128, 1), (129, 128, 2), (1000, 256, 4), (16384, 256, 64)):
        assert schedule.fwd_grid(1, 1, N, bm)[0] == want


def test_bwd_grid_worked_by_hand():
    """One backward worker per 128-key column block: ceil(N / 128) blocks, so
    N = 1 and N = 128 give one block, N = 129 two, N = 16384 exactly 128 (a
    floor division would give 0, 1, 1 and 128), with (batch, heads) after it."""
    for (B, H, N), want in (((1, 1, 1), (1, 1, 1)), ((2, 3, 128), (1, 2, 3)),
                            ((1, 1, 129), (2, 1, 1)), ((1, 2, 16384), (128, 1, 2)),
                            ((4, 32, 8192), (64, 4, 32)), ((1, 1, 1000), (8, 1, 1))):
        assert schedule.bwd_grid(B, H, N, 128) == want
    # The pages' grid has one block per column of the tile grid: the column
    # ranges of the blocks cover every key exactly once.
    for N in (1, 127, 128, 129, 255, 256, 257, 1000):
        nb = schedule.bwd_grid(1, 1, N, 128)[0]
        keys = [k for n in range(nb) for k in range(n * 128, min(N, (n + 1) * 128))]
        assert keys == list(range(N))
        assert nb * 128 >= N > (nb - 1) * 128


@pytest.mark.parametrize("N,bm,bn", [(1, 128, 128), (127, 64, 128), (300, 128, 128),
                                     (1000, 256, 128), (777, 64, 32)])
def test_tile_ranges_match_element_level_brute_force(N, bm, bn):
    """A tile pair is visited iff some (query, key) element in it is unmasked."""
    for causal in (False, True):
        for m in range(schedule.ceil_div(N, bm)):
            j0, j1 = schedule.fwd_kv_tile_range(m, N, bm, bn, causal)
            for j in range(schedule.ceil_div(N, bn)):
                visible = any((not causal) or kk <= qq
                              for qq in range(m * bm, min(N, (m + 1) * bm))
                              for kk in range(j * bn, min(N, (j + 1) * bn)))
                assert (j0 <= j < j1) == visible, (m, j, causal)
        for n in range(schedule.ceil_div(N, bn)):
            i0, i1 = schedule.bwd_q_tile_range(n, N, bm, bn, causal)
            for i in range(schedule.ceil_div(N, bm)):
                visible = any((not causal) or kk <= qq
                              for qq in range(i * bm, min(N, (i + 1) * bm))
                              for kk in range(n * bn, min(N, (n + 1) * bn)))
                assert (i0 <= i < i1) == visible, (n, i, causal)


def test_causal_skips_about_half_the_tiles():
    N, bm, bn = 4096, 128, 128
    full = sum(schedule.fwd_kv_tile_range(m, N, bm, bn, False)[1] for m in range(N // bm))
    causal = sum(schedule.fwd_kv_tile_range(m, N, bm, bn, True)[1] for m in range(N // bm))
    nb = N // bm
    assert full == nb * nb
    assert causal == nb * (nb + 1) // 2


# ---- KV split ("大猿搬砖简记", thread-block section: num_splits_heuristic_fwd) ----

def test_split_utilisation_closed_forms():
    # One full wave, a partial wave, and a wave and a third.
    assert schedule.split_utilisation(152, 152, 1) == 1.0
    assert schedule.split_utilisation(128, 152, 1) == pytest.approx(128 / 152)
    assert schedule.split_utilisation(100, 152, 2) == pytest.approx(200 / 152 / 2)
    assert schedule.split_utilisation(76, 152, 4) == 1.0


def test_num_splits_worked_by_hand():
    """128 workers (2 heads x 64 row blocks of 256) on 152 SMs, 128 K/V tiles.
    Utilisation of s parts is (16s/19) / ceil(16s/19): 16/19 = 0.842 for
    s = 1..6 (16s/19 = 0.84, 1.68, 2.53, 3.37, 4.21, 5.05), 112/114 = 0.982
    for s = 7, and 1 at s = 19 (16 full waves). The best is 1; the smallest
    s reaching 0.95 of it is 7."""
    assert schedule.num_splits_heuristic(128, 152, 128, 128) == 7


def test_num_splits_is_one_when_the_grid_fills_whole_waves():
    for k in (1, 2, 5):
        assert schedule.num_splits_heuristic(152 * k, 152, 64, 128) == 1


def test_num_splits_capped_by_tiles_and_max():
    # Two K/V tiles: at most two parts, whatever the fill.
    assert schedule.num_splits_heuristic(1, 152, 2, 128) <= 2
    assert schedule.num_splits_heuristic(3, 152, 100, 4) <= 4


def test_num_splits_follows_the_stated_rule():
    """The choice has utilisation >= 0.95 of the best candidate and no smaller
    candidate has (the page's selection rule, checked over a sweep)."""
    for workers in (1, 3, 17, 64, 128, 151, 153, 300):
        for nb in (1, 2, 7, 64, 128):
            s = schedule.num_splits_heuristic(workers, 152, nb, 128)
            top = min(128, 152, nb)
            eff = [schedule.split_utilisation(workers, 152, c) for c in range(1, top + 1)]
            assert eff[s - 1] >= 0.95 * max(eff)
            assert all(eff[c - 1] < 0.95 * max(eff) for c in range(1, s))


def test_greedy_makespan_by_hand():
    # [3, 3, 2, 2, 2] on 2 SMs: 3 | 3, then 2 -> 5 | 3, 2 -> 5 | 5, 2 -> 7 | 5.
    assert schedule.greedy_makespan([3, 3, 2, 2, 2], 2) == 7
    # One long CTA and five short ones: the short ones fill the other SM.
    assert schedule.greedy_makespan([5, 1, 1, 1, 1, 1], 2) == 5
    assert schedule.greedy_makespan([4, 4, 4], 4) == 4
    assert schedule.greedy_makespan([], 3) == 0


def test_split_launch_order():
    """Blocks in the given order, each block's parts in order, heads fastest;
    a block with one part is not marked split."""
    got = schedule.split_launch([4, 2], 2, 2)
    assert got == [(2, True), (2, True), (2, True), (2, True), (2, False), (2, False)]
    assert schedule.split_launch([5], 1, 2) == [(2, True), (3, True)]
    assert schedule.split_launch([3, 1], 1, 1) == [(3, False), (1, False)]


def test_makespan_utilisation_by_hand():
    """Two causal row blocks of 4 and 2 tiles, one head, 4 SMs, no costs:
    s = 1 runs [4, 2] (makespan 4, 6 / 16); s = 2 cuts only the first block,
    [2, 2, 2] (makespan 2, 6 / 8); s = 4 gives [1, 1, 1, 1, 1, 1] (makespan 2,
    6 / 8). With the fixed costs (1 per CTA, 6 more per split part): s = 1
    costs [5, 3] (6 / 20); s = 2 costs [9, 9, 3] (6 / 36); s = 4 costs six
    CTAs of 8 on 4 SMs (makespan 16, 6 / 64)."""
    u = schedule.split_utilisation_makespan
    assert u([4, 2], 1, 4, 1, 0, 0) == 6 / 16
    assert u([4, 2], 1, 4, 2, 0, 0) == 6 / 8
    assert u([4, 2], 1, 4, 4, 0, 0) == 6 / 8
    assert u([4, 2], 1, 4, 1) == 6 / 20
    assert u([4, 2], 1, 4, 2) == 6 / 36
    assert u([4, 2], 1, 4, 4) == 6 / 64
    # Splitting pays when one long block would keep one SM busy alone:
    # 64 tiles on 4 SMs, s = 1, 2, 4 take 65, 39 (2 x 32 + 7) and 23 (4 x 16 + 7).
    assert [u([64], 1, 4, c) for c in (1, 2, 4)] == [64 / 260, 64 / 156, 64 / 92]
    assert schedule.num_splits_makespan([64], 1, 4, 128) == 4
    assert schedule.num_splits_makespan([4, 2], 1, 4, 128) == 1


def test_makespan_reading_reduces_to_waves():
    """Equal workers and no costs: the makespan utilisation is the filled
    fraction of the waves."""
    for workers in (1, 7, 64, 152, 153, 300):
        for sms in (4, 152):
            for s in (1, 2, 3):
                got = schedule.split_utilisation_makespan([6] * workers, 1, sms, s, 0, 0)
                assert got == pytest.approx(schedule.split_utilisation(workers, sms, s)), (workers, sms, s)


def test_makespan_rule_follows_the_stated_rule():
    """The choice has utilisation >= 0.95 of the best candidate and no smaller
    candidate has, over causal and equal block sets."""
    for tiles in ([8, 6, 4, 2], [16] * 3, [32, 30, 28, 26, 24, 22, 20, 18, 16, 14, 12, 10, 8, 6, 4, 2]):
        for BH in (1, 2, 5):
            for sms in (8, 16, 152):
                s = schedule.num_splits_makespan(tiles, BH, sms, 128)
                top = min(128, sms, max(tiles))
                eff = [schedule.split_utilisation_makespan(tiles, BH, sms, c) for c in range(1, top + 1)]
                assert eff[s - 1] >= 0.95 * max(eff)
                assert all(eff[c - 1] < 0.95 * max(eff) for c in range(1, s))


@pytest.mark.parametrize("j0,j1", [(0, 1), (0, 5), (3, 17), (0, 128)])
def test_split_part_range_partitions_the_range(j0, j1):
    for p in range(1, j1 - j0 + 1):
        parts = [schedule.split_part_range(j0, j1, p, s) for s in range(p)]
        covered = [j for lo, hi in parts for j in range(lo, hi)]
        assert covered == list(range(j0, j1))  # disjoint, in order, complete
        lens = [hi - lo for lo, hi in parts]
        assert min(lens) >= 1 and max(lens) - min(lens) <= 1


def test_split_num_parts_rule():
    """The longest worker gets num_splits parts (fewer only if it has fewer
    tiles); shorter workers get no more, none gets an empty part, and no part
    of any worker is longer than ceil(n_max / num_splits) tiles."""
    for n_max in (1, 2, 7, 19, 64, 128):
        for S in range(1, 20):
            assert schedule.split_num_parts(n_max, S, n_max) == min(S, n_max)
            cap = schedule.ceil_div(n_max, S)
            prev = 0
            for n in range(1, n_max + 1):
                p = schedule.split_num_parts(n, S, n_max)
                assert 1 <= p <= min(n, S) and p >= prev
                prev = p
                longest = max(hi - lo for lo, hi in
                              (schedule.split_part_range(0, n, p, s) for s in range(p)))
                assert longest <= cap
    assert schedule.split_num_parts(0, 7, 128) == 0
    assert schedule.split_num_parts(5, 1, 128) == 1


def test_split_parts_of_the_two_head_long_sequence():
    """B=1 H=2 N=16384 causal, 7 splits: 256-row block m has 2m+2 tiles of 128
    keys (n_max = 128). Counted by hand from the thresholds p = k for
    128(k-1)/7 < 2m+2 <= 128k/7: nine even tile counts in each of the first
    six intervals (2..18, 20..36, ..., 92..108) and ten in the last
    (110..128), 9*(1+...+6) + 7*10 = 259 parts per head."""
    counts = [schedule.split_num_parts(2 * m + 2, 7, 128) for m in range(64)]
    by_k = {k: counts.count(k) for k in range(1, 8)}
    assert by_k == {1: 9, 2: 9, 3: 9, 4: 9, 5: 9, 6: 9, 7: 10}
    assert sum(counts) == 259


@pytest.mark.parametrize("N,Nk", [(1, 300), (300, 1), (130, 500), (500, 130), (256, 257)])
def test_cross_length_tile_ranges_match_element_level_brute_force(N, Nk):
    """Query length N, key length Nk: a tile pair is visited iff some (query,
    key) element in it is visible (top-left causal: key <= query)."""
    bm = bn = 128
    for causal in (False, True):
        for m in range(schedule.ceil_div(N, bm)):
            j0, j1 = schedule.fwd_kv_tile_range(m, N, bm, bn, causal, n_k=Nk)
            for j in range(schedule.ceil_div(Nk, bn)):
                visible = any((not causal) or kk <= qq
                              for qq in range(m * bm, min(N, (m + 1) * bm))
                              for kk in range(j * bn, min(Nk, (j + 1) * bn)))
                assert (j0 <= j < j1) == visible, (m, j, causal)
        for n in range(schedule.ceil_div(Nk, bn)):
            i0, i1 = schedule.bwd_q_tile_range(n, N, bm, bn, causal, n_k=Nk)
            for i in range(schedule.ceil_div(N, bm)):
                visible = any((not causal) or kk <= qq
                              for qq in range(i * bm, min(N, (i + 1) * bm))
                              for kk in range(n * bn, min(Nk, (n + 1) * bn)))
                assert (i0 <= i < i1) == visible, (n, i, causal)
