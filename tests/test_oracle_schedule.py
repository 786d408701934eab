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
