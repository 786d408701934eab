"""The library's host-side work mapping against the oracle's (CPU only):
integer work, compared exactly."""

import pytest

from oracle import schedule


@pytest.mark.parametrize("B,H,N", [(1, 2, 512), (2, 3, 1), (1, 1, 1000), (4, 32, 8192),
                                   (1, 2, 16384), (8, 16, 2048)])
def test_fwd_grid_matches_oracle(fa2_lib, B, H, N):
    (gx, gy, gz), rows = fa2_lib.fwd_grid(B, H, N)
    assert (gx, gy, gz) == schedule.fwd_grid(B, H, N, rows)


@pytest.mark.parametrize("N", [1, 2, 127, 128, 255, 256, 257, 1000, 2048, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_block_work_matches_oracle(fa2_lib, N, causal):
    (gx, _, _), rows = fa2_lib.fwd_grid(1, 1, N)
    seen = []
    prev = None
    for bx in range(gx):
        r0, r1, tiles = fa2_lib.fwd_block_work(bx, N, causal)
        m = r0 // rows
        assert r0 == m * rows and r1 == min(N, r0 + rows)
        j0, j1 = schedule.fwd_kv_tile_range(m, N, rows, 128, causal)
        assert j0 == 0 and tiles == j1
        seen.append(m)
        if causal and prev is not None:
            assert tiles <= prev  # longest first
        prev = tiles
    assert sorted(seen) == list(range(gx))
    if not causal:
        assert seen == list(range(gx))  # the pages' order, row block fastest


@pytest.mark.parametrize("N", [1, 63, 64, 65, 128, 129, 1000, 4096])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_block_work_matches_oracle(fa2_lib, N, d, causal):
    (gx, gy, gz), keys, qrows = fa2_lib.bwd_grid(2, 3, N, d)
    assert (gx, gy, gz) == schedule.bwd_grid(2, 3, N, keys)
    for bx in range(gx):
        k0, k1, i0, i1 = fa2_lib.bwd_block_work(bx, N, d, causal)
        assert (k0, k1) == (bx * keys, min(N, (bx + 1) * keys))
        assert (i0, i1) == schedule.bwd_q_tile_range(bx, N, qrows, keys, causal)


def _block_tiles(N, causal):
    """K/V tiles of every 256-row forward worker in launch order (causal:
    longest first), from the oracle's brute-force tile ranges."""
    nm = schedule.ceil_div(N, 256)
    order = range(nm - 1, -1, -1) if causal else range(nm)
    return [schedule.fwd_kv_tile_range(m, N, 256, 128, causal)[1] for m in order]


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 16384), (4, 32, 8192), (2, 3, 1000),
                                   (1, 1, 100000), (8, 16, 2048), (1, 5, 4096), (1, 4, 8192),
                                   (2, 4, 1024)])
@pytest.mark.parametrize("num_sms", [1, 132, 152, 160])
def test_num_splits_matches_oracle(fa2_lib, B, H, N, num_sms):
    """The library's K/V split count equals the oracle's rule (makespan
    utilisation of the same launch: one forward CTA per 256 query rows, 128
    keys per tile, row blocks longest first under the causal mask)."""
    lib = fa2_lib.load_library()
    for causal in (0, 1):
        want = schedule.num_splits_makespan(_block_tiles(N, causal), B * H, num_sms, 128)
        assert lib.fa2_num_splits(B, H, N, 128, causal, num_sms) == want, causal


def test_num_splits_of_the_two_head_long_sequence(fa2_lib):
    """B=1 H=2 N=16384 causal on GB300's 152 SMs: 4 parts (the fastest split
    count measured on that shape)."""
    assert fa2_lib.load_library().fa2_num_splits(1, 2, 16384, 128, 1, 152) == 4


def test_num_splits_rejects_bad_arguments(fa2_lib):
    lib = fa2_lib.load_library()
    assert lib.fa2_num_splits(0, 1, 128, 128, 0, 152) == 0
    assert lib.fa2_num_splits(1, 1, 128, 96, 0, 152) == 0
    assert lib.fa2_num_splits(1, 1, 128, 128, 2, 152) == 0
    assert lib.fa2_num_splits(1, 1, 128, 128, 0, 0) == 0


def test_split_workspace_size(fa2_lib):
    lib = fa2_lib.load_library()

    def up(x):
        return -(-x // 256) * 256

    for B, H, N, d, S in ((1, 2, 16384, 128, 7), (2, 3, 1000, 64, 3), (1, 1, 1, 64, 1)):
        rows = S * B * H * N
        counters = B * H * (-(-N // 256)) * 2 * 4
        assert (lib.fa2_fwd_split_workspace_size(B, H, N, d, S)
                == up(rows * d * 4) + up(rows * 4) + up(counters))
    assert lib.fa2_fwd_split_workspace_size(1, 1, 128, 128, 0) == 0
    assert lib.fa2_fwd_split_workspace_size(1, 1, 128, 128, 129) == 0


def test_kv_outer_workspace_size(fa2_lib):
    lib = fa2_lib.load_library()

    def up(x):
        return -(-x // 256) * 256

    for B, H, N, d in ((4, 32, 8192, 128), (2, 3, 1000, 64), (1, 1, 1, 64)):
        rows = B * H * N
        assert lib.fa2_fwd_kv_outer_workspace_size(B, H, N, d) == up(rows * d * 4) + 2 * up(rows * 4)
    assert lib.fa2_fwd_kv_outer_workspace_size(1, 1, 128, 96) == 0
    assert lib.fa2_fwd_kv_outer_workspace_size(0, 1, 128, 64) == 0


def _persistent_loads(fa2_lib, B, H, N, causal, num_sms):
    """Per-CTA lists of the unsplit forward's persistent grid, checked for
    coverage, and each CTA's load in K/V tiles (the oracle's tile ranges)."""
    G, cta, pos = fa2_lib.fwd_schedule(B, H, N, causal, num_sms)
    tiles = _block_tiles(N, causal)  # per rank (launch order)
    nm = len(tiles)
    assert 1 <= G <= num_sms and len(cta) == B * H * nm
    lists = {}
    for i, (c, p) in enumerate(zip(cta, pos)):
        assert 0 <= c < G
        lists.setdefault(c, []).append(p)
    assert len(lists) == G  # no idle CTA
    for ps in lists.values():
        assert sorted(ps) == list(range(len(ps)))
    loads = [0] * G
    for i, c in enumerate(cta):
        loads[c] += tiles[i % nm]
    return G, loads, tiles


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 1, 300), (2, 3, 1000), (3, 5, 640), (1, 2, 16384),
                                   (4, 32, 8192), (8, 16, 2048), (2, 16, 8192), (4, 8, 4096),
                                   (9, 40, 2500), (1, 1, 100000)])
@pytest.mark.parametrize("num_sms", [1, 7, 148, 152])
@pytest.mark.parametrize("causal", [0, 1])
def test_fwd_schedule_runs_every_row_block_once(fa2_lib, B, H, N, num_sms, causal):
    """Every row block of the grid is in exactly one CTA's list, at one
    position, and every CTA has work."""
    _persistent_loads(fa2_lib, B, H, N, causal, num_sms)


def test_fwd_schedule_without_mask_is_round_robin(fa2_lib):
    """Without a causal mask the row blocks are dealt in grid order: block i
    to CTA i mod G, at position i div G."""
    G, cta, pos = fa2_lib.fwd_schedule(8, 16, 2048, False, 152)
    assert G == 152
    assert cta == [i % 152 for i in range(1024)] and pos == [i // 152 for i in range(1024)]


@pytest.mark.parametrize("B,H,N,want", [
    # 128 heads x 32 row blocks: 2048 pairs of 2(32 + 1) = 66 tiles on 152
    # CTAs = 13 rounds + 72 pairs; the 72 leftover pairs are the middle pairs
    # (blocks 15 and 16: 32 and 34 tiles) of the last 72 heads, run as halves.
    (4, 32, 8192, 13 * 66 + 34),
    # 128 heads x 8 row blocks: 512 pairs of 18 tiles = 3 rounds + 56 pairs,
    # whose halves are blocks 3 and 4 (8 and 10 tiles).
    (8, 16, 2048, 3 * 18 + 10),
    # 32 heads x 32 row blocks: 512 pairs = 3 rounds + 56; two middle pairs in
    # each of the last 28 heads, the larger halves being block 17 (36 tiles).
    (2, 16, 8192, 3 * 66 + 36),
])
def test_fwd_schedule_causal_balance(fa2_lib, B, H, N, want):
    """Causal makespans (K/V tiles of the busiest CTA) on 152 SMs, derived by
    hand from the pair rule; each within a few percent of the mean load."""
    G, loads, _ = _persistent_loads(fa2_lib, B, H, N, 1, 152)
    assert max(loads) == want
    assert max(loads) <= 1.07 * sum(loads) / 152


def test_fwd_schedule_small_grid_is_one_block_per_cta(fa2_lib):
    """With no more row blocks than SMs every block gets a CTA of its own."""
    G, cta, pos = fa2_lib.fwd_schedule(2, 4, 1024, True, 152)
    assert G == 32 and sorted(cta) == list(range(32)) and set(pos) == {0}


def test_fwd_schedule_rejects_bad_arguments(fa2_lib):
    import ctypes
    lib = fa2_lib.load_library()
    g = ctypes.c_int()
    for args in ((0, 1, 128, 0, 152), (1, 1, 0, 0, 152), (1, 1, 128, 2, 152), (1, 1, 128, 0, 0)):
        assert lib.fa2_fwd_schedule(*args, ctypes.byref(g), None, None) != 0
    assert lib.fa2_fwd_schedule(1, 1, 128, 0, 152, None, None, None) != 0
    assert lib.fa2_fwd_schedule(1, 1, 128, 0, 152, ctypes.byref(g), None, None) == 0 and g.value == 1
