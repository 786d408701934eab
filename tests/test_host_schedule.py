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
