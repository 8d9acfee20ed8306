"""The tcgen05 GEMM's tile order (host-side restatement, no GPU).

The kernel walks its tiles in token-tile groups: with kTokGroup = 8, tile index
i maps to (token tile, weight tile) so that within a group of 8 token tiles the
token tile is fastest, and the groups follow one another.  This restates that
mapping (csrc/gemm_tc.cu, tile_coords) and checks what the kernel relies on:
every (token tile, weight tile) pair is visited exactly once for any tile
counts, and the CTAs running at once (consecutive tile indices) share weight
tiles while touching at most one group of token tiles.
"""

import pytest

K_TOK_GROUP = 8


def tile_coords(tile, t_tiles, n_tiles, group=K_TOK_GROUP):
    gsize = group * n_tiles
    g, r = divmod(tile, gsize)
    rows = min(group, t_tiles - g * group)
    return g * group + r % rows, r // rows


@pytest.mark.parametrize("t_tiles", [1, 2, 7, 8, 9, 16, 17, 23, 40])
@pytest.mark.parametrize("n_tiles", [1, 3, 43, 112])
def test_every_tile_once(t_tiles, n_tiles):
    seen = [tile_coords(i, t_tiles, n_tiles) for i in range(t_tiles * n_tiles)]
    assert sorted(seen) == [(t, n) for t in range(t_tiles) for n in range(n_tiles)]


@pytest.mark.parametrize("t_tiles,n_tiles,window", [(16, 112, 74), (8, 43, 74), (21, 86, 148)])
def test_running_window(t_tiles, n_tiles, window):
    """A window of consecutive tiles (the CTAs or pairs running at once)
    reuses each weight tile across all the token tiles of its group (up to 8),
    and spans at most two adjacent token-tile groups (it may straddle a group
    boundary)."""
    total = t_tiles * n_tiles
    for start in range(0, total - window + 1, max(1, window // 3)):
        coords = [tile_coords(i, t_tiles, n_tiles) for i in range(start, start + window)]
        groups = {t // K_TOK_GROUP for t, _ in coords}
        assert len(groups) <= 2 and max(groups) - min(groups) <= 1
        weights = {n for _, n in coords}
        rows = min(min(K_TOK_GROUP, t_tiles - g * K_TOK_GROUP) for g in groups)
        assert len(weights) <= window // rows + 2


def test_single_group_is_token_fastest():
    """With at most 8 token tiles (one group) the order is the plain
    token-tile-fastest walk."""
    for t_tiles in range(1, K_TOK_GROUP + 1):
        for i in range(t_tiles * 5):
            assert tile_coords(i, t_tiles, 5) == (i % t_tiles, i // t_tiles)
