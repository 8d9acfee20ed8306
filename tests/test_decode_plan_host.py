"""The decode path's launch plan (host-side restatement, no GPU).

A decode call whose channels exceed one wave of the kernel's resident CTAs is
split over at most three launches (csrc/decode.cu, launch_decode): nl =
ceil(N / wave) launches over equal shares of ceil(N / nl) channels.  Within a
launch the resident CTAs (whole clusters of kc) share the channels evenly,
with no more CTAs than one per 8 channels (rounded up to whole clusters).  This restates that arithmetic and checks what the kernels
rely on: the launches' channel ranges tile [0, N) exactly and in order, no CTA
gets more channels than the wave allows, and every launched CTA has at least
one channel.
"""

import pytest


def plan(N, ctas, cap, kc):
    wave = ctas * cap
    nl = (N + wave - 1) // wave
    share = (N + nl - 1) // nl
    launches = []
    nb = 0
    while nb < N:
        nn = min(share, N - nb)
        want = min(ctas, ((nn + 7) // 8 + kc - 1) // kc * kc)
        rows = (nn + want - 1) // want
        used = (nn + rows - 1) // rows
        grid = (used + kc - 1) // kc * kc
        launches.append((nb, nb + nn, rows, grid, used))
        nb += share
    return nl, launches


@pytest.mark.parametrize("N", [1, 7, 8, 9, 40, 1000, 3900, 4096, 4200, 4201, 5000, 5920, 5921,
                               11008, 12600, 17000, 17760])
@pytest.mark.parametrize("ctas,cap,kc", [(147, 40, 1), (148, 40, 1), (120, 35, 8), (112, 35, 16),
                                         (132, 35, 4), (120, 40, 8)])
def test_launches_tile_the_channels(N, ctas, cap, kc):
    nl, launches = plan(N, ctas, cap, kc)
    assert len(launches) == nl
    assert launches[0][0] == 0 and launches[-1][1] == N
    for (a0, a1, *_), (b0, *_rest) in zip(launches, launches[1:]):
        assert a1 == b0  # contiguous, in order
    for n0, n1, rows, grid, used in launches:
        assert 1 <= rows <= cap  # a CTA's slice fits its shared memory
        assert used <= grid <= ctas and grid % kc == 0  # whole clusters, resident at once
        assert (used - 1) * rows < n1 - n0 <= used * rows  # every launched slice non-empty
        assert n1 - n0 <= ctas * cap  # one launch is one wave of the resident CTAs
        # no more CTAs than one per 8 channels, rounded up to whole clusters
        assert used <= -(-(-(-(n1 - n0) // 8)) // kc) * kc


def test_three_launches_at_most_within_the_limit():
    """The host takes the decode path only while three launches hold N."""
    for ctas, cap, kc in [(148, 40, 1), (120, 35, 8)]:
        wave = ctas * cap
        assert plan(3 * wave, ctas, cap, kc)[0] == 3
        assert plan(2 * wave + 1, ctas, cap, kc)[0] == 3
        assert plan(wave, ctas, cap, kc)[0] == 1
