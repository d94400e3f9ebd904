"""The backward's per-CTA work schedule (host code of the library, no GPU):
every (key tile, head) item is run exactly once, each CTA runs its items
longest first, and the schedule's makespan under the same cost model (11
units per query tile, 8 per item boundary) beats the round-robin snake it
replaces, which is recomputed here from its definition."""

import pytest

from transformer_attention_ggd_gb300 import bam_attn as ba

TILE, BOUNDARY = 11, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        ba.load_library()
    except RuntimeError as e:
        pytest.skip(str(e))


def _cost(sizes):
    return sum(sizes) * TILE + max(len(sizes) - 1, 0) * BOUNDARY


def _snake(nkb, bh, g):
    per = [[] for _ in range(g)]
    total = nkb * bh
    r = 0
    while r * g < total:
        for c in range(g):
            idx = r * g + ((g - 1 - c) if r & 1 else c)
            if idx < total:
                per[c].append(nkb - idx // bh)
        r += 1
    return max(_cost(p) for p in per)


@pytest.mark.parametrize("B,H,T,grid", [(8, 12, 512, 152), (1, 12, 4096, 152), (8, 12, 1024, 152),
                                        (16, 16, 512, 152), (3, 5, 640, 152), (2, 3, 300, 148)])
def test_schedule_covers_every_item_once_and_beats_the_snake(B, H, T, grid):
    nkb = (T + 127) // 128
    bh = B * H
    total = nkb * bh
    g = min(grid, total)
    lists = ba.bam_attn_bwd_schedule(B, H, T, True, grid)
    snake = _snake(nkb, bh, g)
    if lists is None:
        return  # the kernel keeps its own round-robin deal
    assert len(lists) == g
    flat = sorted(w for lst in lists for w in lst)
    assert flat == list(range(total))
    worst = 0
    for lst in lists:
        sizes = [nkb - w // bh for w in lst]  # causal: key tile kb sees nkb - kb query tiles
        assert sizes == sorted(sizes, reverse=True)
        worst = max(worst, _cost(sizes))
    assert worst < snake


def test_training_shape_packs_to_the_lower_bound():
    # 96 heads x key tiles of 4, 3, 2, 1 query tiles on 152 CTAs: the snake's
    # worst CTA runs 4 + 2 + 1 tiles (93 units).  85 is the optimum: under 85
    # a CTA holding a 4-tile item takes at most two more tiles and any other
    # CTA at most six, so 96 x 6 + 56 x 6 = 912 < 960 tiles would fit.
    lists = ba.bam_attn_bwd_schedule(8, 12, 512, True, 152)
    assert lists is not None
    costs = [_cost([4 - w // 96 for w in lst]) for lst in lists]
    assert max(costs) == 85
    assert _snake(4, 96, 152) == 93
    # 960 tiles on 152 CTAs of at most six tiles leave 48 tiles over: at
    # least 48 CTAs run seven (4+3, 85 units); the schedule has no more.
    assert costs.count(85) == 48


def test_noncausal_large_and_bad_arguments():
    assert ba.bam_attn_bwd_schedule(8, 12, 512, False, 152) is None
    # more than 1024 items: the kernel's own round-robin deal
    assert ba.bam_attn_bwd_schedule(1, 12, 32768, True, 152) is None
    with pytest.raises(ba.BamError):
        ba.bam_attn_bwd_schedule(0, 12, 512, True, 152)
