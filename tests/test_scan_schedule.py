"""The chunk scan's CTA split, checked on the host through ssm_debug_scan_schedule (no GPU call).

The chunk scan's CTAs take the tiles (batch, chunk, group, row tile) in order, in up to three
tiers with a different number of CTAs per tile; a CTA decodes its tile and run of heads from
its index the way `decode` below does.  Every (tile, head) must be computed by exactly one CTA,
the two row tiles of a chunk must stay in the same tier (adjacent, so that they run at the same
time), and a plan's heads per CTA bounds every run."""
import ctypes

import numpy as np
import pytest

from selective_state_space_mamba_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def schedule(lib, tiles, rt, hpg, sms, plan_heads):
    out = np.zeros(6, dtype=np.int64)
    grid = lib.ssm_debug_scan_schedule(tiles, rt, hpg, sms, plan_heads, out.ctypes.data_as(ctypes.c_void_p))
    return grid, [(int(out[2 * k]), int(out[2 * k + 1])) for k in range(3)]


def decode(tiers, hpg, cta):
    """CTA index -> (tile, first head, heads), as the kernel does it."""
    tile0 = 0
    for s, (nt, ni) in enumerate(tiers):
        if cta < nt * ni or s == 2:
            k = cta % ni
            run, rem = divmod(hpg, ni)  # the first `rem` CTAs of a tile take one head more
            return tile0 + cta // ni, k * run + min(k, rem), run + (1 if k < rem else 0)
        cta -= nt * ni
        tile0 += nt
    raise AssertionError("unreachable")


SHAPES = [(256, 2, 80, 152), (128, 2, 24, 152), (8192, 2, 4, 152), (64, 1, 2, 152), (2, 1, 2, 152),
          (256, 2, 80, 148), (512, 2, 32, 152), (300, 1, 16, 152), (40, 2, 80, 152), (1024, 2, 8, 132)]


@pytest.mark.parametrize("tiles,rt,hpg,sms", SHAPES)
@pytest.mark.parametrize("plan_heads", [0, 1, 3, 20, 1000])
def test_every_tile_head_once(lib, tiles, rt, hpg, sms, plan_heads):
    grid, tiers = schedule(lib, tiles, rt, hpg, sms, plan_heads)
    assert grid == sum(nt * ni for nt, ni in tiers)
    assert sum(nt for nt, _ in tiers) == tiles
    for nt, ni in tiers:
        assert nt % rt == 0, "a chunk's row tiles split between tiers"
        assert nt == 0 or 1 <= ni <= hpg, "a CTA without heads"
    if plan_heads > 0:
        assert tiers[1][0] == 0 and tiers[2][0] == 0
        assert -(-hpg // tiers[0][1]) <= min(plan_heads, hpg) or tiers[0][0] == 0
    count = np.zeros((tiles, hpg), dtype=np.int32)
    for cta in range(grid):
        tile, first, n = decode(tiers, hpg, cta)
        assert 0 <= tile < tiles and n >= 1 and first + n <= hpg
        if plan_heads > 0:
            assert n <= plan_heads
        count[tile, first:first + n] += 1
    assert (count == 1).all()


def test_headline_split_puts_large_runs_first(lib):
    """At b4 L8192 nh80 chunk 256 (256 tiles of 80 heads) on 152 SMs the model splits the tiles
    in tiers, with runs shrinking from the first tier to the last."""
    grid, tiers = schedule(lib, 256, 2, 80, 152, 0)
    used = [(nt, ni) for nt, ni in tiers if nt > 0]
    assert len(used) > 1
    assert all(a[1] <= b[1] for a, b in zip(used, used[1:]))
    assert grid == schedule(lib, 256, 2, 80, 152, 0)[0]  # cached: the same answer again


def test_invalid_sizes_refused(lib):
    assert lib.ssm_debug_scan_schedule(-1, 2, 80, 152, 0, None) == -1
    assert lib.ssm_debug_scan_schedule(3, 2, 80, 152, 0, None) == -1  # not whole chunks
    assert lib.ssm_debug_scan_schedule(4, 3, 80, 152, 0, None) == -1
    assert lib.ssm_debug_scan_schedule(4, 2, 0, 152, 0, None) == -1
    assert lib.ssm_debug_scan_schedule(4, 2, 8, 0, 0, None) == -1
    assert lib.ssm_debug_scan_schedule(4, 2, 8, 152, -1, None) == -1
