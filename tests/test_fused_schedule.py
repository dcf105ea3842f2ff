"""The fused state pass's work split, checked on the host through ssm_debug_fused_schedule
(the same functions the kernel runs, compiled for the host as well; no GPU needed).

With more (batch, head pair) chains than SMs each CTA takes an equal range of the chain-major
(chain, chunk) units: the head of a chain that ends inside the range first (publishing its
final state), then whole chains, then the tail of a chain that starts inside the range
(starting from the state the previous CTA published).  A CTA waits for that state only as long
as its predecessor's head runs past the point where this CTA reaches its tail."""
import ctypes

import numpy as np
import pytest

from selective_state_space_mamba_gb300 import _lib

SHAPES = [(160, 32, 152), (168, 8, 152), (153, 5, 152), (192, 8, 152), (300, 4, 152), (1000, 3, 152),
          (160, 1, 152), (96, 8, 152), (16, 512, 152), (152, 7, 152), (7, 9, 4), (5, 100, 4), (0, 8, 152),
          (40, 0, 152)]


def schedule(chains, nchunks, sms, split=False):
    lib = _lib.load()
    n = lib.ssm_debug_fused_schedule(chains, nchunks, sms, int(split), None, 0)
    assert n >= 0
    rows = np.zeros((max(n, 1), 6), dtype=np.int64)
    got = lib.ssm_debug_fused_schedule(chains, nchunks, sms, int(split), rows.ctypes.data_as(ctypes.c_void_p), n)
    assert got == n
    return rows[:n]


@pytest.mark.parametrize("chains,nchunks,sms", SHAPES)
def test_every_unit_once_in_order(chains, nchunks, sms):
    rows = schedule(chains, nchunks, sms)
    grid = chains if (chains <= sms or nchunks == 0) else sms
    seen = np.zeros((chains, nchunks), dtype=np.int64)
    for cta, chain, c0, c1, from_carry, to_carry in rows:
        assert 0 <= cta < grid and 0 <= chain < chains and 0 <= c0 < c1 <= nchunks
        seen[chain, c0:c1] += 1
        # a segment starts from a published state exactly when it starts inside its chain, and
        # publishes exactly when it ends inside its chain
        assert bool(from_carry) == (c0 > 0) and bool(to_carry) == (c1 < nchunks)
    assert (seen == 1).all()
    units = chains * nchunks
    for k in range(grid):
        mine = rows[rows[:, 0] == k]
        assert sum(c1 - c0 for _, _, c0, c1, _, _ in mine) == (k + 1) * units // grid - k * units // grid
        kinds = ["head" if r[5] else ("tail" if r[4] else "whole") for r in mine]
        assert kinds == sorted(kinds, key=["head", "whole", "tail"].index), f"CTA {k}: {kinds}"
        assert kinds.count("head") <= 1 and kinds.count("tail") <= 1


@pytest.mark.parametrize("chains,nchunks,sms", SHAPES)
def test_carry_published_before_it_is_needed(chains, nchunks, sms):
    rows = schedule(chains, nchunks, sms)
    publish, need = {}, {}
    for k in np.unique(rows[:, 0]) if len(rows) else []:
        t = 0  # units this CTA has run before the segment
        for cta, chain, c0, c1, from_carry, to_carry in rows[rows[:, 0] == k]:
            if from_carry:
                need[chain] = (k, t)
            t += c1 - c0
            if to_carry:
                publish[chain] = (k, t)
    assert set(need) == set(publish)
    for chain, (k, t_need) in need.items():
        kp, t_pub = publish[chain]
        assert kp == k - 1, f"chain {chain}: published by CTA {kp}, needed by CTA {k}"
        # in units of work: the predecessor has published by the time this CTA reaches its tail
        assert t_pub <= t_need, f"chain {chain}: published after {t_pub} units, needed after {t_need}"


def split_grid(chains, nchunks, sms):
    """Split chains: the same number of equal pieces for every chain, as many as fit the SMs (at
    most one per chunk), so that pieces of different chains line up; one range per SM when
    there are more chains than SMs."""
    return chains * min(sms // chains, nchunks) if chains <= sms else sms


SPLIT_SHAPES = [(16, 512, 152), (2, 64, 152), (1, 4, 152), (1, 1000, 152), (7, 9, 4), (76, 64, 152), (3, 152, 152),
                (160, 32, 152), (5, 30, 148)]


@pytest.mark.parametrize("chains,nchunks,sms", SPLIT_SHAPES)
def test_split_chains_every_unit_once(chains, nchunks, sms):
    """Split chains: ranges of equal length (see split_grid); a segment
    starts from zero exactly when it starts inside its chain and publishes (into its CTA's slot)
    exactly when it ends inside it, so every range publishes at most once."""
    rows = schedule(chains, nchunks, sms, split=True)
    units = chains * nchunks
    grid = split_grid(chains, nchunks, sms)
    assert int(rows[:, 0].max()) + 1 == grid
    seen = np.zeros((chains, nchunks), dtype=np.int64)
    for cta, chain, c0, c1, from_zero, publish in rows:
        assert 0 <= cta < grid and 0 <= chain < chains and 0 <= c0 < c1 <= nchunks
        seen[chain, c0:c1] += 1
        assert bool(from_zero) == (c0 > 0) and bool(publish) == (c1 < nchunks)
    assert (seen == 1).all()
    for k in range(grid):
        mine = rows[rows[:, 0] == k]
        assert sum(c1 - c0 for _, _, c0, c1, _, _ in mine) == (k + 1) * units // grid - k * units // grid
        assert int(mine[:, 5].sum()) <= 1


@pytest.mark.parametrize("chains,nchunks,sms", [(16, 512, 152), (1, 1000, 152), (7, 9, 4), (3, 152, 152)])
def test_split_chains_compose_to_the_recurrence(chains, nchunks, sms):
    """The pieces' own results and the composition the fix-up kernel applies give the chain's
    recurrence h[c+1] = d_c h[c] + s_c, on scalar chains with random decays and increments
    (float64 here; the kernels do the same in f32 per state entry)."""
    rng = np.random.default_rng(7)
    rows = schedule(chains, nchunks, sms, split=True)
    units = chains * nchunks
    grid = split_grid(chains, nchunks, sms)
    lg = -rng.random((chains, nchunks)) * 0.5  # log2 decays
    inc = rng.standard_normal((chains, nchunks))
    h0 = rng.standard_normal(chains)
    ref = np.zeros((chains, nchunks + 1))
    ref[:, 0] = h0
    for c in range(nchunks):
        ref[:, c + 1] = 2.0 ** lg[:, c] * ref[:, c] + inc[:, c]
    # the fused pass: every segment from h0 (chain start) or zero, its end published by its CTA
    hin = np.zeros((chains, nchunks + 1))
    slot = np.zeros(grid)
    for cta, chain, c0, c1, from_zero, publish in rows:
        h = 0.0 if from_zero else h0[chain]
        for c in range(c0, c1):
            hin[chain, c] = h
            h = 2.0 ** lg[chain, c] * h + inc[chain, c]
        if publish:
            slot[cta] = h
        if c1 == nchunks:
            hin[chain, nchunks] = h  # h_final
    # the fix-up: the state entering the piece that range k starts inside chain z
    u = lambda j: j * units // grid
    for k in range(1, grid):
        if u(k) % nchunks == 0:
            continue
        z, zc = divmod(u(k), nchunks)[0], (u(k) // nchunks) * nchunks
        acc, lgs, j = slot[k - 1], 0.0, k - 1
        while u(j) > zc:
            lgs += lg[z, u(j) - zc:u(j + 1) - zc].sum()
            acc += 2.0 ** lgs * slot[j - 1]
            j -= 1
        b, e = u(k) - zc, min(u(k + 1), zc + nchunks) - zc
        dec = 0.0
        for c in range(b, e):
            hin[z, c] += 2.0 ** dec * acc
            dec += lg[z, c]
        if e == nchunks:
            hin[z, nchunks] += 2.0 ** dec * acc
    np.testing.assert_allclose(hin, ref, rtol=1e-12, atol=1e-12)


def test_invalid_sizes():
    lib = _lib.load()
    assert lib.ssm_debug_fused_schedule(-1, 8, 152, 0, None, 0) == -1
    assert lib.ssm_debug_fused_schedule(8, 8, 0, 0, None, 0) == -1
