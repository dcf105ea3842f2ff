"""Pins for the SSD and scan oracles: checks that do not reuse the oracle's formula.

Each ``pin_*`` function takes an oracle callable with the signature of
``oracle.ssd.ssd_fwd`` (or ``oracle.linscan.linscan``) and raises
AssertionError when the oracle disagrees with what the pages or the
mathematics fix.  The same pins run against the numpy oracle, the C oracle
and deliberately broken copies of the oracle (which they must reject).

Sources: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
NVIDIA CUDA Tile" (the Mamba-2 cuTile post) and "Selective-scan CUDA kernels"
(the scan README).
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

RTOL = 1e-11


def _close(got, want, what, rtol=RTOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    scale = max(1.0, float(np.max(np.abs(want)))) if want.size else 1.0
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    assert err <= rtol * scale, f"{what}: max abs err {err:.3e} > {rtol:.0e} * {scale:.3e}"


def small_problem(rng, batch=2, L=37, nh=4, H=3, S=5, G=2, h0=True, a_scale=1.0):
    """Random float64 problem with H != S (so a transposed operand cannot type-check by accident)."""
    x = rng.standard_normal((batch, L, nh, H))
    dt = np.log1p(np.exp(rng.standard_normal((batch, L, nh)) - 1.0))
    A = -np.exp(rng.uniform(0, np.log(16), nh)) * a_scale
    B = rng.standard_normal((batch, L, G, S)) / np.sqrt(S)
    C = rng.standard_normal((batch, L, G, S)) / np.sqrt(S)
    D = rng.uniform(0.5, 1.5, nh)
    hz = rng.standard_normal((batch, nh, H, S)) * 0.3 if h0 else np.zeros((batch, nh, H, S))
    # float32-exact values, so the float32-input C oracle sees exactly what the numpy one does
    return tuple(np.asarray(v, np.float32).astype(np.float64) for v in (x, dt, A, B, C, D, hz))


# ---------------------------------------------------------------------------
# SSD pins
# ---------------------------------------------------------------------------

def chunked_closed_form(x, dt, A, B, C, D, h0, T):
    """The post's chunked form with decay, section "Mamba-2 architecture":

        Y = exp(G) C h_k  +  (exp(G_i - G_j) . (C B^T) . M) X  +  D X
        h_{k+1} = exp(G_last) h_k + X^T (exp(G_last - G) . B)

    per chunk of T tokens, with G the within-chunk inclusive cumsum of
    a = A dt, B already scaled by dt (b_t = dt_t B_t) and M the causal mask
    (i >= j).  Written with matrix products, independently of the
    token-by-token loop.
    """
    batch, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    hpg = nh // G
    y = np.zeros((batch, L, nh, H))
    hf = np.zeros((batch, nh, H, S))
    for bi in range(batch):
        for h in range(nh):
            g = h // hpg
            state = h0[bi, h].copy()                       # H x S
            for s in range(0, L, T):
                e = min(s + T, L)
                a = A[h] * dt[bi, s:e, h]
                Gc = np.cumsum(a)
                Xc = x[bi, s:e, h]                         # T x H
                Bc = dt[bi, s:e, h][:, None] * B[bi, s:e, g]   # T x S
                Cc = C[bi, s:e, g]                         # T x S
                n = e - s
                ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
                expo = np.where(ii >= jj, Gc[:, None] - Gc[None, :], -np.inf)
                Lmat = np.exp(expo)                         # masked decay, 0 above the diagonal
                CB = Cc @ Bc.T
                y[bi, s:e, h] = (np.exp(Gc)[:, None] * (Cc @ state.T)
                                 + (Lmat * CB) @ Xc + D[h] * Xc)
                state = np.exp(Gc[-1]) * state + Xc.T @ (np.exp(Gc[-1] - Gc)[:, None] * Bc)
            hf[bi, h] = state
    return y, hf


def pin_chunked(ssd, rng):
    prob = small_problem(rng)
    y, hf = ssd(*prob)
    for T in (1, 4, 16, prob[0].shape[1]):
        yc, hc = chunked_closed_form(*prob, T)
        _close(y, yc, f"y vs chunked form T={T}")
        _close(hf, hc, f"h_final vs chunked form T={T}")


def pin_linear_attention(ssd, rng):
    """a == 0 (A = 0): Mamba-2 reduces to causal linear attention (the post's no-decay form
    Y = C h_t + ((C B^T) . M) X + D X), brute force over (i, j) pairs."""
    x, dt, A, B, C, D, h0 = small_problem(rng, batch=1, L=9, nh=2, H=3, S=4, G=1)
    A = np.zeros_like(A)
    y, hf = ssd(x, dt, A, B, C, D, h0)
    L, nh, H = x.shape[1], x.shape[2], x.shape[3]
    want = np.zeros_like(y)
    for h in range(nh):
        for i in range(L):
            acc = h0[0, h] @ C[0, i, 0] + D[h] * x[0, i, h]
            for j in range(i + 1):
                acc = acc + float(C[0, i, 0] @ (dt[0, j, h] * B[0, j, 0])) * x[0, j, h]
            want[0, i, h] = acc
    _close(y, want, "y vs causal linear attention")
    want_h = h0.copy()
    for h in range(nh):
        for j in range(L):
            want_h[0, h] += np.outer(x[0, j, h], dt[0, j, h] * B[0, j, 0])
    _close(hf, want_h, "h_final vs sum of outer products")


def pin_skip_only(ssd, rng):
    """B == 0: the state never receives input.  With h0 = 0, y = D x and h_final = 0 exactly;
    with h0 != 0, y_t = exp(sum_{k<=t} a_k) h0 c_t + D x_t and h_final = exp(sum a) h0."""
    x, dt, A, B, C, D, h0 = small_problem(rng, batch=2, L=11, nh=2, H=3, S=4, G=1)
    B = np.zeros_like(B)
    y, hf = ssd(x, dt, A, B, C, D, np.zeros_like(h0))
    assert np.array_equal(np.asarray(y), D[None, None, :, None] * x), "B=0, h0=0: y != D x exactly"
    assert not np.any(np.asarray(hf)), "B=0, h0=0: h_final != 0"
    y, hf = ssd(x, dt, A, B, C, D, h0)
    cum = np.cumsum(A[None, None, :] * dt, axis=1)         # [b, L, nh]
    want = (np.exp(cum)[..., None] * np.einsum("bnps,blns->blnp", h0, C[:, :, [0] * x.shape[2]])
            + D[None, None, :, None] * x)
    _close(y, want, "B=0: y vs decayed h0 readout + D x")
    _close(hf, np.exp(cum[:, -1])[..., None, None] * h0, "B=0: h_final vs exp(sum a) h0")


def pin_scalar_state(ssd, linscan_fn, rng):
    """H = S = 1: the SSD is the scalar scan with a_t = exp(A dt_t), b_t = dt_t B_t x_t,
    and y_t = c_t h_t + D x_t (cross-pins the two oracles)."""
    x, dt, A, B, C, D, h0 = small_problem(rng, batch=2, L=40, nh=3, H=1, S=1, G=1, h0=False)
    y, hf = ssd(x, dt, A, B, C, D, h0)
    for bi in range(2):
        for h in range(3):
            a = np.exp(A[h] * dt[bi, :, h])
            bb = dt[bi, :, h] * B[bi, :, 0, 0] * x[bi, :, h, 0]
            hs = linscan_fn(a[None], bb[None])[0]
            _close(np.asarray(y)[bi, :, h, 0], C[bi, :, 0, 0] * hs + D[h] * x[bi, :, h, 0], "scalar-state y")
            _close(np.asarray(hf)[bi, h, 0, 0], hs[-1], "scalar-state h_final")


def pin_state_carry(ssd, rng):
    """Splitting the sequence and feeding h_final back as h0 equals the full run (the post's
    note that the final state can be the next call's initial state)."""
    prob = small_problem(rng, L=30)
    x, dt, A, B, C, D, h0 = prob
    y, hf = ssd(*prob)
    L1 = 13
    y1, h1 = ssd(x[:, :L1], dt[:, :L1], A, B[:, :L1], C[:, :L1], D, h0)
    y2, h2 = ssd(x[:, L1:], dt[:, L1:], A, B[:, L1:], C[:, L1:], D, h1)
    _close(np.concatenate([y1, y2], axis=1), y, "split-run y")
    _close(h2, hf, "split-run h_final")


def pin_group_mapping(ssd, rng):
    """Head h reads B/C group h // (nheads / ngroups): each head alone, with its group's B/C
    sliced out, reproduces the grouped run."""
    x, dt, A, B, C, D, h0 = small_problem(rng, nh=6, G=3, L=12)
    y, hf = ssd(x, dt, A, B, C, D, h0)
    for h in range(6):
        g = h // 2
        s = slice(h, h + 1)
        yh, hh = ssd(x[:, :, s], dt[:, :, s], A[s], B[:, :, g:g + 1], C[:, :, g:g + 1], D[s], h0[:, s])
        _close(np.asarray(y)[:, :, s], yh, f"head {h} alone: y")
        _close(np.asarray(hf)[:, s], hh, f"head {h} alone: h_final")


def check_ssd_golden(ssd, fixture, rtol=1e-6):
    """Hand-derived worked examples.  A = -ln 2 is not exact in float32 (the C oracle's input
    type), which moves the decays 1/2 and 1/4 by ~3e-8 relative; every planted mistake moves
    a value by O(1), so 1e-6 still separates them."""
    inp = fixture["inputs"]
    arr = {k: np.asarray(v, np.float64) for k, v in inp.items()}
    y, hf = ssd(arr["x"], arr["dt"], arr["A"], arr["B"], arr["C"], arr["D"], arr["h0"])
    _close(y, np.asarray(fixture["expected"]["y"]), f"golden {fixture['name']}: y", rtol=rtol)
    _close(hf, np.asarray(fixture["expected"]["h_final"]), f"golden {fixture['name']}: h_final", rtol=rtol)


SSD_PINS = ("pin_chunked", "pin_linear_attention", "pin_skip_only", "pin_state_carry", "pin_group_mapping")


# ---------------------------------------------------------------------------
# decode-step pins: a step callable has the signature of oracle.ssd.ssd_step,
# (state, x_t, dt_t, A, B_t, C_t, D) -> (y_t, new state)
# ---------------------------------------------------------------------------

def pin_step_chain(step, ssd, rng):
    """Stepping token by token from h0 reproduces the sequential forward over the same tokens,
    and so does a prefill of the first tokens followed by steps from its final state (the
    post's note that a final state can start the next call).  ``ssd`` is the pinned forward."""
    x, dt, A, B, C, D, h0 = small_problem(rng, batch=2, L=12, nh=6, H=3, S=5, G=3)
    y_ref, h_ref = ssd(x, dt, A, B, C, D, h0)
    for start in (0, 7):
        if start:
            _, state = ssd(x[:, :start], dt[:, :start], A, B[:, :start], C[:, :start], D, h0)
        else:
            state = h0
        ys = []
        for t in range(start, x.shape[1]):
            yt, state = step(state, x[:, t], dt[:, t], A, B[:, t], C[:, t], D)
            ys.append(np.asarray(yt))
        _close(np.stack(ys, axis=1), np.asarray(y_ref)[:, start:], f"steps after {start} prefill tokens: y")
        _close(state, h_ref, f"steps after {start} prefill tokens: state")


def pin_step_from_zero(step, rng):
    """From a zero state one step gives the rank-one state dt x (outer) B and the readout
    dt (B . C) x + D x, written out per head with the group of head h at h // (nh / G)."""
    x, dt, A, B, C, D, _ = small_problem(rng, batch=2, L=1, nh=6, H=3, S=5, G=3)
    x, dt, B, C = x[:, 0], dt[:, 0], B[:, 0], C[:, 0]
    y, h = step(None, x, dt, A, B, C, D)
    y, h = np.asarray(y), np.asarray(h)
    for bi in range(2):
        for hd in range(6):
            g = hd // 2
            _close(h[bi, hd], np.outer(x[bi, hd], dt[bi, hd] * B[bi, g]), f"zero state: h[{bi},{hd}]")
            bc = sum(B[bi, g, s] * C[bi, g, s] for s in range(5))
            _close(y[bi, hd], dt[bi, hd] * bc * x[bi, hd] + D[hd] * x[bi, hd], f"zero state: y[{bi},{hd}]")


def pin_step_no_input(step, rng):
    """dt = 0 leaves the state exactly as it was (decay 1, no input) and reads it out;
    x = 0 only decays it: new state = exp(A dt) state, y = exp(A dt) (state . c)."""
    x, dt, A, B, C, D, h0 = small_problem(rng, batch=2, L=1, nh=4, H=3, S=5, G=2)
    x, dt, B, C = x[:, 0], dt[:, 0], B[:, 0], C[:, 0]
    y, h = step(h0, x, np.zeros_like(dt), A, B, C, D)
    assert np.array_equal(np.asarray(h), h0), "dt = 0: state changed"
    want = np.empty_like(x)
    for bi in range(2):
        for hd in range(4):
            g = hd // 2
            for p in range(3):
                want[bi, hd, p] = sum(h0[bi, hd, p, s] * C[bi, g, s] for s in range(5)) + D[hd] * x[bi, hd, p]
    _close(y, want, "dt = 0: y")
    y, h = step(h0, np.zeros_like(x), dt, A, B, C, D)
    dec = np.exp(A[None, :] * dt)
    _close(h, dec[:, :, None, None] * h0, "x = 0: state")
    for bi in range(2):
        for hd in range(4):
            g = hd // 2
            for p in range(3):
                want[bi, hd, p] = dec[bi, hd] * sum(h0[bi, hd, p, s] * C[bi, g, s] for s in range(5))
    _close(y, want, "x = 0: y")


STEP_PINS = ("pin_step_chain", "pin_step_from_zero", "pin_step_no_input")


# ---------------------------------------------------------------------------
# scan pins
# ---------------------------------------------------------------------------

def _dyadic(rng, n, lo, hi, denom=8):
    return [Fraction(int(v), denom) for v in rng.integers(lo * denom, hi * denom + 1, n)]


def bracketings(items, op):
    """Every value obtainable by fully bracketing op over the ordered items (Catalan many)."""
    if len(items) == 1:
        return [items[0]]
    out = []
    for k in range(1, len(items)):
        for left in bracketings(items[:k], op):
            for right in bracketings(items[k:], op):
                out.append(op(left, right))
    return out


def pin_scan_brute_force(linscan_fn, combine_fn, scan_pairs_fn, rng):
    """Exact rational folds: for L <= 6 every bracketing of the pair combine gives the same
    prefix (associativity), and it equals the sequential oracle exactly (dyadic inputs make
    every float64 step exact)."""
    for L in range(1, 7):
        a = _dyadic(rng, L, -2, 2)
        b = _dyadic(rng, L, -3, 3)
        pairs = list(zip(a, b))
        h = linscan_fn(np.array([[float(v) for v in a]]), np.array([[float(v) for v in b]]))[0]
        for t in range(L):
            vals = bracketings(pairs[: t + 1], combine_fn)
            assert all(v == vals[0] for v in vals), f"combine not associative at L={t + 1}"
            assert float(vals[0][1]) == h[t], f"prefix {t}: fold {vals[0][1]} != oracle {h[t]}"
        seq = scan_pairs_fn(a, b, combine_fn)
        assert [float(p[1]) for p in seq] == list(h), "scan_pairs != sequential oracle"


def pin_scan_closed_forms(linscan_fn, rng):
    """a == 1: the scan is a running sum (np.cumsum); a == 0: h = b; constant a = alpha,
    b = beta: h[t] = beta (1 - alpha^(t+1)) / (1 - alpha); a random dyadic case checked
    against exact rational arithmetic."""
    b = rng.standard_normal((3, 50)).astype(np.float32).astype(np.float64)
    _close(linscan_fn(np.ones_like(b), b), np.cumsum(b, axis=1), "a=1 vs cumsum")
    assert np.array_equal(linscan_fn(np.zeros_like(b), b), b), "a=0: h != b"
    alpha, beta = 0.9375, 1.25
    t = np.arange(200)
    _close(linscan_fn(np.full((1, 200), alpha), np.full((1, 200), beta))[0],
           beta * (1 - alpha ** (t + 1)) / (1 - alpha), "constant a,b closed form")


SCAN_PINS = ("pin_scan_brute_force", "pin_scan_closed_forms")
