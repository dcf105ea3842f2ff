"""CPU pins of the decode-step oracle (oracle.ssd.ssd_step), and planted mistakes they must reject."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import native
from oracle import ssd as ossd


def _run_pin(step, pin):
    fn = getattr(P, pin)
    rng = np.random.default_rng(11)
    if pin == "pin_step_chain":
        fn(step, ossd.ssd_fwd, rng)
    else:
        fn(step, rng)


@pytest.mark.parametrize("pin", P.STEP_PINS)
def test_step_pins(pin):
    _run_pin(ossd.ssd_step, pin)


def test_c_oracle_one_token_is_the_step():
    # the C oracle run on one token from a float64 state is the step (the bench's CPU leg uses it)
    rng = np.random.default_rng(12)
    x, dt, A, B, C, D, h0 = P.small_problem(rng, batch=2, L=1, nh=4, H=3, S=5, G=2)
    y, hf = native.ssd_fwd(x, dt, A, B, C, D, h0)
    ys, hs = ossd.ssd_step(h0, x[:, 0], dt[:, 0], A, B[:, 0], C[:, 0], D)
    P._close(y.reshape(2, 4, 3), ys, "C one-token y", rtol=1e-12)
    P._close(hf.reshape(2, 4, 3, 5), hs, "C one-token state", rtol=1e-12)


def test_step_rejects_bad_groups():
    with pytest.raises(ValueError):
        ossd.ssd_step(None, np.zeros((1, 3, 2)), np.zeros((1, 3)), np.zeros(3), np.zeros((1, 2, 4)),
                      np.zeros((1, 2, 4)), np.zeros(3))


def _mutant(kind):
    def step_bad(state, x, dt, A, B, C, D):
        x, dt, A, B, C, D = (np.asarray(v, np.float64) for v in (x, dt, A, B, C, D))
        batch, nh, H = x.shape
        G, S = B.shape[1], B.shape[2]
        gh = np.arange(nh) % G if kind == "group_modulo" else np.arange(nh) // (nh // G)
        h = np.zeros((batch, nh, H, S)) if state is None else np.asarray(state, np.float64)
        a = A[None] * dt
        if kind == "decay_sign":
            a = -a
        Bt, Ct = B[:, gh], C[:, gh]
        if kind == "swap_bc":
            Bt, Ct = Ct, Bt
        bt = Bt if kind == "no_dt_on_b" else dt[:, :, None] * Bt
        upd = x[..., None] * bt[:, :, None, :]
        if kind == "decay_after_input":
            h_new = np.exp(a)[..., None, None] * (h + upd)
        else:
            h_new = np.exp(a)[..., None, None] * h + upd
        readout = h if kind == "exclusive" else h_new
        y = np.einsum("bnps,bns->bnp", readout, Ct)
        if kind != "drop_d":
            y = y + D[None, :, None] * x
        return y, h_new
    return step_bad


MUTANTS = ["exclusive", "drop_d", "decay_sign", "swap_bc", "no_dt_on_b", "group_modulo", "decay_after_input"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_step_pins_reject_planted_mistake(kind):
    bad = _mutant(kind)
    caught = []
    for pin in P.STEP_PINS:
        try:
            _run_pin(bad, pin)
        except AssertionError:
            caught.append(pin)
    assert caught, f"planted mistake {kind!r} passed every step pin"


def test_step_mutant_harness_is_faithful():
    good = _mutant("none")
    rng = np.random.default_rng(13)
    x, dt, A, B, C, D, h0 = P.small_problem(rng, batch=2, L=1, nh=4, H=3, S=5, G=2)
    args = (h0, x[:, 0], dt[:, 0], A, B[:, 0], C[:, 0], D)
    y1, h1 = good(*args)
    y2, h2 = ossd.ssd_step(*args)
    P._close(y1, y2, "unmutated y", rtol=1e-13)
    P._close(h1, h2, "unmutated state", rtol=1e-13)
