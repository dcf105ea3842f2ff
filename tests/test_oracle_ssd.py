"""CPU pins of the SSD oracle (numpy and C twins), and planted mistakes they must reject."""
import json
import os

import numpy as np
import pytest

import oracle_pins as P
from oracle import linscan as olin
from oracle import native
from oracle import ssd as ossd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ssd_worked_examples.json")


def c_ssd(x, dt, A, B, C, D, h0=None):
    """C oracle wrapped to the numpy oracle's signature (all units)."""
    batch, L, nh, H = np.shape(x)
    S = np.shape(B)[3]
    y, hf = native.ssd_fwd(x, dt, A, B, C, D, h0)
    return y.reshape(batch, nh, L, H).transpose(0, 2, 1, 3), hf.reshape(batch, nh, H, S)


def c_linscan(a, b):
    return native.linscan(np.atleast_2d(a), np.atleast_2d(b))


ORACLES = {"numpy": ossd.ssd_fwd, "c": c_ssd}
SCANS = {"numpy": olin.linscan, "c": c_linscan}


@pytest.fixture(params=sorted(ORACLES))
def ssd(request):
    return ORACLES[request.param]


@pytest.mark.parametrize("pin", P.SSD_PINS)
def test_ssd_pins(ssd, pin):
    getattr(P, pin)(ssd, np.random.default_rng(7))


def test_ssd_scalar_state_is_linscan(ssd):
    # float64 decays exp(A dt) feed the scan, so the float64-input numpy scan is the partner;
    # the float32-input C scan is tied to it by test_oracle_linscan.py
    P.pin_scalar_state(ssd, olin.linscan, np.random.default_rng(8))


def test_ssd_golden(ssd):
    for fx in json.load(open(GOLDEN))["fixtures"]:
        P.check_ssd_golden(ssd, fx)


def test_ssd_golden_float64_tight():
    # with float64 inputs the numpy oracle reproduces the hand derivations to rounding
    for fx in json.load(open(GOLDEN))["fixtures"]:
        P.check_ssd_golden(ossd.ssd_fwd, fx, rtol=1e-14)


def test_c_matches_numpy_random():
    rng = np.random.default_rng(3)
    prob = P.small_problem(rng, batch=2, L=70, nh=4, H=8, S=16, G=2)
    prob32 = [np.asarray(v, np.float32) for v in prob]   # the C oracle reads float32 inputs
    y1, h1 = ossd.ssd_fwd(*prob32)
    y2, h2 = c_ssd(*prob32)
    P._close(y2, y1, "C vs numpy y", rtol=1e-12)
    P._close(h2, h1, "C vs numpy h_final", rtol=1e-12)


def test_c_unit_selection():
    rng = np.random.default_rng(4)
    x, dt, A, B, C, D, h0 = P.small_problem(rng, batch=2, L=20, nh=4, H=3, S=5, G=2)
    y, hf = ossd.ssd_fwd(*(np.asarray(v, np.float32) for v in (x, dt, A, B, C, D, h0)))
    units = np.array([7, 0, 5])
    yu, hu = native.ssd_fwd(x, dt, A, B, C, D, h0, units=units)
    for k, u in enumerate(units):
        bi, h = divmod(int(u), 4)
        P._close(yu[k], y[bi, :, h], "unit y", rtol=1e-12)
        P._close(hu[k], hf[bi, h], "unit h_final", rtol=1e-12)


def test_c_rejects_bad_args():
    x = np.zeros((1, 4, 3, 2), np.float32)
    with pytest.raises(ValueError):   # nheads not a multiple of ngroups
        native.ssd_fwd(x, np.zeros((1, 4, 3)), np.zeros(3), np.zeros((1, 4, 2, 2)), np.zeros((1, 4, 2, 2)),
                       np.zeros(3), None)
    with pytest.raises(ValueError):
        native.ssd_fwd(x, np.zeros((1, 4, 3)), np.zeros(3), np.zeros((1, 4, 1, 2)), np.zeros((1, 4, 1, 2)),
                       np.zeros(3), None, units=np.array([3]))


# ---------------------------------------------------------------------------
# planted mistakes: each broken copy of the oracle must fail at least one pin
# ---------------------------------------------------------------------------

def _mutant(kind):
    def ssd_bad(x, dt, A, B, C, D, h0=None):
        x, dt, A, B, C, D = (np.asarray(v, np.float64) for v in (x, dt, A, B, C, D))
        batch, L, nh, H = x.shape
        G, S = B.shape[2], B.shape[3]
        gh = np.arange(nh) % G if kind == "group_modulo" else np.arange(nh) // (nh // G)
        state = np.zeros((batch, nh, H, S)) if h0 is None else np.array(h0, np.float64)
        y = np.empty((batch, L, nh, H))
        for t in range(L):
            a = A[None] * dt[:, t]
            if kind == "decay_sign":
                a = -a
            Bt, Ct = B[:, t, gh], C[:, t, gh]
            if kind == "swap_bc":
                Bt, Ct = Ct, Bt
            bt = Bt if kind == "no_dt_on_b" else dt[:, t, :, None] * Bt
            prev = state
            upd = x[:, t][..., None] * bt[:, :, None, :]
            if kind == "decay_after_input":
                state = np.exp(a)[..., None, None] * (state + upd)
            else:
                state = np.exp(a)[..., None, None] * state + upd
            readout = prev if kind == "exclusive" else state
            y[:, t] = np.einsum("bnps,bns->bnp", readout, Ct)
            if kind != "drop_d":
                y[:, t] += D[None, :, None] * x[:, t]
        return y, state
    return ssd_bad


MUTANTS = ["exclusive", "drop_d", "decay_sign", "swap_bc", "no_dt_on_b", "group_modulo", "decay_after_input"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_reject_planted_mistake(kind):
    bad = _mutant(kind)
    caught = []
    for pin in P.SSD_PINS:
        try:
            getattr(P, pin)(bad, np.random.default_rng(7))
        except AssertionError:
            caught.append(pin)
    try:
        for fx in json.load(open(GOLDEN))["fixtures"]:
            P.check_ssd_golden(bad, fx)
    except AssertionError:
        caught.append("golden")
    assert caught, f"planted mistake {kind!r} passed every pin"


def test_mutant_harness_is_faithful():
    # the mutant generator with no mutation equals the oracle (so the rejections above are real)
    good = _mutant("none")
    prob = P.small_problem(np.random.default_rng(5))
    y1, h1 = good(*prob)
    y2, h2 = ossd.ssd_fwd(*prob)
    P._close(y1, y2, "unmutated y", rtol=1e-13)
    P._close(h1, h2, "unmutated h", rtol=1e-13)
