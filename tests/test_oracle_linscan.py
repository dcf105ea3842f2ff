"""CPU pins of the scalar-scan oracle (numpy and C twins), and the operand-swapped combine
that the suite must reject (selective-scan README, "The problem": the combine is associative,
not commutative, and an operand swap is a silent wrong answer)."""
import json
import os

import numpy as np
import pytest

import oracle_pins as P
from oracle import linscan as olin
from oracle import native

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "linscan_worked_examples.json")


def c_linscan(a, b):
    return native.linscan(np.atleast_2d(a), np.atleast_2d(b))


SCANS = {"numpy": olin.linscan, "c": c_linscan}


@pytest.mark.parametrize("name", sorted(SCANS))
def test_scan_brute_force(name):
    P.pin_scan_brute_force(SCANS[name], olin.combine, olin.scan_pairs, np.random.default_rng(11))


@pytest.mark.parametrize("name", sorted(SCANS))
def test_scan_closed_forms(name):
    P.pin_scan_closed_forms(SCANS[name], np.random.default_rng(12))


@pytest.mark.parametrize("name", sorted(SCANS))
def test_scan_golden(name):
    for fx in json.load(open(GOLDEN))["fixtures"]:
        h = SCANS[name](np.array([fx["a"]]), np.array([fx["b"]]))[0]
        assert list(h) == fx["h"], fx["name"]
        pairs = olin.scan_pairs(fx["a"], fx["b"])
        assert [p[1] for p in pairs] == fx["h"], fx["name"] + " (pair fold)"


def test_c_matches_numpy_rows():
    rng = np.random.default_rng(2)
    a = rng.uniform(0.9, 0.9999, (5, 3001)).astype(np.float32)
    b = rng.standard_normal((5, 3001)).astype(np.float32)
    P._close(c_linscan(a, b), olin.linscan(a, b), "C vs numpy scan", rtol=1e-13)
    sel = native.linscan(a, b, rows=np.array([4, 1]))
    P._close(sel, olin.linscan(a, b)[[4, 1]], "row selection", rtol=1e-13)


def test_empty_row():
    assert olin.linscan(np.zeros((2, 0)), np.zeros((2, 0))).shape == (2, 0)
    assert native.linscan(np.zeros((2, 0)), np.zeros((2, 0))).shape == (2, 0)


def swapped_combine(p, q):
    """Planted mistake: operands of the second component swapped, (a1 a2, a1 b2 + b1)."""
    a1, b1 = p
    a2, b2 = q
    return (a1 * a2, a1 * b2 + b1)


def test_swapped_combine_is_rejected():
    with pytest.raises(AssertionError):
        P.pin_scan_brute_force(olin.linscan, swapped_combine, olin.scan_pairs, np.random.default_rng(11))
    fx = json.load(open(GOLDEN))["fixtures"][1]
    assert [p[1] for p in olin.scan_pairs(fx["a"], fx["b"], swapped_combine)] != fx["h"]


def test_off_by_one_scan_is_rejected():
    def shifted(a, b):   # planted mistake: decay of the previous step applied
        a = np.asarray(a, np.float64)
        return olin.linscan(np.concatenate([np.ones_like(a[..., :1]), a[..., :-1]], axis=-1), b)
    with pytest.raises(AssertionError):
        P.pin_scan_brute_force(shifted, olin.combine, olin.scan_pairs, np.random.default_rng(11))
