"""Scalar selective scan h[t] = a[t] h[t-1] + b[t], the plain definition.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): never called by the
product path.

Source: "Selective-scan CUDA kernels" (README of selective-scan-cuda),
section "The problem": the forward pass is h[t] = a[t]*h[t-1] + b[t] with
h[-1] = 0, and each step is an affine map, so the recurrence is a prefix scan
under the pair combine

    combine((a1, b1), (a2, b2)) = (a1*a2, a2*b1 + b2)

which is associative but not commutative (the left operand is the earlier
segment).
"""
from __future__ import annotations

import numpy as np


def linscan(a, b):
    """Sequential float64 scan over the last axis; rows are independent.

    a, b: arrays of identical shape [..., L].  Returns h (float64, same shape)
    with h[..., t] = a[..., t] * h[..., t-1] + b[..., t] and h[..., -1] = 0.
    """
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.shape != b.shape:
        raise ValueError("a and b must have the same shape")
    h = np.empty(a.shape)
    prev = np.zeros(a.shape[:-1])
    for t in range(a.shape[-1]):
        prev = a[..., t] * prev + b[..., t]
        h[..., t] = prev
    return h


def combine(p, q):
    """Compose two affine segments: first p = (a1, b1), then q = (a2, b2).

    Applying p then q to h gives a2*(a1*h + b1) + b2 = (a1*a2)*h + (a2*b1 + b2).
    Works on scalars, numpy arrays and fractions.Fraction values alike.
    """
    a1, b1 = p
    a2, b2 = q
    return (a1 * a2, a2 * b1 + b2)


def scan_pairs(a, b, op=combine):
    """Inclusive prefix of the pairs (a[t], b[t]) under ``op``, left to right.

    Returns the list of prefix pairs; the b-component of prefix t is h[t]
    (the a-component is the product of the decays so far).  Element type is
    whatever a and b hold (floats or fractions.Fraction), so a test can fold
    exactly.
    """
    out = []
    acc = None
    for p in zip(a, b):
        acc = p if acc is None else op(acc, p)
        out.append(acc)
    return out
