"""Mamba-2 SSD forward, the plain definition (float64, sequential in t).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): never called by the
product path.

Source: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
NVIDIA CUDA Tile" (cuTile blog post), section "Mamba-2 architecture":

    h_t = exp(a_t) h_{t-1} + b_t x_t^T,   a_t = A dt_t,   b_t = dt_t B_t
    y_t = c_t^T h_t + D x_t

with x_t of size H (per head), B_t and c_t of size S (per group), dt_t one
scalar per head and token, A and D one scalar per head, and the state a
matrix per head.

Readings taken where the post is ambiguous:
  * inclusive output: y_t reads h_t (the state after token t).  The post's
    first statement of the output uses h_{t-1}, but its chunked form, the
    no-decay expansion and the kernel's causal mask (i >= j) all use h_t.
  * the state is stored H x S (S contiguous), as the post's kernels index
    it; the prose's "S,H" is the transpose and only changes storage order.
  * dt is taken as given (positive, already passed through softplus by the
    caller); A < 0, so a_t = A dt_t < 0.
  * head h reads B/C group g = h // (nheads / ngroups).
"""
from __future__ import annotations

import numpy as np


def ssd_fwd(x, dt, A, B, C, D, h0=None):
    """Sequential float64 SSD forward.

    Args (any float dtype, upcast to float64):
      x  [batch, L, nheads, H]
      dt [batch, L, nheads]
      A  [nheads]
      B  [batch, L, ngroups, S]
      C  [batch, L, ngroups, S]
      D  [nheads]
      h0 [batch, nheads, H, S] or None (zeros)
    Returns (y [batch, L, nheads, H], h_final [batch, nheads, H, S]), float64.

    All (batch, head) units are independent; they are advanced together, one
    token at a time.
    """
    x = np.asarray(x, np.float64)
    dt = np.asarray(dt, np.float64)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    D = np.asarray(D, np.float64)
    batch, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    if nh % G:
        raise ValueError("nheads must be a multiple of ngroups")
    group_of_head = np.arange(nh) // (nh // G)
    if h0 is None:
        state = np.zeros((batch, nh, H, S))
    else:
        state = np.array(h0, np.float64).reshape(batch, nh, H, S)
    y = np.empty((batch, L, nh, H))
    for t in range(L):
        a_t = A[None, :] * dt[:, t, :]                     # [batch, nh]
        b_t = dt[:, t, :, None] * B[:, t, group_of_head]   # [batch, nh, S]
        c_t = C[:, t, group_of_head]                       # [batch, nh, S]
        x_t = x[:, t]                                      # [batch, nh, H]
        # h_t = exp(a_t) h_{t-1} + x_t (outer) b_t   (H x S storage)
        state = np.exp(a_t)[:, :, None, None] * state + x_t[:, :, :, None] * b_t[:, :, None, :]
        # y_t = h_t c_t + D x_t
        y[:, t] = np.einsum("bnps,bns->bnp", state, c_t) + D[None, :, None] * x_t
    return y, state


def ssd_step(state, x, dt, A, B, C, D):
    """One token of the recurrence with a carried state: the decode step.

    Same definition and readings as ssd_fwd (the post's section "Mamba-2
    architecture"), applied to a single new token.  The post contrasts this
    recurrent form, one state update per token, with the chunked form used
    for whole sequences; its note that the final state of one call can start
    the next is what lets a prefill hand its state to the decode loop.

    Args (any float dtype, upcast to float64):
      state [batch, nheads, H, S] or None (zeros: the first token)
      x     [batch, nheads, H]
      dt    [batch, nheads]
      A, D  [nheads]
      B, C  [batch, ngroups, S]
    Returns (y [batch, nheads, H], new state [batch, nheads, H, S]), float64:
      new state = exp(A dt) state + x (dt B)^T      (H x S per head)
      y         = new state . c + D x                (inclusive reading)
    """
    x = np.asarray(x, np.float64)
    dt = np.asarray(dt, np.float64)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    D = np.asarray(D, np.float64)
    batch, nh, H = x.shape
    G, S = B.shape[1], B.shape[2]
    if nh % G:
        raise ValueError("nheads must be a multiple of ngroups")
    group_of_head = np.arange(nh) // (nh // G)
    if state is None:
        h = np.zeros((batch, nh, H, S))
    else:
        h = np.asarray(state, np.float64).reshape(batch, nh, H, S)
    decay = np.exp(A[None, :] * dt)                        # [batch, nh]
    b = dt[:, :, None] * B[:, group_of_head]               # [batch, nh, S]
    c = C[:, group_of_head]                                # [batch, nh, S]
    h_new = decay[:, :, None, None] * h + x[:, :, :, None] * b[:, :, None, :]
    y = np.einsum("bnps,bns->bnp", h_new, c) + D[None, :, None] * x
    return y, h_new
