"""Shared helpers of the GPU parity tests: device transfer and the tolerance rules.

Tolerances (fixed for this method, written here once):
  float32 workloads: max |GPU - oracle| <= 1e-4 * max |oracle|, per output tensor (the scan:
    per row).  Relative error is undefined at zero crossings, so "max relative error 1e-4"
    is read normwise.
  bf16-input workloads (float32 accumulation): |dy| <= 2e-2 * RMS(y_oracle) + 2^-8 |y_oracle|
    per element, and max |dh_final| <= 1e-2 * RMS(h_final_oracle).  y is returned in bf16 (the
    inputs' dtype), whose own rounding alone moves an element by up to 2^-8 of its size: more
    than 2e-2 * RMS wherever |y| exceeds about 5 RMS (an element of -8.03 at RMS 1.02 rounds to
    -8.0), so the stated 2e-2 * RMS bounds the computation and the output's rounding is added.
    h_final is float32 and has no such term.
"""
from __future__ import annotations

import numpy as np

F32_RTOL = 1e-4
BF16_Y_RMS = 2e-2
BF16_H_RMS = 1e-2
BF16_OUT_U = 2.0 ** -8  # unit roundoff of a bf16 output (8 significand bits, round to nearest)


def to_dev(arr, dtype="f32", device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def err_report(got, ref):
    d = np.abs(np.asarray(got, np.float64) - ref)
    i = np.unravel_index(int(np.argmax(d)), d.shape) if d.size else ()
    return d, i


def assert_f32_close(got, ref, what):
    if ref.size == 0:
        return
    d, i = err_report(got, ref)
    scale = float(np.max(np.abs(ref)))
    assert d[i] <= F32_RTOL * scale or d[i] == 0.0, (
        f"{what}: max|d|={d[i]:.3e} at {i} (gpu {np.asarray(got)[i]!r}, oracle {ref[i]!r}) > 1e-4*{scale:.3e}")


def assert_rows_close(got, ref, what):
    """Per-row normwise float32 rule for the scan: max_t |got - ref| <= 1e-4 max_t |ref| per row."""
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    d = np.abs(np.asarray(got, np.float64) - ref).reshape(ref.shape[0], -1)
    scale = np.max(np.abs(ref), axis=1) if ref.ndim > 1 else np.abs(ref)
    dmax = d.max(axis=1)
    bad = ~((dmax <= F32_RTOL * scale) | (dmax == 0.0))
    if bad.any():
        r = int(np.argmax(bad))
        assert_f32_close(np.asarray(got)[r], ref[r], f"{what} row {r}")


def assert_bf16_close(got, ref, what, rms_tol, out_u=0.0):
    """max |got - ref| - out_u |ref| <= rms_tol * RMS(ref): out_u is the output format's unit
    roundoff (BF16_OUT_U for a bf16 output, 0 for a float32 one)."""
    if ref.size == 0:
        return
    ref = np.asarray(ref, np.float64)
    d = np.abs(np.asarray(got, np.float64) - ref) - out_u * np.abs(ref)
    i = np.unravel_index(int(np.argmax(d)), d.shape)
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert d[i] <= rms_tol * rms, (
        f"{what}: |d| - {out_u:.3g}|ref| = {d[i]:.3e} at {i} (gpu {np.asarray(got)[i]!r}, oracle {ref[i]!r}) > "
        f"{rms_tol}*RMS {rms:.3e}")


def assert_ssd_close(dtype, y, y_ref, hf, hf_ref, what):
    if dtype == "f32":
        assert_f32_close(y, y_ref, f"{what} y")
        if hf_ref is not None:
            assert_f32_close(hf, hf_ref, f"{what} h_final")
    else:
        assert_bf16_close(y, y_ref, f"{what} y", BF16_Y_RMS, BF16_OUT_U)
        if hf_ref is not None:
            assert_bf16_close(hf, hf_ref, f"{what} h_final", BF16_H_RMS)


def assert_step_close(dtype, y, y_ref, h, h_ref, h_in, c_heads, dx, what):
    """Per-element rule for the decode step, from its arithmetic (all f32, one token):

    state: each element is one fma of exp(A dt) h and dt x B (dt x B is exact in f32 for bf16
      inputs); with expf within a few ulp, |dh| <= 2e-6 * scale_h, scale_h = max(|h_ref|, |h_in|).
    y: a 128-term f32 dot product (a 4-term chain and a 5-level tree) of the new state with c,
      plus D x: |dy_i| <= 1e-5 * (sum_s |h_ref[i,s] c_s| + scale_h sum_s |c_s| + |D x_i|), and
      for bf16 output also the rounding to bf16, u = 2^-8: + 2^-8 |y_ref_i| (each term x 1.01).
    c_heads [b, nh, S] is C per head (its group's row), dx [b, nh, H] is D x.
    """
    h_ref = np.asarray(h_ref, np.float64)
    scale_h = max(float(np.max(np.abs(h_ref))) if h_ref.size else 0.0,
                  float(np.max(np.abs(h_in))) if h_in is not None and np.size(h_in) else 0.0, 1e-30)
    dh = np.abs(np.asarray(h, np.float64) - h_ref)
    if dh.size:
        i = np.unravel_index(int(np.argmax(dh)), dh.shape)
        assert dh[i] <= 2e-6 * scale_h, f"{what}: state max|d|={dh[i]:.3e} at {i} > 2e-6*{scale_h:.3e}"
    ca = np.abs(np.asarray(c_heads, np.float64))
    tol = 1e-5 * (np.einsum("bnps,bns->bnp", np.abs(h_ref), ca) + scale_h * ca.sum(-1)[..., None]
                  + np.abs(np.asarray(dx, np.float64)))
    if dtype == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(np.asarray(y_ref, np.float64))
    tol = 1.01 * tol
    dy = np.abs(np.asarray(y, np.float64) - np.asarray(y_ref, np.float64))
    bad = dy > tol
    if bad.any():
        i = np.unravel_index(int(np.argmax(dy - tol)), dy.shape)
        raise AssertionError(f"{what}: y |d|={dy[i]:.3e} at {i} (gpu {np.asarray(y)[i]!r}, oracle "
                             f"{np.asarray(y_ref)[i]!r}) > bound {tol[i]:.3e}; {int(bad.sum())} elements over")
