"""The debug library (libssm_gb300_debug.so, compiled with -DSSM_DEBUG): the same kernels with their
device index checks compiled in, the stand-in for a memory sanitizer on a pool where
compute-sanitizer is not available.  A failed check records SSM_ERR_BOUNDS in the call's status
word and skips the access; nothing traps.

The ragged shapes of the guard tests run through the debug library: every check must pass
(status SSM_OK) and the outputs must match the float64 oracle.  The test hook
ssm_debug_set_bounds_fault then makes one check fail on purpose (the chunk cumsum's store bound
is lowered by a few elements, so the stores it rejects are in-bounds ones that are simply
skipped), and the status word must report SSM_ERR_BOUNDS.
"""
import ctypes

import numpy as np
import pytest

import parity as P
from oracle import linscan as olin
from oracle import ssd as ossd
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    from selective_state_space_mamba_gb300 import _lib
    lib = _lib.load_debug()
    assert lib.ssm_debug_build() == 1
    return lib


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def run_ssd(lib, inp, shape):
    """One forward through the given library; returns (status word, y, h_final) on the host."""
    import torch
    from selective_state_space_mamba_gb300 import _lib
    b, L, nh, H, S, G, T = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.chunk
    x, dt, B, C = (P.to_dev(inp[k], shape.dtype) for k in ("x", "dt", "B", "C"))
    A, D, h0 = P.to_dev(inp["A"]), P.to_dev(inp["D"]), P.to_dev(inp["h0"])
    code = _lib.SSM_BF16 if shape.dtype == "bf16" else _lib.SSM_F32
    wsb = lib.ssm_ssd_fwd_workspace_bytes(b, L, nh, H, S, G, T, code)
    ws = torch.zeros(max(wsb, 1), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    hf = torch.empty((b, nh, H, S), dtype=torch.float32, device="cuda")
    st = lib.ssm_ssd_fwd(_p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(h0), _p(y), _p(hf), b, L, nh, H, S, G, T, code,
                         _p(ws), wsb, _stream())
    assert st == _lib.SSM_OK
    dev_status = lib.ssm_check_device_status(_p(ws), _stream())
    return dev_status, P.to_np(y), P.to_np(hf)


SHAPES = [
    ("f32_L63_T64_G2", 2, 63, 2, 64, 128, 2, 64, "f32"),
    ("f32_L777_T256_nh6_G2", 2, 777, 6, 64, 128, 2, 256, "f32"),
    ("bf16_L1_T256", 1, 1, 4, 64, 128, 1, 256, "bf16"),
    ("bf16_L65_T64", 1, 65, 2, 64, 64, 1, 64, "bf16"),
    ("bf16_L777_T256_nh3", 2, 777, 3, 64, 128, 1, 256, "bf16"),
    ("bf16_L777_T128_nh9_G3", 1, 777, 9, 64, 128, 3, 128, "bf16"),
    ("bf16_L2000_T256_nh4_fused", 2, 2000, 4, 64, 128, 1, 256, "bf16"),
]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s[0])
def test_debug_build_ssd_checks_pass(cuda_lib, dbg, spec):
    from selective_state_space_mamba_gb300 import _lib
    name, b, L, nh, H, S, G, T, dtype = spec
    shape = synth.SSDShape(name, b, L, nh, H, S, G, T, dtype, h0=True)
    inp = synth.ssd_inputs(shape, seed=3 + L % 89)
    status, y, hf = run_ssd(dbg, inp, shape)
    assert status == _lib.SSM_OK, _lib.status_string(status)
    y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    P.assert_ssd_close(dtype, y, y_ref, hf, hf_ref, f"debug build {name}")


def test_debug_build_scan_checks_pass(cuda_lib, dbg):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    for rows, length in [(3, 1), (4, 4097), (2, 65537)]:
        inp = synth.scan_inputs(rows, length, seed=rows)
        a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
        h = torch.empty_like(a)
        wsb = dbg.ssm_linscan_workspace_bytes(rows, length)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        assert dbg.ssm_linscan_fwd(_p(a), _p(b), _p(h), rows, length, _p(ws), wsb, _stream()) == _lib.SSM_OK
        assert dbg.ssm_check_device_status(_p(ws), _stream()) == _lib.SSM_OK
        P.assert_rows_close(P.to_np(h), olin.linscan(inp["a"], inp["b"]), f"debug build scan {rows}x{length}")


def test_debug_build_reports_a_failed_check(cuda_lib, dbg):
    from selective_state_space_mamba_gb300 import _lib
    shape = synth.SSDShape("bounds_hook", 1, 300, 2, 64, 64, 1, 64, "f32", h0=True)
    inp = synth.ssd_inputs(shape, seed=17)
    assert dbg.ssm_debug_set_bounds_fault(3) == _lib.SSM_OK
    try:
        status, _, _ = run_ssd(dbg, inp, shape)
    finally:
        assert dbg.ssm_debug_set_bounds_fault(0) == _lib.SSM_OK
    assert status == _lib.SSM_ERR_BOUNDS, _lib.status_string(status)
    status, y, hf = run_ssd(dbg, inp, shape)  # the hook off again: clean
    assert status == _lib.SSM_OK
    y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    P.assert_ssd_close("f32", y, y_ref, hf, hf_ref, "after the hook")


def test_release_build_has_no_checks(cuda_lib):
    from selective_state_space_mamba_gb300 import _lib
    lib = _lib.load()
    assert lib.ssm_debug_build() == 0
    assert lib.ssm_debug_set_bounds_fault(1) == _lib.SSM_ERR_UNSUPPORTED
