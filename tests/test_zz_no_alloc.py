"""The allocation-free scan entry point (ssm_linscan_fwd_noalloc) against the regular one.

Some callers cannot allocate device memory while they run: a framework that reserves all of
its device memory up front, a real-time loop that cannot take the implicit device
synchronisation of cudaMalloc / cudaFree, or a host with no allocator to provide a workspace.
For them the library keeps the scan's scratch in a fixed device array of its own.  This test
calls that entry point through the C ABI, twice in a row on different problems (so the second
call starts from whatever the first left in the shared scratch), and compares each result
with ssm_linscan_fwd's under the scan's float32 tolerance.  It also checks that a scan larger
than the fixed scratch is refused without launching anything.

Named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import parity as P
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_ELEMS = 1 << 26


def _noalloc(lib, a, b, h):
    import torch
    rows, length = a.shape
    st = lib.ssm_linscan_fwd_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                     ctypes.c_void_p(h.data_ptr()), rows, length,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    for rows, length, seed in [(384, 65536, 31), (5, 3 * 4096 + 17, 32)]:
        inp = synth.scan_inputs(rows, length, seed=seed)
        a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
        want = P.to_np(ssm.linscan_fwd(a, b))
        assert ssm.check_device_status(kind="linscan") == 0
        h = torch.full_like(a, float("nan"))
        assert _noalloc(cuda_lib, a, b, h) == _lib.SSM_OK
        P.assert_rows_close(P.to_np(h), want, f"noalloc {rows}x{length}")


def test_noalloc_refuses_oversize_and_accepts_empty(cuda_lib):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    x = torch.zeros(16, device="cuda")
    big_rows = MAX_ELEMS // 1024 + 1
    st = cuda_lib.ssm_linscan_fwd_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                          ctypes.c_void_p(x.data_ptr()), big_rows, 1024, None)
    assert st == _lib.SSM_ERR_UNSUPPORTED
    assert cuda_lib.ssm_linscan_fwd_noalloc(None, None, None, 0, 10, None) == _lib.SSM_OK
    assert cuda_lib.ssm_linscan_fwd_noalloc(None, None, None, -1, 10, None) == _lib.SSM_ERR_INVALID_ARG
