"""The allocation-free scan entry point (ssm_linscan_fwd_noalloc) against the regular one and the
float64 oracle.

Some callers cannot allocate device memory while they run: a framework that reserves all of
its device memory up front, a real-time loop that cannot take the implicit device
synchronisation of cudaMalloc / cudaFree, or a host with no allocator to provide a workspace.
For them the library keeps the scan's scratch in a fixed device array of its own.  This test
calls that entry point through the C ABI, twice in a row on different problems (so the second
call starts from whatever the first left in the shared scratch), and compares each result with
ssm_linscan_fwd's and with the oracle's under the scan's float32 tolerance.  Bit equality with
ssm_linscan_fwd is not required: the look-back combines a tile's predecessors up to the nearest
one whose prefix is already published, so the association, and with it the rounding, can differ
from run to run.  The largest accepted scan (rows * len = 2^26) runs too, with no change in the
device memory in use around the call; one element more is refused without launching anything.

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


def test_noalloc_matches_workspace_entry_point_and_oracle_twice(cuda_lib):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from oracle import native
    from selective_state_space_mamba_gb300 import _lib
    for rows, length, seed in [(384, 65536, 31), (5, 3 * 4096 + 17, 32)]:
        inp = synth.scan_inputs(rows, length, seed=seed)
        a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
        want = P.to_np(ssm.linscan_fwd(a, b))
        assert ssm.check_device_status(kind="linscan") == 0
        h = torch.full_like(a, float("nan"))
        assert _noalloc(cuda_lib, a, b, h) == _lib.SSM_OK
        got = P.to_np(h)
        P.assert_rows_close(got, want, f"noalloc {rows}x{length} vs ssm_linscan_fwd")
        P.assert_rows_close(got, native.linscan(inp["a"], inp["b"]), f"noalloc {rows}x{length} vs oracle")


def test_noalloc_largest_size_allocates_nothing(cuda_lib):
    """rows * len = 2^26 exactly, rows of a ragged length (16 x 4,194,304 = 2^26; 1024 x 65536
    also 2^26): the result matches ssm_linscan_fwd's, and the device memory in use (the
    driver's free-memory count and torch's allocator) does not change around a call."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    for rows, length, seed in [(1024, 65536, 33), (16, 1 << 22, 34)]:
        assert rows * length == MAX_ELEMS
        inp = synth.scan_inputs(rows, length, seed=seed)
        a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
        want = P.to_np(ssm.linscan_fwd(a, b))
        h = torch.full_like(a, float("nan"))
        assert _noalloc(cuda_lib, a, b, h) == _lib.SSM_OK  # a first call may load the device code
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        h.fill_(float("nan"))
        assert _noalloc(cuda_lib, a, b, h) == _lib.SSM_OK
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
        P.assert_rows_close(P.to_np(h), want, f"noalloc {rows}x{length}")
        del a, b, h


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
