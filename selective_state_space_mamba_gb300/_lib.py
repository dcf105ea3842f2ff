"""ctypes view of the C ABI in include/ssm.h (libssm_gb300.so, built in-tree).

Argument marshalling only: every step of the computation runs in the CUDA library.  Loading
fails loudly when the library is missing and cannot be built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_ALIGNMENT, SSM_ERR_WORKSPACE, SSM_ERR_CUDA, \
    SSM_ERR_TIMEOUT, SSM_ERR_BOUNDS = range(8)
SSM_F32, SSM_BF16 = 0, 1
SSM_SCAN_BLELLOCH, SSM_SCAN_THREE_PASS, SSM_SCAN_LOOKBACK_SERIAL, SSM_SCAN_LOOKBACK_WARP, SSM_SCAN_HILLIS_STEELE = \
    1, 2, 3, 4, 5

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("ssm_status_string", "ssm_version", "ssm_ssd_fwd_workspace_bytes", "ssm_ssd_fwd",
           "ssm_linscan_workspace_bytes", "ssm_linscan_fwd", "ssm_check_device_status",
           "ssm_debug_set_lookback_fault", "ssm_profile_begin", "ssm_profile_end", "ssm_linscan_fwd_noalloc",
           "ssm_ssd_step", "ssm_linscan_baseline_workspace_bytes", "ssm_linscan_baseline", "ssm_ssd_fwd_tune",
           "ssm_ssd_fwd_set_plan", "ssm_ssd_fwd_get_plan", "ssm_ssd_fwd_clear_plans", "ssm_debug_fused_schedule",
           "ssm_debug_scan_schedule",
           "ssm_debug_build", "ssm_debug_set_bounds_fault", "ssm_linscan_fwd_tune", "ssm_linscan_set_shape",
           "ssm_linscan_get_shape", "ssm_linscan_clear_shapes")
PROFILE_KERNELS = ("linscan_lookback", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
                   "ssd_state_fused", "ssd_step", "linscan_baseline", "ssd_state_fixup")

_lib = None
_lock = threading.Lock()


class SsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def _declare(lib):
    vp, i64, u64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
    lib.ssm_status_string.argtypes = [i32]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_version.argtypes = []
    lib.ssm_version.restype = ctypes.c_char_p
    lib.ssm_ssd_fwd_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, i32, i32, i32]
    lib.ssm_ssd_fwd_workspace_bytes.restype = sz
    lib.ssm_ssd_fwd.argtypes = [vp] * 9 + [i64, i64, i32, i32, i32, i32, i32, i32, vp, sz, vp]
    lib.ssm_ssd_fwd.restype = i32
    lib.ssm_ssd_fwd_tune.argtypes = [vp] * 9 + [i64, i64, i32, i32, i32, i32, i32, i32, vp, sz, vp, i32, vp, vp]
    lib.ssm_ssd_fwd_tune.restype = i32
    lib.ssm_debug_fused_schedule.argtypes = [i64, i64, i32, i32, vp, i64]
    lib.ssm_debug_fused_schedule.restype = i64
    lib.ssm_debug_scan_schedule.argtypes = [i64, i32, i32, i32, i32, vp]
    lib.ssm_debug_scan_schedule.restype = i64
    lib.ssm_ssd_fwd_set_plan.argtypes = [i64, i64, i32, i32, i32, i32, i32, i32, i32]
    lib.ssm_ssd_fwd_set_plan.restype = i32
    lib.ssm_ssd_fwd_get_plan.argtypes = [i64, i64, i32, i32, i32, i32, i32, i32, vp]
    lib.ssm_ssd_fwd_get_plan.restype = i32
    lib.ssm_ssd_fwd_clear_plans.argtypes = []
    lib.ssm_ssd_fwd_clear_plans.restype = None
    lib.ssm_ssd_step.argtypes = [vp] * 9 + [i64, i32, i32, i32, i32, i32, vp]
    lib.ssm_ssd_step.restype = i32
    lib.ssm_linscan_baseline_workspace_bytes.argtypes = [i32, i64, i64]
    lib.ssm_linscan_baseline_workspace_bytes.restype = sz
    lib.ssm_linscan_baseline.argtypes = [i32, vp, vp, vp, i64, i64, vp, sz, vp]
    lib.ssm_linscan_baseline.restype = i32
    lib.ssm_linscan_workspace_bytes.argtypes = [i64, i64]
    lib.ssm_linscan_workspace_bytes.restype = sz
    lib.ssm_linscan_fwd.argtypes = [vp, vp, vp, i64, i64, vp, sz, vp]
    lib.ssm_linscan_fwd.restype = i32
    lib.ssm_linscan_fwd_tune.argtypes = [vp, vp, vp, i64, i64, vp, sz, vp, i32, vp, vp]
    lib.ssm_linscan_fwd_tune.restype = i32
    lib.ssm_linscan_set_shape.argtypes = [i64, i64, i32]
    lib.ssm_linscan_set_shape.restype = i32
    lib.ssm_linscan_get_shape.argtypes = [i64, i64, vp]
    lib.ssm_linscan_get_shape.restype = i32
    lib.ssm_linscan_clear_shapes.argtypes = []
    lib.ssm_linscan_clear_shapes.restype = None
    lib.ssm_check_device_status.argtypes = [vp, vp]
    lib.ssm_check_device_status.restype = i32
    lib.ssm_debug_set_lookback_fault.argtypes = [i64, u64]
    lib.ssm_debug_set_lookback_fault.restype = None
    lib.ssm_debug_build.argtypes = []
    lib.ssm_debug_build.restype = i32
    lib.ssm_debug_set_bounds_fault.argtypes = [i64]
    lib.ssm_debug_set_bounds_fault.restype = i32
    lib.ssm_linscan_fwd_noalloc.argtypes = [vp, vp, vp, i64, i64, vp]
    lib.ssm_linscan_fwd_noalloc.restype = i32
    lib.ssm_profile_begin.argtypes = [i32]
    lib.ssm_profile_begin.restype = i32
    lib.ssm_profile_end.argtypes = [vp, vp]
    lib.ssm_profile_end.restype = i32


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the CUDA library (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing:
                try:
                    path = _build.build()
                except Exception as e:  # noqa: BLE001 - re-raised with context
                    if not os.path.exists(_build.LIB):
                        raise RuntimeError(f"CUDA library {_build.LIB} is missing and could not be built: {e}") from e
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing (run __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib = lib
    return _lib


_lib_debug = None


def load_debug():
    """Load the debug library (libssm_gb300_debug.so: the same kernels with device index checks,
    built by __graft_entry__.build()), building it first if it is missing or stale.  It is a
    separate library with its own state; only the tests use it."""
    global _lib_debug
    with _lock:
        if _lib_debug is None:
            path = _build.build(debug=True)
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib_debug = lib
    return _lib_debug


def status_string(status: int) -> str:
    return load().ssm_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != SSM_OK:
        raise SsmError(status, where)
