"""GB300 (sm_103a) selective state-space forward: Mamba-2 chunked SSD and the scalar scan.

Python entry points with the names of the C ABI (include/ssm.h).  They only marshal torch
CUDA tensors into the C calls; every step of the computation runs in the library's CUDA
kernels, enqueued on the current torch stream.  PyTorch supplies device memory and streams.

    y, h_final = ssd_fwd(x, dt, A, B, C, D, h0=None, chunk=256)
    y_t, state = ssd_step(x_t, dt_t, A, B_t, C_t, D, state)     # one decode token
    h = linscan_fwd(a, b)

Importing the package does not load the library; the first call does (and fails loudly if
it cannot).
"""
from __future__ import annotations

from . import _lib
from ._lib import SSM_BF16, SSM_F32, SsmError

__all__ = ["ssd_fwd", "ssd_step", "linscan_fwd", "linscan_baseline", "tune_ssd_fwd", "set_ssd_fwd_plan",
           "get_ssd_fwd_plan", "clear_ssd_fwd_plans", "plan_id", "tune_linscan_fwd",
           "set_linscan_shape", "get_linscan_shape", "clear_linscan_shapes", "Workspace", "check_device_status", "ssd_fwd_workspace_bytes",
           "linscan_workspace_bytes", "SsmError", "version"]


def version() -> str:
    return _lib.load().ssm_version().decode()


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _stream_ptr(device):
    torch = _torch()
    return ctypes_void(torch.cuda.current_stream(device).cuda_stream)


def ctypes_void(v):
    import ctypes
    return ctypes.c_void_p(v) if v else None


def _ptr(t):
    return ctypes_void(t.data_ptr()) if t is not None else None


class Workspace:
    """Zero-initialised device scratch buffer for the C calls, grown on demand.

    The library leaves a workspace ready for reuse after every call.  One Workspace must not
    serve two calls that can run concurrently on different streams.
    """

    def __init__(self, device=None, nbytes: int = 0):
        torch = _torch()
        self.device = torch.device(device if device is not None else "cuda")
        self.buf = None
        if nbytes:
            self.ensure(nbytes)

    def ensure(self, nbytes: int):
        torch = _torch()
        if self.buf is None or self.buf.numel() < nbytes:
            # round up so that small growth does not reallocate every call
            n = max(int(nbytes), 1 << 20)
            self.buf = torch.zeros(n, dtype=torch.uint8, device=self.device)
        return self.buf

    @property
    def nbytes(self) -> int:
        return 0 if self.buf is None else self.buf.numel()

    def ptr(self):
        return _ptr(self.buf)


_default_ws = {}


def _workspace(kind: str, device, nbytes: int) -> Workspace:
    torch = _torch()
    key = (kind, torch.device(device).index)
    ws = _default_ws.get(key)
    if ws is None:
        ws = _default_ws[key] = Workspace(device)
    ws.ensure(nbytes)
    return ws


def ssd_fwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype_code) -> int:
    return int(_lib.load().ssm_ssd_fwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                                                       dtype_code))


def linscan_workspace_bytes(rows, length) -> int:
    return int(_lib.load().ssm_linscan_workspace_bytes(rows, length))


def _require(cond, msg):
    if not cond:
        raise ValueError(msg)


def ssd_fwd(x, dt, A, B, C, D, h0=None, chunk: int = 256, *, y=None, h_final=None, return_final_state=True,
            workspace: Workspace | None = None):
    """Mamba-2 chunked SSD forward on one GPU (see include/ssm.h, ssm_ssd_fwd).

    x [b, L, nh, H], dt [b, L, nh], B/C [b, L, G, S] (all float32 or all bfloat16);
    A, D [nh] float32; h0 [b, nh, H, S] float32 or None.  Returns (y, h_final) with y like x
    and h_final float32 [b, nh, H, S] (None when return_final_state is False).
    """
    torch = _torch()
    lib = _lib.load()
    code = _dtype_code(x)
    _require(x.dim() == 4 and dt.dim() == 3 and B.dim() == 4 and C.dim() == 4, "bad ranks")
    b, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    _require(tuple(dt.shape) == (b, L, nh), "dt must be [b, L, nh]")
    _require(tuple(B.shape) == (b, L, G, S) and tuple(C.shape) == (b, L, G, S), "B, C must be [b, L, G, S]")
    _require(tuple(A.shape) == (nh,) and tuple(D.shape) == (nh,), "A, D must be [nh]")
    for name, t in (("dt", dt), ("B", B), ("C", C)):
        _require(t.dtype == x.dtype, f"{name} must have x's dtype")
    _require(A.dtype == torch.float32 and D.dtype == torch.float32, "A, D must be float32")
    ts = [x, dt, A, B, C, D] + ([h0] if h0 is not None else [])
    for t in ts:
        _require(t.is_cuda and t.is_contiguous(), "all tensors must be contiguous CUDA tensors")
    if h0 is not None:
        _require(tuple(h0.shape) == (b, nh, H, S) and h0.dtype == torch.float32, "h0 must be f32 [b, nh, H, S]")
    if y is None:
        y = torch.empty_like(x)
    if return_final_state and h_final is None:
        h_final = torch.empty((b, nh, H, S), dtype=torch.float32, device=x.device)
    if not return_final_state:
        h_final = None
    need = lib.ssm_ssd_fwd_workspace_bytes(b, L, nh, H, S, G, chunk, code)
    ws = workspace if workspace is not None else _workspace("ssd", x.device, max(need, 1))
    if workspace is not None:
        ws.ensure(need)
    st = lib.ssm_ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(y),
                         _ptr(h_final), b, L, nh, H, S, G, chunk, code, ws.ptr(), ws.nbytes, _stream_ptr(x.device))
    _lib.check(st, "ssm_ssd_fwd")
    return y, h_final


def _ssd_sizes(x, B, chunk):
    b, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    return b, L, nh, H, S, G, chunk, _dtype_code(x)


def plan_id(fused: int = -1, sequential: int = -1, heads_per_cta: int = 0, fused_ring: int = 0) -> int:
    """Pack a plan for ssd_fwd (see include/ssm.h): each flag 1, 0 or -1 (rule of thumb), fused
    also 2 (the fused pass with split chains); fused_ring 1, 2 or 3 picks the fused pass's X + B
    slot split (4 + 3, 3 + 4, 5 + 2), 0 its rule."""
    return (fused + 1) | ((sequential + 1) << 2) | (heads_per_cta << 4) | (fused_ring << 20)


def tune_ssd_fwd(x, dt, A, B, C, D, h0=None, chunk: int = 256, reps: int = 5, *, y=None, h_final=None,
                 workspace: Workspace | None = None):
    """Time every plan of ssd_fwd for these sizes on these tensors and keep the fastest for later
    ssd_fwd calls of the same sizes (ssm_ssd_fwd_tune).  Returns (plan id, median ms)."""
    import ctypes
    torch = _torch()
    lib = _lib.load()
    b, L, nh, H, S, G, chunk, code = _ssd_sizes(x, B, chunk)
    if y is None:
        y = torch.empty_like(x)
    if h_final is None:
        h_final = torch.empty((b, nh, H, S), dtype=torch.float32, device=x.device)
    need = lib.ssm_ssd_fwd_workspace_bytes(b, L, nh, H, S, G, chunk, code)
    ws = workspace if workspace is not None else _workspace("ssd", x.device, max(need, 1))
    if workspace is not None:
        ws.ensure(need)
    plan = ctypes.c_int(-1)
    ms = ctypes.c_float(0.0)
    st = lib.ssm_ssd_fwd_tune(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(y),
                              _ptr(h_final), b, L, nh, H, S, G, chunk, code, ws.ptr(), ws.nbytes,
                              _stream_ptr(x.device), int(reps), ctypes.byref(plan), ctypes.byref(ms))
    _lib.check(st, "ssm_ssd_fwd_tune")
    return plan.value, ms.value


def set_ssd_fwd_plan(x, B, chunk: int, plan: int) -> None:
    """Store `plan` (-1: remove) for ssd_fwd calls with the sizes of x and B (ssm_ssd_fwd_set_plan)."""
    _lib.check(_lib.load().ssm_ssd_fwd_set_plan(*_ssd_sizes(x, B, chunk), int(plan)), "ssm_ssd_fwd_set_plan")


def get_ssd_fwd_plan(x, B, chunk: int) -> int:
    """The stored plan for these sizes, or -1 (ssm_ssd_fwd_get_plan)."""
    import ctypes
    plan = ctypes.c_int(-1)
    _lib.check(_lib.load().ssm_ssd_fwd_get_plan(*_ssd_sizes(x, B, chunk), ctypes.byref(plan)),
               "ssm_ssd_fwd_get_plan")
    return plan.value


def clear_ssd_fwd_plans() -> None:
    _lib.load().ssm_ssd_fwd_clear_plans()


def ssd_step(x, dt, A, B, C, D, state=None, *, y=None, state_out=None, inplace: bool = False):
    """Mamba-2 decode step: one new token per sequence (see include/ssm.h, ssm_ssd_step).

    x [b, nh, H], dt [b, nh], B/C [b, G, S] (all float32 or all bfloat16); A, D [nh] float32;
    state [b, nh, H, S] float32 or None (zeros).  Returns (y, new_state): y like x, new_state
    float32 [b, nh, H, S].  With ``inplace=True`` the new state overwrites ``state``.
    """
    torch = _torch()
    lib = _lib.load()
    code = _dtype_code(x)
    _require(x.dim() == 3 and dt.dim() == 2 and B.dim() == 3 and C.dim() == 3, "bad ranks")
    b, nh, H = x.shape
    G, S = B.shape[1], B.shape[2]
    _require(tuple(dt.shape) == (b, nh), "dt must be [b, nh]")
    _require(tuple(B.shape) == (b, G, S) and tuple(C.shape) == (b, G, S), "B, C must be [b, G, S]")
    _require(tuple(A.shape) == (nh,) and tuple(D.shape) == (nh,), "A, D must be [nh]")
    for name, t in (("dt", dt), ("B", B), ("C", C)):
        _require(t.dtype == x.dtype, f"{name} must have x's dtype")
    _require(A.dtype == torch.float32 and D.dtype == torch.float32, "A, D must be float32")
    for t in [x, dt, A, B, C, D] + ([state] if state is not None else []):
        _require(t.is_cuda and t.is_contiguous(), "all tensors must be contiguous CUDA tensors")
    if state is not None:
        _require(tuple(state.shape) == (b, nh, H, S) and state.dtype == torch.float32,
                 "state must be f32 [b, nh, H, S]")
    if inplace:
        _require(state is not None and state_out is None, "inplace needs a state and no state_out")
        state_out = state
    if state_out is None:
        state_out = torch.empty((b, nh, H, S), dtype=torch.float32, device=x.device)
    if y is None:
        y = torch.empty_like(x)
    st = lib.ssm_ssd_step(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state), _ptr(state_out),
                          _ptr(y), b, nh, H, S, G, code, _stream_ptr(x.device))
    _lib.check(st, "ssm_ssd_step")
    return y, state_out


def linscan_fwd(a, b, *, h=None, workspace: Workspace | None = None):
    """Scalar selective scan h[t] = a[t] h[t-1] + b[t] per row of [rows, L] float32 tensors."""
    torch = _torch()
    lib = _lib.load()
    _require(a.shape == b.shape and a.dim() == 2, "a, b must be [rows, L] and equal")
    _require(a.dtype == torch.float32 and b.dtype == torch.float32, "a, b must be float32")
    _require(a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous(), "contiguous CUDA tensors")
    rows, L = a.shape
    if h is None:
        h = torch.empty_like(a)
    need = lib.ssm_linscan_workspace_bytes(rows, L)
    ws = workspace if workspace is not None else _workspace("linscan", a.device, max(need, 1))
    if workspace is not None:
        ws.ensure(need)
    st = lib.ssm_linscan_fwd(_ptr(a), _ptr(b), _ptr(h), rows, L, ws.ptr(), ws.nbytes, _stream_ptr(a.device))
    _lib.check(st, "ssm_linscan_fwd")
    return h


def tune_linscan_fwd(a, b, *, h=None, reps: int = 5, workspace: Workspace | None = None):
    """Time every CTA shape of linscan_fwd for these sizes on these tensors and keep the fastest
    for later calls of the same sizes (ssm_linscan_fwd_tune).  Returns (shape, median ms)."""
    import ctypes
    torch = _torch()
    lib = _lib.load()
    _require(a.shape == b.shape and a.dim() == 2, "a, b must be [rows, L] and equal")
    _require(a.dtype == torch.float32 and b.dtype == torch.float32, "a, b must be float32")
    _require(a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous(), "contiguous CUDA tensors")
    rows, L = a.shape
    if h is None:
        h = torch.empty_like(a)
    need = lib.ssm_linscan_workspace_bytes(rows, L)
    ws = workspace if workspace is not None else _workspace("linscan", a.device, max(need, 1))
    if workspace is not None:
        ws.ensure(need)
    shape, ms = ctypes.c_int(-1), ctypes.c_float(0.0)
    _lib.check(lib.ssm_linscan_fwd_tune(_ptr(a), _ptr(b), _ptr(h), rows, L, ws.ptr(), ws.nbytes, _stream_ptr(a.device),
                                        int(reps), ctypes.byref(shape), ctypes.byref(ms)), "ssm_linscan_fwd_tune")
    return shape.value, ms.value


def set_linscan_shape(rows: int, length: int, shape: int) -> None:
    """Store a CTA shape (1 .. 4; -1 removes) for linscan_fwd calls of these sizes."""
    _lib.check(_lib.load().ssm_linscan_set_shape(int(rows), int(length), int(shape)), "ssm_linscan_set_shape")


def get_linscan_shape(rows: int, length: int) -> int:
    """The stored CTA shape for these sizes, or -1 (the rule applies)."""
    import ctypes
    v = ctypes.c_int(-1)
    _lib.check(_lib.load().ssm_linscan_get_shape(int(rows), int(length), ctypes.byref(v)), "ssm_linscan_get_shape")
    return v.value


def clear_linscan_shapes() -> None:
    _lib.load().ssm_linscan_clear_shapes()


SCAN_BASELINES = {"blelloch": _lib.SSM_SCAN_BLELLOCH, "three_pass": _lib.SSM_SCAN_THREE_PASS,
                  "lookback_serial": _lib.SSM_SCAN_LOOKBACK_SERIAL, "lookback_warp": _lib.SSM_SCAN_LOOKBACK_WARP,
                  "hillis_steele": _lib.SSM_SCAN_HILLIS_STEELE}


def linscan_baseline(a, b, algo: str, *, h=None, workspace: Workspace | None = None):
    """The scalar scan by one of the reference page's baseline levels (see include/ssm.h,
    ssm_linscan_baseline): "blelloch", "three_pass", "lookback_serial", "lookback_warp" or
    "hillis_steele"."""
    torch = _torch()
    lib = _lib.load()
    _require(algo in SCAN_BASELINES, f"algo must be one of {sorted(SCAN_BASELINES)}")
    code = SCAN_BASELINES[algo]
    _require(a.shape == b.shape and a.dim() == 2, "a, b must be [rows, L] and equal")
    _require(a.dtype == torch.float32 and b.dtype == torch.float32, "a, b must be float32")
    _require(a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous(), "contiguous CUDA tensors")
    rows, L = a.shape
    if h is None:
        h = torch.empty_like(a)
    need = lib.ssm_linscan_baseline_workspace_bytes(code, rows, L)
    ws = workspace if workspace is not None else _workspace("scan_" + algo, a.device, max(need, 1))
    if workspace is not None:
        ws.ensure(need)
    st = lib.ssm_linscan_baseline(code, _ptr(a), _ptr(b), _ptr(h), rows, L, ws.ptr(), ws.nbytes,
                                  _stream_ptr(a.device))
    _lib.check(st, "ssm_linscan_baseline")
    return h


def check_device_status(workspace: Workspace | None = None, kind: str = "ssd", device=None) -> int:
    """Synchronise and return (and clear) the device status word of a workspace (0 = OK)."""
    torch = _torch()
    lib = _lib.load()
    if workspace is None:
        dev = torch.device(device if device is not None else "cuda")
        workspace = _default_ws.get((kind, dev.index if dev.index is not None else torch.cuda.current_device()))
        if workspace is None:
            return 0
    return int(lib.ssm_check_device_status(workspace.ptr(), _stream_ptr(workspace.device)))


def debug_set_lookback_fault(stall_tile: int = -1, spin_limit_ns: int = 0) -> None:
    """Test hook: see ssm_debug_set_lookback_fault in include/ssm.h."""
    _lib.load().ssm_debug_set_lookback_fault(int(stall_tile), int(spin_limit_ns))


class KernelTimer:
    """Per-kernel device times of the library's launches inside a ``with`` block.

    Uses the library's own CUDA events, recorded on the stream of each launch
    (ssm_profile_begin / ssm_profile_end in include/ssm.h).  After the block, ``ms`` maps kernel
    name -> summed milliseconds and ``launches`` kernel name -> launch count.
    """

    def __init__(self, max_launches: int = 4096):
        self.max_launches = max_launches
        self.ms = {}
        self.launches = {}

    def __enter__(self):
        _lib.check(_lib.load().ssm_profile_begin(self.max_launches), "ssm_profile_begin")
        return self

    def __exit__(self, *exc):
        import ctypes
        n = len(_lib.PROFILE_KERNELS)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        _lib.check(_lib.load().ssm_profile_end(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p)),
                   "ssm_profile_end")
        self.ms = {k: float(ms[i]) for i, k in enumerate(_lib.PROFILE_KERNELS)}
        self.launches = {k: int(cnt[i]) for i, k in enumerate(_lib.PROFILE_KERNELS)}
        return False
