"""Guard canaries around every output and workspace buffer: the out-of-bounds check that stands in
for a memory sanitizer (compute-sanitizer is not available on the GPU pool).

Each output (y, h_final, the scan's h, the decode step's state and y) and each workspace is the
middle of a larger device allocation whose margins are filled with a sentinel byte; the call
goes through the C ABI with pointers to the middles.  Afterwards every margin byte must still be
the sentinel, and the outputs must match the float64 oracle.  The shapes are ragged (L = 1, 63,
65, 777, 65,537; odd head counts; chunk 64, 128 and 256; rows of one element and of one element
more than a tile), so that the tails of tiles, chunks and rows sit at the edges of the buffers,
where a store past the end would land in a margin ("Selective-scan CUDA kernels", section
"Two real bugs the tests caught": an overflow that passed for the wrong reason).
"""
import ctypes

import numpy as np
import pytest

import parity as P
from oracle import linscan as olin
from oracle import native
from oracle import ssd as ossd
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu

MARGIN = 64 << 10  # bytes on each side (16-byte alignment kept)
SENTINEL = 0xA5


class Guarded:
    """`nbytes` of device memory between two sentinel-filled margins; the middle is zeroed."""

    def __init__(self, nbytes):
        import torch
        self.nbytes = int(nbytes)
        self.buf = torch.full((MARGIN + self.nbytes + MARGIN,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.buf[MARGIN:MARGIN + self.nbytes].zero_()

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + MARGIN)

    def view(self, dtype, shape):
        return self.buf[MARGIN:MARGIN + self.nbytes].view(dtype).reshape(shape)

    def check(self, what):
        import torch
        torch.cuda.synchronize()
        lo = self.buf[:MARGIN].cpu().numpy()
        hi = self.buf[MARGIN + self.nbytes:].cpu().numpy()
        for name, m in (("before", lo), ("after", hi)):
            bad = np.nonzero(m != SENTINEL)[0]
            assert bad.size == 0, (f"{what}: {bad.size} margin bytes {name} the buffer changed, first at offset "
                                   f"{int(bad[0]) - (MARGIN if name == 'before' else 0)}")


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


SSD_SHAPES = [
    # (name, b, L, nh, H, S, G, T, dtype)
    ("f32_L1_T64", 1, 1, 3, 64, 64, 1, 64, "f32"),
    ("f32_L63_T64_G2", 2, 63, 2, 64, 128, 2, 64, "f32"),
    ("f32_L65_T128_nh5_G5", 1, 65, 5, 64, 64, 5, 128, "f32"),
    ("f32_L777_T256_nh6_G2", 2, 777, 6, 64, 128, 2, 256, "f32"),
    ("f32_L65537_T256", 1, 65537, 2, 64, 64, 1, 256, "f32"),
    ("bf16_L1_T256", 1, 1, 4, 64, 128, 1, 256, "bf16"),
    ("bf16_L63_T128_G2", 2, 63, 4, 64, 128, 2, 128, "bf16"),
    ("bf16_L65_T64", 1, 65, 2, 64, 64, 1, 64, "bf16"),
    ("bf16_L777_T256_nh3", 2, 777, 3, 64, 128, 1, 256, "bf16"),
    ("bf16_L777_T128_nh9_G3", 1, 777, 9, 64, 128, 3, 128, "bf16"),
    ("bf16_L65537_T256_nh4", 1, 65537, 4, 64, 128, 1, 256, "bf16"),
]


@pytest.mark.parametrize("spec", SSD_SHAPES, ids=lambda s: s[0])
def test_ssd_fwd_outputs_and_workspace_guarded(cuda_lib, spec):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    name, b, L, nh, H, S, G, T, dtype = spec
    shape = synth.SSDShape(name, b, L, nh, H, S, G, T, dtype, h0=True)
    inp = synth.ssd_inputs(shape, seed=7 + L % 97)
    x, dt, B, C = (P.to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C"))
    A, D, h0 = P.to_dev(inp["A"]), P.to_dev(inp["D"]), P.to_dev(inp["h0"])
    code = _lib.SSM_BF16 if dtype == "bf16" else _lib.SSM_F32
    lib = _lib.load()
    wsb = lib.ssm_ssd_fwd_workspace_bytes(b, L, nh, H, S, G, T, code)
    y = Guarded(x.numel() * x.element_size())
    hf = Guarded(b * nh * H * S * 4)
    ws = Guarded(wsb)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for call in range(2):  # a second call reuses the workspace as the first left it
        st = lib.ssm_ssd_fwd(p(x), p(dt), p(A), p(B), p(C), p(D), p(h0), y.ptr(), hf.ptr(), b, L, nh, H, S, G, T,
                             code, ws.ptr(), wsb, _stream())
        assert st == _lib.SSM_OK
        for g, what in ((y, "y"), (hf, "h_final"), (ws, "workspace")):
            g.check(f"{name} call {call} {what}")
        assert lib.ssm_check_device_status(ws.ptr(), _stream()) == _lib.SSM_OK
    y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"]) \
        if b * L * nh <= 200000 else native.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                                     inp["h0"])
    if y_ref.shape != (b, L, nh, H):  # the C oracle returns [units, L, H]
        y_ref = y_ref.reshape(b, nh, L, H).transpose(0, 2, 1, 3)
        hf_ref = hf_ref.reshape(b, nh, H, S)
    ty = torch.bfloat16 if dtype == "bf16" else torch.float32
    P.assert_ssd_close(dtype, P.to_np(y.view(ty, (b, L, nh, H))), y_ref, P.to_np(hf.view(torch.float32, (b, nh, H, S))),
                       hf_ref, name)


@pytest.mark.parametrize("rows,length", [(3, 1), (5, 4095), (4, 4097), (2, 65537), (384, 1000), (1, 1 << 20)])
def test_linscan_output_and_workspace_guarded(cuda_lib, rows, length):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    lib = _lib.load()
    inp = synth.scan_inputs(rows, length, seed=rows + length)
    a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    wsb = lib.ssm_linscan_workspace_bytes(rows, length)
    h = Guarded(rows * length * 4)
    ws = Guarded(wsb)
    for call in range(2):
        st = lib.ssm_linscan_fwd(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), h.ptr(), rows, length,
                                 ws.ptr(), wsb, _stream())
        assert st == _lib.SSM_OK
        h.check(f"{rows}x{length} call {call} h")
        ws.check(f"{rows}x{length} call {call} workspace")
        assert lib.ssm_check_device_status(ws.ptr(), _stream()) == _lib.SSM_OK
    ref = native.linscan(inp["a"], inp["b"]) if rows * length > 100000 else olin.linscan(inp["a"], inp["b"])
    P.assert_rows_close(P.to_np(h.view(torch.float32, (rows, length))), ref, f"linscan {rows}x{length}")


@pytest.mark.parametrize("algo", ["blelloch", "three_pass", "lookback_serial", "lookback_warp", "hillis_steele"])
def test_scan_baselines_output_and_workspace_guarded(cuda_lib, algo):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    import selective_state_space_mamba_gb300 as ssm
    lib = _lib.load()
    rows, length = (5, 2047) if algo == "blelloch" else (3, 2 * 2048 + 257)
    inp = synth.scan_inputs(rows, length, seed=11)
    a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    code = ssm.SCAN_BASELINES[algo]
    wsb = lib.ssm_linscan_baseline_workspace_bytes(code, rows, length)
    h = Guarded(rows * length * 4)
    ws = Guarded(max(wsb, 16))
    st = lib.ssm_linscan_baseline(code, ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), h.ptr(), rows,
                                  length, ws.ptr(), wsb, _stream())
    assert st == _lib.SSM_OK
    h.check(f"{algo} h")
    ws.check(f"{algo} workspace")
    P.assert_rows_close(P.to_np(h.view(torch.float32, (rows, length))), olin.linscan(inp["a"], inp["b"]), algo)


@pytest.mark.parametrize("dtype,nh,G,H,S", [("bf16", 5, 5, 64, 128), ("f32", 3, 1, 48, 64), ("bf16", 80, 1, 64, 128)])
def test_decode_step_outputs_guarded(cuda_lib, dtype, nh, G, H, S):
    import torch
    from selective_state_space_mamba_gb300 import _lib
    lib = _lib.load()
    shape = synth.StepShape(f"guard_step_{dtype}_{nh}", 3, nh, H, S, G, dtype)
    inp = synth.step_inputs(shape, seed=13)
    x, dt, B, C = (P.to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C"))
    A, D, state = P.to_dev(inp["A"]), P.to_dev(inp["D"]), P.to_dev(inp["state"])
    code = _lib.SSM_BF16 if dtype == "bf16" else _lib.SSM_F32
    y = Guarded(x.numel() * x.element_size())
    so = Guarded(state.numel() * 4)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.ssm_ssd_step(p(x), p(dt), p(A), p(B), p(C), p(D), p(state), so.ptr(), y.ptr(), 3, nh, H, S, G, code,
                          _stream())
    assert st == _lib.SSM_OK
    y.check("step y")
    so.check("step state_out")
    y_ref, h_ref = ossd.ssd_step(inp["state"], inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"])
    ty = torch.bfloat16 if dtype == "bf16" else torch.float32
    got_y = P.to_np(y.view(ty, tuple(x.shape)))
    got_h = P.to_np(so.view(torch.float32, tuple(state.shape)))
    nhg = np.arange(nh) // (nh // G)
    P.assert_step_close(dtype, got_y, y_ref, got_h, h_ref, inp["state"], inp["C"][:, nhg],
                        inp["D"][None, :, None].astype(np.float64) * inp["x"], "guarded step")
