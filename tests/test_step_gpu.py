"""GPU parity of the decode step (ssm_ssd_step, through the C ABI) against the float64 oracle.

Small shapes (both dtypes, both state sizes, head sizes 16..256, grouped B/C, with and without
a carried state, in place) are compared on every output with the per-element rule derived in
parity.assert_step_close; so is the full decode workload (b128 nh80 H64 S128 bf16, the launch
the benchmark times).  A prefill by ssd_fwd followed by decode steps
is compared with the oracle's forward over all tokens.
"""
import zlib

import numpy as np
import pytest

import parity as P
from oracle import ssd as ossd
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu


def gpu_step(inp, dtype, state=True, inplace=False):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    x, dt, B, C = (P.to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C"))
    A, D = P.to_dev(inp["A"]), P.to_dev(inp["D"])
    st = P.to_dev(inp["state"]) if state else None
    y, h = ssm.ssd_step(x, dt, A, B, C, D, st, inplace=inplace)
    if inplace:
        assert h.data_ptr() == st.data_ptr()
    torch.cuda.synchronize()
    return P.to_np(y), P.to_np(h)


def per_head(arr_g, nh):
    """[b, G, S] -> [b, nh, S]: each head's group row (head h reads group h // (nh / G))."""
    G = arr_g.shape[1]
    return arr_g[:, np.arange(nh) // (nh // G)]


def check(dtype, inp, y, h, what, state=True):
    h_in = inp["state"] if state else None
    y_ref, h_ref = ossd.ssd_step(h_in, inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"])
    nh = inp["x"].shape[1]
    dx = inp["D"][None, :, None].astype(np.float64) * inp["x"]
    P.assert_step_close(dtype, y, y_ref, h, h_ref, h_in, per_head(inp["C"], nh), dx, what)


SHAPES = []
for dtype in ("f32", "bf16"):
    for (b, nh, G, H, S) in [(1, 2, 1, 64, 128), (3, 6, 2, 64, 64), (2, 4, 4, 16, 128), (2, 3, 1, 80, 64),
                             (5, 8, 2, 256, 128), (7, 5, 5, 48, 64)]:
        SHAPES.append(synth.StepShape(f"step_{dtype}_b{b}_nh{nh}_G{G}_H{H}_S{S}", b, nh, H, S, G, dtype))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_step_small_all_outputs(cuda_lib, shape):
    inp = synth.step_inputs(shape, seed=zlib.crc32(shape.name.encode()) & 0xFFFF)
    y, h = gpu_step(inp, shape.dtype)
    check(shape.dtype, inp, y, h, shape.name)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_zero_state_and_in_place(cuda_lib, dtype):
    shape = synth.StepShape("step_edge", 3, 6, 64, 128, 3, dtype)
    inp = synth.step_inputs(shape, seed=31)
    y, h = gpu_step(inp, dtype, state=False)
    check(dtype, inp, y, h, "state None (zeros)", state=False)
    y, h = gpu_step(inp, dtype, inplace=True)
    check(dtype, inp, y, h, "in place")


def test_step_dt_zero_keeps_state_exactly(cuda_lib):
    # dt = 0: decay exp(0) = 1 and no input, so the f32 state comes back bit for bit
    shape = synth.StepShape("step_dt0", 2, 4, 64, 128, 2, "bf16")
    inp = synth.step_inputs(shape, seed=32)
    inp["dt"] = np.zeros_like(inp["dt"])
    y, h = gpu_step(inp, "bf16")
    assert np.array_equal(h, inp["state"].astype(np.float64))
    check("bf16", inp, y, h, "dt = 0")


def test_step_full_workload_every_unit(cuda_lib):
    shape = synth.STEP_B128
    inp = synth.step_inputs(shape)
    y, h = gpu_step(inp, shape.dtype)
    assert np.isfinite(y).all() and np.isfinite(h).all()
    # every (batch, head) unit, 16 sequences at a time (the rule is per element)
    for b0 in range(0, shape.batch, 16):
        sl = slice(b0, min(shape.batch, b0 + 16))
        sub = {k: inp[k][sl] for k in ("x", "dt", "B", "C", "state")}
        sub.update(A=inp["A"], D=inp["D"])
        check(shape.dtype, sub, y[sl], h[sl], f"{shape.name} batch {b0}..")


def test_step_deterministic(cuda_lib):
    shape = synth.StepShape("step_det", 4, 8, 64, 128, 2, "bf16")
    inp = synth.step_inputs(shape, seed=33)
    y1, h1 = gpu_step(inp, "bf16")
    y2, h2 = gpu_step(inp, "bf16")
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


def test_step_batch_zero(cuda_lib):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    dev = "cuda"
    x = torch.empty((0, 4, 64), device=dev)
    y, h = ssm.ssd_step(x, torch.empty((0, 4), device=dev), torch.zeros(4, device=dev),
                        torch.empty((0, 1, 128), device=dev), torch.empty((0, 1, 128), device=dev),
                        torch.zeros(4, device=dev))
    assert y.shape == (0, 4, 64) and h.shape == (0, 4, 64, 128)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode_equals_forward(cuda_lib, dtype):
    """ssd_fwd over a prompt hands its final state to ssd_step; the decode outputs and the final
    state match the oracle's forward over prompt + decoded tokens."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    L0, K = 300, 6
    shape = synth.SSDShape(f"prefill_{dtype}", 2, L0 + K, 4, 64, 128, 2, 128, dtype, h0=True)
    inp = synth.ssd_inputs(shape, seed=41)
    dev = {k: P.to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C")}
    A, D, h0 = P.to_dev(inp["A"]), P.to_dev(inp["D"]), P.to_dev(inp["h0"])
    _, state = ssm.ssd_fwd(dev["x"][:, :L0].contiguous(), dev["dt"][:, :L0].contiguous(), A,
                           dev["B"][:, :L0].contiguous(), dev["C"][:, :L0].contiguous(), D, h0, chunk=shape.chunk)
    ys = []
    for t in range(L0, L0 + K):
        yt, state = ssm.ssd_step(dev["x"][:, t].contiguous(), dev["dt"][:, t].contiguous(), A,
                                 dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(), D, state, inplace=True)
        ys.append(P.to_np(yt))
    torch.cuda.synchronize()
    assert ssm.check_device_status(kind="ssd") == 0
    y_ref, h_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    P.assert_ssd_close(dtype, np.stack(ys, axis=1), y_ref[:, L0:], P.to_np(state), h_ref, "prefill + decode")


def test_decode_loop_matches_forward_f32(cuda_lib):
    """Forty decode steps from h0 in f32 reproduce the oracle's forward over the same tokens."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    shape = synth.SSDShape("decode_loop_f32", 3, 40, 6, 64, 64, 3, 64, "f32", h0=True)
    inp = synth.ssd_inputs(shape, seed=42)
    dev = {k: P.to_dev(inp[k]) for k in ("x", "dt", "B", "C")}
    A, D = P.to_dev(inp["A"]), P.to_dev(inp["D"])
    state = P.to_dev(inp["h0"])
    ys = []
    for t in range(shape.seqlen):
        yt, state = ssm.ssd_step(dev["x"][:, t].contiguous(), dev["dt"][:, t].contiguous(), A,
                                 dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(), D, state)
        ys.append(P.to_np(yt))
    torch.cuda.synchronize()
    y_ref, h_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    P.assert_ssd_close("f32", np.stack(ys, axis=1), y_ref, P.to_np(state), h_ref, "decode loop")
