"""The C-ABI calls captured into CUDA graphs and replayed with new inputs each time.

A replay repeats the captured kernels with the captured arguments, so nothing a call decides
on the host (such as a per-call tag) may change between replays.  The look-back kernels take
their flag epoch from the workspace, which each launch advances, so replay after replay their
flags stay distinct; these tests refill the inputs before every replay and check every
output against the float64 oracle.
"""
import numpy as np
import pytest

import parity as P
from oracle import linscan as olin
from oracle import ssd as ossd
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu


def test_linscan_graph_replays(cuda_lib):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    rows, length = 3, 3 * 4096 + 17  # several look-back tiles per row and a ragged tail
    a = torch.empty((rows, length), device="cuda")
    b = torch.empty_like(a)
    h = torch.empty_like(a)
    first = synth.scan_inputs(rows, length, seed=61)
    a.copy_(torch.from_numpy(first["a"]))
    b.copy_(torch.from_numpy(first["b"]))
    ssm.linscan_fwd(a, b, h=h)  # warm-up: workspace and launch set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ssm.linscan_fwd(a, b, h=h)
    for rep in range(4):
        inp = synth.scan_inputs(rows, length, seed=62 + rep)
        a.copy_(torch.from_numpy(inp["a"]))
        b.copy_(torch.from_numpy(inp["b"]))
        g.replay()
        torch.cuda.synchronize()
        assert ssm.check_device_status(kind="linscan") == 0
        P.assert_rows_close(h.cpu().numpy().astype(np.float64), olin.linscan(inp["a"], inp["b"]), f"replay {rep}")


@pytest.mark.parametrize("shape", [
    synth.SSDShape("graph_bf16", 2, 700, 8, 64, 128, 2, 256, "bf16", h0=True),
    # few state entries: the look-back state-passing kernel (flags in the workspace)
    synth.SSDShape("graph_lookback_f32", 1, 4096, 2, 64, 64, 1, 64, "f32", h0=True),
], ids=lambda s: s.name)
def test_ssd_fwd_graph_replays(cuda_lib, shape):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp0 = synth.ssd_inputs(shape, seed=71)
    d = {k: P.to_dev(v, shape.dtype if k in ("x", "dt", "B", "C") else "f32") for k, v in inp0.items()}
    y = torch.empty_like(d["x"])
    hf = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.dstate), device="cuda")

    def call():
        ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk, y=y, h_final=hf)

    call()  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for rep in range(3):
        inp = synth.ssd_inputs(shape, seed=72 + rep)
        for k, v in inp.items():
            d[k].copy_(P.to_dev(v, shape.dtype if k in ("x", "dt", "B", "C") else "f32"))
        g.replay()
        torch.cuda.synchronize()
        assert ssm.check_device_status(kind="ssd") == 0
        y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
        P.assert_ssd_close(shape.dtype, P.to_np(y), y_ref, P.to_np(hf), hf_ref, f"{shape.name} replay {rep}")


def test_decode_step_graph_loop(cuda_lib):
    """One captured in-place decode step, replayed token after token with the next token's
    inputs copied in: the loop equals the oracle's forward over those tokens."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    shape = synth.SSDShape("graph_decode", 2, 12, 4, 64, 128, 2, 64, "bf16", h0=True)
    inp = synth.ssd_inputs(shape, seed=81)
    x = P.to_dev(inp["x"][:, 0], "bf16")
    dt = P.to_dev(inp["dt"][:, 0], "bf16")
    B = P.to_dev(inp["B"][:, 0], "bf16")
    C = P.to_dev(inp["C"][:, 0], "bf16")
    A, D = P.to_dev(inp["A"]), P.to_dev(inp["D"])
    state = P.to_dev(inp["h0"])
    y = torch.empty_like(x)
    ssm.ssd_step(x, dt, A, B, C, D, state.clone(), y=y)  # warm-up on a copy of the state
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ssm.ssd_step(x, dt, A, B, C, D, state, y=y, inplace=True)
    ys = []
    for t in range(shape.seqlen):
        x.copy_(P.to_dev(inp["x"][:, t], "bf16"))
        dt.copy_(P.to_dev(inp["dt"][:, t], "bf16"))
        B.copy_(P.to_dev(inp["B"][:, t], "bf16"))
        C.copy_(P.to_dev(inp["C"][:, t], "bf16"))
        g.replay()
        ys.append(P.to_np(y))
    torch.cuda.synchronize()
    y_ref, h_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    P.assert_ssd_close("bf16", np.stack(ys, axis=1), y_ref, P.to_np(state), h_ref, "graph decode loop")


def test_fused_split_chains_graph_replays(cuda_lib):
    """The fused state pass with more chains than SMs inside a CUDA graph: the states a CTA
    publishes for its successor are flagged with the epoch kept in the workspace, which every
    launch moves on, so a replay never takes a flag of the replay before it."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from oracle import native
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nh = 2 * (sms + 8)
    shape = synth.SSDShape("graph_fused_split", 1, 520, nh, 64, 128, 1, 64, "bf16", h0=True)
    inp0 = synth.ssd_inputs(shape, seed=91)
    d = {k: P.to_dev(v, "bf16" if k in ("x", "dt", "B", "C") else "f32") for k, v in inp0.items()}
    y = torch.empty_like(d["x"])
    hf = torch.empty((1, nh, 64, 128), device="cuda")

    def call():
        ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk, y=y, h_final=hf)

    try:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, ssm.plan_id(1, -1, 0))
        call()  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        units = np.arange(nh)
        for rep in range(3):
            inp = synth.ssd_inputs(shape, seed=92 + rep)
            for k, v in inp.items():
                d[k].copy_(P.to_dev(v, "bf16" if k in ("x", "dt", "B", "C") else "f32"))
            g.replay()
            torch.cuda.synchronize()
            assert ssm.check_device_status(kind="ssd") == 0
            y_ref, hf_ref = native.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                                           units=units)
            yn, hn = P.to_np(y), P.to_np(hf)
            yu = np.stack([yn[0, :, u] for u in units])
            hu = np.stack([hn[0, u] for u in units])
            P.assert_ssd_close("bf16", yu, y_ref, hu, hf_ref, f"{shape.name} replay {rep}")
    finally:
        ssm.clear_ssd_fwd_plans()


def test_split_chains_graph_replays(cuda_lib):
    """The fused pass with split chains (every piece from a zero state, then the fix-up kernel
    adds the state each piece enters with) inside a CUDA graph: 2 chains of 65 chunks, so the
    pieces are single chunks and each fix-up composes up to 64 earlier pieces' end states."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    shape = synth.SSDShape("graph_split_chains", 1, 65 * 64 - 3, 4, 64, 128, 1, 64, "bf16", h0=True)
    inp0 = synth.ssd_inputs(shape, seed=95)
    d = {k: P.to_dev(v, "bf16" if k in ("x", "dt", "B", "C") else "f32") for k, v in inp0.items()}
    y = torch.empty_like(d["x"])
    hf = torch.empty((1, shape.nheads, 64, 128), device="cuda")

    def call():
        ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk, y=y, h_final=hf)

    try:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, ssm.plan_id(2, -1, 0))
        call()  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        for rep in range(3):
            inp = synth.ssd_inputs(shape, seed=96 + rep)
            for k, v in inp.items():
                d[k].copy_(P.to_dev(v, "bf16" if k in ("x", "dt", "B", "C") else "f32"))
            g.replay()
            torch.cuda.synchronize()
            assert ssm.check_device_status(kind="ssd") == 0
            y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
            P.assert_ssd_close("bf16", P.to_np(y), y_ref, P.to_np(hf), hf_ref, f"{shape.name} replay {rep}")
    finally:
        ssm.clear_ssd_fwd_plans()
