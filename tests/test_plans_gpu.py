"""GPU tests of the per-shape plans of ssd_fwd (ssm_ssd_fwd_tune / _set_plan / _get_plan): every
candidate plan computes the forward within the parity rules, and tuning stores a plan that
later calls use."""
import numpy as np
import pytest

import parity as P
from oracle import ssd as ossd
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu


def dev_inputs(inp, dtype):
    d = {k: P.to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C")}
    d.update(A=P.to_dev(inp["A"]), D=P.to_dev(inp["D"]), h0=P.to_dev(inp["h0"]))
    return d


def run(ssm, d, chunk):
    import torch
    y, hf = ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=chunk)
    torch.cuda.synchronize()
    assert ssm.check_device_status(kind="ssd") == 0
    return P.to_np(y), P.to_np(hf)


@pytest.mark.parametrize("dtype,hpg", [("bf16", 4), ("f32", 2)])
def test_every_plan_is_correct(cuda_lib, dtype, hpg):
    import selective_state_space_mamba_gb300 as ssm
    G = 2
    shape = synth.SSDShape(f"plans_{dtype}", 2, 700, G * hpg, 64, 128, G, 256, dtype, h0=True)
    inp = synth.ssd_inputs(shape, seed=51)
    d = dev_inputs(inp, dtype)
    y_ref, hf_ref = ossd.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    plans = [ssm.plan_id(0, 1, 0), ssm.plan_id(0, 0, 0)]
    if dtype == "bf16":
        plans += [ssm.plan_id(1, -1, 0)] + [ssm.plan_id(f, 1 - f, h) for f in (0, 1) for h in (1, 2, hpg)]
        plans += [ssm.plan_id(1, -1, h, ring) for ring in (1, 2, 3) for h in (0, 1)]  # the fused pass's ring splits
        plans += [ssm.plan_id(2, -1, h, ring) for ring in (0, 2) for h in (0, 1)]  # split chains
    try:
        for plan in plans:
            ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, plan)
            assert ssm.get_ssd_fwd_plan(d["x"], d["B"], shape.chunk) == plan
            y, hf = run(ssm, d, shape.chunk)
            P.assert_ssd_close(dtype, y, y_ref, hf, hf_ref, f"plan {plan}")
        ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, -1)
        assert ssm.get_ssd_fwd_plan(d["x"], d["B"], shape.chunk) == -1
    finally:
        ssm.clear_ssd_fwd_plans()


def test_tune_stores_the_fastest_plan(cuda_lib):
    import selective_state_space_mamba_gb300 as ssm
    shape = synth.SSD_B8_L2048
    inp = synth.ssd_inputs(shape)
    d = dev_inputs(inp, shape.dtype)
    try:
        plan, ms = ssm.tune_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk, reps=3)
        assert plan >= 0 and ms > 0
        assert ssm.get_ssd_fwd_plan(d["x"], d["B"], shape.chunk) == plan
        y, hf = run(ssm, d, shape.chunk)
        units = [0, 57, 191]
        from oracle import native
        y_ref, hf_ref = native.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                                       units=np.asarray(units))
        nh = shape.nheads
        P.assert_ssd_close(shape.dtype, np.stack([y[u // nh, :, u % nh] for u in units]), y_ref,
                           np.stack([hf[u // nh, u % nh] for u in units]), hf_ref, f"tuned plan {plan}")
    finally:
        ssm.clear_ssd_fwd_plans()


def test_invalid_plan_rejected(cuda_lib):
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    import torch
    x = torch.zeros((1, 256, 2, 64), device="cuda", dtype=torch.bfloat16)
    B = torch.zeros((1, 256, 1, 128), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ssm.SsmError) as e:
        ssm.set_ssd_fwd_plan(x, B, 256, 3 << 2)   # sequential field 3 is not a choice
    assert e.value.status == _lib.SSM_ERR_INVALID_ARG
    with pytest.raises(ssm.SsmError) as e:
        ssm.set_ssd_fwd_plan(x, B, 256, 4 << 20)  # ring field 4 is not a choice
    assert e.value.status == _lib.SSM_ERR_INVALID_ARG


@pytest.mark.parametrize("rows,length", [(3, 1), (5, 4095), (4, 4097), (384, 1000), (2, 65537), (384, 65536)])
def test_every_scan_shape_is_correct(cuda_lib, rows, length):
    """Each CTA shape of the scan (consumer groups x ring depth x CTAs per SM) against the oracle."""
    import selective_state_space_mamba_gb300 as ssm
    from oracle import native
    inp = synth.scan_inputs(rows, length, seed=rows * 7 + length)
    a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    ref = native.linscan(inp["a"], inp["b"])
    try:
        for shape in (1, 2, 3, 4):
            ssm.set_linscan_shape(rows, length, shape)
            assert ssm.get_linscan_shape(rows, length) == shape
            h = ssm.linscan_fwd(a, b)
            assert ssm.check_device_status(kind="linscan") == 0
            P.assert_rows_close(P.to_np(h), ref, f"scan shape {shape} {rows}x{length}")
    finally:
        ssm.clear_linscan_shapes()
    assert ssm.get_linscan_shape(rows, length) == -1


def test_scan_tune_stores_the_fastest_shape(cuda_lib):
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    from oracle import native
    inp = synth.scan_inputs(96, 65536, seed=77)
    a, b = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    try:
        shape, ms = ssm.tune_linscan_fwd(a, b, reps=3)
        assert 1 <= shape <= 4 and ms > 0
        assert ssm.get_linscan_shape(96, 65536) == shape
        h = ssm.linscan_fwd(a, b)
        P.assert_rows_close(P.to_np(h), native.linscan(inp["a"], inp["b"]), f"tuned scan shape {shape}")
        with pytest.raises(ssm.SsmError) as e:
            ssm.set_linscan_shape(96, 65536, 5)
        assert e.value.status == _lib.SSM_ERR_INVALID_ARG
    finally:
        ssm.clear_linscan_shapes()


def _sm_count():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("extra_chains,seqlen,chunk,G,h0,final,ring", [(8, 520, 64, 1, True, True, 0),
                                                                      (1, 300, 64, 1, True, True, 2),
                                                                      (40, 1000, 128, 2, True, True, 0),
                                                                      (148, 200, 64, 4, True, True, 3),
                                                                      (8, 700, 128, 1, False, False, 0),
                                                                      (8, 200, 256, 1, True, True, 2),
                                                                      (40, 1000, 256, 1, True, True, 3)])
def test_fused_pass_with_more_chains_than_sms(cuda_lib, extra_chains, seqlen, chunk, G, h0, final, ring):
    """The fused state pass with more (batch, head pair) chains than SMs: one CTA per SM runs an
    equal range of chunks, so chains are split between CTAs and the CTA that runs a chain's
    tail starts from the state its predecessor publishes (with one chunk per chain the ranges
    hold whole chains only).  Every output is compared with the float64 oracle, and a second
    call (a new flag epoch) gives the same result."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from oracle import native
    chains = _sm_count() + extra_chains
    nh = 2 * chains
    while nh % G or (nh // G) % 2:
        nh += 2
    shape = synth.SSDShape(f"fused_split_{chains}", 1, seqlen, nh, 64, 128, G, chunk, "bf16", h0=h0)
    inp = synth.ssd_inputs(shape, seed=61 + extra_chains)
    d = dev_inputs(inp, "bf16")
    units = np.arange(shape.batch * nh)
    y_ref, hf_ref = native.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["h0"] if h0 else None, units=units)
    try:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], chunk, ssm.plan_id(1, -1, 0, ring))
        first = None
        for rep in range(2):
            y, hf = ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"] if h0 else None,
                                chunk=chunk, return_final_state=final)
            torch.cuda.synchronize()
            assert ssm.check_device_status(kind="ssd") == 0
            y = P.to_np(y)
            yu = np.stack([y[u // nh, :, u % nh] for u in units])
            if final:
                hf = P.to_np(hf)
                hu = np.stack([hf[u // nh, u % nh] for u in units])
                P.assert_ssd_close("bf16", yu, y_ref, hu, hf_ref, f"{shape.name} call {rep}")
            else:
                assert hf is None
                P.assert_ssd_close("bf16", yu, y_ref, None, None, f"{shape.name} call {rep}")
            if first is None:
                first = (y, hf)
            else:
                assert np.array_equal(first[0], y) and (not final or np.array_equal(first[1], hf))
    finally:
        ssm.clear_ssd_fwd_plans()


def test_fused_pass_with_large_B(cuda_lib):
    """The fused state pass where the group's B rows exceed 32 MB (b2 L65600 G1: 33.6 MB): its B
    loads then carry no evict-last priority (the lines would keep it after the pass).  Every
    output is compared with the float64 oracle."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    from oracle import native
    shape = synth.SSDShape("fused_large_B", 2, 65600, 4, 64, 128, 1, 256, "bf16", h0=True)
    assert shape.batch * shape.seqlen * shape.ngroups * 128 * 2 > 32 << 20
    inp = synth.ssd_inputs(shape, seed=79)
    d = dev_inputs(inp, "bf16")
    y_ref, hf_ref = native.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    try:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, ssm.plan_id(1, -1, 0))
        y, hf = run(ssm, d, shape.chunk)
        nh = shape.nheads
        yu = np.stack([y[u // nh, :, u % nh] for u in range(shape.batch * nh)])
        hu = np.stack([hf[u // nh, u % nh] for u in range(shape.batch * nh)])
        P.assert_ssd_close("bf16", yu, y_ref, hu, hf_ref, shape.name)
    finally:
        ssm.clear_ssd_fwd_plans()


def test_fused_pass_shares_the_gpu(cuda_lib):
    """The fused state pass while bf16 matmuls on another stream hold SMs.  Its CTAs take their
    ranges in claim order, not by block index, so a CTA that waits for the state its
    predecessor publishes waits for a CTA that is already running, whichever SMs are free when
    the CTAs start.  The result is bit-identical to the same call on an idle GPU."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    chains = _sm_count() + 40
    shape = synth.SSDShape("fused_shared", 1, 1000, 2 * chains, 64, 128, 1, 128, "bf16", h0=True)
    inp = synth.ssd_inputs(shape, seed=77)
    d = dev_inputs(inp, "bf16")
    try:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, ssm.plan_id(1, -1, 0))
        y0, hf0 = run(ssm, d, shape.chunk)
        a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16) / 64
        busy, mine = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        for rep in range(3):
            with torch.cuda.stream(busy):
                prods = [a @ a for _ in range(4)]
            with torch.cuda.stream(mine):
                y, hf = ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk)
            torch.cuda.synchronize()
            del prods
            assert ssm.check_device_status(kind="ssd") == 0
            assert np.array_equal(P.to_np(y), y0) and np.array_equal(P.to_np(hf), hf0), f"call {rep}"
    finally:
        ssm.clear_ssd_fwd_plans()
