"""GPU parity of linscan_lookback (through the C ABI) against the float64 oracle.

Cases follow the scan README's coverage ("Correctness"): ragged tails, L = 1, decay near 1,
very long rows (2^22), long look-back chains (up to 32,768 tiles), repeated runs; plus the
full 384 x 65,536 workload and its ragged companions, and a bounded-wait timeout.
"""
import numpy as np
import pytest

import parity as P
from oracle import linscan as olin
from oracle import native
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu
TILE = 4096


def gpu_scan(a, b, stream=None):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    ta, tb = P.to_dev(a), P.to_dev(b)
    if stream is None:
        h = ssm.linscan_fwd(ta, tb)
    else:
        with torch.cuda.stream(stream):
            h = ssm.linscan_fwd(ta, tb)
        stream.synchronize()
    assert ssm.check_device_status(kind="linscan") == 0
    return P.to_np(h)


def test_full_384x65536(cuda_lib):
    s = synth.SCAN_384x65536
    inp = synth.scan_inputs(s.rows, s.length, seed=synth.WORKLOAD_SEED[s.name])
    h = gpu_scan(inp["a"], inp["b"])
    ref = native.linscan(inp["a"], inp["b"])
    P.assert_rows_close(h, ref, s.name)


@pytest.mark.parametrize("shape", synth.SCAN_RAGGED, ids=lambda s: s.name)
def test_ragged_workloads(cuda_lib, shape):
    inp = synth.scan_inputs(shape.rows, shape.length, seed=synth.BASE_SEED + 11)
    h = gpu_scan(inp["a"], inp["b"])
    ref = native.linscan(inp["a"], inp["b"])
    P.assert_rows_close(h, ref, shape.name)


@pytest.mark.parametrize("rows,length", [(1, 1), (7, 3), (5, TILE - 1), (5, TILE), (5, TILE + 1), (2, 2 * TILE - 1),
                                         (3, 3 * TILE + 17), (4, 4 * TILE - 1), (3, 4 * TILE + 17), (1, 12345),
                                         (33, 1000), (2, 64 * TILE + 5)])
def test_small_and_ragged(cuda_lib, rows, length):
    inp = synth.scan_inputs(rows, length, seed=rows * 1000003 + length)
    h = gpu_scan(inp["a"], inp["b"])
    P.assert_rows_close(h, olin.linscan(inp["a"], inp["b"]), f"{rows}x{length}")


def test_long_chain_32768_tiles(cuda_lib):
    n = 32768 * TILE
    inp = synth.scan_inputs(1, n, seed=5, a_low=0.999, a_high=1.0)
    h = gpu_scan(inp["a"], inp["b"])
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), "1x2^27")


def test_decay_one_is_cumsum_and_zero_is_reset(cuda_lib):
    rng = np.random.default_rng(1)
    b = rng.standard_normal((3, 3 * TILE + 5)).astype(np.float32)
    a = np.ones_like(b)
    P.assert_rows_close(gpu_scan(a, b), native.linscan(a, b), "a=1")
    a = rng.uniform(0.5, 1.0, b.shape).astype(np.float32)
    a[:, ::97] = 0.0  # exact zeros reset the recurrence: h = b there
    h = gpu_scan(a, b)
    P.assert_rows_close(h, native.linscan(a, b), "a with zeros")
    assert np.array_equal(h[:, ::97], b[:, ::97].astype(np.float64))


def test_empty(cuda_lib):
    for shape in [(0, 10), (10, 0)]:
        z = np.zeros(shape, np.float32)
        assert gpu_scan(z, z).shape == shape


def test_side_stream(cuda_lib):
    import torch
    inp = synth.scan_inputs(4, 5 * TILE + 3, seed=9)
    h = gpu_scan(inp["a"], inp["b"], stream=torch.cuda.Stream())
    P.assert_rows_close(h, olin.linscan(inp["a"], inp["b"]), "side stream")


def test_repeated_runs(cuda_lib):
    """Look-back composition order depends on which flags a tile observes, so bit equality
    across runs is not promised; every run must meet the tolerance (the count of
    bit-identical runs is printed)."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp = synth.scan_inputs(1, 1 << 22, seed=17)
    ref = native.linscan(inp["a"], inp["b"])
    ta, tb = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    first = ssm.linscan_fwd(ta, tb).clone()
    same = 0
    for _ in range(100):
        h = ssm.linscan_fwd(ta, tb)
        same += int(torch.equal(h, first))
        P.assert_rows_close(P.to_np(h), ref, "repeat")
    assert ssm.check_device_status(kind="linscan") == 0
    print(f"bit-identical runs: {same}/100")


def test_bounded_wait_timeout(cuda_lib):
    """A tile that never publishes makes its successors give up after the limit and report
    SSM_ERR_TIMEOUT; the next call is clean."""
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    inp = synth.scan_inputs(1, 256 * TILE, seed=3)
    ta, tb = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    try:
        ssm.debug_set_lookback_fault(stall_tile=5, spin_limit_ns=20_000_000)
        ssm.linscan_fwd(ta, tb)
        assert ssm.check_device_status(kind="linscan") == _lib.SSM_ERR_TIMEOUT
    finally:
        ssm.debug_set_lookback_fault(-1, 0)
    h = P.to_np(ssm.linscan_fwd(ta, tb))
    assert ssm.check_device_status(kind="linscan") == 0
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), "after timeout")


def test_many_rows_bounded_wait_timeout(cuda_lib):
    """The same on many ragged rows (400 x 5000: look-back tiles that straddle rows and stop at
    row starts): a tile that never publishes makes its successors in the row give up after the
    limit and report SSM_ERR_TIMEOUT, and the next call is clean."""
    import selective_state_space_mamba_gb300 as ssm
    from selective_state_space_mamba_gb300 import _lib
    inp = synth.scan_inputs(400, 5000, seed=4)
    ta, tb = P.to_dev(inp["a"]), P.to_dev(inp["b"])
    try:
        ssm.debug_set_lookback_fault(stall_tile=5, spin_limit_ns=20_000_000)
        ssm.linscan_fwd(ta, tb)
        assert ssm.check_device_status(kind="linscan") == _lib.SSM_ERR_TIMEOUT
    finally:
        ssm.debug_set_lookback_fault(-1, 0)
    h = P.to_np(ssm.linscan_fwd(ta, tb))
    assert ssm.check_device_status(kind="linscan") == 0
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), "after timeout")
