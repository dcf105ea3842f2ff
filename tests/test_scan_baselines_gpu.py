"""GPU parity of the baseline scans (ssm_linscan_baseline: the reference page's Levels 1, 2,
3 and 3b) against the float64 oracle, under the same per-row float32 rule as linscan_fwd."""
import numpy as np
import pytest

import parity as P
from oracle import linscan as olin
from oracle import native
from selective_state_space_mamba_gb300 import synth

pytestmark = pytest.mark.gpu

ALGOS = ["blelloch", "three_pass", "lookback_serial", "lookback_warp", "hillis_steele"]


def run(algo, rows, length, seed=3, a_low=0.90):
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp = synth.scan_inputs(rows, length, seed=seed, a_low=a_low)
    a = torch.from_numpy(inp["a"]).cuda()
    b = torch.from_numpy(inp["b"]).cuda()
    h = ssm.linscan_baseline(a, b, algo)
    torch.cuda.synchronize()
    if algo.startswith("lookback"):
        assert ssm.check_device_status(kind="scan_" + algo) == 0
    return inp, h.cpu().numpy().astype(np.float64)


def shapes(algo):
    if algo == "blelloch":
        return [(3, 1), (5, 31), (4, 1000), (7, 2048), (64, 1024)]
    return [(3, 1), (5, 255), (4, 257), (384, 1000), (3, 4096 * 3 + 17), (2, 65537)]


@pytest.mark.parametrize("algo", ALGOS)
def test_baseline_small_shapes(cuda_lib, algo):
    for rows, length in shapes(algo):
        inp, h = run(algo, rows, length)
        ref = olin.linscan(inp["a"], inp["b"])
        P.assert_rows_close(h, ref, f"{algo} {rows}x{length}")


@pytest.mark.parametrize("algo", ["three_pass", "lookback_serial", "lookback_warp", "hillis_steele"])
def test_baseline_full_workload_every_row(cuda_lib, algo):
    shape = synth.SCAN_384x65536
    inp, h = run(algo, shape.rows, shape.length, seed=synth.WORKLOAD_SEED[shape.name])
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), f"{algo} 384x65536")


def test_blelloch_rows_of_2048_every_row(cuda_lib):
    inp, h = run("blelloch", 12288, 2048, seed=5)
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), "blelloch 12288x2048")


@pytest.mark.parametrize("algo", ["lookback_serial", "lookback_warp"])
def test_lookback_long_chain(cuda_lib, algo):
    # one row of 2^22 elements: a chain of 16,384 tiles through the look-back
    inp, h = run(algo, 1, 1 << 22, seed=6, a_low=0.999)
    P.assert_rows_close(h, native.linscan(inp["a"], inp["b"]), f"{algo} 1x2^22")


def test_baselines_agree_with_each_other(cuda_lib):
    # every level is a different association of the same combine: all match the production scan
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp = synth.scan_inputs(64, 2048, seed=7)
    a = torch.from_numpy(inp["a"]).cuda()
    b = torch.from_numpy(inp["b"]).cuda()
    ref = ssm.linscan_fwd(a, b).cpu().numpy().astype(np.float64)
    for algo in ALGOS:
        P.assert_rows_close(ssm.linscan_baseline(a, b, algo).cpu().numpy().astype(np.float64), ref, algo)
