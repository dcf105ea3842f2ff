"""CPU tests of the C ABI: the library builds, loads, exports every symbol include/ssm.h declares,
and rejects bad arguments on the host before anything is enqueued (no GPU needed)."""
import ctypes
import os
import re

import pytest

from selective_state_space_mamba_gb300 import _build, _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ssm.h")


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SSM_API\s+[\w\s\*]*?\b(ssm_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert declared_symbols() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {_build.LIB}").read()
    exported = set(re.findall(r"\bT (ssm_\w+)", out))
    assert set(declared_symbols()) <= exported
    assert all(s.startswith("ssm_") for s in exported), "only the C ABI is exported"


def test_debug_library_exports_every_declared_symbol():
    # the debug variant (device index checks) is the same ABI; building it is host-only work
    import ctypes
    from selective_state_space_mamba_gb300 import _build as b
    path = b.build(debug=True)
    dl = ctypes.CDLL(path)
    for name in _lib.EXPORTS:
        assert hasattr(dl, name), name


def test_library_targets_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_status_strings(lib):
    for code in range(8):
        s = _lib.status_string(code)
        assert s.startswith("SSM_")
    assert _lib.status_string(_lib.SSM_ERR_BOUNDS).startswith("SSM_ERR_BOUNDS")
    assert _lib.status_string(99) == "unknown ssm_status"
    assert lib.ssm_version().decode().count(".") == 2


def test_workspace_sizes(lib):
    # 0 for invalid / unsupported shapes
    assert lib.ssm_ssd_fwd_workspace_bytes(1, 256, 2, 32, 64, 1, 64, 0) == 0   # headdim 32
    assert lib.ssm_ssd_fwd_workspace_bytes(1, 256, 3, 64, 64, 2, 64, 0) == 0   # nh % G
    assert lib.ssm_ssd_fwd_workspace_bytes(1, 256, 2, 64, 64, 1, 100, 0) == 0  # chunk
    assert lib.ssm_linscan_workspace_bytes(-1, 5) == 0
    # grows with the problem and holds at least the per-chunk states
    w3 = lib.ssm_ssd_fwd_workspace_bytes(4, 8192, 80, 64, 128, 1, 256, 1)
    states = 4 * 32 * 80 * 64 * 128
    assert w3 >= states * 4 + states * 2
    assert w3 % 256 == 0
    # header + one 16-byte descriptor per 4096-element tile
    assert lib.ssm_linscan_workspace_bytes(384, 65536) >= 256 + (384 * 65536 // 4096) * 16


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _ssd(lib, **kw):
    args = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=FAKE, h0=None, y=FAKE, hf=None, batch=1, L=256, nh=2,
                H=64, S=64, G=1, T=64, dtype=0, ws=FAKE, wsb=1 << 40)
    args.update(kw)
    return lib.ssm_ssd_fwd(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["h0"], args["y"],
                           args["hf"], args["batch"], args["L"], args["nh"], args["H"], args["S"], args["G"],
                           args["T"], args["dtype"], args["ws"], args["wsb"], None)


def test_ssd_host_validation(lib):
    assert _ssd(lib, H=32) == _lib.SSM_ERR_UNSUPPORTED
    assert _ssd(lib, S=96) == _lib.SSM_ERR_UNSUPPORTED
    assert _ssd(lib, T=32) == _lib.SSM_ERR_UNSUPPORTED
    assert _ssd(lib, nh=3, G=2) == _lib.SSM_ERR_INVALID_ARG
    assert _ssd(lib, batch=-1) == _lib.SSM_ERR_INVALID_ARG
    assert _ssd(lib, L=-5) == _lib.SSM_ERR_INVALID_ARG
    assert _ssd(lib, dtype=7) == _lib.SSM_ERR_INVALID_ARG
    assert _ssd(lib, x=None) == _lib.SSM_ERR_INVALID_ARG
    assert _ssd(lib, x=FAKE + 4) == _lib.SSM_ERR_ALIGNMENT
    assert _ssd(lib, h0=FAKE + 8) == _lib.SSM_ERR_ALIGNMENT
    assert _ssd(lib, ws=None) == _lib.SSM_ERR_WORKSPACE
    assert _ssd(lib, wsb=1024) == _lib.SSM_ERR_WORKSPACE
    assert _ssd(lib, ws=FAKE + 16) == _lib.SSM_ERR_ALIGNMENT
    # no tokens and no final state requested: nothing to enqueue
    assert _ssd(lib, L=0, hf=None) == _lib.SSM_OK
    assert _ssd(lib, batch=0, hf=None) == _lib.SSM_OK


def test_linscan_host_validation(lib):
    f = lib.ssm_linscan_fwd
    assert f(FAKE, FAKE, FAKE, -1, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 3, -1, FAKE, 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 0, 10, None, 0, None) == _lib.SSM_OK   # empty: nothing enqueued
    assert f(FAKE, FAKE, FAKE, 10, 0, None, 0, None) == _lib.SSM_OK
    assert f(None, FAKE, FAKE, 3, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, FAKE, 3, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_ALIGNMENT
    assert f(FAKE, FAKE, FAKE, 3, 10, FAKE, 16, None) == _lib.SSM_ERR_WORKSPACE
    assert f(FAKE, FAKE, FAKE, 3, 10, FAKE + 128, 1 << 30, None) == _lib.SSM_ERR_ALIGNMENT


def test_product_package_does_not_import_oracle():
    pkg = os.path.dirname(_lib.__file__)
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                text = open(os.path.join(root, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), fn
            if fn.endswith((".cu", ".cuh", ".h")):
                assert "ssm_oracle" not in open(os.path.join(root, fn)).read(), fn


def _step(lib, **kw):
    args = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=FAKE, sin=None, sout=FAKE, y=FAKE, batch=2, nh=4, H=64,
                S=128, G=2, dtype=1)
    args.update(kw)
    return lib.ssm_ssd_step(args["x"], args["dt"], args["A"], args["B"], args["C"], args["D"], args["sin"],
                            args["sout"], args["y"], args["batch"], args["nh"], args["H"], args["S"], args["G"],
                            args["dtype"], None)


def test_step_host_validation(lib):
    assert _step(lib, H=24) == _lib.SSM_ERR_UNSUPPORTED    # headdim not a multiple of 16
    assert _step(lib, S=96) == _lib.SSM_ERR_UNSUPPORTED
    assert _step(lib, nh=3, G=2) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, batch=-1) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, dtype=5) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, sout=None) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, y=None) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, B=FAKE + 2) == _lib.SSM_ERR_ALIGNMENT
    assert _step(lib, sin=FAKE + 0x100008) == _lib.SSM_ERR_ALIGNMENT
    state_bytes = 2 * 4 * 64 * 128 * 4
    # in place is allowed (it would launch, so it is only checked on a GPU); partial overlap is not
    assert _step(lib, sin=FAKE, sout=FAKE + state_bytes - 16) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, sin=FAKE + 16, sout=FAKE) == _lib.SSM_ERR_INVALID_ARG
    assert _step(lib, batch=0) == _lib.SSM_OK                # nothing to enqueue


def test_scan_baseline_host_validation(lib):
    f = lib.ssm_linscan_baseline
    ws = lib.ssm_linscan_baseline_workspace_bytes
    assert f(9, FAKE, FAKE, FAKE, 3, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG   # unknown algorithm
    assert f(_lib.SSM_SCAN_BLELLOCH, FAKE, FAKE, FAKE, 3, 2049, None, 0, None) == _lib.SSM_ERR_UNSUPPORTED
    assert f(_lib.SSM_SCAN_THREE_PASS, FAKE, FAKE, FAKE, 1, 4194305, FAKE, 1 << 40, None) == _lib.SSM_ERR_UNSUPPORTED
    assert f(_lib.SSM_SCAN_THREE_PASS, FAKE, FAKE, FAKE, 65536, 16, FAKE, 1 << 40, None) == _lib.SSM_ERR_UNSUPPORTED
    assert f(_lib.SSM_SCAN_LOOKBACK_WARP, FAKE, FAKE, FAKE, -1, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_INVALID_ARG
    assert f(_lib.SSM_SCAN_LOOKBACK_WARP, FAKE, FAKE, FAKE, 0, 10, None, 0, None) == _lib.SSM_OK
    assert f(_lib.SSM_SCAN_LOOKBACK_SERIAL, FAKE + 4, FAKE, FAKE, 3, 10, FAKE, 1 << 30, None) == _lib.SSM_ERR_ALIGNMENT
    assert f(_lib.SSM_SCAN_LOOKBACK_SERIAL, FAKE, FAKE, FAKE, 3, 10, FAKE, 16, None) == _lib.SSM_ERR_WORKSPACE
    assert ws(_lib.SSM_SCAN_BLELLOCH, 3, 100) == 0
    # three-pass: one float per element plus the tile aggregates; look-back: header + 16 B per 256 elements
    assert ws(_lib.SSM_SCAN_THREE_PASS, 2, 5000) >= 4 * 10000 + 8 * 2 * 3
    assert ws(_lib.SSM_SCAN_LOOKBACK_WARP, 4, 1000) >= 256 + 16 * 16


def test_plan_host_validation(lib):
    # size checks come before any device query, so they run without a GPU
    assert lib.ssm_ssd_fwd_set_plan(1, 256, 2, 32, 64, 1, 64, 0, 0) == _lib.SSM_ERR_UNSUPPORTED   # headdim 32
    assert lib.ssm_ssd_fwd_set_plan(1, 256, 3, 64, 64, 2, 64, 0, 0) == _lib.SSM_ERR_INVALID_ARG   # nh % G
    assert lib.ssm_ssd_fwd_get_plan(1, 256, 2, 64, 64, 1, 100, 0, None) == _lib.SSM_ERR_UNSUPPORTED  # chunk
    args = [FAKE] * 9 + [1, 256, 2, 64, 64, 1, 64, 0, FAKE, 1 << 40, None]
    assert lib.ssm_ssd_fwd_tune(*args, 0, None, None) == _lib.SSM_ERR_INVALID_ARG      # reps < 1
    assert lib.ssm_ssd_fwd_tune(*args[:9], 1, 256, 2, 64, 64, 1, 64, 0, FAKE + 16, 1 << 40, None, 3, None,
                                None) == _lib.SSM_ERR_ALIGNMENT                        # workspace alignment


def test_plan_id_packing():
    import selective_state_space_mamba_gb300 as ssm
    assert ssm.plan_id() == 0 | (0 << 2)                    # all rules of thumb
    assert ssm.plan_id(1, -1, 0) == 2
    assert ssm.plan_id(0, 1, 20) == 1 | (2 << 2) | (20 << 4)
    assert ssm.plan_id(2, -1, 0) == 3                        # the fused pass with split chains
