"""Seeded synthetic inputs for the SSD forward and the scalar selective scan.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the method's arithmetic, so both the CUDA path (tests, bench)
and the float64 oracle can consume exactly the same values.

Storage convention: every array is returned as numpy ``float32``.  For the
bf16 workloads the values have already been rounded (round-to-nearest-even)
to bf16, so a float32 array holds them exactly and the conversion to a torch
``bfloat16`` tensor is exact.  ``A``, ``D`` and ``h0`` are float32 in every
workload (the state dtype of the Mamba-2 cuTile post's benchmark spec).

Distributions (the Mamba-2 cuTile post, "Mamba-2 architecture": A < 0 per
head, dt > 0 per token and head, B and C of size S, x of size H):
  x ~ N(0, 1); B, C ~ N(0, 1)/sqrt(S); dt = softplus(N(0, 1) - dt_shift);
  A = -exp(U(0, ln 16)); D ~ U(0.5, 1.5); h0 = 0 or N(0, 0.1^2).
Scan (selective-scan CUDA README, "The problem"): a ~ U(0.90, 0.9999),
b ~ N(0, 1).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class SSDShape:
    """Shape and recipe of one SSD forward workload."""

    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str  # "f32" or "bf16"
    dt_shift: float = 2.0
    h0: bool = False  # draw h0 ~ N(0, 0.1^2) instead of zeros

    @property
    def nchunks(self) -> int:
        return -(-self.seqlen // self.chunk)

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def replace(self, **kw) -> "SSDShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class ScanShape:
    """Shape of one scalar-scan workload: ``rows`` independent rows of ``length``."""

    name: str
    rows: int
    length: int


# The five workloads of the hot path, by index.
SSD_SMALL_F32 = SSDShape("ssd_b1_L256_nh2_H64_S64_T64_f32", 1, 256, 2, 64, 64, 1, 64, "f32")
SCAN_384x65536 = ScanShape("linscan_384x65536_f32", 384, 65536)
SCAN_RAGGED = (ScanShape("linscan_384x1_f32", 384, 1),
               ScanShape("linscan_384x1000_f32", 384, 1000),
               ScanShape("linscan_384x65537_f32", 384, 65537),
               ScanShape("linscan_1x4194304_f32", 1, 1 << 22))
SSD_B8_L2048 = SSDShape("ssd_b8_L2048_nh24_H64_S128_T256_bf16", 8, 2048, 24, 64, 128, 1, 256, "bf16")
SSD_B4_L8192 = SSDShape("ssd_b4_L8192_nh80_H64_S128_T256_bf16", 4, 8192, 80, 64, 128, 1, 256, "bf16",
                        h0=True)
SSD_B1_L131072 = SSDShape("ssd_b1_L131072_nh32_H64_S128_G8_T256_bf16", 1, 131072, 32, 64, 128, 8, 256,
                          "bf16", dt_shift=4.0, h0=True)


@dataclasses.dataclass(frozen=True)
class StepShape:
    """Shape of one decode-step workload: one new token for each of ``batch`` sequences."""

    name: str
    batch: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    dtype: str  # "f32" or "bf16"
    dt_shift: float = 2.0

    def replace(self, **kw) -> "StepShape":
        return dataclasses.replace(self, **kw)


# Decode: the model shape of the b4 L8192 forward (80 heads of 64 x 128, one group) with a
# batch of 128 sequences, so that the carried f32 state (335.5 MB) is larger than L2.
STEP_B128 = StepShape("ssd_step_b128_nh80_H64_S128_bf16", 128, 80, 64, 128, 1, "bf16")

WORKLOAD_SEED = {
    SSD_SMALL_F32.name: BASE_SEED + 0,
    SCAN_384x65536.name: BASE_SEED + 1,
    SSD_B8_L2048.name: BASE_SEED + 2,
    SSD_B4_L8192.name: BASE_SEED + 3,
    SSD_B1_L131072.name: BASE_SEED + 4,
    STEP_B128.name: BASE_SEED + 5,
}


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    NaN/inf are not produced by the generators, so no special casing is done.
    """
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def _store(v: np.ndarray, dtype: str) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return round_to_bf16(v) if dtype == "bf16" else v


def _softplus(z: np.ndarray) -> np.ndarray:
    # numerically safe log(1 + e^z), part of the input recipe only
    return np.logaddexp(0.0, z)


def ssd_inputs(shape: SSDShape, seed: int | None = None) -> dict:
    """Draw one SSD workload.

    Returns float32 arrays: x [b,L,nh,H], dt [b,L,nh], A [nh], B [b,L,G,S],
    C [b,L,G,S], D [nh], h0 [b,nh,H,S] (zeros unless ``shape.h0``).
    """
    if seed is None:
        seed = WORKLOAD_SEED.get(shape.name, BASE_SEED)
    rng = np.random.Generator(np.random.PCG64(seed))
    b, L, nh, H, S, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    x = rng.standard_normal((b, L, nh, H), dtype=np.float32)
    Bm = rng.standard_normal((b, L, G, S), dtype=np.float32) * np.float32(1.0 / math.sqrt(S))
    Cm = rng.standard_normal((b, L, G, S), dtype=np.float32) * np.float32(1.0 / math.sqrt(S))
    dt = _softplus(rng.standard_normal((b, L, nh)) - shape.dt_shift)
    A = -np.exp(rng.uniform(0.0, math.log(16.0), nh))
    D = rng.uniform(0.5, 1.5, nh)
    if shape.h0:
        h0 = rng.standard_normal((b, nh, H, S), dtype=np.float32) * np.float32(0.1)
    else:
        h0 = np.zeros((b, nh, H, S), np.float32)
    return {
        "x": _store(x, shape.dtype),
        "dt": _store(dt, shape.dtype),
        "A": np.ascontiguousarray(A, np.float32),
        "B": _store(Bm, shape.dtype),
        "C": _store(Cm, shape.dtype),
        "D": np.ascontiguousarray(D, np.float32),
        "h0": np.ascontiguousarray(h0, np.float32),
    }


def step_inputs(shape: StepShape, seed: int | None = None) -> dict:
    """Draw one decode-step workload, with the same distributions as ssd_inputs.

    Returns float32 arrays: x [b,nh,H], dt [b,nh], A [nh], B [b,G,S], C [b,G,S], D [nh] and
    the carried state [b,nh,H,S] ~ N(0, 0.1^2).
    """
    if seed is None:
        seed = WORKLOAD_SEED.get(shape.name, BASE_SEED)
    rng = np.random.Generator(np.random.PCG64(seed))
    b, nh, H, S, G = shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    x = rng.standard_normal((b, nh, H), dtype=np.float32)
    Bm = rng.standard_normal((b, G, S), dtype=np.float32) * np.float32(1.0 / math.sqrt(S))
    Cm = rng.standard_normal((b, G, S), dtype=np.float32) * np.float32(1.0 / math.sqrt(S))
    dt = _softplus(rng.standard_normal((b, nh)) - shape.dt_shift)
    A = -np.exp(rng.uniform(0.0, math.log(16.0), nh))
    D = rng.uniform(0.5, 1.5, nh)
    state = rng.standard_normal((b, nh, H, S), dtype=np.float32) * np.float32(0.1)
    return {
        "x": _store(x, shape.dtype),
        "dt": _store(dt, shape.dtype),
        "A": np.ascontiguousarray(A, np.float32),
        "B": _store(Bm, shape.dtype),
        "C": _store(Cm, shape.dtype),
        "D": np.ascontiguousarray(D, np.float32),
        "state": np.ascontiguousarray(state, np.float32),
    }


def scan_inputs(rows: int, length: int, seed: int = BASE_SEED + 1,
                a_low: float = 0.90, a_high: float = 0.9999) -> dict:
    """Draw one scalar-scan workload: a ~ U(a_low, a_high), b ~ N(0,1), both [rows, length] f32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.uniform(a_low, a_high, (rows, length)).astype(np.float32)
    bv = rng.standard_normal((rows, length), dtype=np.float32)
    return {"a": np.ascontiguousarray(a), "b": np.ascontiguousarray(bv)}
