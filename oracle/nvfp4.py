"""NVFP4 decoding, written from the format definitions (oracle; test infrastructure).

NVFP4, NVIDIA's 4-bit floating-point format, is the weight format of the
Edge0 expert pool ("Edge0-145B en local", introduction; "Edge0-145B Review",
section "Q3_K oder NVFP4", which notes it is aimed at Blackwell).  A weight is

    w = e2m1(code) * e4m3(scale of its 16-element block along K) * g

with ``g`` one fp32 per matrix.  E2M1 and E4M3 follow the OCP Microscaling
(MX) v1.0 element definitions: E2M1 has 1 sign, 2 exponent (bias 1) and 1
mantissa bit; E4M3 (the "FN" variant) has 1 sign, 4 exponent (bias 7) and 3
mantissa bits, no infinities, and NaN at S.1111.111.

Everything here decodes exactly into fp64.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code: (-1)^s * 2^(e-1) * (1 + m/2), or m/2 if e == 0."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def e4m3_value(byte: int) -> float:
    """Value of one E4M3FN byte: (-1)^s * 2^(e-7) * (1 + m/8), or m/8 * 2^-6 if e == 0."""
    s = (byte >> 7) & 1
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> uint8 [..., K]; the low nibble is the even element."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0x0F
    out[..., 1::2] = codes >> 4
    return out


def dequantize(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """Exact fp64 matrix [rows, K] from codes [rows, K/2], scales [rows, K/16], g."""
    vals = E2M1_TABLE[unpack_nibbles(codes)]
    sc = E4M3_TABLE[np.asarray(scales, dtype=np.uint8)]
    if np.isnan(sc).any():
        raise ValueError("E4M3 NaN scale in an expert record")
    rows, K = vals.shape
    assert sc.shape == (rows, K // 16)
    return vals * np.repeat(sc, 16, axis=1) * float(np.float32(g))


def quantize(w: np.ndarray, g: float = 1.0):
    """NVFP4 quantisation of an fp32 matrix [rows, K] (K % 16 == 0), by definition.

    The pages fix the format but not the quantiser; this is the plain reading:
      * per 16-element block, scale = E4M3 round-to-nearest-even of
        amax / (6 g) (6 = largest E2M1 magnitude), saturating at 448;
      * each element's code = the E2M1 value nearest to w / (scale g), ties
        to the even code (the one whose mantissa bit is 0), saturating at 6;
      * an all-zero block (or a block whose scale rounds to 0) gets scale 0
        and codes 0.
    Division and comparison happen in fp64 from fp32 inputs.
    Returns (codes uint8 [rows, K/2], scales uint8 [rows, K/16]).
    """
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    rows, K = w.shape
    assert K % 16 == 0
    gd = float(np.float32(g))
    blocks = w.reshape(rows, K // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    target = amax / (6.0 * gd)
    # E4M3 RNE by nearest-grid search over the 127 finite non-negative codes
    grid = E4M3_TABLE[:127]                           # 0x00..0x7E, increasing
    sb = _nearest_even_code(target, grid)
    sval = grid[sb]
    denom = sval * gd
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(denom[..., None] > 0, blocks / denom[..., None], 0.0)
    mag_grid = E2M1_TABLE[:8]                         # 0, .5, 1, 1.5, 2, 3, 4, 6
    mcode = _nearest_even_code(np.abs(r), mag_grid)
    sign = (r < 0) & (mcode > 0)
    code = (mcode | (sign.astype(np.int64) << 3)).reshape(rows, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb.astype(np.uint8)


def _nearest_even_code(x: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to x (grid increasing, x >= 0).

    Ties go to the even index (for E2M1 magnitudes and E4M3 bytes the even
    index is the one with the low mantissa bit clear).  Values past the last
    grid point saturate to it.
    """
    x = np.asarray(x, dtype=np.float64)
    hi = np.clip(np.searchsorted(grid, x, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    dlo = np.abs(x - grid[lo])
    dhi = np.abs(grid[hi] - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.int64)
