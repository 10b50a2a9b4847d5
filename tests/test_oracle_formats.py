"""Pins of the oracle's NVFP4 decoding and quantiser (no GPU)."""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_pairs(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            a, b = line.split()[:2]
            rows.append((int(a), float(b)))
    return rows


def test_e2m1_table_matches_ocp_values():
    for code, val in _golden_pairs("e2m1_values.txt"):
        got = nvfp4.E2M1_TABLE[code]
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e4m3_table_matches_torch_float8_e4m3fn():
    b = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = nvfp4.E4M3_TABLE
    nan = np.isnan(b)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(b[~nan], ours[~nan])
    assert np.array_equal(np.signbit(b[~nan]), np.signbit(ours[~nan]))
    # subnormals are m * 2^-9 and the largest finite is 448
    assert all(ours[m] == m * 2.0 ** -9 for m in range(8))
    assert np.nanmax(ours) == 448.0


def test_unpack_low_nibble_first():
    out = nvfp4.unpack_nibbles(np.array([[0x21, 0xF7]], dtype=np.uint8))
    assert out.tolist() == [[1, 2, 7, 15]]


def test_dequantize_hand_example():
    # one row, K=32: block 0 scale 1.0 (0x38), block 1 scale 2^-9 (0x01); g = 2
    codes = np.zeros((1, 16), dtype=np.uint8)
    codes[0, 0] = 0xF7          # element 0: low nibble 7 (6.0); element 1: 15 (-6.0)
    codes[0, 8] = 0x03          # element 16: code 3 = 1.5
    scales = np.array([[0x38, 0x01]], dtype=np.uint8)
    w = nvfp4.dequantize(codes, scales, 2.0)
    assert w.shape == (1, 32)
    assert w[0, 0] == 12.0 and w[0, 1] == -12.0
    assert w[0, 16] == 1.5 * 2.0 ** -9 * 2.0
    assert np.count_nonzero(w) == 3


def test_dequantize_rejects_nan_scale():
    with pytest.raises(ValueError):
        nvfp4.dequantize(np.zeros((1, 8), np.uint8), np.array([[0x7F]], np.uint8), 1.0)


def test_quantize_exact_roundtrip(rng):
    # blocks whose amax is 6*s for an E4M3 s and whose elements are e2m1 * s
    rows, K = 8, 64
    sbytes = rng.integers(0x10, 0x60, size=(rows, K // 16))
    s = nvfp4.E4M3_TABLE[sbytes]
    codes = rng.integers(0, 16, size=(rows, K))
    codes[:, ::16] = 7                      # make 6.0 the block maximum
    w = nvfp4.E2M1_TABLE[codes] * np.repeat(s, 16, axis=1)
    qc, qs = nvfp4.quantize(w.astype(np.float32), 1.0)
    assert np.array_equal(qs, sbytes.astype(np.uint8))
    assert np.array_equal(nvfp4.dequantize(qc, qs, 1.0), w)


def test_quantize_scale_rounding_matches_torch_e4m3(rng):
    w = rng.standard_normal((16, 256)).astype(np.float32) * 3.0
    g = 0.5
    _, qs = nvfp4.quantize(w, g)
    amax = np.abs(w.astype(np.float64).reshape(16, 16, 16)).max(axis=2)
    target = torch.from_numpy(amax / (6.0 * g))
    ref = target.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(qs, ref)


def test_quantize_codes_are_nearest_brute_force(rng):
    w = (rng.standard_normal((4, 64)) * rng.uniform(0.1, 10, size=(4, 1))).astype(np.float32)
    g = 1.0
    qc, qs = nvfp4.quantize(w, g)
    codes = nvfp4.unpack_nibbles(qc)
    s = np.repeat(nvfp4.E4M3_TABLE[qs], 16, axis=1)
    mags = [0, .5, 1, 1.5, 2, 3, 4, 6]
    for r in range(4):
        for k in range(64):
            x = float(w[r, k]) / (s[r, k] * g)
            # brute force: every magnitude, smallest distance, tie -> even index
            best = min(range(8), key=lambda i: (abs(abs(x) - mags[i]), i % 2))
            got = int(codes[r, k])
            assert got & 7 == best, (r, k, x, got, best)
            if best:
                assert (got >> 3) == (1 if x < 0 else 0)
