"""Checks of the seeded input generator (no GPU)."""
import numpy as np
import torch

import synth


def test_splitmix64_reference_values():
    # SplitMix64 stream seeded with 0 (Steele, Lea, Flood 2014): first outputs
    got = [int(v) for v in synth.splitmix64(np.array([0, 0x9E3779B97F4A7C15], dtype=np.uint64))]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_e4m3_encode_matches_torch(rng):
    v = np.concatenate([rng.uniform(0.0, 448.0, 5000), rng.uniform(0, 0.02, 5000),
                        [0.0, 2.0 ** -10, 3 * 2.0 ** -10, 0.002, 0.01, 448.0]])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.e4m3_encode_rne(v), ref)


def test_expert_scale_distribution():
    codes, scales, glob = synth.expert_bytes(0, 0, 3, 1792)
    assert codes.size == 3 * 640 * 1792 // 2 and scales.size == 3 * 640 * 1792 // 16
    assert set(np.unique(scales).tolist()) <= {1, 2, 3, 4, 5}
    freq = np.bincount(scales, minlength=6)[1:] / scales.size
    # uniform on [0.002, 0.01] rounded to the 2^-9 grid
    expect = np.array([1.5 - 1.024, 1, 1, 1, 5.12 - 4.5]) / (5.12 - 1.024)
    assert np.allclose(freq, expect, atol=0.005)
    nib = np.concatenate([codes & 15, codes >> 4])
    assert np.allclose(np.bincount(nib, minlength=16) / nib.size, 1 / 16, atol=0.002)
    assert np.array_equal(glob, np.ones(3, np.float32))


def test_generator_is_deterministic_and_keyed():
    a = synth.expert_bytes(4, 1, 7, 1280)
    b = synth.expert_bytes(4, 1, 7, 1280)
    c = synth.expert_bytes(4, 1, 8, 1280)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])


def test_dense_inputs_distribution():
    lay = synth.make_layer(synth.LayerSpec(seed=0, layer=0, latent=1280))
    D = synth.bf16_bits_to_f32(lay.D)
    assert D.shape == (1280, 2560)
    assert abs(D.std() * np.sqrt(2560) - 1) < 0.01
    zb = synth.zipf_bias(3, 0)
    assert sorted(np.round(np.exp(-zb / 1.1)).astype(int).tolist()) == list(range(1, 513))
