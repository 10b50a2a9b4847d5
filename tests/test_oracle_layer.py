"""Pins of the oracle's layer pieces against library routines and invariants (no GPU)."""
import os

import numpy as np
import torch

import synth
from oracle import moe, nvfp4, record
from conftest import oracle_layer, tiny_spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def test_swiglu_expert_matches_torch(rng):
    L, F, n = 48, 32, 5
    z = rng.standard_normal((n, L))
    Wg, Wu, Wd = rng.standard_normal((F, L)), rng.standard_normal((F, L)), rng.standard_normal((L, F))
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(_t(z), _t(Wg))) *
        torch.nn.functional.linear(_t(z), _t(Wu)), _t(Wd)).numpy()
    assert np.allclose(moe.swiglu_expert(z, Wg, Wu, Wd), ref, rtol=1e-12, atol=1e-12)


def test_rmsnorm_matches_torch(rng):
    v = rng.standard_normal((6, 2560)) * 3
    ref = torch.nn.functional.rms_norm(_t(v), (2560,), eps=1e-6).numpy()
    assert np.allclose(moe.rmsnorm(v, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_bf16_rounding_is_nearest_even_brute_force(rng):
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-3, 4, 4000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]])
    got = moe.bf16_to_f64(moe.f64_to_bf16(x))
    for xi, gi in zip(x, got):
        e = np.floor(np.log2(abs(xi)))
        ulp = 2.0 ** (e - 7)
        lo = np.floor(abs(xi) / ulp) * ulp
        hi = lo + ulp
        dlo, dhi = abs(xi) - lo, hi - abs(xi)
        mag = lo if (dlo < dhi or (dlo == dhi and (lo / ulp) % 2 == 0)) else hi
        assert gi == np.copysign(mag, xi), (xi, gi)
    assert np.array_equal(moe.bf16_to_f64(synth.f32_to_bf16_bits(np.float32([1.5, -2.25]))), [1.5, -2.25])


def test_zero_routed_experts_give_shared_path_only(rng):
    spec = tiny_spec(seed=5)
    inp = synth.make_layer(spec)
    zero = lambda e: (np.zeros_like(inp.expert(e)[0]), inp.expert(e)[1], inp.expert(e)[2])
    lay = moe.Layer(inp.D, inp.U, inp.R, inp.bias, zero, inp.shared,
                    spec.latent, spec.ffn, spec.top_k)
    x = synth.tokens_bf16(7, 9, spec.hidden)
    y = moe.layer_forward(lay, x)["y"]
    # independent shared-expert-only path with library ops
    xs = _t(moe.bf16_to_f64(x))
    D, U = _t(moe.bf16_to_f64(inp.D)), _t(moe.bf16_to_f64(inp.U))
    c, s, g = inp.shared()
    L, F = spec.latent, spec.ffn
    Wg = _t(nvfp4.dequantize(c[:F * L // 2].reshape(F, -1), s[:F * L // 16].reshape(F, -1), g[0]))
    Wu = _t(nvfp4.dequantize(c[F * L // 2:F * L].reshape(F, -1), s[F * L // 16:F * L // 8].reshape(F, -1), g[1]))
    Wd = _t(nvfp4.dequantize(c[F * L:].reshape(L, -1), s[F * L // 8:].reshape(L, -1), g[2]))
    z = xs @ D.T
    ref = ((torch.nn.functional.silu(z @ Wg.T) * (z @ Wu.T)) @ Wd.T) @ U.T
    assert np.allclose(y, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_token_permutation_invariance():
    spec = tiny_spec(seed=9, zipf=1.1)
    lay = oracle_layer(synth.make_layer(spec))
    x = synth.tokens_bf16(3, 13, spec.hidden)
    p = np.random.default_rng(0).permutation(13)
    y = moe.layer_forward(lay, x)["y"]
    yp = moe.layer_forward(lay, x[p])["y"]
    assert np.array_equal(yp, y[p])


def test_teacher_forcing_with_own_indices_is_identity():
    spec = tiny_spec(seed=2)
    lay = oracle_layer(synth.make_layer(spec))
    x = synth.tokens_bf16(4, 6, spec.hidden)
    out = moe.layer_forward(lay, x, want=("idx",))
    again = moe.layer_forward(lay, x, idx_override=out["idx"])
    assert np.array_equal(out["y"], again["y"])


def test_teacher_forcing_with_other_indices_matches_brute_force():
    """idx_override with experts the oracle would not pick: y and w must follow the
    given indices, with weights renormalised from the fp64 logits over exactly those
    experts (per-token torch/scipy composition).  An override that was ignored, or
    weights taken from the oracle's own top-k, fails here."""
    import scipy.special
    spec = tiny_spec(seed=31, n_experts=16, top_k=3, zipf=0.7)
    inp = synth.make_layer(spec)
    lay = oracle_layer(inp)
    T = 5
    x = synth.tokens_bf16(12, T, spec.hidden)
    own = moe.layer_forward(lay, x, want=("idx", "logits"))
    # J: ranks 3..5 of each token's ordering (never the oracle's choice), in a
    # rotated order so that the rank order of J differs from the logits' order too
    J = np.empty((T, 3), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(16), -own["logits"][t]))
        J[t] = np.roll(order[3:6], t)
        assert not set(J[t]) & set(own["idx"][t])
    out = moe.layer_forward(lay, x, idx_override=J, want=("idx", "w"))
    assert np.array_equal(out["idx"], J)
    L, F = spec.latent, spec.ffn

    def mats(src):
        c, s, g = src
        return (_t(nvfp4.dequantize(c[:F * L // 2].reshape(F, -1), s[:F * L // 16].reshape(F, -1), g[0])),
                _t(nvfp4.dequantize(c[F * L // 2:F * L].reshape(F, -1), s[F * L // 16:F * L // 8].reshape(F, -1), g[1])),
                _t(nvfp4.dequantize(c[F * L:].reshape(L, -1), s[F * L // 8:].reshape(L, -1), g[2])))

    D, U, R = (_t(moe.bf16_to_f64(a)) for a in (inp.D, inp.U, inp.R))
    for t in range(T):
        zt = D @ _t(moe.bf16_to_f64(x[t]))
        lt = (R @ zt).numpy() + inp.bias.astype(np.float64)
        p = scipy.special.softmax(lt)[J[t]]
        wt = p / p.sum()
        assert np.allclose(out["w"][t], wt, rtol=1e-12, atol=0)
        Wg, Wu, Wd = mats(inp.shared())
        ct = Wd @ (torch.nn.functional.silu(Wg @ zt) * (Wu @ zt))
        for j, e in enumerate(J[t]):
            Wg, Wu, Wd = mats(inp.expert(int(e)))
            ct = ct + wt[j] * (Wd @ (torch.nn.functional.silu(Wg @ zt) * (Wu @ zt)))
        assert np.allclose(out["y"][t], (U @ ct).numpy(), rtol=1e-10, atol=1e-12)
    # and the override changes the answer: the oracle's own routing gives another y
    assert not np.allclose(out["y"], own["y"], rtol=1e-3, atol=1e-6)


def test_combine_is_linear_in_routed_outputs():
    """Halving every routed expert's down global halves the routed part of c."""
    spec = tiny_spec(seed=11)
    inp = synth.make_layer(spec)
    half = lambda e: (inp.expert(e)[0], inp.expert(e)[1], inp.expert(e)[2] * np.float32([1, 1, 0.5]))
    lay = oracle_layer(inp)
    lay_h = moe.Layer(inp.D, inp.U, inp.R, inp.bias, half, inp.shared, spec.latent, spec.ffn, spec.top_k)
    x = synth.tokens_bf16(8, 5, spec.hidden)
    a = moe.layer_forward(lay, x, want=("c", "o_shared"))
    b = moe.layer_forward(lay_h, x, want=("c", "o_shared"))
    assert np.allclose(b["c"] - b["o_shared"], 0.5 * (a["c"] - a["o_shared"]), rtol=1e-12, atol=1e-14)


def _page_sizes():
    out = {}
    for line in open(os.path.join(GOLDEN, "page_sizes.txt")):
        line = line.split("#")[0].strip()
        if line:
            name, val = line.split()[:2]
            out[name] = float(val)
    return out


def test_shapes_reproduce_page_figures():
    p = _page_sizes()
    for L, tag in ((1792, "145b"), (1280, "120b")):
        assert p["latent_" + tag] == L
        pool = 48 * 512 * 3 * 640 * L
        assert round(pool / 1e9, 1) == p["expert_pool_" + tag] / 1e9
        active = 48 * 10 * 3 * 640 * L
        assert round(active / 1e9, 2) == p["active_expert_params_" + tag] / 1e9
        # the printed fixed record is the Q3_K one: 910 bytes per latent row
        assert L * 910 == p["q3k_record_" + tag]
    # NVFP4 record (4 bits + one 8-bit scale per 16 weights) x 48 x 512 = experts.bin
    body = record.record_body_bytes(1792, 640)
    assert body == 1_935_360
    assert round(48 * 512 * record.record_bytes(1792, 640) / 1e9, 1) == p["nvfp4_experts_bin_gb"]
    assert round(48 * 512 * 1792 * 910 / 1e9, 1) == p["q3k_experts_bin_gb"]


def test_stack_post_norm_two_layers():
    spec0, spec1 = tiny_spec(seed=1, layer=0), tiny_spec(seed=1, layer=1)
    l0, l1 = oracle_layer(synth.make_layer(spec0)), oracle_layer(synth.make_layer(spec1))
    x = synth.tokens_bf16(1, 3, spec0.hidden)
    xf, trace = moe.stack_forward([l0, l1], x)
    y0 = moe.f64_to_bf16(moe.layer_forward(l0, x)["y"])
    x1 = moe.f64_to_bf16(moe.rmsnorm(moe.bf16_to_f64(x) + moe.bf16_to_f64(y0)))
    assert np.array_equal(trace[1][0], x1)
    r = moe.bf16_to_f64(xf)
    assert np.allclose(np.sqrt(np.mean(r * r, axis=1)), 1.0, atol=1e-2)


def test_layer_matches_per_token_brute_force():
    """Per-token composition with library routines on a tiny layer: torch fp64
    matmuls, brute-force top-k, scipy softmax, torch silu, explicit sum over k."""
    import scipy.special
    from test_oracle_routing import _brute_topk
    spec = tiny_spec(seed=21, n_experts=8, top_k=3, zipf=1.1)
    inp = synth.make_layer(spec)
    lay = oracle_layer(inp)
    x = synth.tokens_bf16(5, 4, spec.hidden)
    y = moe.layer_forward(lay, x)["y"]
    L, F = spec.latent, spec.ffn

    def mats(src):
        c, s, g = src
        return (_t(nvfp4.dequantize(c[:F * L // 2].reshape(F, -1), s[:F * L // 16].reshape(F, -1), g[0])),
                _t(nvfp4.dequantize(c[F * L // 2:F * L].reshape(F, -1), s[F * L // 16:F * L // 8].reshape(F, -1), g[1])),
                _t(nvfp4.dequantize(c[F * L:].reshape(L, -1), s[F * L // 8:].reshape(L, -1), g[2])))

    D, U, R = (_t(moe.bf16_to_f64(a)) for a in (inp.D, inp.U, inp.R))
    for t in range(4):
        zt = D @ _t(moe.bf16_to_f64(x[t]))
        lt = (R @ zt).numpy() + inp.bias.astype(np.float64)
        sel = _brute_topk(lt.tolist(), spec.top_k)
        p = scipy.special.softmax(lt)[sel]
        wt = p / p.sum()
        Wg, Wu, Wd = mats(inp.shared())
        ct = Wd @ (torch.nn.functional.silu(Wg @ zt) * (Wu @ zt))
        for j, e in enumerate(sel):
            Wg, Wu, Wd = mats(inp.expert(e))
            ct = ct + wt[j] * (Wd @ (torch.nn.functional.silu(Wg @ zt) * (Wu @ zt)))
        assert np.allclose(y[t], (U @ ct).numpy(), rtol=1e-10, atol=1e-12)


def test_bf16_ulp_of_the_parity_check():
    import parity
    v = np.array([1.0, 1.5, -0.065, 3.0e-3, 0.0])
    # 8 significant bits: ulp = 2^(exponent - 7)
    assert np.array_equal(parity.bf16_ulp(v), [2.0 ** -7, 2.0 ** -7, 2.0 ** -11, 2.0 ** -16, 0.0])
