"""Parity of grouped latent projections (G D/U pairs per layer, a group label per
expert) with the oracle's ``grouped_layer_forward``, through the C ABI.

A grouped layer runs the prefill kernels at every T (one token up), so the cases
span T = 1 .. 16 as well as several 64-token chunks and token tiles."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext
from oracle import moe
from conftest import oracle_layer
from parity import check_layer

pytestmark = pytest.mark.gpu

SMALL = dict(latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)


@pytest.fixture(scope="module")
def dev():
    from synth import device
    return device


@pytest.fixture(scope="module")
def small(dev):
    inp = synth.make_layer(synth.LayerSpec(seed=41, layer=0, zipf=0.7, groups=4, shared_group=1, **SMALL))
    d = dev.DeviceLayer(inp, max_tokens=300)
    yield d, oracle_layer(inp)
    d.close()


@pytest.mark.parametrize("T", [1, 2, 7, 16, 17, 64, 65, 300])
def test_grouped_layer_matches_oracle(small, dev, T):
    d, lay = small
    x_bits = synth.tokens_bf16(500 + T, T, d.spec.hidden)
    y = d.forward(dev.bf16_tensor(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    r = d.routing(T)
    # the tokens' experts span several groups
    assert max(len(set(lay.labels[row])) for row in r["idx"]) > 1
    m = check_layer(d, lay, x_bits, dev.bf16_bits(y), r)
    assert m["tokens"] == T


@pytest.mark.parametrize("T", [5, 130])
def test_grouped_stage_tensors(small, dev, T):
    d, lay = small
    x_bits = synth.tokens_bf16(77 + T, T, d.spec.hidden)
    d.forward(dev.bf16_tensor(x_bits))
    torch.cuda.synchronize()
    ref = moe.grouped_layer_forward(lay, x_bits, want=("z", "logits"))
    # z of every group, f16 times a power of two per token
    z = d.debug_tensor(0, T)
    assert z.shape == ref["z"].shape == (T, 4 * d.spec.latent)
    ratio = (z * ref["z"]).sum(axis=1) / (ref["z"] ** 2).sum(axis=1)
    scale = 2.0 ** np.round(np.log2(ratio))
    zz = z / scale[:, None]
    assert np.all(np.abs(zz - ref["z"]) <= 2.0 ** -10 * np.abs(ref["z"]) + 1e-6 / scale[:, None])
    # each expert's logit scores its own group's latent (folded router, two bf16 halves)
    lg = d.debug_tensor(1, T)
    assert np.abs(lg - ref["logits"]).max() <= 1e-4 * max(1.0, np.abs(ref["logits"]).max())
    # c per group (bf16), against the oracle on the GPU's routing; unused groups are zero
    r = d.routing(T)
    c_ref = moe.grouped_layer_forward(lay, x_bits, idx_override=r["idx"], want=("c",))["c"]
    c = d.debug_tensor(2, T)
    assert np.linalg.norm(c - c_ref) / np.linalg.norm(c_ref) < 5e-3
    assert np.array_equal(c == 0, c_ref == 0)


def test_grouped_deterministic_and_token_order(small, dev):
    d, _ = small
    T = 40
    x_bits = synth.tokens_bf16(91, T, d.spec.hidden)
    y = dev.bf16_bits(d.forward(dev.bf16_tensor(x_bits)))
    assert np.array_equal(y, dev.bf16_bits(d.forward(dev.bf16_tensor(x_bits))))
    p = np.random.default_rng(5).permutation(T)
    assert np.array_equal(dev.bf16_bits(d.forward(dev.bf16_tensor(x_bits[p]))), y[p])


def test_grouped_stack_chains_the_layer_forwards(dev):
    """The stack call on grouped layers is the layer forwards with the residual norm
    between them, bit for bit."""
    ds = [dev.DeviceLayer(synth.make_layer(synth.LayerSpec(seed=50 + i, layer=i, groups=2, **SMALL)),
                          max_tokens=16) for i in range(2)]
    T, H = 3, SMALL["hidden"]
    x = dev.bf16_tensor(synth.tokens_bf16(4, T, H))
    y = torch.empty_like(x)
    ext.edge0_moe_stack_forward([d.handle for d in ds], x, y, T, 1e-6)
    cur, tmp = x.clone(), torch.empty_like(x)
    for d in ds:
        d.forward(cur, tmp)
        ext.edge0_residual_rmsnorm(cur, tmp, cur, T, H, 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(dev.bf16_bits(y), dev.bf16_bits(cur))
    for d in ds:
        d.close()


def test_grouped_layer_145b_shapes(dev):
    """Eight groups of 64 experts at the 145B widths (latent 1792, 512 experts, top 10)."""
    spec = synth.LayerSpec(seed=7, layer=0, latent=synth.LATENT_145B, groups=8, shared_group=3)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=64)
    lay = oracle_layer(inp)
    for T in (1, 8, 64):
        x_bits = synth.tokens_bf16(40 + T, T, spec.hidden)
        y = d.forward(dev.bf16_tensor(x_bits))
        torch.cuda.synchronize()
        r = d.routing(T)
        tokens = None if T <= 8 else np.array([0, 21, 63])
        check_layer(d, lay, x_bits, dev.bf16_bits(y), r, tokens=tokens)
    d.close()


def test_grouped_argument_checks(small, dev):
    d, _ = small
    s = d.spec
    # a label outside [0, G) is refused when the handle is made (read back on the host)
    bad = torch.from_numpy(np.where(np.arange(s.n_experts) == 5, 4, d.inputs.labels).astype(np.int32)).cuda()
    with pytest.raises(ext.Edge0Error) as ei:
        ext.MoELayer(hidden=s.hidden, latent=s.latent, n_experts=s.n_experts, top_k=s.top_k, ffn=s.ffn,
                     max_tokens=16, D=d.D, U=d.U, router=d.R, router_bias=d.bias, experts=d.records,
                     expert_stride=d.stride, shared_expert=d.shared, n_groups=4, expert_group=bad,
                     shared_group=0)
    assert ei.value.status == ext.EDGE0_ERR_INVALID_ARG
    # residency tiering and the allocation-free entry serve one group only
    host = torch.empty(1, dtype=torch.uint8).pin_memory()
    assert ext.lib().edge0_moe_tier_attach(d.handle, ctypes.c_void_p(host.data_ptr()), 1, None) == \
        ext.EDGE0_ERR_UNSUPPORTED
    x = dev.bf16_tensor(synth.tokens_bf16(1, 1, s.hidden))
    y = torch.empty_like(x)
    desc = ext.edge0_moe_desc(s.hidden, s.latent, s.n_experts, s.top_k, s.ffn, 0, d.D.data_ptr(),
                              d.U.data_ptr(), d.R.data_ptr(), d.bias.data_ptr(), d.records.data_ptr(),
                              d.stride, d.shared.data_ptr(), 4, d.labels.data_ptr(), 1)
    assert ext.lib().edge0_moe_forward_noalloc(ctypes.byref(desc), ctypes.c_void_p(x.data_ptr()),
                                               ctypes.c_void_p(y.data_ptr()), 1, None, None) == \
        ext.EDGE0_ERR_UNSUPPORTED
