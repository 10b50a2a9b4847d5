"""Parity of the CUDA prefill path (T > 16) with the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext
from oracle import moe
from conftest import oracle_layer
from parity import check_layer, error_metrics, routing_flips

pytestmark = pytest.mark.gpu

SMALL = dict(latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)


def small_spec(seed=0, layer=0, zipf=0.0, **over):
    kw = dict(SMALL)
    kw.update(over)
    return synth.LayerSpec(seed=seed, layer=layer, zipf=zipf, **kw)


def dev_bf16(b):
    from synth import device
    return device.bf16_tensor(b)


def bits(t):
    from synth import device
    return device.bf16_bits(t)


@pytest.fixture(scope="module")
def dev():
    from synth import device
    return device


@pytest.fixture(scope="module")
def small(dev):
    inp = synth.make_layer(small_spec(seed=17, zipf=0.7))
    d = dev.DeviceLayer(inp, max_tokens=1100)
    yield d, oracle_layer(inp)
    d.close()


@pytest.mark.parametrize("T", [17, 40, 64, 65, 300, 1000, 1100])
def test_prefill_small_shapes(small, T):
    """Whole-tensor parity; T spans one chunk, ragged chunks and several token tiles."""
    d, lay = small
    x_bits = synth.tokens_bf16(300 + T, T, d.spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    m = check_layer(d, lay, x_bits, bits(y), d.routing(T))
    assert m["tokens"] == T


def test_prefill_stage_tensors(small):
    d, lay = small
    T = 130
    x_bits = synth.tokens_bf16(11, T, d.spec.hidden)
    d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    ref = moe.layer_forward(lay, x_bits, want=("z", "logits", "c", "idx"))
    # z is emitted in f16 times a power of two per token (below 1 in magnitude):
    # within one f16 rounding of the exact value (plus fp32 sums)
    z = d.debug_tensor(0, T)
    assert np.abs(z).max() < 1.0
    ratio = (z * ref["z"]).sum(axis=1) / (ref["z"] ** 2).sum(axis=1)
    scale = 2.0 ** np.round(np.log2(ratio))
    zz = z / scale[:, None]
    assert np.all(np.abs(zz - ref["z"]) <= 2.0 ** -10 * np.abs(ref["z"]) + 1e-6 / scale[:, None])
    # logits from the folded router in two bf16 halves, fp32 accumulation
    lg = d.debug_tensor(1, T)
    assert np.abs(lg - ref["logits"]).max() <= 1e-4 * max(1.0, np.abs(ref["logits"]).max())
    r = d.routing(T)
    c_ref = moe.layer_forward(lay, x_bits, idx_override=r["idx"], want=("c",))["c"]
    c = d.debug_tensor(2, T)
    assert np.linalg.norm(c - c_ref) / np.linalg.norm(c_ref) < 5e-3


def test_prefill_deterministic_and_token_order(small):
    d, _ = small
    T = 200
    x_bits = synth.tokens_bf16(78, T, d.spec.hidden)
    y = bits(d.forward(dev_bf16(x_bits)))
    y2 = bits(d.forward(dev_bf16(x_bits)))
    assert np.array_equal(y, y2)                       # run-to-run deterministic
    p = np.random.default_rng(2).permutation(T)
    yp = bits(d.forward(dev_bf16(x_bits[p])))
    # a token's result does not depend on where the other tokens sit
    assert np.array_equal(yp, y[p])


def test_prefill_every_token_on_the_same_experts(dev):
    """A dominant bias sends all T tokens to experts 0..k-1: groups of T rows,
    several 256-row token tiles each, ragged last tile, all other groups empty."""
    spec = small_spec(seed=3)
    inp = synth.make_layer(spec)
    inp.bias = np.zeros(spec.n_experts, np.float32)
    inp.bias[:spec.top_k] = 100.0 + 20.0 * np.arange(spec.top_k, 0, -1, dtype=np.float32)
    T = 600
    d = dev.DeviceLayer(inp, max_tokens=T)
    lay = oracle_layer(inp)
    x_bits = synth.tokens_bf16(5, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    r = d.routing(T)
    assert np.array_equal(r["idx"], np.tile(np.arange(spec.top_k), (T, 1)))
    assert r["counts"][:spec.top_k].tolist() == [T] * spec.top_k and r["counts"][spec.top_k:].sum() == 0
    check_layer(d, lay, x_bits, bits(y), r)
    d.close()


def test_prefill_zero_routed_experts_leave_the_shared_path(dev):
    spec = small_spec(seed=8)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=100)
    stride = d.stride
    L, F = spec.latent, spec.ffn
    nc = synth.expert_sizes(L, F)[0]
    # zero every code byte of each routed record (scales and globals stay)
    gu_row, d_pair = 9 * L // 8, 9 * F // 8
    for e in range(spec.n_experts):
        base = e * stride
        rec = d.records[base:base + F * gu_row].view(F, gu_row)
        rec[:, :L].zero_()
        dblk = d.records[base + F * gu_row:base + F * gu_row + (L // 2) * d_pair].view(L // 2, d_pair)
        dblk[:, :F].zero_()
    zero = lambda e: (np.zeros_like(inp.expert(e)[0]), inp.expert(e)[1], inp.expert(e)[2])
    lay = moe.Layer(inp.D, inp.U, inp.R, inp.bias, zero, inp.shared, L, F, spec.top_k)
    T = 100
    x_bits = synth.tokens_bf16(9, T, spec.hidden)
    y = bits(d.forward(dev_bf16(x_bits)))
    ref = moe.layer_forward(lay, x_bits)["y"]
    rel, mx = error_metrics(y, ref)
    assert rel < 1e-2 and mx < 3e-2
    assert nc > 0
    d.close()


def test_prefill_invalid_arguments(small):
    d, _ = small
    T = 1101
    x = torch.zeros((T, d.spec.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(ext.Edge0Error) as ei:
        ext.edge0_moe_forward(d.handle, x, y, T)        # above max_tokens
    assert ei.value.status == ext.EDGE0_ERR_INVALID_ARG
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK


def test_prefill_stack_chain(dev):
    """T > 16 stacks chain layer calls and the residual norm; compare with the oracle
    stack forced to each layer's GPU routing (per-layer calls reproduce the stack bits)."""
    from parity import chain_amplification, check_layer as _cl, stack_chain, stack_e2e_bound
    n_layers, T = 3, 48
    specs = [small_spec(seed=5, layer=l, zipf=(0.0 if l % 2 == 0 else 1.1)) for l in range(n_layers)]
    inps = [synth.make_layer(s) for s in specs]
    devs = [dev.DeviceLayer(i, max_tokens=T) for i in inps]
    lays = [oracle_layer(i) for i in inps]
    H = specs[0].hidden
    x_bits = synth.tokens_bf16(6, T, H)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ext.edge0_moe_stack_forward([d.handle for d in devs], dev_bf16(x_bits), y, T, 1e-6)
    torch.cuda.synchronize()
    cur, idx_layers, rels = dev_bf16(x_bits), [], []
    for l, d in enumerate(devs):
        yl = d.forward(cur)
        torch.cuda.synchronize()
        r = d.routing(T)
        idx_layers.append(r["idx"])
        rels.append(_cl(d, lays[l], bits(cur), bits(yl), r, check_perm=False)["rel_l2"])
        nx = torch.empty_like(cur)
        ext.edge0_residual_rmsnorm(cur, yl, nx, T, H, 1e-6)
        cur = nx
    torch.cuda.synchronize()
    assert np.array_equal(bits(cur), bits(y))
    xf, _, _ = stack_chain(lays, x_bits, idx_layers)
    got, ref = moe.bf16_to_f64(bits(y)), moe.bf16_to_f64(xf)
    bound = stack_e2e_bound(rels, chain_amplification(lays, x_bits[:8], [r[:8] for r in idx_layers]))
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= bound
    for d in devs:
        d.close()


def _full_routing_check(lay, x_bits, r):
    """Routing of every token against the oracle's fp64 logits (flips only at near-ties)."""
    x = moe.bf16_to_f64(x_bits)
    logits = moe.router_logits(moe.d_projection(x, lay.D), lay.R, lay.bias)
    flipped, bad = routing_flips(r["idx"], logits, lay.k)
    assert not bad, f"routing differs beyond near-ties at tokens {bad[:8]}"
    counts, offsets, perm, pos = moe.permutation(r["idx"], lay.n_experts)
    assert np.array_equal(r["counts"], counts)
    assert np.array_equal(r["offsets"], offsets)
    assert np.array_equal(r["perm"], perm)
    assert np.array_equal(r["pos"], pos)
    return len(flipped)


def test_layer_145b_t4096_zipf(dev):
    spec = synth.LayerSpec(seed=3, layer=0, latent=1792, zipf=1.1)
    inp = synth.make_layer(spec)
    T = 4096
    d = dev.DeviceLayer(inp, max_tokens=T)
    lay = oracle_layer(inp)
    x_bits = synth.tokens_bf16(3, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    r = d.routing(T)
    flips = _full_routing_check(lay, x_bits, r)
    # the largest group spans many token tiles; sample its tokens and others
    rng = np.random.default_rng(33)
    big = int(np.argmax(r["counts"]))
    in_big = np.nonzero((r["idx"] == big).any(axis=1))[0]
    sel = np.unique(np.concatenate([rng.choice(in_big, 64, replace=False), rng.choice(T, 128, replace=False),
                                    [0, T - 1]]))
    m = check_layer(d, lay, x_bits, bits(y), r, tokens=sel, check_perm=False)
    print("layer145b_t4096_zipf", m, "flips(all tokens)", flips, "max group", int(r["counts"].max()))
    d.close()


def test_layer_145b_t16384_uniform(dev):
    spec = synth.LayerSpec(seed=4, layer=0, latent=1792)
    inp = synth.make_layer(spec)
    T = 16384
    d = dev.DeviceLayer(inp, max_tokens=T)
    lay = oracle_layer(inp)
    x_bits = synth.tokens_bf16(4, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    r = d.routing(T)
    flips = _full_routing_check(lay, x_bits, r)
    sel = np.unique(np.concatenate([np.random.default_rng(44).choice(T, 96, replace=False), [0, T - 1]]))
    m = check_layer(d, lay, x_bits, bits(y), r, tokens=sel, check_perm=False)
    print("layer145b_t16384", m, "flips(all tokens)", flips)
    d.close()


def test_prefill_generic_topk_path(dev):
    """E = 96 (not a power-of-two multiple of 32) takes the shared-memory top-k kernel."""
    spec = small_spec(seed=21, n_experts=96, top_k=6, zipf=0.9)
    inp = synth.make_layer(spec)
    T = 150
    d = dev.DeviceLayer(inp, max_tokens=T)
    x_bits = synth.tokens_bf16(31, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    check_layer(d, oracle_layer(inp), x_bits, bits(y), d.routing(T))
    d.close()


@pytest.mark.parametrize("zipf", [0.0, 1.1])
def test_prefill_t16384_bit_reproducible(dev, zipf):
    """Repeated forwards of a full-size layer give identical bits (every tile of
    every stage writes each output once; no cross-stage buffer is reused early)."""
    spec = synth.LayerSpec(seed=4, layer=1, latent=1792, zipf=zipf)
    T = 16384
    d = dev.DeviceLayer(synth.make_layer(spec), max_tokens=T)
    x = dev_bf16(synth.tokens_bf16(4000, T, spec.hidden))
    ys = []
    for _ in range(6):
        y = torch.empty_like(x)
        ext.edge0_moe_forward(d.handle, x, y, T)
        torch.cuda.synchronize()
        ys.append(bits(y))
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    d.close()


@pytest.mark.parametrize("T", [17, 64, 65, 300, 800])
def test_prefill_partial_output_tiles(dev, T):
    """hidden = 576 is two 256-column output tiles and a partial third: the D GEMM's
    latent and router columns and the U GEMM's columns end inside a tile, with the
    tokens on the MMA's N side (T <= 64), the U GEMM split along K (T <= 768) and
    neither (T = 800)."""
    inp = synth.make_layer(small_spec(seed=29, hidden=576, zipf=0.4))
    d = dev.DeviceLayer(inp, max_tokens=800)
    lay = oracle_layer(inp)
    x_bits = synth.tokens_bf16(70 + T, T, 576)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    sel = None if T <= 300 else np.arange(0, T, 7)
    # outputs here reach 5x their rms, where half a bf16 ulp is already 1 % of it
    m = check_layer(d, lay, x_bits, bits(y), d.routing(T), tokens=sel, out_ulp=True)
    assert m["tokens"] == (T if sel is None else len(sel))
    d.close()
