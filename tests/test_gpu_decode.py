"""Parity of the CUDA decode path (T <= 16) with the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext
from oracle import moe, nvfp4, record
from conftest import oracle_layer
from parity import check_layer, error_metrics

pytestmark = pytest.mark.gpu

SMALL = dict(latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)


def small_spec(seed=0, layer=0, zipf=0.0, **over):
    kw = dict(SMALL)
    kw.update(over)
    return synth.LayerSpec(seed=seed, layer=layer, zipf=zipf, **kw)


@pytest.fixture(scope="module")
def dev():
    from synth import device
    return device


@pytest.fixture(scope="module")
def small(dev):
    inp = synth.make_layer(small_spec(seed=7, zipf=0.5))
    d = dev.DeviceLayer(inp, max_tokens=16)
    yield d, oracle_layer(inp)
    d.close()


def test_device_fill_matches_host_generator(dev):
    for latent, ffn, seed, layer, e0 in ((256, 128, 3, 1, 5), (1792, 640, 0, 0, 511)):
        codes, scales, glob = dev.fill_experts(seed, layer, e0, 2, latent, ffn)
        nc, ns = synth.expert_sizes(latent, ffn)
        for i in range(2):
            hc, hs, hg = synth.expert_bytes(seed, layer, e0 + i, latent, ffn)
            assert np.array_equal(codes[i * nc:(i + 1) * nc].cpu().numpy(), hc)
            assert np.array_equal(scales[i * ns:(i + 1) * ns].cpu().numpy(), hs)
            assert np.array_equal(glob[i * 3:(i + 1) * 3].cpu().numpy(), hg)


def test_device_packer_matches_record_layout(dev):
    L, F = 256, 128
    codes, scales, glob = dev.fill_experts(11, 2, 0, 3, L, F)
    glob.copy_(torch.tensor([0.5, 2.0, 1.25] * 3, device="cuda"))
    stride = ext.edge0_expert_record_stride(L, F)
    rec = torch.full((3 * stride,), 0xAB, dtype=torch.uint8, device="cuda")
    ext.edge0_pack_experts(codes, scales, glob, 3, L, F, rec, stride)
    torch.cuda.synchronize()
    nc, ns = synth.expert_sizes(L, F)
    rb = rec.cpu().numpy()
    for i in range(3):
        c, s, g = record.read_record(rb[i * stride:(i + 1) * stride], L, F)
        assert np.array_equal(c, codes[i * nc:(i + 1) * nc].cpu().numpy())
        assert np.array_equal(s, scales[i * ns:(i + 1) * ns].cpu().numpy())
        assert np.array_equal(g, np.float32([0.5, 2.0, 1.25]))
        # bytes past the record up to the stride are untouched
        assert np.all(rb[i * stride + record.record_bytes(L, F):(i + 1) * stride] == 0xAB)


def test_quantizer_matches_oracle_bit_exact():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 50, size=(64, 1))).astype(np.float32)
    w[3, :16] = 0.0                       # an all-zero block
    w[4, 5] = 1e6                         # saturating scale
    for g in (1.0, 0.37):
        wt = torch.from_numpy(w).cuda()
        codes = torch.empty(64 * 256, dtype=torch.uint8, device="cuda")
        scales = torch.empty(64 * 32, dtype=torch.uint8, device="cuda")
        ext.edge0_quantize_nvfp4(wt, 64, 512, g, codes, scales)
        torch.cuda.synchronize()
        qc, qs = nvfp4.quantize(w, g)
        assert np.array_equal(scales.cpu().numpy().reshape(64, 32), qs)
        assert np.array_equal(codes.cpu().numpy().reshape(64, 256), qc)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 13, 16])
def test_decode_small_shapes(small, T):
    d, lay = small
    x_bits = synth.tokens_bf16(100 + T, T, d.spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    r = d.routing(T)
    m = check_layer(d, lay, x_bits, bits(y), r)
    assert m["tokens"] == T


def dev_bf16(b):
    from synth import device
    return device.bf16_tensor(b)


def bits(t):
    from synth import device
    return device.bf16_bits(t)


def test_stage_tensors_match_oracle(small):
    d, lay = small
    T = 4
    x_bits = synth.tokens_bf16(42, T, d.spec.hidden)
    d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    ref = moe.layer_forward(lay, x_bits, want=("z", "logits", "c", "idx"))
    z = d.debug_tensor(0, T)
    assert np.abs(z - ref["z"]).max() <= 1e-5 * np.abs(ref["z"]).max()
    lg = d.debug_tensor(1, T)
    assert np.abs(lg - ref["logits"]).max() <= 1e-5 * max(1.0, np.abs(ref["logits"]).max())
    r = d.routing(T)
    c_ref = moe.layer_forward(lay, x_bits, idx_override=r["idx"], want=("c",))["c"]
    c = d.debug_tensor(2, T)
    assert np.linalg.norm(c - c_ref) / np.linalg.norm(c_ref) < 5e-3


def test_token_permutation_invariance_bit_exact(small):
    d, _ = small
    T = 9
    x_bits = synth.tokens_bf16(77, T, d.spec.hidden)
    p = np.random.default_rng(1).permutation(T)
    y = bits(d.forward(dev_bf16(x_bits)))
    yp = bits(d.forward(dev_bf16(x_bits[p])))
    assert np.array_equal(yp, y[p])
    y2 = bits(d.forward(dev_bf16(x_bits)))
    assert np.array_equal(y, y2)                       # run-to-run deterministic


@pytest.mark.parametrize("shape", ["small", "145b"])
def test_every_token_on_the_same_experts(dev, shape):
    """A router bias that dominates the logits sends every token to experts 0..k-1: at
    T = 16 every routed group has 16 tokens (two token tiles in the MMAs) and, at
    Edge0-145B shapes, every down group spans two units of the ring."""
    spec = small_spec(seed=3) if shape == "small" else synth.LayerSpec(seed=3, layer=0, latent=1792)
    inp = synth.make_layer(spec)
    inp.bias = np.zeros(spec.n_experts, np.float32)
    inp.bias[:spec.top_k] = 100.0 + 20.0 * np.arange(spec.top_k, 0, -1, dtype=np.float32)
    d = dev.DeviceLayer(inp, max_tokens=16)
    lay = oracle_layer(inp)
    T = 16
    x_bits = synth.tokens_bf16(5, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    r = d.routing(T)
    assert np.array_equal(r["idx"], np.tile(np.arange(spec.top_k), (T, 1)))
    assert r["counts"][:spec.top_k].tolist() == [T] * spec.top_k and r["counts"][spec.top_k:].sum() == 0
    check_layer(d, lay, x_bits, bits(y), r)
    d.close()


def test_exact_logit_ties_rank_by_lower_index(dev):
    """Exact ties repeated in every 32-expert chunk (router weights zero, logits = bias):
    the top-k ranks by (logit descending, index ascending), as the oracle does."""
    spec = small_spec(seed=4, n_experts=256, top_k=16)
    inp = synth.make_layer(spec)
    inp.R = np.zeros_like(inp.R)                   # logits are the bias exactly
    inp.bias = np.full(spec.n_experts, -100.0, np.float32)
    for c in range(spec.n_experts // 32):
        inp.bias[c * 32:c * 32 + 16] = 100.0 - np.arange(16, dtype=np.float32)
    d = dev.DeviceLayer(inp, max_tokens=16)
    lay = oracle_layer(inp)
    for T in (1, 5):
        x_bits = synth.tokens_bf16(31 + T, T, spec.hidden)
        y = d.forward(dev_bf16(x_bits))
        torch.cuda.synchronize()
        r = d.routing(T)
        want = np.concatenate([np.arange(0, 256, 32), np.arange(1, 256, 32)])
        assert np.array_equal(r["idx"], np.tile(want, (T, 1)))
        check_layer(d, lay, x_bits, bits(y), r)
    d.close()


def test_zero_routed_experts_leave_the_shared_path(dev):
    """Zeroed routed records (all codes 0): y equals U * shared(z), as in the oracle."""
    spec = small_spec(seed=8)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=16)
    stride = d.stride
    L, F = spec.latent, spec.ffn
    nc = synth.expert_sizes(L, F)[0]
    for e in range(spec.n_experts):
        d.records[e * stride:e * stride + nc].zero_()
    zero = lambda e: (np.zeros_like(inp.expert(e)[0]), inp.expert(e)[1], inp.expert(e)[2])
    lay = moe.Layer(inp.D, inp.U, inp.R, inp.bias, zero, inp.shared, L, F, spec.top_k)
    T = 3
    x_bits = synth.tokens_bf16(9, T, spec.hidden)
    y = bits(d.forward(dev_bf16(x_bits)))
    ref = moe.layer_forward(lay, x_bits)["y"]
    rel, mx = error_metrics(y, ref)
    assert rel < 1e-2 and mx < 3e-2
    d.close()


def test_residual_rmsnorm_matches_oracle():
    T, H = 5, 2560
    x = synth.tokens_bf16(1, T, H)
    y = synth.tokens_bf16(2, T, H)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ext.edge0_residual_rmsnorm(dev_bf16(x), dev_bf16(y), out, T, H, 1e-6)
    torch.cuda.synchronize()
    ref = moe.bf16_to_f64(moe.residual_rmsnorm(x, y))
    got = moe.bf16_to_f64(bits(out))
    # both round to bf16: at most one bf16 step apart
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)
    assert np.mean(got == ref) > 0.99


def test_invalid_arguments(small):
    d, _ = small
    x = torch.zeros((17, d.spec.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(ext.Edge0Error) as ei:
        ext.edge0_moe_forward(d.handle, x, y, 17)      # max_tokens is 16 for this handle
    assert ei.value.status == ext.EDGE0_ERR_INVALID_ARG
    with pytest.raises(ext.Edge0Error):
        ext.edge0_moe_forward(d.handle, x, x, 2)       # x and y overlap
    ext.edge0_moe_forward(d.handle, x, y, 0)          # T = 0 is a no-op
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK


def test_layer_145b_t1(dev):
    spec = synth.LayerSpec(seed=0, layer=0, latent=1792)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=16)
    x_bits = synth.tokens_bf16(0, 1, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    m = check_layer(d, oracle_layer(inp), x_bits, bits(y), d.routing(1))
    print("layer145b_t1", m)
    d.close()


@pytest.mark.parametrize("T", [4, 8, 11, 16])
def test_layer_145b_large_buckets(dev, T):
    """Verify-window buckets at Edge0-145B shapes: several waves of gate/up units
    through the ring, down units packing several experts, and at T = 16 the shared
    expert's slots split over two down units where its h rows do not fit one slot."""
    spec = synth.LayerSpec(seed=17, layer=0, latent=1792)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=16)
    x_bits = synth.tokens_bf16(170 + T, T, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    m = check_layer(d, oracle_layer(inp), x_bits, bits(y), d.routing(T))
    print(f"layer145b T={T}", m)
    d.close()


def test_layer_120b_t4(dev):
    spec = synth.LayerSpec(seed=1, layer=0, latent=1280)
    inp = synth.make_layer(spec)
    d = dev.DeviceLayer(inp, max_tokens=16)
    x_bits = synth.tokens_bf16(1, 4, spec.hidden)
    y = d.forward(dev_bf16(x_bits))
    torch.cuda.synchronize()
    m = check_layer(d, oracle_layer(inp), x_bits, bits(y), d.routing(4))
    print("layer120b_t4", m)
    d.close()


def test_stack_teacher_forced_and_end_to_end(dev):
    from parity import chain_amplification, layer_check_metrics, stack_chain, stack_e2e_bound
    n_layers, T = 4, 2
    specs = [small_spec(seed=2, layer=l, zipf=(0.0 if l % 2 == 0 else 1.1)) for l in range(n_layers)]
    inps = [synth.make_layer(s) for s in specs]
    devs = [dev.DeviceLayer(i, max_tokens=16) for i in inps]
    lays = [oracle_layer(i) for i in inps]
    x_bits = synth.tokens_bf16(2, T, specs[0].hidden)
    H, K = specs[0].hidden, specs[0].top_k
    tx = torch.empty((n_layers, T, H), dtype=torch.bfloat16, device="cuda")
    ty = torch.empty_like(tx)
    ti = torch.empty((n_layers, T, K), dtype=torch.int32, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ext.edge0_moe_stack_forward_trace([d.handle for d in devs], dev_bf16(x_bits), y, T, 1e-6, tx, ty, ti)
    torch.cuda.synchronize()
    txb, tyb, tib = bits(tx), bits(ty), ti.cpu().numpy()
    assert np.array_equal(txb[0], x_bits)
    rels = []
    for l in range(n_layers):
        # each layer checked on the GPU's own input to it and on its own routing
        rel, mx, _, bad = layer_check_metrics(lays[l], txb[l], tyb[l], tib[l])
        assert not bad and rel <= 1e-2 and mx <= 3e-2, (l, rel, mx, bad)
        rels.append(rel)
        if l + 1 < n_layers:
            nxt = moe.residual_rmsnorm(txb[l], tyb[l])
            assert np.mean(nxt == txb[l + 1]) > 0.99
    # the last layer's routing is also published through edge0_moe_debug_routing
    assert np.array_equal(devs[0].routing(T)["idx"], tib[-1])
    # end to end through the oracle stack forced to the GPU's routing
    xf, _, _ = stack_chain(lays, x_bits, tib)
    got = moe.bf16_to_f64(bits(y))
    ref = moe.bf16_to_f64(xf)
    bound = stack_e2e_bound(rels, chain_amplification(lays, x_bits, tib))
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= bound
    # the same stack through per-layer calls gives the same bits
    cur = dev_bf16(x_bits)
    for d in devs:
        yl = d.forward(cur)
        nx = torch.empty_like(cur)
        ext.edge0_residual_rmsnorm(cur, yl, nx, T, H, 1e-6)
        cur = nx
    torch.cuda.synchronize()
    assert np.array_equal(bits(cur), bits(y))
    for d in devs:
        d.close()


def test_stack_forward_replays_from_a_cuda_graph(dev):
    """A stack call captured into a CUDA graph (after one uncaptured call with the
    same layers) replays to the same bits as the direct call."""
    n_layers, T = 3, 1
    specs = [small_spec(seed=40, layer=l) for l in range(n_layers)]
    devs = [dev.DeviceLayer(synth.make_layer(s), max_tokens=16) for s in specs]
    handles = [d.handle for d in devs]
    H = specs[0].hidden
    x = dev_bf16(synth.tokens_bf16(41, T, H))
    y_direct = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ext.edge0_moe_stack_forward(handles, x, y_direct, T, 1e-6)
    torch.cuda.synchronize()
    y = torch.empty_like(y_direct)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ext.edge0_moe_stack_forward(handles, x, y, T, 1e-6, s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), bits(y_direct))
    assert ext.edge0_moe_get_error(handles[0]) == ext.EDGE0_OK
    del g
    for d in devs:
        d.close()
