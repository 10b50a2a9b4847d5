"""Expert residency tiering on the GPU: the layer's records in pinned host memory,
some of them cached in device slots.  Every decode forward must give the same bits
as the handle that reads all records from device memory, whatever is resident; the
miss counters must match the routing; rebalancing promotes the most-used experts."""
import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("shape", ["small", "145b"])
def test_tiered_forwards_match_the_resident_handle(shape):
    from synth import device
    if shape == "small":
        spec = synth.LayerSpec(seed=31, layer=0, latent=256, hidden=512, n_experts=64, top_k=4, ffn=128, zipf=1.1)
    else:
        spec = synth.LayerSpec(seed=3, layer=0, latent=1792, zipf=1.1)
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=16)
    host = torch.empty(dl.records.numel(), dtype=torch.uint8, pin_memory=True)
    host.copy_(dl.records.cpu())
    tl = ext.MoELayer(hidden=spec.hidden, latent=spec.latent, n_experts=spec.n_experts, top_k=spec.top_k,
                      ffn=spec.ffn, max_tokens=16, D=dl.D, U=dl.U, router=dl.R, router_bias=dl.bias,
                      experts=dl.records, expert_stride=dl.stride, shared_expert=dl.shared)
    E, K = spec.n_experts, spec.top_k
    n_slots = E // 4
    ext.edge0_moe_tier_attach(tl.handle, host, n_slots)
    xs = [device.bf16_tensor(synth.tokens_bf16(400 + i, T, spec.hidden)) for i, T in enumerate((1, 3, 16, 1, 4))]
    expected_misses = 0

    def run_all(resident):
        nonlocal expected_misses
        for x in xs:
            T = x.shape[0]
            ref = dl.forward(x)
            y = torch.empty_like(x)
            ext.edge0_moe_forward(tl.handle, x, y, T)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(y), _bits(ref))
            used = set(np.unique(dl.routing(T)["idx"]).tolist())
            expected_misses += len(used - resident)

    run_all(set())                                        # nothing resident: every expert from host memory
    st = ext.edge0_moe_tier_stats(tl.handle)
    assert st["forwards"] == len(xs) and st["misses"] == expected_misses and st["resident"] == 0
    assert st["host_bytes"] == expected_misses * dl.stride
    place = list(range(0, 2 * n_slots, 2))                # every other expert
    ext.edge0_moe_tier_place(tl.handle, place)
    run_all(set(place))
    assert ext.edge0_moe_tier_stats(tl.handle)["misses"] == expected_misses
    ext.edge0_moe_tier_rebalance(tl.handle)               # the most-used of the 10 forwards so far
    st = ext.edge0_moe_tier_stats(tl.handle)
    assert 0 < st["resident"] <= n_slots
    before = st["misses"]
    for x in xs:
        y = torch.empty_like(x)
        ext.edge0_moe_forward(tl.handle, x, y, x.shape[0])
        assert np.array_equal(_bits(y), _bits(dl.forward(x)))
    torch.cuda.synchronize()
    # the inputs repeat: the experts they use most are now resident, so fewer misses
    assert ext.edge0_moe_tier_stats(tl.handle)["misses"] - before < expected_misses / 2
    assert ext.edge0_moe_get_error(tl.handle) == ext.EDGE0_OK
    ext.edge0_moe_tier_detach(tl.handle)
    y = torch.empty_like(xs[0])
    ext.edge0_moe_forward(tl.handle, xs[0], y, 1)
    assert np.array_equal(_bits(y), _bits(dl.forward(xs[0])))
    tl.close()
    dl.close()


def test_tiering_refuses_what_it_does_not_serve():
    from synth import device
    spec = synth.LayerSpec(seed=32, layer=0, latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=64)
    host = torch.empty(dl.records.numel(), dtype=torch.uint8, pin_memory=True)
    with pytest.raises(ext.Edge0Error) as ei:              # a prefill-capable handle
        ext.edge0_moe_tier_attach(dl.handle, host, 8)
    assert ei.value.status == ext.EDGE0_ERR_UNSUPPORTED
    d16 = device.DeviceLayer(synth.make_layer(spec), max_tokens=16)
    pageable = np.zeros(dl.records.numel(), np.uint8)
    with pytest.raises(ext.Edge0Error) as ei:              # host memory the device cannot map
        ext.edge0_moe_tier_attach(d16.handle, pageable, 8)
    assert ei.value.status == ext.EDGE0_ERR_INVALID_ARG
    with pytest.raises(ext.Edge0Error):                    # not attached
        ext.edge0_moe_tier_rebalance(d16.handle)
    dl.close()
    d16.close()
