"""The allocation-free decode forward against the handle-based forward (GPU).

Some callers cannot call cudaMalloc (a host program that owns all device
memory, a plug-in under a fixed budget, a real-time loop); they use
edge0_moe_forward_noalloc, whose scratch is a static array inside the library.
Collected last so that a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext
from oracle import moe
from parity import MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu


def _noalloc(dl, x, T):
    s = dl.spec
    y = torch.empty_like(x)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ext.edge0_moe_forward_noalloc(s.hidden, s.latent, s.n_experts, s.top_k, s.ffn, dl.D, dl.U, dl.R,
                                  dl.bias, dl.records, dl.stride, dl.shared, x, y, T, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y


def _close(a, b):
    ya = moe.bf16_to_f64(a.view(torch.int16).cpu().numpy().view(np.uint16))
    yb = moe.bf16_to_f64(b.view(torch.int16).cpu().numpy().view(np.uint16))
    rel = np.linalg.norm(ya - yb) / np.linalg.norm(yb)
    mx = np.abs(ya - yb).max() / np.sqrt(np.mean(yb ** 2))
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


@pytest.mark.parametrize("shape", ["small", "145b"])
def test_noalloc_matches_handle_forward_twice(shape):
    from synth import device
    if shape == "small":
        spec = synth.LayerSpec(seed=4, layer=0, latent=256, hidden=512, n_experts=64, top_k=4, ffn=128,
                               zipf=0.5)
        T = 5
    else:
        spec = synth.LayerSpec(seed=0, layer=0, latent=1792)
        T = 1
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=16)
    x = device.bf16_tensor(synth.tokens_bf16(21, T, spec.hidden))
    ref = dl.forward(x)
    torch.cuda.synchronize()
    for _ in range(2):                 # the static scratch keeps the last call's contents
        _close(_noalloc(dl, x, T), ref)
    dl.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from synth import device
    spec = synth.LayerSpec(seed=4, layer=0, latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=32)
    x = torch.zeros((17, spec.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(ext.Edge0Error) as ei:
        ext.edge0_moe_forward_noalloc(spec.hidden, spec.latent, spec.n_experts, spec.top_k, spec.ffn, dl.D,
                                      dl.U, dl.R, dl.bias, dl.records, dl.stride, dl.shared, x, y, 17)
    assert ei.value.status == ext.EDGE0_ERR_UNSUPPORTED
    dl.close()
