"""Failure detection on the GPU without a fault: a bounded device wait that runs
out must come back as EDGE0_ERR_TIMEOUT on the host, and the handle must stay usable."""
import numpy as np
import pytest
import torch

import synth
import latent_sparse_moe_router_b300 as ext
from conftest import oracle_layer
from parity import check_layer

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_the_handle_recovers():
    from synth import device
    spec = synth.LayerSpec(seed=12, layer=0, latent=256, hidden=512, n_experts=64, top_k=4, ffn=128)
    inp = synth.make_layer(spec)
    d = device.DeviceLayer(inp, max_tokens=64)
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    ext.edge0_moe_debug_wait_probe(d.handle)           # waits on an mbarrier nothing arrives at
    torch.cuda.synchronize()                           # the probe returned: the wait was bounded
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_ERR_TIMEOUT
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK   # reading cleared the word
    # both paths still run correctly on the same handle
    for T in (3, 40):
        x_bits = synth.tokens_bf16(900 + T, T, spec.hidden)
        y = d.forward(device.bf16_tensor(x_bits))
        torch.cuda.synchronize()
        check_layer(d, oracle_layer(inp), x_bits, device.bf16_bits(y), d.routing(T))
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    d.close()
