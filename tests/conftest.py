import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


def oracle_layer(inputs):
    """Oracle view of a synth.LayerInputs (exact decode, experts on demand)."""
    from oracle import moe
    s = inputs.spec
    if s.groups > 1:
        return moe.GroupedLayer(inputs.D, inputs.U, inputs.R, inputs.bias, inputs.expert, inputs.shared,
                                s.latent, s.ffn, s.top_k, inputs.labels, s.shared_group)
    return moe.Layer(inputs.D, inputs.U, inputs.R, inputs.bias,
                     inputs.expert, inputs.shared, s.latent, s.ffn, s.top_k)


def tiny_spec(seed=0, layer=0, latent=64, hidden=128, n_experts=16, top_k=3, ffn=32, zipf=0.0, groups=1,
              shared_group=0):
    import synth
    return synth.LayerSpec(seed=seed, layer=layer, latent=latent, hidden=hidden,
                           n_experts=n_experts, top_k=top_k, ffn=ffn, zipf=zipf, groups=groups,
                           shared_group=shared_group)


@pytest.fixture
def rng():
    return np.random.default_rng(1234)
