"""Pins of the oracle's grouped latent projections (``moe.grouped_layer_forward``).

The grouped layer ("Edge0-145B hardware requirements", section "Edge0-145B latent
MoE architecture: how 145B fits one GPU": eight D/U groups per layer, each expert
labelled with its group) is pinned to the ungrouped layer, which its own tests pin:

  * with one group it is the ungrouped layer;
  * with G groups it equals the ungrouped layer of latent width G*l whose D and U
    are the stacked groups, whose router row for expert e sits in e's block and is
    zero elsewhere, and whose expert weights sit in their group's block with zero
    codes and scales elsewhere.  That identity fixes every place a group index is
    used: the router's input, each expert's input, the shared expert's group, the
    per-group combine and the sum over U_g.
"""
import numpy as np
import pytest

import synth
from conftest import oracle_layer, tiny_spec
from oracle import moe


def _embed_expert(src, g: int, G: int, latent: int, ffn: int):
    """Logical NVFP4 arrays of an expert of group g rewritten for latent G*latent."""
    codes, scales, glob = src
    (cg, sg), (cu, su), (cd, sd) = synth.split_expert(codes, scales, latent, ffn)
    l, F, W = latent, ffn, G * latent

    def rows_block(a, per):      # [F][per] -> [F][G*per], block g
        out = np.zeros((a.shape[0], G * per), dtype=np.uint8)
        out[:, g * per:(g + 1) * per] = a
        return out

    def cols_block(a, n):        # [n][x] -> [G*n][x], rows of block g
        out = np.zeros((G * n, a.shape[1]), dtype=np.uint8)
        out[g * n:(g + 1) * n] = a
        return out

    codes2 = np.concatenate([rows_block(cg, l // 2).ravel(), rows_block(cu, l // 2).ravel(),
                             cols_block(cd, l).ravel()])
    scales2 = np.concatenate([rows_block(sg, l // 16).ravel(), rows_block(su, l // 16).ravel(),
                              cols_block(sd, l).ravel()])
    assert codes2.size == 3 * F * W // 2 and scales2.size == 3 * F * W // 16
    return codes2, scales2, glob


def _embedded_layer(inp):
    s = inp.spec
    G, l, E = s.groups, s.latent, s.n_experts
    R2 = np.zeros((E, G * l), dtype=np.uint16)
    for e in range(E):
        g = int(inp.labels[e])
        R2[e, g * l:(g + 1) * l] = inp.R[e]
    ex = {}

    def expert(e):
        if e not in ex:
            ex[e] = _embed_expert(inp.expert(e), int(inp.labels[e]), G, l, s.ffn)
        return ex[e]

    def shared():
        return _embed_expert(inp.shared(), s.shared_group, G, l, s.ffn)

    return moe.Layer(inp.D, inp.U, R2, inp.bias, expert, shared, G * l, s.ffn, s.top_k)


def test_group_labels_split_the_experts_evenly():
    lab = synth.group_labels(3, 1, 512, 8)
    assert np.array_equal(np.bincount(lab, minlength=8), np.full(8, 64))
    assert not np.array_equal(lab, np.repeat(np.arange(8), 64))   # not contiguous blocks
    assert np.array_equal(synth.group_labels(3, 1, 512, 1), np.zeros(512, np.int32))
    one = synth.make_layer(tiny_spec(seed=5))
    assert one.D.shape == (64, 128) and one.U.shape == (128, 64)


def test_one_group_is_the_ungrouped_layer():
    inp = synth.make_layer(tiny_spec(seed=7, zipf=1.1))
    s = inp.spec
    grouped = moe.GroupedLayer(inp.D, inp.U, inp.R, inp.bias, inp.expert, inp.shared, s.latent, s.ffn,
                               s.top_k, np.zeros(s.n_experts), 0)
    x = synth.tokens_bf16(8, 6, s.hidden)
    want = ("z", "logits", "idx", "w", "c")
    a = moe.grouped_layer_forward(grouped, x, want=want)
    b = moe.layer_forward(oracle_layer(inp), x, want=want)
    assert np.array_equal(a["idx"], b["idx"])
    for k in ("y", "z", "logits", "w", "c"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-12 * np.abs(b[k]).max())


@pytest.mark.parametrize("groups,shared_group,zipf", [(4, 0, 0.0), (4, 3, 1.1), (2, 1, 0.0)])
def test_grouped_layer_is_the_block_embedded_layer(groups, shared_group, zipf):
    inp = synth.make_layer(tiny_spec(seed=11 + groups, groups=groups, shared_group=shared_group, zipf=zipf))
    x = synth.tokens_bf16(12, 9, inp.spec.hidden)
    want = ("z", "logits", "idx", "w", "c")
    lay, emb = oracle_layer(inp), _embedded_layer(inp)
    assert isinstance(lay, moe.GroupedLayer)
    a = moe.grouped_layer_forward(lay, x, want=want)
    b = moe.layer_forward(emb, x, want=want)
    assert np.array_equal(a["idx"], b["idx"])
    # the routed experts of a token span several groups (else the test pins little)
    assert max(len(set(inp.labels[row])) for row in a["idx"]) > 1
    for k in ("y", "z", "logits", "w", "c"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-11, atol=1e-11 * np.abs(b[k]).max())
    # teacher forcing through both paths with indices the oracle would not pick
    J = np.stack([np.roll(np.arange(inp.spec.n_experts), t)[: inp.spec.top_k] for t in range(x.shape[0])])
    a = moe.grouped_layer_forward(lay, x, idx_override=J, want=("w", "c"))
    b = moe.layer_forward(emb, x, idx_override=J, want=("w", "c"))
    for k in ("y", "w", "c"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-11, atol=1e-11 * np.abs(b[k]).max())


def test_unused_group_up_projection_has_no_effect():
    inp = synth.make_layer(tiny_spec(seed=21, groups=4, shared_group=0, n_experts=16, top_k=2))
    x = synth.tokens_bf16(13, 1, inp.spec.hidden)
    lay = oracle_layer(inp)
    ref = moe.grouped_layer_forward(lay, x, want=("idx",))
    used = set(int(inp.labels[e]) for e in ref["idx"][0]) | {0}
    l = inp.spec.latent
    for g in range(4):
        U2 = inp.U.copy()
        U2[:, g * l:(g + 1) * l] ^= np.uint16(0x8000)          # negate U_g
        lay2 = moe.GroupedLayer(inp.D, U2, inp.R, inp.bias, inp.expert, inp.shared, l, inp.spec.ffn,
                                inp.spec.top_k, inp.labels, 0)
        y2 = moe.grouped_layer_forward(lay2, x)["y"]
        if g in used:
            assert not np.allclose(y2, ref["y"])
        else:
            assert np.array_equal(y2, ref["y"])
    assert len(used) < 4          # at least one group unused by this token


def test_forward_dispatches_on_the_layer_kind():
    inp = synth.make_layer(tiny_spec(seed=2, groups=2))
    x = synth.tokens_bf16(3, 2, inp.spec.hidden)
    lay = oracle_layer(inp)
    np.testing.assert_array_equal(moe.forward(lay, x)["y"], moe.grouped_layer_forward(lay, x)["y"])
    inp1 = synth.make_layer(tiny_spec(seed=2))
    lay1 = oracle_layer(inp1)
    np.testing.assert_array_equal(moe.forward(lay1, x)["y"], moe.layer_forward(lay1, x)["y"])
