"""Comparison of the CUDA path against the oracle (shared by the GPU tests and smoke).

The tolerances, the routing-flip rule and the teacher-forced stack chain live in
``oracle.compare`` (test infrastructure), which the bench's parity report uses too."""
from __future__ import annotations

import numpy as np

from oracle import moe
from oracle.compare import (GAP, MAX_ABS, REL_L2, error_metrics, layer_check_metrics,  # noqa: F401
                            routing_flips, stack_chain, stack_rel_l2)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """One unit in the last place of bf16 at |v| (8 significant bits; 0 for v = 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    return np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 0.0)


def check_layer(dev, lay, x_bits: np.ndarray, y_gpu_bits: np.ndarray, routing: dict,
                tokens=None, check_perm=True, out_ulp=False):
    """Oracle comparison of one layer forward.  ``tokens`` restricts the y/route
    checks to a sample of token rows (the permutation is always checked whole).
    ``out_ulp``: the max-abs bound also allows one bf16 ulp of each output element (y
    is emitted in bf16), for shapes whose outputs reach many times their rms."""
    T, k = routing["idx"].shape
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ref = moe.forward(lay, x_bits[sel], want=("logits", "idx", "w"))
    gidx = routing["idx"][sel]
    flipped, bad = routing_flips(gidx, ref["logits"], k)
    assert not bad, f"routing differs beyond near-ties at tokens {bad[:8]}"
    if flipped:
        ref = moe.forward(lay, x_bits[sel], idx_override=gidx, want=("logits", "idx", "w"))
    w_ref = moe.routing_weights(ref["logits"], gidx)
    assert np.abs(routing["w"][sel] - w_ref).max() < 1e-5
    if check_perm:
        counts, offsets, perm, pos = moe.permutation(routing["idx"], lay.n_experts)
        assert np.array_equal(routing["counts"], counts)
        assert np.array_equal(routing["offsets"], offsets)
        assert np.array_equal(routing["perm"], perm)
        assert np.array_equal(routing["pos"], pos)
    rel, mx = error_metrics(y_gpu_bits[sel], ref["y"])
    assert rel <= REL_L2, f"rel L2 {rel:.3e}"
    if out_ulp:
        err = np.abs(moe.bf16_to_f64(y_gpu_bits[sel]) - ref["y"]) - bf16_ulp(ref["y"])
        mx = float(max(0.0, err.max()) / np.sqrt(np.mean(ref["y"] ** 2)))
    assert mx <= MAX_ABS, f"max abs / rms {mx:.3e}"
    return dict(rel_l2=rel, max_abs_over_rms=mx, flips=len(flipped), tokens=len(sel))



def chain_amplification(lays, x_bits: np.ndarray, idx_per_layer, seed: int = 99):
    """The oracle stack's own amplification of a rounding-level input change: one bf16
    ulp moved in a seeded tenth of the input elements, routing forced to the given
    indices in both runs.  Returns (relative output change) / (relative input change)."""
    xp = np.array(x_bits, dtype=np.uint16)
    xp[np.random.default_rng(seed).random(xp.shape) < 0.1] ^= np.uint16(1)
    x0, x1 = moe.bf16_to_f64(x_bits), moe.bf16_to_f64(xp)
    d_in = np.linalg.norm(x1 - x0) / np.linalg.norm(x0)
    f0 = moe.bf16_to_f64(stack_chain(lays, x_bits, idx_per_layer)[0])
    f1 = moe.bf16_to_f64(stack_chain(lays, xp, idx_per_layer)[0])
    return float(np.linalg.norm(f1 - f0) / np.linalg.norm(f0) / d_in)


def stack_e2e_bound(layer_rels, amplification: float) -> float:
    """End-to-end error the per-layer checks imply: the measured per-layer errors (each
    on the GPU's own input and routing) add in quadrature and are carried to the output
    with at most the chain's own measured amplification."""
    return float(np.sqrt(np.sum(np.square(layer_rels)))) * max(1.0, amplification)
