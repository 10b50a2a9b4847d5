"""Comparison of the CUDA path against the oracle (shared by the GPU tests and smoke).

The tolerances, the routing-flip rule and the teacher-forced stack chain live in
``oracle.compare`` (test infrastructure), which the bench's parity report uses too."""
from __future__ import annotations

import numpy as np

from oracle import moe
from oracle.compare import (GAP, MAX_ABS, REL_L2, error_metrics, layer_check_metrics,  # noqa: F401
                            routing_flips, stack_chain, stack_rel_l2)


def check_layer(dev, lay, x_bits: np.ndarray, y_gpu_bits: np.ndarray, routing: dict,
                tokens=None, check_perm=True):
    """Oracle comparison of one layer forward.  ``tokens`` restricts the y/route
    checks to a sample of token rows (the permutation is always checked whole)."""
    T, k = routing["idx"].shape
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ref = moe.layer_forward(lay, x_bits[sel], want=("logits", "idx", "w"))
    gidx = routing["idx"][sel]
    flipped, bad = routing_flips(gidx, ref["logits"], k)
    assert not bad, f"routing differs beyond near-ties at tokens {bad[:8]}"
    if flipped:
        ref = moe.layer_forward(lay, x_bits[sel], idx_override=gidx, want=("logits", "idx", "w"))
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
    assert mx <= MAX_ABS, f"max abs / rms {mx:.3e}"
    return dict(rel_l2=rel, max_abs_over_rms=mx, flips=len(flipped), tokens=len(sel))

