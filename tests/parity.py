"""Comparison of the CUDA path against the oracle (shared by the GPU tests and smoke)."""
from __future__ import annotations

import numpy as np

from oracle import moe

GAP = 1e-3        # routing flips allowed only where the oracle's logits are this close
REL_L2 = 1e-2     # relative L2 error of y over the whole output tensor
MAX_ABS = 3e-2    # max |y_gpu - y_oracle| <= MAX_ABS * rms(y_oracle)


def routing_flips(gpu_idx: np.ndarray, logits: np.ndarray, k: int):
    """Tokens whose GPU expert list (in rank order) differs from the oracle's.

    Returns (flipped token indices, bad token indices): a flip is legal only if
    every disagreement is between experts whose oracle logits differ by < GAP
    (an expert kept in place of another, or two experts ranked the other way).
    """
    flipped, bad = [], []
    for t in range(gpu_idx.shape[0]):
        l = logits[t]
        order = np.lexsort((np.arange(l.size), -l))
        ref = order[:k]
        g = gpu_idx[t]
        if np.array_equal(g, ref):
            continue
        flipped.append(t)
        ok = len(set(g.tolist())) == k
        extra = set(g.tolist()) - set(ref.tolist())
        missing = set(ref.tolist()) - set(g.tolist())
        for e in extra:
            for f in missing:
                ok &= (l[f] - l[e]) < GAP
        for i in range(k):
            for j in range(i + 1, k):
                if l[g[i]] < l[g[j]] or (l[g[i]] == l[g[j]] and g[i] > g[j]):
                    ok &= (l[g[j]] - l[g[i]]) < GAP
        if not ok:
            bad.append(t)
    return flipped, bad


def error_metrics(y_gpu_bits: np.ndarray, y_ref: np.ndarray):
    yg = moe.bf16_to_f64(y_gpu_bits)
    d = yg - y_ref
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(y_ref), 1e-300))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    mx = float(np.abs(d).max() / max(rms, 1e-300))
    return rel, mx


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
