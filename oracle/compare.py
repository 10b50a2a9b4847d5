"""Comparison of another implementation's layer outputs with the oracle (test
infrastructure, like the rest of this package).

Tolerances and routing-flip rule of the parity checks:
  * expert indices must equal the oracle's top-k, except where the oracle's logits
    of the experts involved differ by less than GAP (a near-tie; counted as a flip);
  * outputs: relative L2 error <= REL_L2 over the compared tensor, and
    max |y - y_oracle| <= MAX_ABS * rms(y_oracle);
  * where a flip occurred, the oracle is re-run on the other implementation's
    indices (teacher forcing of the routing), so a legal flip is not an error.
"""
from __future__ import annotations

import numpy as np

from . import moe

GAP = 1e-3        # routing flips allowed only where the oracle's logits are this close
REL_L2 = 1e-2     # relative L2 error of y over the whole output tensor
MAX_ABS = 3e-2    # max |y_gpu - y_oracle| <= MAX_ABS * rms(y_oracle)


def stack_rel_l2(n_layers: int) -> float:
    """End-to-end tolerance of an n-layer stack output (post-norm residual chain).

    Every layer is held to REL_L2 against the oracle on the same input and the same
    routing; the residual carries each layer's error forward, and errors of different
    layers are independent, so they add in quadrature: REL_L2 * sqrt(n_layers)."""
    return REL_L2 * float(np.sqrt(n_layers))


def routing_flips(gpu_idx: np.ndarray, logits: np.ndarray, k: int):
    """Tokens whose expert list (in rank order) differs from the oracle's.

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
    """(relative L2 error, max abs error / rms of the reference) of bf16 outputs."""
    yg = moe.bf16_to_f64(y_gpu_bits)
    d = yg - y_ref
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(y_ref), 1e-300))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    mx = float(np.abs(d).max() / max(rms, 1e-300))
    return rel, mx


def layer_check_metrics(lay, x_bits: np.ndarray, y_gpu_bits: np.ndarray, gidx: np.ndarray):
    """One layer on the other implementation's input and routing:
    (rel L2, max abs / rms, flipped token count, bad token list)."""
    ref = moe.forward(lay, x_bits, want=("logits",))
    flipped, bad = routing_flips(gidx, ref["logits"], lay.k)
    if flipped:
        ref = moe.forward(lay, x_bits, idx_override=gidx)
    rel, mx = error_metrics(y_gpu_bits, ref["y"])
    return rel, mx, len(flipped), bad


def stack_chain(lays, x_bits: np.ndarray, idx_per_layer, eps: float = 1e-6):
    """The oracle stack with every layer's routing forced to the given indices
    (teacher forcing of the routing only: each layer runs on the chain's own input).
    Returns (final x bits, flipped token count, bad (layer, token) list): flips compare
    the forced indices with the chain's own fp64 logits at each layer."""
    xb = np.asarray(x_bits, dtype=np.uint16)
    n_flip, bad_all = 0, []
    for l, lay in enumerate(lays):
        idx = np.asarray(idx_per_layer[l], dtype=np.int32)
        out = moe.forward(lay, xb, idx_override=idx, want=("logits",))
        flipped, bad = routing_flips(idx, out["logits"], lay.k)
        n_flip += len(flipped)
        bad_all += [(l, t) for t in bad]
        xb = moe.residual_rmsnorm(xb, moe.f64_to_bf16(out["y"]), eps)
    return xb, n_flip, bad_all
