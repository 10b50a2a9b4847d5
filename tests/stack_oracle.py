"""Oracle work of the full-size stack checks, split into tasks for a process pool.

Each task regenerates the layers it needs from their seeded specs (the bytes are
the same on every call), so only token rows and expert indices cross process
boundaries.  The pool is started with the "spawn" method: the workers never see
a CUDA context.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _init_worker():
    # one BLAS thread per worker: the pool provides the parallelism
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(1)
    except Exception:
        pass


def _oracle_layer(seed: int, layer: int, latent: int, zipf: float):
    import synth
    from oracle import moe
    spec = synth.LayerSpec(seed=seed, layer=layer, latent=latent, zipf=zipf)
    inp = synth.make_layer(spec)
    return moe.Layer(inp.D, inp.U, inp.R, inp.bias, inp.expert, inp.shared, spec.latent, spec.ffn,
                     spec.top_k)


def layer_task(args):
    """Per-layer check on the GPU's input and routing for a set of token rows."""
    from parity import layer_check_metrics
    seed, layer, latent, zipf, x_bits, y_bits, gidx = args
    lay = _oracle_layer(seed, layer, latent, zipf)
    rel, mx, flips, bad = layer_check_metrics(lay, x_bits, y_bits, gidx)
    return layer, rel, mx, flips, bad


def chain_task(args):
    """One token (or a few) through the whole oracle stack, routing forced to the GPU's.

    With ``perturb`` the chain also runs from an input whose bf16 values are moved by
    one unit in the last place in a seeded tenth of the elements, and returns the
    relative size of that input change and of the resulting output change: the
    chain's own amplification of a rounding-level perturbation."""
    from oracle import moe
    from parity import stack_chain
    seed, n_layers, latent, zipfs, x_bits, idx_per_layer, perturb = args
    lays = [_oracle_layer(seed, l, latent, zipfs[l % len(zipfs)]) for l in range(n_layers)]
    xf, flips, bad = stack_chain(lays, x_bits, idx_per_layer)
    if not perturb:
        return xf, flips, bad, None
    xp = np.array(x_bits, dtype=np.uint16)
    sel = np.random.default_rng(seed + 99).random(xp.shape) < 0.1
    xp[sel] ^= np.uint16(1)                       # one ulp of bf16 in those elements
    x0, x1 = moe.bf16_to_f64(x_bits), moe.bf16_to_f64(xp)
    d_in = float(np.linalg.norm(x1 - x0) / np.linalg.norm(x0))
    xpf, _, _ = stack_chain(lays, xp, idx_per_layer)
    f0, f1 = moe.bf16_to_f64(xf), moe.bf16_to_f64(xpf)
    d_out = float(np.linalg.norm(f1 - f0) / np.linalg.norm(f0))
    return xf, flips, bad, (d_in, d_out)


def make_pool():
    n = max(1, min(32, (os.cpu_count() or 2)))
    return mp.get_context("spawn").Pool(n, initializer=_init_worker)
