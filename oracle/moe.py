"""The latent-MoE layer by definition, in fp64 (oracle; test infrastructure).

What one layer computes for a token, as the pages describe it:
  * attention stays at width 2560; a shared down-projection D maps the token
    to a latent of width l (1792 for the 145B model) before the experts and a
    shared up-projection U maps the result back; each layer has 512 routed
    experts and one shared expert, and the router keeps 10 per token
    ("Edge0-145B hardware requirements", section "Edge0-145B latent MoE
    architecture: how 145B fits one GPU");
  * each expert maps l -> 640 -> l, the shared expert runs next to the routed
    ones, the combined latent goes through U, and there is one D and one U
    per layer ("Edge0-145B · Q3_K" model card, section "Architecture":
    diagram caption and config block, SwiGLU width 640);
  * latent widths are 1792 (145B) and 1280 (120B) ("Edge0 Squeezes a 145B
    Coding Agent...", table "Released model variants").

Readings where the pages are silent (each listed in the design notes):
  * one D and one U per layer (the model card's reading) in ``layer_forward``;
    the "eight groups" of the hardware-requirements page are ``GroupedLayer``
    and ``grouped_layer_forward`` (their readings are in that docstring);
  * the router scores the latent z: logits l = R z + b, R [E, l];
  * top-k by (logit descending, expert index ascending); weights are the
    softmax over all E renormalised over the k kept, which equals
    exp(l_k - m) / sum_{j in top} exp(l_j - m) for any m;
  * each expert is SwiGLU: o = W_d (silu(W_g z) * (W_up z)), silu(a) = a / (1 + e^-a);
  * the shared expert is ungated (weight 1), same shape and format;
  * combine c = o_shared + sum_k w_k o_k at width l, then y = U c;
  * stack: x_{l+1} = RMSNorm(x_l + y_l), unit gain, eps 1e-6, bf16 between layers.

Every dot product here is fp64 (numpy matmul on fp64 arrays); inputs are
decoded exactly (bf16 -> fp64, NVFP4 -> fp64).
"""
from __future__ import annotations

import numpy as np

from . import nvfp4


# ---------------------------------------------------------------- bf16 helpers
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values (bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, one round-to-nearest-even step (normal range)."""
    x = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(x))
    b = np.ascontiguousarray(x).view(np.uint64).copy()
    # bf16 keeps 7 of fp64's 52 fraction bits: round away the low 45 bits
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = b + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb
    b &= ~np.uint64((1 << 45) - 1)
    f32 = b.view(np.float64).astype(np.float32)      # exact: value has 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------- layer steps
def d_projection(x: np.ndarray, D: np.ndarray) -> np.ndarray:
    """z = D x for every token: x [T, H], D [l, H] -> z [T, l]."""
    return x @ D.T


def router_logits(z: np.ndarray, R: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """l = R z + b: z [T, l], R [E, l], b [E] or None -> logits [T, E]."""
    logits = z @ R.T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return logits


def top_k(logits: np.ndarray, k: int) -> np.ndarray:
    """Expert indices [T, k]: rank by logit descending, equal logits by index ascending."""
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    ar = np.arange(E)
    for t in range(T):
        order = np.lexsort((ar, -logits[t]))     # primary key last: -logit, then index
        idx[t] = order[:k]
    return idx


def routing_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Renormalised softmax weights over the kept experts [T, k]."""
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    return ex / ex.sum(axis=1, keepdims=True)


def permutation(idx: np.ndarray, n_experts: int):
    """Token -> expert grouping of the T*k slots (slot s = t*k + j).

    counts[e]  = number of slots routed to e
    offsets    = exclusive prefix sum of counts (n_experts + 1 entries)
    perm[p]    = slot at grouped position p; groups in expert order, and
                 within a group slots in ascending (t, j) order
    pos[t, j]  = grouped position of slot (t, j) (the inverse of perm)
    """
    flat = idx.reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=n_experts).astype(np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, pos.reshape(idx.shape)


def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def expert_matrices(codes, scales, glob, latent: int, ffn: int):
    """Dequantised (W_g [F, l], W_up [F, l], W_d [l, F]) of one expert, fp64."""
    L, F = latent, ffn
    cg = codes[: F * L // 2].reshape(F, L // 2)
    cu = codes[F * L // 2: F * L].reshape(F, L // 2)
    cd = codes[F * L:].reshape(L, F // 2)
    sg = scales[: F * L // 16].reshape(F, L // 16)
    su = scales[F * L // 16: F * L // 8].reshape(F, L // 16)
    sd = scales[F * L // 8:].reshape(L, F // 16)
    Wg = nvfp4.dequantize(cg, sg, glob[0])
    Wu = nvfp4.dequantize(cu, su, glob[1])
    Wd = nvfp4.dequantize(cd, sd, glob[2])
    return Wg, Wu, Wd


def swiglu_expert(z: np.ndarray, Wg, Wu, Wd) -> np.ndarray:
    """o = W_d (silu(W_g z) * (W_up z)) for rows z [n, l] -> [n, l]."""
    h = silu(z @ Wg.T) * (z @ Wu.T)
    return h @ Wd.T


def u_projection(c: np.ndarray, U: np.ndarray) -> np.ndarray:
    """y = U c: c [T, l], U [H, l] -> y [T, H]."""
    return c @ U.T


def rmsnorm(v: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) per row, unit gain."""
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------- the layer
class Layer:
    """One layer's parameters in exact form, with experts dequantised on demand.

    ``expert_source(e)`` returns the logical NVFP4 arrays (codes, scales,
    globals) of routed expert e; ``shared_source()`` those of the shared expert.
    """

    def __init__(self, D_bits, U_bits, R_bits, bias, expert_source, shared_source,
                 latent: int, ffn: int, top_k: int):
        self.D = bf16_to_f64(D_bits)
        self.U = bf16_to_f64(U_bits)
        self.R = bf16_to_f64(R_bits)
        self.bias = bias
        self.expert_source = expert_source
        self.shared_source = shared_source
        self.latent, self.ffn, self.k = latent, ffn, top_k
        self.n_experts = self.R.shape[0]

    def matrices(self, e: int):
        src = self.shared_source() if e < 0 else self.expert_source(e)
        return expert_matrices(*src, self.latent, self.ffn)


def layer_forward(layer: Layer, x_bits: np.ndarray, idx_override: np.ndarray | None = None,
                  want: tuple = ()):
    """One latent-MoE layer on tokens x (bf16 bits [T, H]).

    Returns a dict with y (fp64 [T, H]) and whatever of z, logits, idx, w,
    counts, offsets, perm, pos, c, o_shared is listed in ``want``.
    ``idx_override`` replaces the oracle's own top-k choice (teacher forcing
    with another implementation's expert indices); the weights are then the
    renormalised softmax of the oracle's logits over those indices.
    Experts are evaluated expert-major: each used expert is dequantised once.
    """
    x = bf16_to_f64(x_bits)
    z = d_projection(x, layer.D)
    logits = router_logits(z, layer.R, layer.bias)
    idx = top_k(logits, layer.k) if idx_override is None else np.asarray(idx_override, np.int32)
    w = routing_weights(logits, idx)
    T, k = idx.shape
    Wg, Wu, Wd = layer.matrices(-1)
    o_shared = swiglu_expert(z, Wg, Wu, Wd)
    c = o_shared.copy()
    for e in np.unique(idx):
        # a token keeps k distinct experts, so each t appears once per group
        t_sel, j_sel = np.nonzero(idx == e)
        Wg, Wu, Wd = layer.matrices(int(e))
        c[t_sel] += w[t_sel, j_sel][:, None] * swiglu_expert(z[t_sel], Wg, Wu, Wd)
    y = u_projection(c, layer.U)
    out = {"y": y}
    loc = dict(z=z, logits=logits, idx=idx, w=w, c=c, o_shared=o_shared)
    for name in want:
        if name in loc:
            out[name] = loc[name]
    if any(n in want for n in ("counts", "offsets", "perm", "pos")):
        counts, offsets, perm, pos = permutation(idx, layer.n_experts)
        out.update(counts=counts, offsets=offsets, perm=perm, pos=pos)
    return out


def residual_rmsnorm(x_bits: np.ndarray, y_bits: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Post-norm residual between stacked layers: bf16(RMSNorm(x + y))."""
    v = bf16_to_f64(x_bits) + bf16_to_f64(y_bits)
    return f64_to_bf16(rmsnorm(v, eps))


def stack_forward(layers: list, x_bits: np.ndarray, eps: float = 1e-6):
    """x_{l+1} = RMSNorm(x_l + y_l) over the stack; y_l rounded to bf16 as layers emit it.

    Returns (x_final bits, per-layer list of (x_l bits, y_l fp64)).
    """
    trace = []
    xb = np.asarray(x_bits, dtype=np.uint16)
    for layer in layers:
        y = layer_forward(layer, xb)["y"]
        trace.append((xb, y))
        xb = residual_rmsnorm(xb, f64_to_bf16(y), eps)
    return xb, trace


# ---------------------------------------------------------------- grouped latent projections
class GroupedLayer(Layer):
    """A layer whose down and up projections come in G groups.

    "Edge0-145B hardware requirements", section "Edge0-145B latent MoE
    architecture: how 145B fits one GPU": each layer has eight groups of D and U,
    every expert carries a label naming the group it uses, and each group of 64
    experts shares its two matrices; "Edge0-145B · Q3_K" model card, section
    "Architecture" (diagram caption): D maps the token to the latent per routing
    group.

    D_bits [G*l, H]: rows g*l .. g*l + l - 1 are D_g.  U_bits [H, G*l]: columns
    g*l .. g*l + l - 1 are U_g.  labels [E]: the group of each routed expert;
    shared_group: the group of the shared expert.
    """

    def __init__(self, D_bits, U_bits, R_bits, bias, expert_source, shared_source,
                 latent: int, ffn: int, top_k: int, labels, shared_group: int):
        super().__init__(D_bits, U_bits, R_bits, bias, expert_source, shared_source, latent, ffn, top_k)
        self.groups = self.D.shape[0] // latent
        assert self.D.shape[0] == self.groups * latent and self.U.shape[1] == self.groups * latent
        self.labels = np.asarray(labels, dtype=np.int64)
        assert self.labels.shape == (self.n_experts,)
        assert self.labels.min() >= 0 and self.labels.max() < self.groups
        self.shared_group = int(shared_group)
        assert 0 <= self.shared_group < self.groups

    def D_group(self, g: int) -> np.ndarray:
        return self.D[g * self.latent:(g + 1) * self.latent]

    def U_group(self, g: int) -> np.ndarray:
        return self.U[:, g * self.latent:(g + 1) * self.latent]


def grouped_layer_forward(layer: GroupedLayer, x_bits: np.ndarray, idx_override: np.ndarray | None = None,
                          want: tuple = ()):
    """One layer with grouped latent projections on tokens x (bf16 bits [T, H]).

    Readings where the pages leave the step open:
      * z_g = D_g x for every group g (one latent per routing group);
      * expert e's router row scores its own group's latent: l_e = R_e z_{g(e)} + b_e;
      * expert e runs on z_{g(e)}, the shared expert on z of its group;
      * each group combines its own experts: c_g = [g = g_shared] o_shared
        + sum over kept k with g(e_k) = g of w_k o_k (zero for a group nobody used);
      * y = sum_g U_g c_g.
    With one group this is ``layer_forward``.  Returns y and whatever of z, c
    (both [T, G*l], group-major columns), logits, idx, w, o_shared is in ``want``.
    """
    x = bf16_to_f64(x_bits)
    G, l = layer.groups, layer.latent
    T = x.shape[0]
    z = [d_projection(x, layer.D_group(g)) for g in range(G)]
    logits = np.empty((T, layer.n_experts), dtype=np.float64)
    for g in range(G):
        rows = np.nonzero(layer.labels == g)[0]
        logits[:, rows] = router_logits(z[g], layer.R[rows], None)
    if layer.bias is not None:
        logits = logits + np.asarray(layer.bias, dtype=np.float32).astype(np.float64)[None, :]
    idx = top_k(logits, layer.k) if idx_override is None else np.asarray(idx_override, np.int32)
    w = routing_weights(logits, idx)
    c = [np.zeros((T, l), dtype=np.float64) for _ in range(G)]
    Wg, Wu, Wd = layer.matrices(-1)
    o_shared = swiglu_expert(z[layer.shared_group], Wg, Wu, Wd)
    c[layer.shared_group] += o_shared
    for e in np.unique(idx):
        g = int(layer.labels[e])
        t_sel, j_sel = np.nonzero(idx == e)
        Wg, Wu, Wd = layer.matrices(int(e))
        c[g][t_sel] += w[t_sel, j_sel][:, None] * swiglu_expert(z[g][t_sel], Wg, Wu, Wd)
    y = np.zeros((T, layer.U.shape[0]), dtype=np.float64)
    for g in range(G):
        y += u_projection(c[g], layer.U_group(g))
    out = {"y": y}
    loc = dict(z=np.concatenate(z, axis=1), logits=logits, idx=idx, w=w, c=np.concatenate(c, axis=1),
               o_shared=o_shared)
    for name in want:
        if name in loc:
            out[name] = loc[name]
    if any(n in want for n in ("counts", "offsets", "perm", "pos")):
        counts, offsets, perm, pos = permutation(idx, layer.n_experts)
        out.update(counts=counts, offsets=offsets, perm=perm, pos=pos)
    return out


def forward(layer: Layer, x_bits: np.ndarray, idx_override: np.ndarray | None = None, want: tuple = ()):
    """``grouped_layer_forward`` for a GroupedLayer, else ``layer_forward``."""
    if isinstance(layer, GroupedLayer):
        return grouped_layer_forward(layer, x_bits, idx_override, want)
    return layer_forward(layer, x_bits, idx_override, want)
