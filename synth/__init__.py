"""Seeded synthetic inputs for the latent-MoE layer (input generation only).

This module is shared by the oracle tests and by the CUDA-path tests and bench.
It produces the *bytes* of the inputs and holds none of the layer's arithmetic:
no projection, routing, dequantisation or SwiGLU lives here.

Workload shapes follow the pages:
  * hidden 2560, latent 1792 (Edge0-145B) or 1280 (Edge0-120B), 512 routed
    experts + 1 shared, top-10, SwiGLU width 640
    ("Edge0-145B hardware requirements", section "latent MoE architecture";
    "Edge0-145B · Q3_K" model card, section "Architecture";
    "Edge0 Squeezes a 145B Coding Agent...", table "Released model variants").
  * experts in NVFP4 ("Edge0-145B en local", intro: NVIDIA's 4-bit float format).

Distributions (the workload recipe):
  * x ~ N(0, 1); D, U, router ~ N(0, 1/fan_in); all rounded to bf16 (RNE).
    Dense tensors come from numpy ``default_rng`` seeded by (seed, layer, tag).
  * Expert records: E2M1 codes uniform over the 16 nibbles, one E4M3 scale per
    16 weights drawn uniform in [0.002, 0.01] then rounded to nearest-even
    E4M3 (the whole range is E4M3-subnormal: codes 1..5), fp32 global 1.0.
    Those bytes come from a counter-based generator (SplitMix64 of a per-stream
    key plus an index) so that a CUDA fill kernel (``synth/fill.cu``) can write
    the 47 GB stack on the device while this module regenerates any single
    expert bit-identically on the host.
  * Zipf(s) router bias over a seeded expert order: b_e = -s * ln(rank_e).
  * Grouped latent projections (G groups): D [G*l, H] and U [H, G*l] drawn like the
    single D and U (each group's block N(0, 1/fan_in) of that block); group labels
    from a seeded permutation of the experts, E/G experts per group, so that a
    group's experts are not contiguous indices; the shared expert in group
    ``shared_group``.  G = 1 gives the same bytes as the ungrouped layer.

Per-expert logical arrays (the order the generator emits bytes in):
  codes  uint8 [3*F*L/2]  = gate [F][L/2] | up [F][L/2] | down [L][F/2]
  scales uint8 [3*F*L/16] = gate [F][L/16] | up [F][L/16] | down [L][F/16]
  globals fp32 [3]        = gate, up, down
Within a code byte the low nibble is the even element along K.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

HIDDEN = 2560
N_EXPERTS = 512
TOP_K = 10
FFN = 640
LATENT_145B = 1792
LATENT_120B = 1280

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
KIND_CODES = 1
KIND_SCALES = 2


def splitmix64(x):
    """SplitMix64 output function (Steele, Lea, Flood 2014) on uint64 arrays."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, layer: int, expert: int, kind: int) -> np.uint64:
    """Key of one byte stream: chained SplitMix64 over (seed, layer, expert, kind).

    ``expert`` = n_experts addresses the shared expert of the layer.
    """
    k = splitmix64(np.uint64(seed))
    k = splitmix64(k ^ np.uint64(layer))
    k = splitmix64(k ^ np.uint64(expert))
    k = splitmix64(k ^ np.uint64(kind))
    return np.uint64(k)


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """Round positive finite fp64 values to E4M3 (OCP E4M3FN, bias 7) bytes, RNE.

    Input preparation only (the layer never encodes); saturates at 448.
    """
    v = np.asarray(v, dtype=np.float64)
    assert np.all(v >= 0.0) and np.all(np.isfinite(v))
    out = np.zeros(v.shape, dtype=np.uint8)
    sub = v < 2.0 ** -6
    # subnormal grid m * 2^-9; m == 8 lands on the first normal (byte 0x08)
    out[sub] = np.rint(v[sub] * 512.0).astype(np.uint8)
    nv = v[~sub]
    if nv.size:
        fr, ex = np.frexp(nv)                     # nv = fr * 2^ex, fr in [0.5, 1)
        e = ex - 1                                # nv = (2*fr) * 2^e
        mant = np.rint((2.0 * fr - 1.0) * 8.0)   # 0..8 (RNE on the 3-bit grid)
        bump = mant == 8.0
        e = np.where(bump, e + 1, e)
        mant = np.where(bump, 0.0, mant)
        code = ((e + 7) << 3).astype(np.int64) + mant.astype(np.int64)
        code = np.minimum(code, 0x7E)
        out[~sub] = code.astype(np.uint8)
    return out


def expert_sizes(latent: int, ffn: int = FFN):
    """(code bytes, scale bytes) of one expert's logical arrays."""
    return 3 * ffn * latent // 2, 3 * ffn * latent // 16


def expert_bytes(seed: int, layer: int, expert: int, latent: int, ffn: int = FFN):
    """Logical NVFP4 arrays of one expert: (codes u8, scales u8, globals f32[3])."""
    n_codes, n_scales = expert_sizes(latent, ffn)
    assert n_codes % 8 == 0
    kc = stream_key(seed, layer, expert, KIND_CODES)
    with np.errstate(over="ignore"):
        words = splitmix64(kc + np.arange(n_codes // 8, dtype=np.uint64))
    codes = words.astype("<u8").view(np.uint8).copy()
    ks = stream_key(seed, layer, expert, KIND_SCALES)
    with np.errstate(over="ignore"):
        h = splitmix64(ks + np.arange(n_scales, dtype=np.uint64))
    u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    # two separately rounded IEEE operations (no fused multiply-add)
    v = np.multiply(u, 0.008)
    v = np.add(v, 0.002)
    scales = e4m3_encode_rne(v)
    glob = np.ones(3, dtype=np.float32)
    return codes, scales, glob


def split_expert(codes, scales, latent: int, ffn: int = FFN):
    """Views of one expert's logical arrays as per-matrix 2-D arrays."""
    L, F = latent, ffn
    cg = codes[: F * L // 2].reshape(F, L // 2)
    cu = codes[F * L // 2: F * L].reshape(F, L // 2)
    cd = codes[F * L:].reshape(L, F // 2)
    sg = scales[: F * L // 16].reshape(F, L // 16)
    su = scales[F * L // 16: F * L // 8].reshape(F, L // 16)
    sd = scales[F * L // 8:].reshape(L, F // 16)
    return (cg, sg), (cu, su), (cd, sd)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (b >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(seed, layer, tag, shape, std):
    rng = np.random.default_rng([seed, layer, tag])
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a)


TAG_X, TAG_D, TAG_U, TAG_R, TAG_ZIPF, TAG_GROUP = 1, 2, 3, 4, 5, 6


def tokens_bf16(seed: int, T: int, hidden: int = HIDDEN, tag_layer: int = 0):
    """x ~ N(0,1) as bf16 bits [T, hidden]."""
    return _normal_bf16(seed, tag_layer, TAG_X, (T, hidden), 1.0)


def zipf_bias(seed: int, layer: int, n_experts: int = N_EXPERTS, s: float = 1.1):
    """Router bias b_e = -s ln(rank_e), rank over a seeded permutation of experts."""
    order = np.random.default_rng([seed, layer, TAG_ZIPF]).permutation(n_experts)
    rank = np.empty(n_experts, dtype=np.float64)
    rank[order] = np.arange(1, n_experts + 1, dtype=np.float64)
    return (-s * np.log(rank)).astype(np.float32)


def group_labels(seed: int, layer: int, n_experts: int, groups: int) -> np.ndarray:
    """Group of each expert: a seeded permutation split into G equal parts."""
    labels = np.zeros(n_experts, dtype=np.int32)
    if groups > 1:
        order = np.random.default_rng([seed, layer, TAG_GROUP]).permutation(n_experts)
        labels[order] = (np.arange(n_experts) * groups // n_experts).astype(np.int32)
    return labels


@dataclass
class LayerSpec:
    seed: int
    layer: int
    latent: int
    hidden: int = HIDDEN
    n_experts: int = N_EXPERTS
    top_k: int = TOP_K
    ffn: int = FFN
    zipf: float = 0.0          # 0 = uniform routing (no bias)
    groups: int = 1            # latent groups (D/U pairs)
    shared_group: int = 0      # group of the shared expert


@dataclass
class LayerInputs:
    """Dense bf16 tensors (bit patterns) plus an on-demand expert source."""
    spec: LayerSpec
    D: np.ndarray              # u16 [L, H]
    U: np.ndarray              # u16 [H, L]
    R: np.ndarray              # u16 [E, L]
    bias: np.ndarray | None    # f32 [E] or None
    labels: np.ndarray = None  # i32 [E] group of each expert (all 0 for one group)
    _cache: dict = field(default_factory=dict, repr=False)

    def expert(self, e: int):
        """Logical arrays of routed expert e (e == n_experts: the shared expert)."""
        if e not in self._cache:
            s = self.spec
            self._cache[e] = expert_bytes(s.seed, s.layer, e, s.latent, s.ffn)
        return self._cache[e]

    def shared(self):
        return self.expert(self.spec.n_experts)


def make_layer(spec: LayerSpec) -> LayerInputs:
    L, H, E, G = spec.latent, spec.hidden, spec.n_experts, spec.groups
    assert G >= 1 and E % G == 0 and 0 <= spec.shared_group < G
    D = _normal_bf16(spec.seed, spec.layer, TAG_D, (G * L, H), 1.0 / math.sqrt(H))
    U = _normal_bf16(spec.seed, spec.layer, TAG_U, (H, G * L), 1.0 / math.sqrt(L))
    R = _normal_bf16(spec.seed, spec.layer, TAG_R, (E, L), 1.0 / math.sqrt(L))
    bias = zipf_bias(spec.seed, spec.layer, E, spec.zipf) if spec.zipf > 0 else None
    return LayerInputs(spec, D, U, R, bias, group_labels(spec.seed, spec.layer, E, G))


# The five seeded workloads (shapes and seeds of the stated configurations).
WORKLOADS = {
    "layer145b_t1": dict(latent=LATENT_145B, T=1, seed=0, layers=1, zipf=(0.0,)),
    "layer120b_t4": dict(latent=LATENT_120B, T=4, seed=1, layers=1, zipf=(0.0,)),
    "stack48_145b_t1x256": dict(latent=LATENT_145B, T=1, seed=2, layers=48, zipf=(0.0,),
                                tokens=256),
    "layer145b_t4096_zipf": dict(latent=LATENT_145B, T=4096, seed=3, layers=1, zipf=(1.1,)),
    "prefill4x145b_t16384": dict(latent=LATENT_145B, T=16384, seed=4, layers=4,
                                 zipf=(0.0, 1.1, 0.0, 1.1)),
}
