"""Python binding of libedge0_moe.so, the latent-MoE layer library for B300 (sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C names of ``include/edge0_moe.h``; device
buffers are passed as torch CUDA tensors (or raw integer addresses), streams
as ``torch.cuda.Stream`` (default: torch's current stream).  A missing or
unloadable library raises immediately; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libedge0_moe.so")

EDGE0_OK = 0
EDGE0_ERR_INVALID_ARG = 1
EDGE0_ERR_UNSUPPORTED = 2
EDGE0_ERR_CUDA = 3
EDGE0_ERR_OOM = 4
EDGE0_ERR_TIMEOUT = 5

EXPORTED = (
    "edge0_expert_record_bytes", "edge0_expert_record_stride", "edge0_pack_expert_host",
    "edge0_pack_experts", "edge0_quantize_nvfp4", "edge0_moe_create", "edge0_moe_forward",
    "edge0_moe_debug_routing", "edge0_moe_debug_tensor", "edge0_residual_rmsnorm",
    "edge0_moe_stack_forward", "edge0_moe_stack_forward_trace", "edge0_moe_get_error",
    "edge0_status_string", "edge0_moe_destroy", "edge0_moe_forward_noalloc", "edge0_gemm_bf16_tn",
    "edge0_moe_profile_stages", "edge0_moe_stage_times", "edge0_moe_debug_wait_probe",
    "edge0_moe_profile_decode", "edge0_moe_decode_phase_times", "edge0_moe_tier_attach",
    "edge0_moe_tier_place", "edge0_moe_tier_rebalance", "edge0_moe_tier_stats", "edge0_moe_tier_detach",
    "edge0_tier_plan",
)

EDGE0_PREFILL_STAGES = 10
# kernels one prefill forward launches (token scale, x -> [z | logits], top-k +
# histogram, scan, offsets, scatter, row gather, gate/up, down, combine, U)
PREFILL_KERNELS_PER_FORWARD = 11
U_SPLIT_MAX_TOKENS = 768          # prefill forwards up to this T split the U GEMM along K (one more kernel)
PREFILL_STAGE_NAMES = ("xz_gemm", "topk_hist", "scan_chunks", "offsets", "scatter", "gather_rows",
                       "gate_up_grouped", "down_grouped", "combine", "u_gemm")


class Edge0Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_text(status)} ({status})")


class edge0_moe_desc(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("latent", ctypes.c_int), ("n_experts", ctypes.c_int),
        ("top_k", ctypes.c_int), ("ffn", ctypes.c_int), ("max_tokens", ctypes.c_int),
        ("D", ctypes.c_void_p), ("U", ctypes.c_void_p), ("router", ctypes.c_void_p),
        ("router_bias", ctypes.c_void_p), ("experts", ctypes.c_void_p),
        ("expert_stride", ctypes.c_size_t), ("shared_expert", ctypes.c_void_p),
        ("n_groups", ctypes.c_int), ("expert_group", ctypes.c_void_p), ("shared_group", ctypes.c_int),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the in-tree shared library (built by ``build.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with latent_sparse_moe_router_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        sig = {
            "edge0_expert_record_bytes": (sz, [i, i]),
            "edge0_expert_record_stride": (sz, [i, i]),
            "edge0_pack_expert_host": (i, [vp, vp, vp, i, i, vp]),
            "edge0_pack_experts": (i, [vp, vp, vp, i, i, i, vp, sz, vp]),
            "edge0_quantize_nvfp4": (i, [vp, i, i, f, vp, vp, vp]),
            "edge0_moe_create": (i, [ctypes.POINTER(edge0_moe_desc), ctypes.POINTER(vp)]),
            "edge0_moe_forward": (i, [vp, vp, vp, i, vp]),
            "edge0_moe_debug_routing": (i, [vp, vp, vp, vp, vp, vp, vp, vp]),
            "edge0_moe_debug_tensor": (i, [vp, i, vp, sz, vp]),
            "edge0_residual_rmsnorm": (i, [vp, vp, vp, i, i, f, vp]),
            "edge0_moe_stack_forward": (i, [vp, i, vp, vp, i, f, vp]),
            "edge0_moe_stack_forward_trace": (i, [vp, i, vp, vp, i, f, vp, vp, vp, vp]),
            "edge0_moe_get_error": (i, [vp]),
            "edge0_status_string": (ctypes.c_char_p, [i]),
            "edge0_moe_destroy": (None, [vp]),
            "edge0_moe_forward_noalloc": (i, [ctypes.POINTER(edge0_moe_desc), vp, vp, i, vp, vp]),
            "edge0_gemm_bf16_tn": (i, [vp, vp, vp, i, i, i, vp, vp]),
            "edge0_moe_profile_stages": (i, [vp, i]),
            "edge0_moe_debug_wait_probe": (i, [vp, vp]),
            "edge0_moe_stage_times": (i, [vp, vp, i, vp]),
            "edge0_moe_profile_decode": (i, [vp, i]),
            "edge0_moe_decode_phase_times": (i, [vp, vp, i, vp]),
            "edge0_moe_tier_attach": (i, [vp, vp, i, vp]),
            "edge0_moe_tier_place": (i, [vp, vp, vp]),
            "edge0_moe_tier_rebalance": (i, [vp, vp]),
            "edge0_moe_tier_stats": (i, [vp, vp]),
            "edge0_moe_tier_detach": (i, [vp]),
            "edge0_tier_plan": (i, [vp, i, i, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_text(status: int) -> str:
    return lib().edge0_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != EDGE0_OK:
        raise Edge0Error(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ record format
def edge0_expert_record_bytes(latent: int, ffn: int) -> int:
    return lib().edge0_expert_record_bytes(latent, ffn)


def edge0_expert_record_stride(latent: int, ffn: int) -> int:
    return lib().edge0_expert_record_stride(latent, ffn)


def edge0_pack_expert_host(codes, scales, globals_, latent: int, ffn: int):
    """Host packer: numpy uint8 codes/scales and float32[3] globals -> uint8 record."""
    import numpy as np
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    globals_ = np.ascontiguousarray(globals_, dtype=np.float32)
    out = np.zeros(edge0_expert_record_bytes(latent, ffn), dtype=np.uint8)
    _check(lib().edge0_pack_expert_host(_ptr(codes), _ptr(scales), _ptr(globals_), latent, ffn,
                                        _ptr(out)), "edge0_pack_expert_host")
    return out


def edge0_pack_experts(codes, scales, globals_, n_experts, latent, ffn, records, stride, stream=None):
    _check(lib().edge0_pack_experts(_ptr(codes), _ptr(scales), _ptr(globals_), n_experts, latent, ffn,
                                    _ptr(records), stride, _stream(stream)), "edge0_pack_experts")


def edge0_quantize_nvfp4(w, rows, K, g, codes, scales, stream=None):
    _check(lib().edge0_quantize_nvfp4(_ptr(w), rows, K, float(g), _ptr(codes), _ptr(scales),
                                      _stream(stream)), "edge0_quantize_nvfp4")


# ------------------------------------------------------------------ layer
def edge0_moe_create(hidden, latent, n_experts, top_k, ffn, max_tokens, D, U, router, router_bias,
                     experts, expert_stride, shared_expert, n_groups=1, expert_group=None,
                     shared_group=0) -> int:
    d = edge0_moe_desc(hidden, latent, n_experts, top_k, ffn, max_tokens, _ptr(D), _ptr(U),
                       _ptr(router), _ptr(router_bias), _ptr(experts), expert_stride,
                       _ptr(shared_expert), n_groups, _ptr(expert_group), shared_group)
    h = ctypes.c_void_p()
    _check(lib().edge0_moe_create(ctypes.byref(d), ctypes.byref(h)), "edge0_moe_create")
    return h.value


def edge0_moe_forward(handle, x, y, T, stream=None):
    _check(lib().edge0_moe_forward(handle, _ptr(x), _ptr(y), T, _stream(stream)), "edge0_moe_forward")


def edge0_moe_debug_routing(handle, idx=None, w=None, counts=None, offsets=None, perm=None, pos=None,
                            stream=None):
    _check(lib().edge0_moe_debug_routing(handle, _ptr(idx), _ptr(w), _ptr(counts), _ptr(offsets),
                                         _ptr(perm), _ptr(pos), _stream(stream)),
           "edge0_moe_debug_routing")


def edge0_moe_debug_tensor(handle, what, dst, nbytes, stream=None):
    _check(lib().edge0_moe_debug_tensor(handle, what, _ptr(dst), nbytes, _stream(stream)),
           "edge0_moe_debug_tensor")


def edge0_gemm_bf16_tn(A, B, C, M, N, K, err=None, stream=None):
    """C = A B^T (bf16 in, fp32 out) on the tcgen05 tensor cores."""
    _check(lib().edge0_gemm_bf16_tn(_ptr(A), _ptr(B), _ptr(C), M, N, K, _ptr(err), _stream(stream)),
           "edge0_gemm_bf16_tn")


def edge0_residual_rmsnorm(x, y, out, T, hidden, eps, stream=None):
    _check(lib().edge0_residual_rmsnorm(_ptr(x), _ptr(y), _ptr(out), T, hidden, float(eps),
                                        _stream(stream)), "edge0_residual_rmsnorm")


def _handle_array(handles):
    arr = (ctypes.c_void_p * len(handles))(*handles)
    return arr


def edge0_moe_stack_forward(handles, x, y, T, eps, stream=None):
    arr = _handle_array(handles)
    _check(lib().edge0_moe_stack_forward(ctypes.cast(arr, ctypes.c_void_p), len(handles), _ptr(x),
                                         _ptr(y), T, float(eps), _stream(stream)),
           "edge0_moe_stack_forward")


def edge0_moe_stack_forward_trace(handles, x, y, T, eps, trace_x, trace_y, trace_idx=None, stream=None):
    arr = _handle_array(handles)
    _check(lib().edge0_moe_stack_forward_trace(ctypes.cast(arr, ctypes.c_void_p), len(handles),
                                               _ptr(x), _ptr(y), T, float(eps), _ptr(trace_x),
                                               _ptr(trace_y), _ptr(trace_idx), _stream(stream)),
           "edge0_moe_stack_forward_trace")


def edge0_moe_forward_noalloc(hidden, latent, n_experts, top_k, ffn, D, U, router, router_bias, experts,
                              expert_stride, shared_expert, x, y, T, status=None, stream=None):
    """Decode forward with no device allocation (scratch in the library's static
    array); for callers that cannot call cudaMalloc.  See the C header."""
    d = edge0_moe_desc(hidden, latent, n_experts, top_k, ffn, 0, _ptr(D), _ptr(U), _ptr(router),
                       _ptr(router_bias), _ptr(experts), expert_stride, _ptr(shared_expert))
    _check(lib().edge0_moe_forward_noalloc(ctypes.byref(d), _ptr(x), _ptr(y), T, _ptr(status),
                                           _stream(stream)), "edge0_moe_forward_noalloc")


def edge0_moe_debug_wait_probe(handle, stream=None):
    """Make one bounded device wait run out (nothing faults); see the C header."""
    _check(lib().edge0_moe_debug_wait_probe(handle, _stream(stream)), "edge0_moe_debug_wait_probe")


def edge0_moe_profile_stages(handle, enable: bool):
    _check(lib().edge0_moe_profile_stages(handle, int(bool(enable))), "edge0_moe_profile_stages")


def edge0_moe_stage_times(handle):
    """Per-stage milliseconds of the last (timed) prefill forward, as a list."""
    buf = (ctypes.c_float * EDGE0_PREFILL_STAGES)()
    n = ctypes.c_int()
    _check(lib().edge0_moe_stage_times(handle, ctypes.cast(buf, ctypes.c_void_p), EDGE0_PREFILL_STAGES,
                                       ctypes.byref(n)), "edge0_moe_stage_times")
    return [float(buf[i]) for i in range(n.value)]


EDGE0_DECODE_PHASES = 19
DECODE_PHASE_NAMES = ("p0", "p0_spread", "barrier1", "routing", "p1_gate_up", "p1_spread", "barrier2",
                      "p2_down_combine", "p2_spread", "barrier3", "p3_u", "p3_spread", "barrier4", "layer_total",
                      "routing_loads", "routing_topk", "p1_issue", "p2_h_staging", "p2_down_mma")


def edge0_moe_profile_decode(handle, enable: bool):
    _check(lib().edge0_moe_profile_decode(handle, int(bool(enable))), "edge0_moe_profile_decode")


def edge0_moe_decode_phase_times(handle, n_layers: int = 1):
    """Per-layer phase microseconds of the last profiled decode launch: a list of
    dicts keyed by DECODE_PHASE_NAMES."""
    n_max = EDGE0_DECODE_PHASES * n_layers
    buf = (ctypes.c_float * n_max)()
    n = ctypes.c_int()
    _check(lib().edge0_moe_decode_phase_times(handle, ctypes.cast(buf, ctypes.c_void_p), n_max, ctypes.byref(n)),
           "edge0_moe_decode_phase_times")
    vals = [float(buf[i]) for i in range(n.value)]
    return [dict(zip(DECODE_PHASE_NAMES, vals[l * EDGE0_DECODE_PHASES:(l + 1) * EDGE0_DECODE_PHASES]))
            for l in range(n.value // EDGE0_DECODE_PHASES)]


# ------------------------------------------------------------------ residency tiering
def edge0_moe_tier_attach(handle, host_records, n_slots, stream=None):
    """host_records: pinned host tensor (or address) of the layer's records at the handle's stride."""
    _check(lib().edge0_moe_tier_attach(handle, _ptr(host_records), int(n_slots), _stream(stream)),
           "edge0_moe_tier_attach")


def edge0_moe_tier_place(handle, slot_expert, stream=None):
    import numpy as np
    arr = np.ascontiguousarray(slot_expert, dtype=np.int32)
    _check(lib().edge0_moe_tier_place(handle, arr.ctypes.data, _stream(stream)), "edge0_moe_tier_place")


def edge0_moe_tier_rebalance(handle, stream=None):
    _check(lib().edge0_moe_tier_rebalance(handle, _stream(stream)), "edge0_moe_tier_rebalance")


def edge0_moe_tier_stats(handle):
    """dict(forwards, misses, host_bytes, resident)."""
    buf = (ctypes.c_ulonglong * 4)()
    _check(lib().edge0_moe_tier_stats(handle, ctypes.cast(buf, ctypes.c_void_p)), "edge0_moe_tier_stats")
    return dict(forwards=buf[0], misses=buf[1], host_bytes=buf[2], resident=buf[3])


def edge0_moe_tier_detach(handle):
    _check(lib().edge0_moe_tier_detach(handle), "edge0_moe_tier_detach")


def edge0_tier_plan(use, n_slots, cur):
    """The residency policy on the host: returns (slot -> expert array, slots changed)."""
    import numpy as np
    use = np.ascontiguousarray(use, dtype=np.uint32)
    cur = np.ascontiguousarray(cur, dtype=np.int32)
    nxt = np.full(int(n_slots), -1, dtype=np.int32)
    n = lib().edge0_tier_plan(use.ctypes.data, use.size, int(n_slots), cur.ctypes.data, nxt.ctypes.data)
    if n < 0:
        raise Edge0Error(EDGE0_ERR_INVALID_ARG, "edge0_tier_plan")
    return nxt, n


def edge0_moe_get_error(handle) -> int:
    return lib().edge0_moe_get_error(handle)


def edge0_status_string(status: int) -> str:
    return status_text(status)


def edge0_moe_destroy(handle):
    if handle:
        lib().edge0_moe_destroy(handle)


class MoELayer:
    """A layer handle plus references to the device tensors it borrows."""

    def __init__(self, *, hidden, latent, n_experts, top_k, ffn, max_tokens, D, U, router,
                 router_bias, experts, expert_stride, shared_expert, n_groups=1, expert_group=None,
                 shared_group=0):
        self._keep = (D, U, router, router_bias, experts, shared_expert)
        self.hidden, self.latent, self.n_experts, self.top_k, self.ffn = hidden, latent, n_experts, top_k, ffn
        self.max_tokens = max_tokens
        self.n_groups = n_groups
        self.handle = edge0_moe_create(hidden, latent, n_experts, top_k, ffn, max_tokens, D, U, router,
                                       router_bias, experts, expert_stride, shared_expert, n_groups,
                                       expert_group, shared_group)

    def forward(self, x, y, T=None, stream=None):
        edge0_moe_forward(self.handle, x, y, x.shape[0] if T is None else T, stream)
        return y

    def close(self):
        if self.handle:
            edge0_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
