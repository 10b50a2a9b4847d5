"""Device copies of the seeded workloads (input generation for tests and bench).

Dense tensors are generated on the host (``synth``) and uploaded; expert bytes
are written on the device by ``synth/fill.cu`` (the same counter streams as
``synth.expert_bytes``) and packed into records by the library's own packer
(``edge0_pack_experts``), the way a user of the library would load weights.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

import synth
import latent_sparse_moe_router_b300 as ext

_FILL = None


def _fill_lib():
    global _FILL
    if _FILL is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_synth_fill.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run latent_sparse_moe_router_b300.build.build()")
        L = ctypes.CDLL(path)
        L.synth_fill_experts.restype = ctypes.c_int
        L.synth_fill_experts.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
        _FILL = L
    return _FILL


def fill_experts(seed: int, layer: int, expert0: int, n: int, latent: int, ffn: int, device="cuda"):
    """Logical NVFP4 arrays of experts [expert0, expert0+n) on the device."""
    nc, ns = synth.expert_sizes(latent, ffn)
    codes = torch.empty(n * nc, dtype=torch.uint8, device=device)
    scales = torch.empty(n * ns, dtype=torch.uint8, device=device)
    glob = torch.empty(n * 3, dtype=torch.float32, device=device)
    rc = _fill_lib().synth_fill_experts(seed, layer, expert0, n, latent, ffn, codes.data_ptr(),
                                        scales.data_ptr(), glob.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    if rc:
        raise RuntimeError(f"synth_fill_experts failed ({rc})")
    return codes, scales, glob


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def pack_layer_records(spec: synth.LayerSpec, records: torch.Tensor | None = None,
                       shared: torch.Tensor | None = None, chunk: int = 128):
    """Generate and pack the E routed + 1 shared records of one layer on the device."""
    L, F, E = spec.latent, spec.ffn, spec.n_experts
    stride = ext.edge0_expert_record_stride(L, F)
    if records is None:
        records = torch.empty(E * stride, dtype=torch.uint8, device="cuda")
    if shared is None:
        shared = torch.empty(stride, dtype=torch.uint8, device="cuda")
    for e0 in range(0, E + 1, chunk):
        n = min(chunk, E + 1 - e0)
        codes, scales, glob = fill_experts(spec.seed, spec.layer, e0, n, L, F)
        n_routed = max(0, min(n, E - e0))
        if n_routed:
            ext.edge0_pack_experts(codes, scales, glob, n_routed, L, F,
                                   records.data_ptr() + e0 * stride, stride)
        if e0 + n > E:           # the shared expert is stream index E
            i = E - e0
            nc, ns = synth.expert_sizes(L, F)
            ext.edge0_pack_experts(codes.data_ptr() + i * nc, scales.data_ptr() + i * ns,
                                   glob.data_ptr() + i * 12, 1, L, F, shared, stride)
    return records, shared, stride


class DeviceLayer:
    """One seeded layer resident on the device, with its library handle."""

    def __init__(self, inputs: synth.LayerInputs, max_tokens: int = 16, records=None, shared=None):
        s = inputs.spec
        self.inputs = inputs
        self.spec = s
        self.D = bf16_tensor(inputs.D)
        self.U = bf16_tensor(inputs.U)
        self.R = bf16_tensor(inputs.R)
        self.bias = None if inputs.bias is None else torch.from_numpy(inputs.bias).cuda()
        self.records, self.shared, self.stride = pack_layer_records(s, records, shared)
        self.labels = torch.from_numpy(inputs.labels).cuda() if s.groups > 1 else None
        self.layer = ext.MoELayer(hidden=s.hidden, latent=s.latent, n_experts=s.n_experts, top_k=s.top_k,
                                  ffn=s.ffn, max_tokens=max_tokens, D=self.D, U=self.U, router=self.R,
                                  router_bias=self.bias, experts=self.records,
                                  expert_stride=self.stride, shared_expert=self.shared,
                                  n_groups=s.groups, expert_group=self.labels, shared_group=s.shared_group)

    @property
    def handle(self):
        return self.layer.handle

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        ext.edge0_moe_forward(self.handle, x, y, x.shape[0], stream)
        return y

    def routing(self, T: int):
        K, E = self.spec.top_k, self.spec.n_experts
        idx = torch.empty(T * K, dtype=torch.int32, device="cuda")
        w = torch.empty(T * K, dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
        pos = torch.empty(T * K, dtype=torch.int32, device="cuda")
        ext.edge0_moe_debug_routing(self.handle, idx, w, counts, offsets, perm, pos)
        torch.cuda.synchronize()
        return dict(idx=idx.cpu().numpy().reshape(T, K), w=w.cpu().numpy().reshape(T, K),
                    counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                    perm=perm.cpu().numpy(), pos=pos.cpu().numpy().reshape(T, K))

    def debug_tensor(self, what: int, T: int):
        """Stage tensor of the last forward as float64 [T, n]: z (0), logits (1), c (2).
        z and c are fp32 on the decode path (T <= 16); on the prefill path (and at
        every T for grouped layers) z is f16 times a per-token power of two and c is
        bf16, both G * latent wide."""
        GL = self.spec.groups * self.spec.latent
        n = {0: GL, 1: self.spec.n_experts, 2: GL}[what]
        if (T > 16 or self.spec.groups > 1) and what in (0, 2):
            # prefill: z as f16 scaled by a power of two per token, c as bf16
            out = torch.empty(T * n, dtype=torch.float16 if what == 0 else torch.bfloat16, device="cuda")
            ext.edge0_moe_debug_tensor(self.handle, what, out, out.numel() * 2)
            torch.cuda.synchronize()
            return out.float().cpu().numpy().astype(np.float64).reshape(T, n)
        out = torch.empty(T * n, dtype=torch.float32, device="cuda")
        ext.edge0_moe_debug_tensor(self.handle, what, out, out.numel() * 4)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64).reshape(T, n)

    def close(self):
        self.layer.close()
