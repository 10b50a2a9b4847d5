"""Reader of one packed NVFP4 expert record (oracle; test infrastructure).

Written from the record layout the library documents for its packer (the
pages fix the format, NVFP4 with one E4M3 scale per 16 weights along K and an
fp32 scale per matrix, but no byte layout; the model card's "Architecture"
section only says each expert is one fixed-size record).  For latent L and
SwiGLU width F the record holds, in order, with no gaps:

  gate codes  [F][L/2]   up codes  [F][L/2]   down codes  [L][F/2]
  gate scales [F][L/16]  up scales [F][L/16]  down scales [L][F/16]
  globals fp32 little-endian: gate, up, down

Codes: two E2M1 nibbles per byte, low nibble first along K.  Records sit in an
array at a caller-chosen stride (the library's default rounds the size up to
a multiple of 256 bytes).
"""
from __future__ import annotations

import numpy as np


def record_body_bytes(latent: int, ffn: int) -> int:
    """Bytes of codes and scales: 3 matrices of L*F weights at 4 + 8/16 bits each."""
    return 3 * latent * ffn // 2 + 3 * latent * ffn // 16


def record_bytes(latent: int, ffn: int) -> int:
    return record_body_bytes(latent, ffn) + 12


def read_record(buf: np.ndarray, latent: int, ffn: int):
    """Split one record (uint8 buffer) into the logical (codes, scales, globals)."""
    L, F = latent, ffn
    buf = np.asarray(buf, dtype=np.uint8)
    n_codes = 3 * F * L // 2
    n_scales = 3 * F * L // 16
    codes = buf[:n_codes]
    scales = buf[n_codes:n_codes + n_scales]
    glob = buf[n_codes + n_scales:n_codes + n_scales + 12].view("<f4").astype(np.float32)
    return codes, scales, glob
