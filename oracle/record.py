"""Reader of one packed NVFP4 expert record (oracle; test infrastructure).

Written from the record layout the library documents for its packer.  The
pages fix the format (NVFP4: E2M1 elements, an E4M3 scale per 16 weights along
K, an fp32 scale per matrix) and say each expert is one fixed-size record
("Edge0-145B · Q3_K" model card, section "Architecture"), but print no byte
layout.  For latent L and SwiGLU width F the record holds, with no gaps:

  GU block: F rows of 9L/8 bytes; row f = gate codes f (L/2) | up codes f (L/2)
            | gate scales f (L/16) | up scales f (L/16)
  D block:  L/2 row pairs of 9F/8 bytes; pair p = down codes rows 2p, 2p+1
            (F/2 each) | down scales rows 2p, 2p+1 (F/16 each)
  globals:  fp32 little-endian gate, up, down

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
    """Split one record (uint8 buffer) into the logical (codes, scales, globals).

    Logical order: codes = gate [F][L/2] | up [F][L/2] | down [L][F/2];
    scales = gate [F][L/16] | up [F][L/16] | down [L][F/16].
    """
    L, F = latent, ffn
    buf = np.asarray(buf, dtype=np.uint8)
    gu_row, d_pair = 9 * L // 8, 9 * F // 8
    gu = buf[:F * gu_row].reshape(F, gu_row)
    dd = buf[F * gu_row:F * gu_row + (L // 2) * d_pair].reshape(L // 2, d_pair)
    g_codes, u_codes = gu[:, :L // 2], gu[:, L // 2:L]
    g_scales, u_scales = gu[:, L:L + L // 16], gu[:, L + L // 16:]
    d_codes = dd[:, :F].reshape(L, F // 2)
    d_scales = dd[:, F:].reshape(L, F // 16)
    codes = np.concatenate([g_codes.ravel(), u_codes.ravel(), d_codes.ravel()])
    scales = np.concatenate([g_scales.ravel(), u_scales.ravel(), d_scales.ravel()])
    body = F * gu_row + (L // 2) * d_pair
    glob = buf[body:body + 12].view("<f4").astype(np.float32)
    return codes, scales, glob
