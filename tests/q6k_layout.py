"""Test-side numpy statement of the customary 210-byte q6_K super-block.

A second, independent statement of the layout (besides the oracle's
decoder and the product's C packer), used to build fixtures.  Layout:
bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits), 192-207 int8
scales (one per 16 weights), 208-209 fp16 d.  Quant q in [-32, 31] is
stored as u = q + 32; element 128n + 32r + l keeps its low nibble in
nibble r // 2 of ql[64n + 32 (r % 2) + l] and its two high bits in bits
2r, 2r + 1 of qh[32n + l].
"""
import numpy as np


def encode(q, sc, d) -> np.ndarray:
    """q [N][K] in -32..31, sc [N][K/16] in -128..127, d [N][K/256] (rounded to fp16)."""
    q = np.asarray(q, np.int64)
    N, K = q.shape
    nsb = K // 256
    u = (q + 32).reshape(N, nsb, 2, 4, 32)          # [N, sb, n, r, l]
    out = np.zeros((N, nsb, 210), np.uint8)
    ql = np.zeros((N, nsb, 2, 2, 32), np.int64)      # [n, r % 2, l]
    qh = np.zeros((N, nsb, 2, 32), np.int64)         # [n, l]
    for r in range(4):
        ql[:, :, :, r % 2, :] |= (u[:, :, :, r, :] & 15) << (4 * (r // 2))
        qh[:, :, :, :] |= (u[:, :, :, r, :] >> 4) << (2 * r)
    out[:, :, 0:128] = ql.reshape(N, nsb, 128)
    out[:, :, 128:192] = qh.reshape(N, nsb, 64)
    out[:, :, 192:208] = np.asarray(sc, np.int64).reshape(N, nsb, 16).astype(np.int8).view(np.uint8)
    out[:, :, 208:210] = np.asarray(d, np.float16).reshape(N, nsb, 1).view(np.uint8)
    return out
