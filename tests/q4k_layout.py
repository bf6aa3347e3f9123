"""Test-side numpy reading of the customary 144-byte q4_K super-block.

A third, independent statement of the byte layout (besides the oracle's C
unpacker and the product's C packer), used to build fixtures and to
cross-check both.  Layout: bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 twelve
bytes s[] of 6-bit scales/mins (sub-blocks 0-3 in the low 6 bits of s[0..3]
and s[4..7]; sub-blocks 4-7 split into a low nibble in s[8..11] and two high
bits in the top of s[0..3] / s[4..7]), 16-143 nibbles (element 64p+32h+l is
nibble h of byte 32p+l).
"""
import numpy as np


def decode(blk: np.ndarray, N: int, K: int):
    b = blk.reshape(N, K // 256, 144)
    d = b[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    s = b[:, :, 4:16].astype(np.int64)
    sc = np.empty((N, K // 256, 8), np.int64)
    m = np.empty((N, K // 256, 8), np.int64)
    sc[:, :, 0:4] = s[:, :, 0:4] & 63
    m[:, :, 0:4] = s[:, :, 4:8] & 63
    sc[:, :, 4:8] = (s[:, :, 8:12] & 15) + 16 * (s[:, :, 0:4] // 64)
    m[:, :, 4:8] = (s[:, :, 8:12] // 16) + 16 * (s[:, :, 4:8] // 64)
    qb = b[:, :, 16:144].reshape(N, K // 256, 4, 32).astype(np.int64)
    v = np.stack([qb & 15, qb >> 4], axis=3)          # [N, sb, p, h, l]
    v = v.reshape(N, K)
    return dict(d=d, dmin=dmin, sc=sc.reshape(N, K // 32), m=m.reshape(N, K // 32), v=v)


def encode(d, dmin, sc, m, v) -> np.ndarray:
    """Fields -> bytes. d, dmin [N][K/256] (float, rounded to fp16);
    sc, m [N][K/32] in 0..63; v [N][K] in 0..15."""
    v = np.asarray(v, np.int64)
    N, K = v.shape
    nsb = K // 256
    sc = np.asarray(sc, np.int64).reshape(N, nsb, 8)
    m = np.asarray(m, np.int64).reshape(N, nsb, 8)
    out = np.zeros((N, nsb, 144), np.uint8)
    out[:, :, 0:2] = np.asarray(d, np.float16).reshape(N, nsb, 1).view(np.uint8)
    out[:, :, 2:4] = np.asarray(dmin, np.float16).reshape(N, nsb, 1).view(np.uint8)
    s = np.zeros((N, nsb, 12), np.int64)
    s[:, :, 0:4] = sc[:, :, 0:4] + 64 * (sc[:, :, 4:8] // 16)
    s[:, :, 4:8] = m[:, :, 0:4] + 64 * (m[:, :, 4:8] // 16)
    s[:, :, 8:12] = (sc[:, :, 4:8] % 16) + 16 * (m[:, :, 4:8] % 16)
    out[:, :, 4:16] = s.astype(np.uint8)
    vv = v.reshape(N, nsb, 4, 2, 32)
    out[:, :, 16:144] = (vv[:, :, :, 0, :] + 16 * vv[:, :, :, 1, :]).reshape(N, nsb, 128).astype(np.uint8)
    return out
