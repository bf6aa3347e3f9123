"""Numpy restatement of the tensor-core operand plane's encoding (the bytes
mmq_quantize_q8_1_tcop writes), for exact tests of the device encoding.

Built from the q8_1 values (q, da, sa) only; every step is one correctly
rounded f32 or fp16 operation (numpy's float32 -> float16 conversion rounds
to nearest even, and an fp16 x fp16 product is exact in float32 before its
single rounding to fp16), so the bits must match the kernel's exactly.
"""
import numpy as np


def _f32(u):
    return np.asarray(u, np.uint32).view(np.float32)


def _u32(f):
    return np.asarray(f, np.float32).view(np.uint32)


def super_block_scale(da):
    """da f32 [M][K/32] -> (inv, g) f32 [M][K/256]: 2^(134-e), 2^(e-134) with e
    the biased exponent of the largest da of the eight chunks, at least 8."""
    M, nb = da.shape
    D = da.reshape(M, nb // 8, 8).max(axis=2)
    eb = np.maximum((_u32(D) >> 23) & 0xFF, 8).astype(np.uint32)
    return _f32((261 - eb) << 23), _f32((eb - 7) << 23)


def encode(q, da, sa):
    """-> (hi, lo uint16 [M][K] in the plane's k order, t2 uint32
    [M][K/256][32], g f32 [M][K/256])."""
    q = np.asarray(q, np.int8)
    M, K = q.shape
    inv, g = super_block_scale(da)
    s = da * np.repeat(inv, 8, axis=1)                          # exact (power of two)
    shi = _f32((_u32(s) + np.uint32(0x00080000)) & np.uint32(0xFFF00000))
    hh = shi.astype(np.float16)
    hl = (s - hh.astype(np.float32)).astype(np.float16)
    qh = q.astype(np.float16)
    hi = (qh * np.repeat(hh, 32, axis=1)).astype(np.float16)   # exact product
    lo = (qh * np.repeat(hl, 32, axis=1)).astype(np.float16)
    perm = np.arange(K).reshape(-1, 4)[:, [0, 2, 1, 3]].reshape(-1)
    am = (da * sa.astype(np.float32)) * np.repeat(inv, 8, axis=1)
    ahi = _f32(_u32(am) & np.uint32(0xFFFFE000))
    alo = am - ahi
    nsb = K // 256
    t2 = np.zeros((M, nsb, 32), np.float32)
    t2[:, :, 0:8] = ahi.reshape(M, nsb, 8)
    t2[:, :, 8:16] = ahi.reshape(M, nsb, 8)
    t2[:, :, 16:24] = alo.reshape(M, nsb, 8)
    return (hi[:, perm].view(np.uint16), lo[:, perm].view(np.uint16), t2.view(np.uint32), g)


def split(buf, M, K):
    """The plane's bytes (uint8 numpy) -> (hi, lo [M][K], t2, g) views, at the
    offsets the library uses (each part 256-byte aligned; the activation part
    holds, per token row and 32-k chunk, 32 hi values then 32 lo values)."""
    up = lambda b: (b + 255) // 256 * 256
    n, nsb = M * K, M * (K // 256)
    o_t2 = up(4 * n)
    o_g = o_t2 + up(nsb * 128)
    a = buf[:4 * n].view(np.uint16).reshape(M, K // 32, 2, 32)
    hi = a[:, :, 0, :].reshape(M, K)
    lo = a[:, :, 1, :].reshape(M, K)
    t2 = buf[o_t2:o_t2 + nsb * 128].view(np.uint32).reshape(M, K // 256, 32)
    g = buf[o_g:o_g + nsb * 4].view(np.float32).reshape(M, K // 256)
    return hi, lo, t2, g
