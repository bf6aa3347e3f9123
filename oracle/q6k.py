"""CPU oracle for q6_K x q8_1 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product library never calls it and
shares no code with it.

q6_K is the next weight family the pages' MMQ line moved to (web page "20 .
r15 -- f32-accumulate mma probe (dead end) + rank-1 term2 rescale", section
"Proof of pattern portability", and its master-table note: the fold was
later reused in the q6_K kernels).  The pages print neither its layout nor
its arithmetic; the readings taken here:

* Layout: the customary 210-byte super-block of 256 weights -- ql[128] (low
  4 bits of each quant), qh[64] (high 2 bits), scales[16] (int8, one per 16
  consecutive weights), d (fp16).  Element e = 128 n + 32 r + l of a
  super-block (n = 0..1, r = 0..3, l = 0..31): low bits = nibble (r >> 1) of
  ql[64 n + 32 (r & 1) + l], high bits = bits 2r..2r+1 of qh[32 n + l];
  quant q = low | high << 4, minus 32 (so q in [-32, 31]); scale index e / 16.
* Arithmetic: weight w = d * sc * q (no minimum, so the second term of the
  q4_K rescale is absent).  Per 16-weight sub-block s the exact integer dot
  S_is = sum_k a_ik * q_jk; per q8_1 block c (two sub-blocks):
      C_ij += da_ic * d_j * (sc_j,2c * S_i,2c + sc_j,2c+1 * S_i,2c+1),
  here in float64, rounded once to float32.

Pins (tests/test_oracle_pins.py): hand-packed bytes against
tests/golden/q6k_bytes.txt, pack/unpack round trips against the tests' own
encoder, S against an int64 einsum, worked single-block examples, and the
identity C == dot(da * q_a, dequant(W)) on brute-force tiny inputs.
"""
from __future__ import annotations

import numpy as np

QK6 = 256
Q6K_BYTES = 210


def unpack_q6K(blk: np.ndarray, N: int, K: int):
    """bytes [N][K/256][210] -> dict(q int8 [N][K], sc int8 [N][K/16], d float64 [N][K/256])."""
    b = np.asarray(blk, np.uint8).reshape(N, K // QK6, Q6K_BYTES)
    ql = b[:, :, 0:128].astype(np.int64)
    qh = b[:, :, 128:192].astype(np.int64)
    sc = b[:, :, 192:208].copy().view(np.int8).reshape(N, K // 16)
    d = b[:, :, 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
    q = np.empty((N, K // QK6, 256), np.int64)
    for n in range(2):
        for r in range(4):
            for l in range(32):
                low = (ql[:, :, 64 * n + 32 * (r & 1) + l] >> (4 * (r >> 1))) & 15
                high = (qh[:, :, 32 * n + l] >> (2 * r)) & 3
                q[:, :, 128 * n + 32 * r + l] = (low | (high << 4)) - 32
    return dict(q=q.reshape(N, K).astype(np.int8), sc=sc, d=d)


def dequant_q6K(blk: np.ndarray, N: int, K: int) -> np.ndarray:
    """w = d * sc * q as float64 [N][K]."""
    u = unpack_q6K(blk, N, K)
    return (np.repeat(u["d"], 256, axis=1) * np.repeat(u["sc"].astype(np.float64), 16, axis=1)
            * u["q"].astype(np.float64))


def block_dots16(qa: np.ndarray, blk: np.ndarray, N: int) -> np.ndarray:
    """Exact per-16-k dots S [M][N][K/16] (int32) of int8 activations with q6_K quants."""
    qa = np.asarray(qa, np.int8)
    M, K = qa.shape
    q = unpack_q6K(blk, N, K)["q"].astype(np.int64)
    A = qa.astype(np.int64).reshape(M, K // 16, 16)
    W = q.reshape(N, K // 16, 16)
    return np.einsum("msk,nsk->mns", A, W).astype(np.int32)


def gemm(qa, da, blk, N: int, rows=None, cols=None):
    """Blockwise q6_K x q8_1 GEMM in float64.  Returns (C float32, C64, T) for
    all outputs [M][N], or for the listed (row, col) pairs; T = sum_k
    |a_k w_k| with a = da * q (the tolerance scale)."""
    qa = np.asarray(qa, np.int8)
    da = np.asarray(da, np.float32).astype(np.float64)
    M, K = qa.shape
    u = unpack_q6K(blk, N, K)
    dsc = np.repeat(u["d"], 16, axis=1) * u["sc"].astype(np.float64)      # [N][K/16]
    if rows is None:
        S = block_dots16(qa, blk, N).astype(np.float64)                    # [M][N][K/16]
        da16 = np.repeat(da, 2, axis=1)                                    # [M][K/16]
        C64 = np.einsum("ms,mns,ns->mn", da16, S, dsc)
        a = np.repeat(da, 32, axis=1) * qa.astype(np.float64)              # [M][K]
        w = np.repeat(dsc, 16, axis=1) * u["q"].astype(np.float64)        # [N][K]
        T = np.abs(a) @ np.abs(w).T
    else:
        rows = np.asarray(rows)
        cols = np.asarray(cols)
        A = qa.astype(np.int64)[rows].reshape(rows.size, K // 16, 16)
        W = u["q"].astype(np.int64)[cols].reshape(cols.size, K // 16, 16)
        S = np.einsum("psk,psk->ps", A, W).astype(np.float64)              # [P][K/16]
        da16 = np.repeat(da[rows], 2, axis=1)
        C64 = np.einsum("ps,ps,ps->p", da16, S, dsc[cols])
        a = np.repeat(da[rows], 32, axis=1) * qa.astype(np.float64)[rows]
        w = np.repeat(dsc[cols], 16, axis=1) * u["q"].astype(np.float64)[cols]
        T = np.einsum("pk,pk->p", np.abs(a), np.abs(w))
    return C64.astype(np.float32), C64, T


def dequant_dot(qa, da, blk, N: int) -> np.ndarray:
    """Brute force D_ij = sum_k (da * q_a)_ik * w_jk in float64."""
    qa = np.asarray(qa, np.int8)
    M, K = qa.shape
    a = np.repeat(np.asarray(da, np.float32).astype(np.float64), 32, axis=1) * qa.astype(np.float64)
    return a @ dequant_q6K(blk, N, K).T
