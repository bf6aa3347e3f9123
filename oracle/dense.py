"""CPU oracle for the dequantize-then-dense control path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product library never calls it and
shares no code with it.

The control path is the f16 GEMM path the pages measure MMQ against (web page
"16 . r12 -- 16-chain warp tile + ldmatrix", the landing note comparing MMQ
with the f16 default path), with its dequantize step as on page "Round 31
Track C Audit: dq_f16 (dense_mm.metal) & DW<F> (mma.metal)", section 2.1
(q4_K weights expanded to an fp16 buffer, then a dense GEMM).

Reading (the pages do not print the arithmetic): each weight is
    w = fp16( f32( d*sc*v - dmin*m ) )
with d*sc*v and dmin*m exact in float32 (at most 21 and 17 significant
bits), the difference rounded once to float32 and then once to float16,
round-to-nearest-even both times -- what a float32 dequantizer writing
fp16 produces.  Activations are rounded from float32 to float16 the same
way.  The GEMM reference sums the exact products of the fp16 values in
float64.

Pins (tests/test_oracle_pins.py): hand-worked values, including one where
rounding to float32 first changes the fp16 result (tests/golden), a q4_K
field sweep against fractions.Fraction, and integer matrices against an
int64 matmul.
"""
from __future__ import annotations

import numpy as np

from . import unpack_q4K


def dequantize_q4K_f16(blk: np.ndarray, N: int, K: int) -> np.ndarray:
    """q4_K bytes -> float16 [N][K]: fp16(f32(d*sc*v - dmin*m))."""
    u = unpack_q4K(blk, N, K)
    d = np.repeat(u["d"].astype(np.float32), 256, axis=1)        # fp16 values: exact in f32
    dmin = np.repeat(u["dmin"].astype(np.float32), 256, axis=1)
    sc = np.repeat(u["sc"].astype(np.float32), 32, axis=1)
    m = np.repeat(u["m"].astype(np.float32), 32, axis=1)
    v = u["v"].astype(np.float32)
    a = d * sc * v            # exact in float32
    b = dmin * m              # exact in float32
    return (a - b).astype(np.float16)   # one float32 rounding, then one float16 rounding


def convert_f16(x: np.ndarray) -> np.ndarray:
    """float32 -> float16, round to nearest even."""
    return np.asarray(x, np.float32).astype(np.float16)


def gemm_f16(a16: np.ndarray, b16: np.ndarray):
    """C = A . B^T of fp16 A [M][K], B [N][K]: exact products summed in float64.
    Returns (C float64 [M][N], T = sum |a*b| float64 [M][N])."""
    A = np.asarray(a16, np.float16).astype(np.float64)
    B = np.asarray(b16, np.float16).astype(np.float64)
    return A @ B.T, np.abs(A) @ np.abs(B).T


def gemm_f16_sampled(a16: np.ndarray, b16: np.ndarray, rows, cols):
    """gemm_f16 at the listed (row, col) pairs only: (C float64, T float64)."""
    A = np.asarray(a16, np.float16).astype(np.float64)[np.asarray(rows)]
    B = np.asarray(b16, np.float16).astype(np.float64)[np.asarray(cols)]
    return np.einsum("ik,ik->i", A, B), np.einsum("ik,ik->i", np.abs(A), np.abs(B))
