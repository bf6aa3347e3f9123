"""CPU oracle for the q4_K x q8_1 quantized GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.  The arithmetic lives in ``oracle.c`` (plain C, built
``-O2 -fno-fast-math -ffp-contract=off`` with OpenMP over rows); this module
only builds it and marshals numpy arrays.

Oracle array layouts (its own, deliberately the plainest ones):
  q  int8  [M][K]          da float32 [M][K/32]      sa int32 [M][K/32]
  blk uint8 [N][K/256][144] (customary q4_K super-blocks)
  S  int32 [M][N][K/32]     C float32 [M][N]          T float64 [M][N]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
          "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            sigs = {
                "oracle_quantize_q8_1": [P, I, I, P, P, P],
                "oracle_unpack_q4K": [P, I, I, P, P, P, P, P],
                "oracle_dequant_q4K": [P, I, I, P],
                "oracle_block_dots": [P, P, I, I, I, P],
                "oracle_gemm": [P, P, P, P, I, I, I, P, P, P],
                "oracle_gemm_sampled": [P, P, P, P, I, I, I, I, P, P, P, P, P],
                "oracle_dequant_dot": [P, P, P, I, I, I, P],
            }
            for name, args in sigs.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def quantize_q8_1(x: np.ndarray):
    """x float32 [M][K] -> (q int8 [M][K], da float32 [M][K/32], sa int32 [M][K/32])."""
    x = _c(x, np.float32)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K), np.int8)
    da = np.empty((M, K // 32), np.float32)
    sa = np.empty((M, K // 32), np.int32)
    _load().oracle_quantize_q8_1(_p(x), M, K, _p(q), _p(da), _p(sa))
    return q, da, sa


def unpack_q4K(blk: np.ndarray, N: int, K: int):
    """q4_K bytes -> dict(d, dmin [N][K/256] f64; sc, m [N][K/32] u8; v [N][K] u8)."""
    blk = _c(blk, np.uint8)
    assert blk.size == N * (K // 256) * 144
    out = dict(d=np.empty((N, K // 256)), dmin=np.empty((N, K // 256)),
               sc=np.empty((N, K // 32), np.uint8), m=np.empty((N, K // 32), np.uint8),
               v=np.empty((N, K), np.uint8))
    _load().oracle_unpack_q4K(_p(blk), N, K, _p(out["d"]), _p(out["dmin"]),
                              _p(out["sc"]), _p(out["m"]), _p(out["v"]))
    return out


def dequant_q4K(blk: np.ndarray, N: int, K: int) -> np.ndarray:
    """w = d*sc*v - dmin*m as float64 [N][K]."""
    blk = _c(blk, np.uint8)
    w = np.empty((N, K))
    _load().oracle_dequant_q4K(_p(blk), N, K, _p(w))
    return w


def block_dots(q: np.ndarray, blk: np.ndarray, N: int) -> np.ndarray:
    """Exact per-32-k int32 dots S [M][N][K/32]."""
    q = _c(q, np.int8)
    blk = _c(blk, np.uint8)
    M, K = q.shape
    S = np.empty((M, N, K // 32), np.int32)
    _load().oracle_block_dots(_p(q), _p(blk), M, N, K, _p(S))
    return S


def gemm(q, da, sa, blk, N: int, want_c64: bool = False, want_bound: bool = True):
    """Blockwise two-term GEMM. Returns (C f32 [M][N], C64 or None, T or None)."""
    q = _c(q, np.int8)
    da = _c(da, np.float32)
    sa = _c(sa, np.int32)
    blk = _c(blk, np.uint8)
    M, K = q.shape
    C = np.empty((M, N), np.float32)
    C64 = np.empty((M, N)) if want_c64 else None
    T = np.empty((M, N)) if want_bound else None
    _load().oracle_gemm(_p(q), _p(da), _p(sa), _p(blk), M, N, K, _p(C), _p(C64), _p(T))
    return C, C64, T


def gemm_sampled(q, da, sa, blk, N: int, rows, cols):
    """Same as gemm() for the listed (row, col) pairs only: (C f32, C64, T)."""
    q = _c(q, np.int8)
    da = _c(da, np.float32)
    sa = _c(sa, np.int32)
    blk = _c(blk, np.uint8)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    M, K = q.shape
    n = rows.size
    C = np.empty(n, np.float32)
    C64 = np.empty(n)
    T = np.empty(n)
    _load().oracle_gemm_sampled(_p(q), _p(da), _p(sa), _p(blk), M, N, K, n,
                                _p(rows), _p(cols), _p(C), _p(C64), _p(T))
    return C, C64, T


def dequant_dot(q, da, blk, N: int) -> np.ndarray:
    """Brute force D_ij = sum_k (da*q)_ik * w_jk in float64 [M][N]."""
    q = _c(q, np.int8)
    da = _c(da, np.float32)
    blk = _c(blk, np.uint8)
    M, K = q.shape
    D = np.empty((M, N))
    _load().oracle_dequant_dot(_p(q), _p(da), _p(blk), M, N, K, _p(D))
    return D


def within_tolerance(C_gpu: np.ndarray, C_ref: np.ndarray, T: np.ndarray,
                     rel: float = 1e-4, abs_: float = 1e-6) -> np.ndarray:
    """Elementwise |C_gpu - C_ref| <= rel * T + abs_ (the stated parity bound)."""
    return np.abs(C_gpu.astype(np.float64) - C_ref.astype(np.float64)) <= rel * T + abs_
