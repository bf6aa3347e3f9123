"""q4_K x q8_1 quantized GEMM (MMQ) for GB300 (sm_103a).

Thin ctypes binding over the C-ABI library ``lib/libmmq.so`` (declared in
``include/mmq.h``).  Functions named ``mmq_*`` mirror the C entry points
one to one and take raw pointers; the snake-case helpers below them only
allocate outputs with PyTorch and pass ``data_ptr()`` and the current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmmq.so")

MMQ_OK = 0
MMQ_ERR_ARG = -1
MMQ_ERR_ALIGN = -2
MMQ_ERR_DEVICE = -3
MMQ_ERR_RESOURCE = -4
MMQ_ERR_CUDA = -5
MMQ_ERR_DEVICE_TIMEOUT = -6

MMQ_PATH_AUTO = 0
MMQ_PATH_MMA_S8 = 1
MMQ_PATH_TC = 2
MMQ_PATH_SMALL_M = 3
MMQ_HOST_NOALLOC_SCRATCH_BYTES = 64 << 20
SMALL_M_MAX = 64
MMQ_GGUF_F32, MMQ_GGUF_F16, MMQ_GGUF_Q4_K, MMQ_GGUF_Q6_K = 0, 1, 12, 14

# Every symbol include/mmq.h declares.
EXPORTS = (
    "mmq_q8_1_bytes", "mmq_q8_1_view", "mmq_quantize_q8_1", "mmq_q4K_bytes",
    "mmq_pack_q4K", "mmq_q4K_gemm", "mmq_q8_1_tcop_bytes", "mmq_quantize_q8_1_tcop", "mmq_q4K_gemm_tcop", "mmq_q6K_gemm_path", "mmq_q6K_gemm_launches", "mmq_q6K_scaled_block_dots", "mmq_q4K_gemm_host_workspace", "mmq_q4K_gemm_host", "mmq_q4K_gemm_host_noalloc", "mmq_q4K_gemm_launches", "mmq_q4K_gemm_path", "mmq_q4K_gemm_q8_1", "mmq_q4K_block_dots", "mmq_q4K_scaled_block_dots",
    "mmq_dequantize_q4K_f16", "mmq_convert_f32_f16", "mmq_gemm_f16",
    "mmq_q4K_gemm_swiglu_q8_1", "mmq_interleave_rows_q4K",
    "mmq_q6K_bytes", "mmq_pack_q6K", "mmq_q6K_dev_bytes", "mmq_repack_q6K", "mmq_q6K_gemm",
    "mmq_q6K_block_dots",
    "mmq_gguf_open", "mmq_gguf_close", "mmq_gguf_tensor_count", "mmq_gguf_find", "mmq_gguf_tensor_info",
    "mmq_gguf_read", "mmq_gguf_write",
    "mmq_status", "mmq_strerror", "mmq_debug_inject_timeout", "mmq_debug_force_gemv_split",
    "mmq_set_programmatic_launch",
)


class mmq_q8_1_t(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("da", ctypes.c_void_p), ("sa", ctypes.c_void_p)]


class MMQError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmmq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libmmq.so not built ({path}); run q4_q8_int8_gb300.build.build()")
            lib = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
            Q = mmq_q8_1_t
            sigs = {
                "mmq_q8_1_bytes": ([I, I], S),
                "mmq_q8_1_view": ([P, I, I, ctypes.POINTER(Q)], ctypes.c_int),
                "mmq_quantize_q8_1": ([P, I, I, Q, P], ctypes.c_int),
                "mmq_q4K_bytes": ([I, I], S),
                "mmq_q8_1_tcop_bytes": ([I, I], S),
                "mmq_quantize_q8_1_tcop": ([P, I, I, Q, P, P], ctypes.c_int),
                "mmq_q4K_gemm_tcop": ([P, P, P, I, I, I, P], ctypes.c_int),
                "mmq_pack_q4K": ([P, P, P, P, P, I, I, P], ctypes.c_int),
                "mmq_q4K_gemm": ([Q, P, P, I, I, I, P], ctypes.c_int),
                "mmq_q4K_gemm_host_workspace": ([I, I, I], S),
                "mmq_q4K_gemm_host": ([P, P, P, I, I, I, P, S, P], ctypes.c_int),
                "mmq_q4K_gemm_host_noalloc": ([P, P, P, I, I, I, P], ctypes.c_int),
                "mmq_q4K_gemm_launches": ([I, I, I, ctypes.c_int], ctypes.c_int),
                "mmq_q4K_gemm_path": ([Q, P, P, I, I, I, ctypes.c_int, P], ctypes.c_int),
                "mmq_q4K_gemm_q8_1": ([Q, P, P, Q, I, I, I, P], ctypes.c_int),
                "mmq_q4K_block_dots": ([Q, P, P, I, I, I, ctypes.c_int, P], ctypes.c_int),
                "mmq_q4K_scaled_block_dots": ([Q, P, P, I, I, I, P], ctypes.c_int),
                "mmq_dequantize_q4K_f16": ([P, P, I, I, P], ctypes.c_int),
                "mmq_convert_f32_f16": ([P, P, I, P], ctypes.c_int),
                "mmq_gemm_f16": ([P, P, P, I, I, I, P], ctypes.c_int),
                "mmq_q4K_gemm_swiglu_q8_1": ([Q, P, P, Q, I, I, I, P], ctypes.c_int),
                "mmq_interleave_rows_q4K": ([P, P, P, I, I, P], ctypes.c_int),
                "mmq_q6K_bytes": ([I, I], S),
                "mmq_pack_q6K": ([P, P, P, I, I, P], ctypes.c_int),
                "mmq_q6K_dev_bytes": ([I, I], S),
                "mmq_repack_q6K": ([P, P, I, I, P], ctypes.c_int),
                "mmq_q6K_gemm": ([Q, P, P, I, I, I, P], ctypes.c_int),
                "mmq_q6K_gemm_path": ([Q, P, P, I, I, I, ctypes.c_int, P], ctypes.c_int),
                "mmq_q6K_gemm_launches": ([I, I, I, ctypes.c_int], ctypes.c_int),
                "mmq_q6K_scaled_block_dots": ([Q, P, P, I, I, I, P], ctypes.c_int),
                "mmq_q6K_block_dots": ([Q, P, P, I, I, I, P], ctypes.c_int),
                "mmq_gguf_open": ([ctypes.c_char_p, ctypes.POINTER(P)], ctypes.c_int),
                "mmq_gguf_close": ([P], None),
                "mmq_gguf_tensor_count": ([P], I),
                "mmq_gguf_find": ([P, ctypes.c_char_p], ctypes.c_int),
                "mmq_gguf_tensor_info": ([P, I, ctypes.c_char_p, S, ctypes.POINTER(ctypes.c_uint32),
                                          ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_uint64)], ctypes.c_int),
                "mmq_gguf_read": ([P, I, P, ctypes.c_uint64], ctypes.c_int),
                "mmq_gguf_write": ([ctypes.c_char_p, I, ctypes.POINTER(ctypes.c_char_p),
                                    ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(P)], ctypes.c_int),
                "mmq_status": ([P], ctypes.c_int),
                "mmq_strerror": ([ctypes.c_int], ctypes.c_char_p),
                "mmq_debug_inject_timeout": ([ctypes.c_int], None),
                "mmq_debug_force_gemv_split": ([ctypes.c_int], ctypes.c_int),
                "mmq_set_programmatic_launch": ([ctypes.c_int], None),
            }
            for name, (args, res) in sigs.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


# ---- one-to-one mirrors of the C entry points (raw pointers) ---------------
def mmq_q8_1_bytes(M, K):
    return load_library().mmq_q8_1_bytes(M, K)


def mmq_q8_1_view(buf, M, K, out):
    return load_library().mmq_q8_1_view(buf, M, K, ctypes.byref(out))


def mmq_quantize_q8_1(x, M, K, aq, stream):
    return load_library().mmq_quantize_q8_1(x, M, K, aq, stream)


def mmq_q4K_bytes(N, K):
    return load_library().mmq_q4K_bytes(N, K)


def mmq_q8_1_tcop_bytes(M, K):
    return load_library().mmq_q8_1_tcop_bytes(M, K)


def mmq_quantize_q8_1_tcop(x, M, K, aq, tcop, stream):
    return load_library().mmq_quantize_q8_1_tcop(x, M, K, aq, tcop, stream)


def mmq_q4K_gemm_tcop(tcop, bq4k, C, M, N, K, stream):
    return load_library().mmq_q4K_gemm_tcop(tcop, bq4k, C, M, N, K, stream)


def mmq_pack_q4K(v, sc, m, d, dmin, N, K, out):
    return load_library().mmq_pack_q4K(v, sc, m, d, dmin, N, K, out)


def mmq_q4K_gemm(aq, bq4k, C, M, N, K, stream):
    return load_library().mmq_q4K_gemm(aq, bq4k, C, M, N, K, stream)


def mmq_q4K_gemm_host_workspace(M, N, K):
    return load_library().mmq_q4K_gemm_host_workspace(M, N, K)


def mmq_q4K_gemm_host(x_host, bq4k, C_host, M, N, K, ws, ws_bytes, stream):
    return load_library().mmq_q4K_gemm_host(x_host, bq4k, C_host, M, N, K, ws, ws_bytes, stream)


def mmq_q4K_gemm_host_noalloc(x_host, bq4k, C_host, M, N, K, stream):
    return load_library().mmq_q4K_gemm_host_noalloc(x_host, bq4k, C_host, M, N, K, stream)


def mmq_q4K_gemm_launches(M, N, K, path):
    return load_library().mmq_q4K_gemm_launches(M, N, K, path)


def mmq_q4K_gemm_path(aq, bq4k, C, M, N, K, path, stream):
    return load_library().mmq_q4K_gemm_path(aq, bq4k, C, M, N, K, path, stream)


def mmq_q4K_gemm_q8_1(aq, bq4k, C, out, M, N, K, stream):
    return load_library().mmq_q4K_gemm_q8_1(aq, bq4k, C, out, M, N, K, stream)


def mmq_q4K_block_dots(aq, bq4k, S, M, N, K, path, stream):
    return load_library().mmq_q4K_block_dots(aq, bq4k, S, M, N, K, path, stream)


def mmq_q4K_scaled_block_dots(aq, bq4k, S, M, N, K, stream):
    return load_library().mmq_q4K_scaled_block_dots(aq, bq4k, S, M, N, K, stream)


def mmq_status(stream):
    return load_library().mmq_status(stream)


def mmq_strerror(code):
    return load_library().mmq_strerror(code).decode()


def mmq_debug_inject_timeout(enable):
    load_library().mmq_debug_inject_timeout(1 if enable else 0)


def mmq_debug_force_gemv_split(ks):
    return load_library().mmq_debug_force_gemv_split(ks)


def mmq_set_programmatic_launch(enable):
    load_library().mmq_set_programmatic_launch(1 if enable else 0)


def strerror(code: int) -> str:
    return mmq_strerror(code)


def _check(rc: int, what: str):
    if rc != MMQ_OK:
        raise MMQError(rc, what)


# ---- PyTorch-facing helpers (memory and streams only) ----------------------
def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def q8_1_struct(qs, da, sa) -> mmq_q8_1_t:
    return mmq_q8_1_t(qs.data_ptr(), da.data_ptr(), sa.data_ptr())


def empty_q8_1(M: int, K: int, device="cuda"):
    """Allocate (qs int8 [M][K], da f32 [M][K/32], sa int32 [M][K/32])."""
    import torch
    return (torch.empty((M, K), dtype=torch.int8, device=device),
            torch.empty((M, K // 32), dtype=torch.float32, device=device),
            torch.empty((M, K // 32), dtype=torch.int32, device=device))


def quantize_q8_1(x, out=None, stream=None):
    """x float32 [M][K] (CUDA, contiguous) -> (qs, da, sa) CUDA tensors."""
    M, K = x.shape
    qs, da, sa = out if out is not None else empty_q8_1(M, K, x.device)
    _check(mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), M, K, q8_1_struct(qs, da, sa),
                             _stream_ptr(stream)), "mmq_quantize_q8_1")
    return qs, da, sa


def empty_tcop(M: int, K: int, device="cuda"):
    """Allocate the tensor-core operand plane of M x K activations (uint8,
    mmq_q8_1_tcop_bytes(M, K) bytes; the caching allocator's blocks are
    256-byte aligned, which the call checks)."""
    import torch
    n = mmq_q8_1_tcop_bytes(M, K)
    if n == 0:
        raise MMQError(MMQ_ERR_ARG, "mmq_q8_1_tcop_bytes")
    return torch.empty((n,), dtype=torch.uint8, device=device)


def quantize_q8_1_tcop(x, out=None, tcop=None, stream=None):
    """x float32 [M][K] (CUDA) -> ((qs, da, sa), tcop): the q8_1 prepass that
    also writes the operand plane for q4K_gemm_tcop."""
    M, K = x.shape
    qs, da, sa = out if out is not None else empty_q8_1(M, K, x.device)
    tcop = tcop if tcop is not None else empty_tcop(M, K, x.device)
    _check(mmq_quantize_q8_1_tcop(ctypes.c_void_p(x.data_ptr()), M, K, q8_1_struct(qs, da, sa),
                                  ctypes.c_void_p(tcop.data_ptr()), _stream_ptr(stream)),
           "mmq_quantize_q8_1_tcop")
    return (qs, da, sa), tcop


def q4K_gemm_tcop(tcop, w, M: int, N: int, K: int, out=None, stream=None):
    """The super-block tcgen05 GEMM on an operand plane -> C float32 [M][N]."""
    import torch
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=w.device)
    _check(mmq_q4K_gemm_tcop(ctypes.c_void_p(tcop.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(C.data_ptr()), M, N, K, _stream_ptr(stream)),
           "mmq_q4K_gemm_tcop")
    return C


def q4K_gemm(aq, w, N: int, path: int = MMQ_PATH_AUTO, out=None, stream=None):
    """aq = (qs, da, sa); w uint8 q4_K bytes of an N x K matrix -> C float32 [M][N]."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=qs.device)
    _check(mmq_q4K_gemm_path(q8_1_struct(qs, da, sa), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(C.data_ptr()), M, N, K, path, _stream_ptr(stream)),
           "mmq_q4K_gemm")
    return C


def q4K_gemm_host(x_host, w, N: int, out=None, workspace=None, stream=None):
    """x_host float32 [M][K] CPU tensor (pinned for overlap) -> C float32 [M][N]
    CPU tensor, through mmq_q4K_gemm_host (chunked copies overlapped with the
    kernels).  Returns after the call is queued; synchronize the stream before
    reading the result.  Without a caller-owned `workspace` (a CUDA uint8
    tensor) one is allocated here and the call synchronizes the stream before
    returning, since the allocator cannot see the library's copy streams."""
    import torch
    M, K = x_host.shape
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    need = mmq_q4K_gemm_host_workspace(M, N, K)
    own = workspace is None
    if own:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=w.device)
    base = (workspace.data_ptr() + 255) // 256 * 256
    avail = workspace.numel() - (base - workspace.data_ptr())
    sp = _stream_ptr(stream)
    _check(mmq_q4K_gemm_host(ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(C.data_ptr()), M, N, K, ctypes.c_void_p(base), avail, sp),
           "mmq_q4K_gemm_host")
    if own:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return C


def q4K_gemm_q8_1(aq, w, N: int, with_c: bool = True, out=None, stream=None):
    """GEMM whose result is also quantized to q8_1 ([M][N] q8_1 triple, ready
    as the next GEMM's activations); returns (C or None, (qs, da, sa))."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    C = torch.empty((M, N), dtype=torch.float32, device=qs.device) if with_c else None
    o = out if out is not None else empty_q8_1(M, N, qs.device)
    _check(mmq_q4K_gemm_q8_1(q8_1_struct(qs, da, sa), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(C.data_ptr() if C is not None else 0), q8_1_struct(*o),
                             M, N, K, _stream_ptr(stream)),
           "mmq_q4K_gemm_q8_1")
    return C, o


def q4K_block_dots(aq, w, N: int, path: int = MMQ_PATH_AUTO, out=None, stream=None):
    """Exact per-chunk int32 dots S [M][N][K/32] from the selected kernel's dot-product code."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    S = out if out is not None else torch.empty((M, N, K // 32), dtype=torch.int32, device=qs.device)
    _check(mmq_q4K_block_dots(q8_1_struct(qs, da, sa), ctypes.c_void_p(w.data_ptr()),
                              ctypes.c_void_p(S.data_ptr()), M, N, K, path, _stream_ptr(stream)),
           "mmq_q4K_block_dots")
    return S


def q4K_scaled_block_dots(aq, w, N: int, out=None, stream=None):
    """sc * S int32 [M][N][K/32] from the tcgen05 kernel's own weight operand."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    S = out if out is not None else torch.empty((M, N, K // 32), dtype=torch.int32, device=qs.device)
    _check(mmq_q4K_scaled_block_dots(q8_1_struct(qs, da, sa), ctypes.c_void_p(w.data_ptr()),
                                     ctypes.c_void_p(S.data_ptr()), M, N, K, _stream_ptr(stream)),
           "mmq_q4K_scaled_block_dots")
    return S


def force_gemv_split(ks: int):
    """Test hook: force the dot-product kernel's K split (1, 2, 4; 0 = automatic)."""
    _check(mmq_debug_force_gemv_split(ks), "mmq_debug_force_gemv_split")


def mmq_dequantize_q4K_f16(bq4k, wh, N, K, stream):
    return load_library().mmq_dequantize_q4K_f16(bq4k, wh, N, K, stream)


def mmq_convert_f32_f16(x, xh, n, stream):
    return load_library().mmq_convert_f32_f16(x, xh, n, stream)


def mmq_gemm_f16(A, B, C, M, N, K, stream):
    return load_library().mmq_gemm_f16(A, B, C, M, N, K, stream)


def mmq_q4K_gemm_swiglu_q8_1(aq, bq4k_gu, hf, out, M, F, K, stream):
    return load_library().mmq_q4K_gemm_swiglu_q8_1(aq, bq4k_gu, hf, out, M, F, K, stream)


def mmq_interleave_rows_q4K(gate, up, out, F, K, stream):
    return load_library().mmq_interleave_rows_q4K(gate, up, out, F, K, stream)


def interleave_rows_q4K(gate, up, F: int, K: int, out=None, stream=None):
    """gate, up: q4_K bytes of F x K matrices (CUDA uint8) -> rows interleaved (2F x K)."""
    import torch
    o = out if out is not None else torch.empty(2 * gate.numel(), dtype=torch.uint8, device=gate.device)
    _check(mmq_interleave_rows_q4K(ctypes.c_void_p(gate.data_ptr()), ctypes.c_void_p(up.data_ptr()),
                                   ctypes.c_void_p(o.data_ptr()), F, K, _stream_ptr(stream)),
           "mmq_interleave_rows_q4K")
    return o


def q4K_gemm_swiglu_q8_1(aq, w_gu, F: int, with_h: bool = False, out=None, stream=None):
    """silu(x.gate^T) * (x.up^T) quantized to q8_1 ([M][F] triple); w_gu from
    interleave_rows_q4K.  Returns (h f32 or None, (qs, da, sa))."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    h = torch.empty((M, F), dtype=torch.float32, device=qs.device) if with_h else None
    o = out if out is not None else empty_q8_1(M, F, qs.device)
    _check(mmq_q4K_gemm_swiglu_q8_1(q8_1_struct(qs, da, sa), ctypes.c_void_p(w_gu.data_ptr()),
                                    ctypes.c_void_p(h.data_ptr() if h is not None else 0), q8_1_struct(*o),
                                    M, F, K, _stream_ptr(stream)),
           "mmq_q4K_gemm_swiglu_q8_1")
    return h, o


def mmq_q6K_bytes(N, K):
    return load_library().mmq_q6K_bytes(N, K)


def mmq_pack_q6K(q, sc, d, N, K, out):
    return load_library().mmq_pack_q6K(q, sc, d, N, K, out)


def mmq_q6K_dev_bytes(N, K):
    return load_library().mmq_q6K_dev_bytes(N, K)


def mmq_repack_q6K(src, dst, N, K, stream):
    return load_library().mmq_repack_q6K(src, dst, N, K, stream)


def mmq_q6K_gemm(aq, w, C, M, N, K, stream):
    return load_library().mmq_q6K_gemm(aq, w, C, M, N, K, stream)


def mmq_q6K_gemm_path(aq, w, C, M, N, K, path, stream):
    return load_library().mmq_q6K_gemm_path(aq, w, C, M, N, K, path, stream)


def mmq_q6K_gemm_launches(M, N, K, path):
    return load_library().mmq_q6K_gemm_launches(M, N, K, path)


def mmq_q6K_scaled_block_dots(aq, w, S, M, N, K, stream):
    return load_library().mmq_q6K_scaled_block_dots(aq, w, S, M, N, K, stream)


def mmq_q6K_block_dots(aq, w, S, M, N, K, stream):
    return load_library().mmq_q6K_block_dots(aq, w, S, M, N, K, stream)


def pack_q6K(q, sc, d_bits):
    """Host packer (numpy): q int8 [N][K], sc int8 [N][K/16], d fp16 bits [N][K/256] -> bytes."""
    import numpy as np
    q = np.ascontiguousarray(q, np.int8)
    N, K = q.shape
    sc = np.ascontiguousarray(sc, np.int8)
    d_bits = np.ascontiguousarray(d_bits, np.uint16)
    out = np.empty((N, K // 256, 210), np.uint8)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(mmq_pack_q6K(ptr(q), ptr(sc), ptr(d_bits), N, K, ptr(out)), "mmq_pack_q6K")
    return out


def repack_q6K(w, N: int, K: int, out=None, stream=None):
    """Customary q6_K bytes (CUDA uint8) -> the device layout the q6_K GEMM reads."""
    import torch
    o = out if out is not None else torch.empty(N * (K // 256) * 224, dtype=torch.uint8, device=w.device)
    _check(mmq_repack_q6K(ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(o.data_ptr()), N, K,
                          _stream_ptr(stream)), "mmq_repack_q6K")
    return o


def q6K_gemm(aq, w_dev, N: int, path: int = MMQ_PATH_AUTO, out=None, stream=None):
    """aq = (qs, da, sa); w_dev q6_K bytes in the device layout -> C float32 [M][N]."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=qs.device)
    _check(mmq_q6K_gemm_path(q8_1_struct(qs, da, sa), ctypes.c_void_p(w_dev.data_ptr()),
                             ctypes.c_void_p(C.data_ptr()), M, N, K, path, _stream_ptr(stream)), "mmq_q6K_gemm")
    return C


def q6K_block_dots(aq, w_dev, N: int, out=None, stream=None):
    """Exact per-16 int32 dots S [M][N][K/16]."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    S = out if out is not None else torch.empty((M, N, K // 16), dtype=torch.int32, device=qs.device)
    _check(mmq_q6K_block_dots(q8_1_struct(qs, da, sa), ctypes.c_void_p(w_dev.data_ptr()),
                              ctypes.c_void_p(S.data_ptr()), M, N, K, _stream_ptr(stream)), "mmq_q6K_block_dots")
    return S


def q6K_scaled_block_dots(aq, w_dev, N: int, out=None, stream=None):
    """The tcgen05 q6_K kernel's exact per-chunk dots S' [M][N][K/32] (int32):
    per 32-k chunk the sum of sc * S16 over its two sub-blocks."""
    import torch
    qs, da, sa = aq
    M, K = qs.shape
    S = out if out is not None else torch.empty((M, N, K // 32), dtype=torch.int32, device=qs.device)
    _check(mmq_q6K_scaled_block_dots(q8_1_struct(qs, da, sa), ctypes.c_void_p(w_dev.data_ptr()),
                                     ctypes.c_void_p(S.data_ptr()), M, N, K, _stream_ptr(stream)),
           "mmq_q6K_scaled_block_dots")
    return S


def gguf_write(path: str, tensors):
    """tensors: list of (name, type, ne0, ne1, numpy buffer) -> a GGUF file."""
    import numpy as np
    lib = load_library()
    n = len(tensors)
    bufs = [np.ascontiguousarray(t[4]) for t in tensors]
    names = (ctypes.c_char_p * n)(*[t[0].encode() for t in tensors])
    types = (ctypes.c_uint32 * n)(*[t[1] for t in tensors])
    dims = (ctypes.c_int64 * (2 * n))(*[v for t in tensors for v in (t[2], t[3])])
    data = (ctypes.c_void_p * n)(*[b.ctypes.data_as(ctypes.c_void_p) for b in bufs])
    _check(lib.mmq_gguf_write(path.encode(), n, names, types, dims, data), "mmq_gguf_write")


def gguf_read(path: str):
    """A GGUF file -> {name: (type, dims tuple, numpy uint8 bytes)} for the
    F32 / F16 / Q4_K / Q6_K tensors (others listed with empty bytes)."""
    import numpy as np
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.mmq_gguf_open(path.encode(), ctypes.byref(h)), "mmq_gguf_open")
    try:
        out = {}
        for i in range(lib.mmq_gguf_tensor_count(h)):
            name = ctypes.create_string_buffer(256)
            t, nd = ctypes.c_uint32(), ctypes.c_uint32()
            dims = (ctypes.c_int64 * 4)()
            nb = ctypes.c_uint64()
            _check(lib.mmq_gguf_tensor_info(h, i, name, 256, ctypes.byref(t), ctypes.byref(nd), dims,
                                            ctypes.byref(nb)), "mmq_gguf_tensor_info")
            buf = np.empty(nb.value, np.uint8)
            if nb.value:
                _check(lib.mmq_gguf_read(h, i, buf.ctypes.data_as(ctypes.c_void_p), nb.value), "mmq_gguf_read")
            out[name.value.decode()] = (t.value, tuple(dims[:nd.value]), buf)
        return out
    finally:
        lib.mmq_gguf_close(h)


def dequantize_q4K_f16(w, N: int, K: int, out=None, stream=None):
    """q4_K bytes of an N x K matrix (CUDA uint8) -> float16 [N][K]."""
    import torch
    wh = out if out is not None else torch.empty((N, K), dtype=torch.float16, device=w.device)
    _check(mmq_dequantize_q4K_f16(ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(wh.data_ptr()), N, K,
                                  _stream_ptr(stream)), "mmq_dequantize_q4K_f16")
    return wh


def convert_f16(x, out=None, stream=None):
    """float32 CUDA tensor -> float16 of the same shape (round to nearest even)."""
    import torch
    xh = out if out is not None else torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check(mmq_convert_f32_f16(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(xh.data_ptr()), x.numel(),
                               _stream_ptr(stream)), "mmq_convert_f32_f16")
    return xh


def gemm_f16(a, b, out=None, stream=None):
    """a float16 [M][K], b float16 [N][K] (CUDA) -> a . b^T as float32 [M][N]."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check(mmq_gemm_f16(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                        ctypes.c_void_p(C.data_ptr()), M, N, K, _stream_ptr(stream)), "mmq_gemm_f16")
    return C


def status(stream=None) -> int:
    return mmq_status(_stream_ptr(stream))


def pack_q4K(v, sc, m, d_bits, dmin_bits):
    """Host packer (numpy arrays): fields -> q4_K bytes [N][K/256][144]."""
    import numpy as np
    v = np.ascontiguousarray(v, np.uint8)
    N, K = v.shape
    sc = np.ascontiguousarray(sc, np.uint8)
    m = np.ascontiguousarray(m, np.uint8)
    d_bits = np.ascontiguousarray(d_bits, np.uint16)
    dmin_bits = np.ascontiguousarray(dmin_bits, np.uint16)
    out = np.empty((N, K // 256, 144), np.uint8)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(mmq_pack_q4K(ptr(v), ptr(sc), ptr(m), ptr(d_bits), ptr(dmin_bits), N, K, ptr(out)),
           "mmq_pack_q4K")
    return out
