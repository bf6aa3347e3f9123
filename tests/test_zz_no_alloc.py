"""mmq_q4K_gemm_host_noalloc: the host-buffer prepass + GEMM for callers that
cannot give the library device memory (code that reaches the GPU only
through this C ABI, or a plug-in whose host process has reserved the device
memory in its own pool).  Its workspace is a fixed device array inside the
library instead of a caller allocation.

The test calls it through the C ABI twice in a row, on two different shapes
and inputs (the second call reuses the array the first one filled), and
compares each result with mmq_q4K_gemm_host given a caller-allocated
workspace, within the GEMM tolerance |dC| <= 1e-4 * sum_k |a_k w_k| + 1e-6.
It also checks that a shape whose workspace does not fit in the array is
refused before any device work.  This file is collected last, so that a
run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _noalloc(mmq, xh, w, Ch, M, N, K):
    import torch
    stream = torch.cuda.current_stream()
    rc = mmq.mmq_q4K_gemm_host_noalloc(ctypes.c_void_p(xh.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                       ctypes.c_void_p(Ch.data_ptr()), M, N, K, mmq._stream_ptr(stream))
    assert rc == mmq.MMQ_OK, mmq.strerror(rc)
    stream.synchronize()


def _with_workspace(mmq, xh, w, M, N, K):
    import torch
    need = mmq.mmq_q4K_gemm_host_workspace(M, N, K)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    Ch = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.current_stream()
    rc = mmq.mmq_q4K_gemm_host(ctypes.c_void_p(xh.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                               ctypes.c_void_p(Ch.data_ptr()), M, N, K, ctypes.c_void_p(base),
                               ws.numel() - (base - ws.data_ptr()), mmq._stream_ptr(stream))
    assert rc == mmq.MMQ_OK, mmq.strerror(rc)
    stream.synchronize()
    return Ch


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    mmq = require_gpu()
    # two calls in a row on different shapes: 300 rows (two row chunks) and
    # 700 rows (three chunks, a larger footprint over the same array)
    for M, K, N, seed in ((300, 1024, 516, 11), (700, 2048, 1028, 12)):
        assert mmq.mmq_q4K_gemm_host_workspace(M, N, K) <= mmq.MMQ_HOST_NOALLOC_SCRATCH_BYTES
        x = synthetic.activations(M, K, 900 + seed, 0.01)
        blk = synthetic.q4K_weights(N, K, 950 + seed)
        w = to_dev(blk.reshape(-1))
        xh = torch.from_numpy(x).pin_memory()
        Ch = torch.full((M, N), float("nan"), dtype=torch.float32, pin_memory=True)
        _noalloc(mmq, xh, w, Ch, M, N, K)
        assert mmq.status() == 0
        C_ws = _with_workspace(mmq, xh, w, M, N, K)
        q, da, sa = oracle.quantize_q8_1(x)
        _, _, T = oracle.gemm(q, da, sa, blk, N)
        C_new, C_old = Ch.numpy().astype(np.float64), C_ws.numpy().astype(np.float64)
        assert np.isfinite(C_new).all()
        assert (np.abs(C_new - C_old) <= RTOL * T + ATOL).all()


def test_noalloc_refuses_a_shape_larger_than_its_array():
    mmq = require_gpu()
    M, N, K = 4096, 16384, 16384
    assert mmq.mmq_q4K_gemm_host_workspace(M, N, K) > mmq.MMQ_HOST_NOALLOC_SCRATCH_BYTES
    # refused during argument checks, before any pointer is used
    dummy = ctypes.c_void_p(0x10000)
    assert mmq.mmq_q4K_gemm_host_noalloc(dummy, dummy, dummy, M, N, K, None) == mmq.MMQ_ERR_ARG
