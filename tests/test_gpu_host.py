"""The host-buffer pipeline (mmq_q4K_gemm_host): activations and result in
host memory, the rows in chunks whose copies overlap the kernels.

C must equal, bit for bit, mmq_quantize_q8_1 + mmq_q4K_gemm applied to each
chunk of rows on the device (the same kernels on the same rows), and be
within the GEMM tolerance |C - C_ref| <= 1e-4 * sum_k |a_k w_k| + 1e-6 of
the oracle; pinned and pageable host memory give the same bits."""
import ctypes

import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu


def _chunks(M):
    """The library's chunking: up to a quarter of the rows rounded up to 128, at least 256."""
    if M <= 256:
        return [(0, M)]
    mc = max(256, ((M + 3) // 4 + 127) // 128 * 128)
    return [(r, min(M, r + mc)) for r in range(0, M, mc)]


@pytest.mark.parametrize("M,N,K", [(1, 4, 256), (300, 260, 768), (1100, 516, 1024), (2048, 4096, 4096)])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_pipeline_bits(M, N, K, pinned):
    import torch
    mmq = require_gpu()
    x = synthetic.activations(M, K, 700 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 701 + N)
    w = to_dev(blk.reshape(-1))
    xh = torch.from_numpy(x)
    if pinned:
        xh = xh.pin_memory()
    Ch = torch.empty((M, N), dtype=torch.float32, pin_memory=pinned)
    mmq.q4K_gemm_host(xh, w, N, out=Ch)
    assert mmq.status() == 0
    xd = to_dev(x)
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for r0, r1 in _chunks(M):
        mmq.q4K_gemm(mmq.quantize_q8_1(xd[r0:r1].contiguous()), w, N, out=ref[r0:r1])
    torch.cuda.synchronize()
    assert torch.equal(Ch.view(torch.int32), ref.cpu().view(torch.int32))
    q, da, sa = oracle.quantize_q8_1(x)
    if M * N <= 600_000:
        C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
        assert oracle.within_tolerance(Ch.numpy(), C_ref, T).all()
    else:
        rows, cols = sample_points(M, N, 1500, 5)
        C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
        assert oracle.within_tolerance(Ch.numpy()[rows, cols], C_ref, T).all()


def test_host_pipeline_caller_workspace_and_stream_order():
    # two calls back to back on one stream with one workspace, then a device
    # kernel on that stream reading what the second call's inputs overwrote
    import torch
    mmq = require_gpu()
    M, N, K = 700, 260, 512
    blk = synthetic.q4K_weights(N, K, 711)
    w = to_dev(blk.reshape(-1))
    xs = [torch.from_numpy(synthetic.activations(M, K, 712 + i, 0.01)).pin_memory() for i in range(2)]
    outs = [torch.empty((M, N), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    need = mmq.mmq_q4K_gemm_host_workspace(M, N, K)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    for i in range(2):
        mmq.q4K_gemm_host(xs[i], w, N, out=outs[i], workspace=ws, stream=s)
    s.synchronize()
    for i in range(2):
        ref = mmq.q4K_gemm_host(xs[i], w, N)
        assert torch.equal(outs[i].view(torch.int32), ref.view(torch.int32))
    assert mmq.status() == 0


def test_host_pipeline_argument_errors():
    import torch
    mmq = require_gpu()
    M, N, K = 300, 8, 256
    need = mmq.mmq_q4K_gemm_host_workspace(M, N, K)
    assert need > 0
    assert mmq.mmq_q4K_gemm_host_workspace(M, 6, K) == 0          # N % 4
    assert mmq.mmq_q4K_gemm_host_workspace(M, N, 250) == 0        # K % 256
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    w = torch.zeros(N * 144, dtype=torch.uint8, device="cuda")
    xh = torch.zeros((M, K), dtype=torch.float32)
    Ch = torch.zeros((M, N), dtype=torch.float32)
    P = lambda v: ctypes.c_void_p(v)
    args = (P(xh.data_ptr()), P(w.data_ptr()), P(Ch.data_ptr()), M, N, K)
    assert mmq.mmq_q4K_gemm_host(*args, P(base), need - 1, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_host(*args, P(base + 16), need, None) == mmq.MMQ_ERR_ALIGN
    assert mmq.mmq_q4K_gemm_host(None, *args[1:], P(base), need, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_host(*args, P(base), need, None) == mmq.MMQ_OK
    torch.cuda.synchronize()
    assert (Ch == 0).all()   # zero weights and zero activations
    assert mmq.status() == 0


def test_host_pipeline_in_cuda_graph():
    # the three-stream pipeline captured into a CUDA graph (its copy streams
    # join the capture through the caller stream's start event) and replayed
    import torch
    mmq = require_gpu()
    M, N, K = 1100, 516, 1024
    blk = synthetic.q4K_weights(N, K, 721)
    w = to_dev(blk.reshape(-1))
    xh = torch.from_numpy(synthetic.activations(M, K, 722, 0.01)).pin_memory()
    ref = mmq.q4K_gemm_host(xh, w, N)
    need = mmq.mmq_q4K_gemm_host_workspace(M, N, K)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    out = torch.zeros((M, N), dtype=torch.float32, pin_memory=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mmq.q4K_gemm_host(xh, w, N, out=out, workspace=ws, stream=s)   # warm-up outside capture
        s.synchronize()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mmq.q4K_gemm_host(xh, w, N, out=out, workspace=ws, stream=s)
        for _ in range(2):
            out.zero_()
            g.replay()
            s.synchronize()
            assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    assert mmq.status() == 0
