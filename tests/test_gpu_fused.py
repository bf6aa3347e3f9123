"""GEMM with the q8_1 output fused (mmq_q4K_gemm_q8_1): the q8_1 triple it
writes must equal, bit for bit, the q8_1 quantization of its own f32 result
(the oracle's quantize on the GPU's C), and C itself must be within the GEMM
tolerance of the oracle."""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _check_q8_of(C, o):
    q, da, sa = oracle.quantize_q8_1(np.ascontiguousarray(C))
    assert (o[0].cpu().numpy() == q).all()
    assert (o[1].cpu().numpy().view(np.uint32) == da.view(np.uint32)).all()
    assert (o[2].cpu().numpy() == sa).all()


@pytest.mark.parametrize("M,N,K", [(200, 256, 512), (130, 4096, 1024), (256, 160, 2816), (37, 96, 512),
                                   (1, 32, 256), (2, 288, 768), (3, 4096, 4096), (4, 11008, 4096),
                                   (4, 4096, 11008), (5, 96, 256), (16, 4096, 4096), (31, 160, 2816),
                                   (64, 11008, 4096), (9, 4096, 11008)])
def test_fused_q8_1_output(M, N, K):
    mmq = require_gpu()
    x = synthetic.activations(M, K, 300 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 400 + N)
    aq = mmq.quantize_q8_1(to_dev(x))
    C, o = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N)
    assert mmq.status() == 0
    Ch = C.cpu().numpy()
    _check_q8_of(Ch, o)
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    assert oracle.within_tolerance(Ch, C_ref, T, RTOL, ATOL).all()
    # without the f32 result: the same q8_1 bits
    _, o2 = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N, with_c=False)
    assert mmq.status() == 0
    for a, b in zip(o, o2):
        assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())


@pytest.mark.parametrize("ks", [1, 2, 4])
@pytest.mark.parametrize("M,N,K", [(1, 256, 11008), (4, 4096, 4096), (2, 288, 2816)])
def test_fused_q8_1_output_every_split(ks, M, N, K):
    # the dot-product kernel's q8_1 epilogue with each K split forced: the
    # q8_1 bits of its own C, and C within tolerance
    mmq = require_gpu()
    x = synthetic.activations(M, K, 500 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 510 + N)
    aq = mmq.quantize_q8_1(to_dev(x))
    mmq.force_gemv_split(ks)
    try:
        C, o = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N)
        assert mmq.status() == 0
    finally:
        mmq.force_gemv_split(0)
    Ch = C.cpu().numpy()
    _check_q8_of(Ch, o)
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    assert oracle.within_tolerance(Ch, C_ref, T, RTOL, ATOL).all()


def test_fused_q8_1_output_full_size():
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs("q_proj")
    M = x.shape[0]
    aq = mmq.quantize_q8_1(to_dev(x))
    C, o = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N)
    assert mmq.status() == 0
    Ch = C.cpu().numpy()
    _check_q8_of(Ch, o)
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 2000, 23)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    assert oracle.within_tolerance(Ch[rows, cols], C_ref, T, RTOL, ATOL).all()


@pytest.mark.parametrize("M", [1, 2, 4])
def test_q8_1_output_special_blocks(M):
    # an all-zero 32-column output block (zero weights: the zero-scale
    # branch), and blocks of a few repeated values (one amax shared by many
    # outputs, each quantized to +-127 or a small multiple)
    import torch
    from tests import q4k_layout
    mmq = require_gpu()
    N, K = 96, 256
    x = np.zeros((M, K), np.float32)
    x[:, :32] = 1.0                                  # a = 127 on chunk 0, zero elsewhere
    v = np.zeros((N, K), np.int64)
    v[32:64, :32] = (np.arange(32)[:, None] % 16)    # row 32 + i: 32 * (i % 16) = sum of its nibbles
    v[64:96, :32] = (np.arange(32)[:, None] * 7 % 16)
    blk = q4k_layout.encode(np.ones((N, 1)), np.zeros((N, 1)), np.ones((N, K // 32)),
                            np.zeros((N, K // 32)), v)
    aq = mmq.quantize_q8_1(to_dev(x))
    C, o = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N)
    torch.cuda.synchronize()
    assert mmq.status() == 0
    Ch = C.cpu().numpy()
    assert (Ch[:, :32] == 0).all() and (o[1].cpu().numpy()[:, 0] == 0).all()
    _check_q8_of(Ch, o)


def test_q8_1_output_chain_programmatic_launch_and_graph():
    # GEMM -> q8_1 -> GEMM at one token: the same bits with the launch mode on
    # and off, directly and from a CUDA graph, and equal to prepass + GEMM
    import torch
    mmq = require_gpu()
    M, K, N1, N2 = 1, 1024, 512, 256
    x = synthetic.activations(M, K, 940, 0.01)
    w1 = to_dev(synthetic.q4K_weights(N1, K, 941).reshape(-1))
    w2 = to_dev(synthetic.q4K_weights(N2, N1, 942).reshape(-1))
    aq = mmq.quantize_q8_1(to_dev(x))

    def chain():
        _, o1 = mmq.q4K_gemm_q8_1(aq, w1, N1, with_c=False)
        C2, o2 = mmq.q4K_gemm_q8_1(o1, w2, N2)
        return C2, o2

    try:
        mmq.mmq_set_programmatic_launch(False)
        ref = chain()
        C1 = mmq.q4K_gemm(aq, w1, N1)
        ref2 = mmq.q4K_gemm(mmq.quantize_q8_1(C1), w2, N2)
        torch.cuda.synchronize()
        assert torch.equal(ref[0].view(torch.int32), ref2.view(torch.int32))
        mmq.mmq_set_programmatic_launch(True)
        got = chain()
        torch.cuda.synchronize()
        assert torch.equal(got[0].view(torch.int32), ref[0].view(torch.int32))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            chain()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                gout = chain()
            for _ in range(3):
                g.replay()
            s.synchronize()
        assert torch.equal(gout[0].view(torch.int32), ref[0].view(torch.int32))
        for a, b in zip(gout[1], ref[1]):
            assert torch.equal(a, b)
        assert mmq.status() == 0
    finally:
        mmq.mmq_set_programmatic_launch(False)
