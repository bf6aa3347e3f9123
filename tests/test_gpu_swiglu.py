"""Fused SwiGLU epilogue (gate and up in one GEMM, q8_1 output) vs the oracle.

h must stay within the GEMM tolerance propagated through silu(g) * u
(oracle.ffn.swiglu_bound, with |C - C_ref| <= 1e-4 * sum_k |a_k w_k| + 1e-6
for g and u); the q8_1 output must equal, bit for bit, the prepass applied
to the kernel's own h (the quantization decision is taken in f32 on both
sides).  The interleaving of gate and up rows must be an exact byte copy.
"""
import numpy as np
import pytest

import oracle
from oracle import ffn
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _interleave_host(gate, up, F, K):
    g = gate.reshape(F, -1)
    u = up.reshape(F, -1)
    out = np.empty((2 * F, g.shape[1]), np.uint8)
    out[0::2] = g
    out[1::2] = u
    return out


def _run(M, F, K, seed, with_h=True):
    mmq = require_gpu()
    x = synthetic.activations(M, K, seed, 0.01)
    gate = synthetic.q4K_weights(F, K, seed + 1)
    up = synthetic.q4K_weights(F, K, seed + 2)
    w_gu = mmq.interleave_rows_q4K(to_dev(gate.reshape(-1)), to_dev(up.reshape(-1)), F, K)
    blk_gu = _interleave_host(gate, up, F, K)
    assert (w_gu.cpu().numpy() == blk_gu.reshape(-1)).all()
    aq = mmq.quantize_q8_1(to_dev(x))
    h, (qs, da, sa) = mmq.q4K_gemm_swiglu_q8_1(aq, w_gu, F, with_h=with_h)
    assert mmq.status() == 0
    return mmq, x, blk_gu, aq, w_gu, h, (qs.cpu().numpy(), da.cpu().numpy(), sa.cpu().numpy())


@pytest.mark.parametrize("M,F,K", [(200, 256, 512), (130, 512, 1024), (37, 96, 512), (1, 32, 256),
                                   (300, 160, 2816), (2, 96, 768), (3, 160, 4096), (4, 256, 2816),
                                   (1, 4096, 4096), (5, 96, 512), (16, 256, 4096), (33, 160, 2816),
                                   (64, 512, 1024)])
def test_swiglu_full(M, F, K):
    mmq, x, blk_gu, aq, w_gu, h, (qs, da, sa) = _run(M, F, K, 400 + M)
    h = h.cpu().numpy()
    q, dq, sq = oracle.quantize_q8_1(x)
    _, C64, T = oracle.gemm(q, dq, sq, blk_gu, 2 * F, want_c64=True)
    g, u = C64[:, 0::2], C64[:, 1::2]
    bound = ffn.swiglu_bound(g, u, RTOL * T[:, 0::2] + ATOL, RTOL * T[:, 1::2] + ATOL)
    err = np.abs(h.astype(np.float64) - ffn.swiglu(g, u))
    assert (err <= bound).all(), f"{(err > bound).sum()} outside; worst ratio {np.max(err / bound):.3f}"
    rq, rda, rsa = oracle.quantize_q8_1(h)
    assert (qs == rq).all() and (da.view(np.uint32) == rda.view(np.uint32)).all() and (sa == rsa).all()


@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("M,F,K", [(1, 128, 11008), (4, 2048, 4096), (3, 160, 2816)])
def test_swiglu_dot_product_every_split(ks, M, F, K):
    # the dot-product kernel's SwiGLU epilogue with each K split it takes
    # (1 and 2) forced: h within the propagated bound, q8_1 bits of its own h
    mmq = require_gpu()
    mmq.force_gemv_split(ks)
    try:
        mmq, x, blk_gu, aq, w_gu, h, (qs, da, sa) = _run(M, F, K, 600 + M)
    finally:
        mmq.force_gemv_split(0)
    h = h.cpu().numpy()
    q, dq, sq = oracle.quantize_q8_1(x)
    _, C64, T = oracle.gemm(q, dq, sq, blk_gu, 2 * F, want_c64=True)
    g, u = C64[:, 0::2], C64[:, 1::2]
    bound = ffn.swiglu_bound(g, u, RTOL * T[:, 0::2] + ATOL, RTOL * T[:, 1::2] + ATOL)
    assert (np.abs(h.astype(np.float64) - ffn.swiglu(g, u)) <= bound).all()
    rq, rda, rsa = oracle.quantize_q8_1(h)
    assert (qs == rq).all() and (da.view(np.uint32) == rda.view(np.uint32)).all() and (sa == rsa).all()


@pytest.mark.parametrize("M", [130, 1, 4, 16, 64])
def test_swiglu_without_h_same_bits(M):
    mmq, x, blk_gu, aq, w_gu, h, o1 = _run(M, 256, 1024, 77, with_h=True)
    _, o2 = mmq.q4K_gemm_swiglu_q8_1(aq, w_gu, 256, with_h=False)
    assert mmq.status() == 0
    for a, b in zip(o1, o2):
        assert (a == b.cpu().numpy()).all()


def test_swiglu_gate_up_full_size_sampled():
    # the 7B FFN: 2048 tokens, 4096 -> 2 x 11008 (cluster-free: 16 x 172 tiles)
    M, F, K = 2048, 11008, 4096
    mmq, x, blk_gu, aq, w_gu, h, (qs, da, sa) = _run(M, F, K, 500)
    h = h.cpu().numpy()
    assert np.isfinite(h).all()
    q, dq, sq = oracle.quantize_q8_1(x)
    rows, fcols = sample_points(M, F, 1500, 9)
    Cg, Cg64, Tg = oracle.gemm_sampled(q, dq, sq, blk_gu, 2 * F, rows, 2 * fcols)
    Cu, Cu64, Tu = oracle.gemm_sampled(q, dq, sq, blk_gu, 2 * F, rows, 2 * fcols + 1)
    bound = ffn.swiglu_bound(Cg64, Cu64, RTOL * Tg + ATOL, RTOL * Tu + ATOL)
    err = np.abs(h[rows, fcols].astype(np.float64) - ffn.swiglu(Cg64, Cu64))
    assert (err <= bound).all()
    rq, rda, rsa = oracle.quantize_q8_1(h)
    assert (qs == rq).all() and (da.view(np.uint32) == rda.view(np.uint32)).all() and (sa == rsa).all()


def test_swiglu_argument_errors():
    import ctypes
    mmq = require_gpu()
    good = mmq.q8_1_struct(*mmq.empty_q8_1(4, 256, "cuda"))
    out = mmq.q8_1_struct(*mmq.empty_q8_1(4, 64, "cuda"))
    import torch
    w = torch.zeros(2 * 64 * 144, dtype=torch.uint8, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    assert mmq.mmq_q4K_gemm_swiglu_q8_1(good, P(w), None, out, 4, 48, 256, None) == mmq.MMQ_ERR_ARG  # F % 32
    assert mmq.mmq_q4K_gemm_swiglu_q8_1(good, P(w), None, out, 4, 64, 250, None) == mmq.MMQ_ERR_ARG  # K % 256
    assert mmq.mmq_interleave_rows_q4K(P(w), None, P(w), 4, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.status() == 0


@pytest.mark.parametrize("M", [1, 4, 16])
def test_swiglu_gate_up_decode_full_size(M):
    # the 7B FFN at a few tokens (the dot-product kernel's cluster epilogue)
    M_, F, K = M, 11008, 4096
    mmq, x, blk_gu, aq, w_gu, h, (qs, da, sa) = _run(M_, F, K, 510 + M)
    h = h.cpu().numpy()
    q, dq, sq = oracle.quantize_q8_1(x)
    rows, fcols = sample_points(M_, F, 3000, 10)
    Cg, Cg64, Tg = oracle.gemm_sampled(q, dq, sq, blk_gu, 2 * F, rows, 2 * fcols)
    Cu, Cu64, Tu = oracle.gemm_sampled(q, dq, sq, blk_gu, 2 * F, rows, 2 * fcols + 1)
    bound = ffn.swiglu_bound(Cg64, Cu64, RTOL * Tg + ATOL, RTOL * Tu + ATOL)
    err = np.abs(h[rows, fcols].astype(np.float64) - ffn.swiglu(Cg64, Cu64))
    assert (err <= bound).all()
    rq, rda, rsa = oracle.quantize_q8_1(h)
    assert (qs == rq).all() and (da.view(np.uint32) == rda.view(np.uint32)).all() and (sa == rsa).all()
