"""q6_K x q8_1 on the GPU vs the CPU oracle (oracle.q6k).

Per-16 block dots S must match bit for bit; C must satisfy
|C - C_ref| <= 1e-4 * sum_k |a_k w_k| + 1e-6 element by element (the q4_K
bound; the q6_K arithmetic is the same rescale without the second term).
The device layout must be the customary bytes padded to 224 per
super-block.
"""
import numpy as np
import pytest

import oracle
from oracle import q6k
from q4_q8_int8_gb300 import synthetic
from tests import q6k_layout
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _dev(blk, N, K):
    mmq = require_gpu()
    w_dev = mmq.repack_q6K(to_dev(blk.reshape(-1)), N, K)
    return mmq, w_dev


def test_repack_layout():
    N, K = 33, 768
    blk = synthetic.q6K_weights(N, K, 601)
    mmq, w_dev = _dev(blk, N, K)
    ref = np.zeros((N, K // 256, 224), np.uint8)
    ref[:, :, :210] = blk
    assert (w_dev.cpu().numpy() == ref.reshape(-1)).all()


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (1, 4, 256), (130, 260, 2816)])
def test_q6k_block_dots_bit_exact(M, N, K):
    x = synthetic.activations(M, K, 610 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 620 + N)
    mmq, w_dev = _dev(blk, N, K)
    aq = mmq.quantize_q8_1(to_dev(x))
    S = mmq.q6K_block_dots(aq, w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    q, _, _ = oracle.quantize_q8_1(x)
    assert (S == q6k.block_dots16(q, blk, N)).all()


@pytest.mark.parametrize("sign", [1, -1])
def test_q6k_block_dots_extremes(sign):
    # a = +-127 everywhere and q = -32 everywhere: |S| = 16 * 127 * 32 = 65024
    M, N, K = 128, 128, 512
    x = np.full((M, K), 2.0 * sign, np.float32)
    blk = q6k_layout.encode(np.full((N, K), -32), np.ones((N, K // 16)), np.ones((N, 2)))
    mmq, w_dev = _dev(blk, N, K)
    S = mmq.q6K_block_dots(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    assert (S == -sign * 65024).all()


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (64, 128, 2816), (2, 132, 768), (3, 260, 4096), (4, 68, 11008),
                                   (1, 36, 1280), (7, 132, 1024), (16, 260, 2816), (12, 4, 256)])
def test_q6k_gemm_full(M, N, K):
    x = synthetic.activations(M, K, 630 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 640 + N)
    mmq, w_dev = _dev(blk, N, K)
    C = mmq.q6K_gemm(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, _ = oracle.quantize_q8_1(x)
    _, C64, T = q6k.gemm(q, da, blk, N)
    ok = np.abs(C.astype(np.float64) - C64) <= RTOL * T + ATOL
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance"


@pytest.mark.parametrize("name", ["q_proj", "down"])
def test_q6k_gemm_full_size_sampled(name):
    M, K, N = synthetic.SHAPES[name]
    x = synthetic.activations(M, K, 650, 0.01)
    blk = synthetic.q6K_weights(N, K, 660)
    mmq, w_dev = _dev(blk, N, K)
    C = mmq.q6K_gemm(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    assert np.isfinite(C).all()
    q, da, _ = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 2000, 11)
    _, C64, T = q6k.gemm(q, da, blk, N, rows=rows, cols=cols)
    assert (np.abs(C[rows, cols].astype(np.float64) - C64) <= RTOL * T + ATOL).all()


@pytest.mark.parametrize("M,N,K", [(1, 11008, 4096), (4, 4096, 11008), (16, 4096, 4096)])
def test_q6k_gemm_decode_size_sampled(M, N, K):
    # decode shapes: the dot-product kernel (M <= 4)
    x = synthetic.activations(M, K, 655 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 665 + M)
    mmq, w_dev = _dev(blk, N, K)
    C = mmq.q6K_gemm(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, _ = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 12)
    _, C64, T = q6k.gemm(q, da, blk, N, rows=rows, cols=cols)
    assert (np.abs(C[rows, cols].astype(np.float64) - C64) <= RTOL * T + ATOL).all()


def test_q6k_worked_examples_exact():
    # x = 1: da = fl(1/127), a = 127; q = 31 (sc 1, d 1), q = 0, q = -32 (sc -128, d 0.5)
    M, N, K = 4, 8, 512
    x = np.ones((M, K), np.float32)
    q = np.array([[31] * K, [0] * K, [-32] * K] + [[31] * K] * 5)
    sc = np.array([[1] * 32, [5] * 32, [-128] * 32] + [[1] * 32] * 5)
    d = np.array([[1.0] * 2, [3.0] * 2, [0.5] * 2] + [[1.0] * 2] * 5)
    blk = q6k_layout.encode(q, sc, d)
    mmq, w_dev = _dev(blk, N, K)
    C = mmq.q6K_gemm(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    da = np.float32(1.0) / np.float32(127.0)
    # 32 sub-block terms da * d * sc * S summed in f32: within a few ulp of the exact total
    assert np.allclose(C[:, 0], 512 * 127 * 31 * np.float64(da), rtol=1e-6)
    assert (C[:, 1] == 0).all()                   # q = 0: every S is 0, no second term
    assert np.allclose(C[:, 2], 512 * 127 * 4096 * 0.5 * np.float64(da), rtol=1e-6)


def test_q6k_every_output_written_and_deterministic():
    import torch
    M, N, K = 200, 516, 1024
    x = synthetic.activations(M, K, 91, 0.01)
    blk = synthetic.q6K_weights(N, K, 92)
    mmq, w_dev = _dev(blk, N, K)
    aq = mmq.quantize_q8_1(to_dev(x))
    buf = torch.full((M * N + 2048,), float("nan"), device="cuda")
    buf[:1024] = 7.0
    buf[-1024:] = 7.0
    C1 = buf[1024:1024 + M * N].view(M, N)
    mmq.q6K_gemm(aq, w_dev, N, out=C1)
    C2 = mmq.q6K_gemm(aq, w_dev, N)
    torch.cuda.synchronize()
    assert torch.isfinite(C1).all()
    assert (buf[:1024] == 7.0).all() and (buf[-1024:] == 7.0).all()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


@pytest.mark.parametrize("ks", [1, 2, 4])
@pytest.mark.parametrize("M,N,K", [(1, 260, 11008), (2, 132, 4096), (4, 68, 2816), (8, 260, 1280), (16, 132, 4096)])
def test_q6k_dot_product_every_split(ks, M, N, K):
    # each K split of the q6_K dot-product kernel (up to 16 tokens), forced,
    # within tolerance of the oracle
    x = synthetic.activations(M, K, 671 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 681 + N)
    mmq, w_dev = _dev(blk, N, K)
    aq = mmq.quantize_q8_1(to_dev(x))
    mmq.force_gemv_split(ks)
    try:
        C = mmq.q6K_gemm(aq, w_dev, N).cpu().numpy()
        assert mmq.status() == 0
    finally:
        mmq.force_gemv_split(0)
    q, da, _ = oracle.quantize_q8_1(x)
    _, C64, T = q6k.gemm(q, da, blk, N)
    ok = np.abs(C.astype(np.float64) - C64) <= RTOL * T + ATOL
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance"


@pytest.mark.parametrize("M,N,K", [(16, 11008, 4096), (8, 4096, 4096), (1, 4096, 4096)])
def test_q6k_dot_product_chosen_split_sampled(M, N, K):
    # the automatic split on decode shapes where the choice differs from the
    # widest split (16 tokens on 4096 -> 11008 takes 2), sampled
    x = synthetic.activations(M, K, 691 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 695 + N)
    mmq, w_dev = _dev(blk, N, K)
    C = mmq.q6K_gemm(mmq.quantize_q8_1(to_dev(x)), w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, _ = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 13)
    _, C64, T = q6k.gemm(q, da, blk, N, rows=rows, cols=cols)
    assert (np.abs(C[rows, cols].astype(np.float64) - C64) <= RTOL * T + ATOL).all()
