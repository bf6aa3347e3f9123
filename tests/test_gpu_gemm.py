"""GEMM kernels on the GPU vs the CPU oracle.

S (exact per-chunk int32 dots) must match bit for bit; C must satisfy
|C - C_ref| <= 1e-4 * sum_k |a_k w_k| + 1e-6 element by element (web page
"20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2 rescale",
section 2.1 for the math, 2.3 for the |S| bound).
"""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests import q4k_layout
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _paths():
    import q4_q8_int8_gb300 as mmq
    return [mmq.MMQ_PATH_MMA_S8, mmq.MMQ_PATH_TC, mmq.MMQ_PATH_TC_PAIR]


def _paths_for(M):
    import q4_q8_int8_gb300 as mmq
    p = _paths()
    if M <= mmq.SMALL_M_MAX:
        p = p + [mmq.MMQ_PATH_SMALL_M]
    return p


def _dev_inputs(x, blk):
    mmq = require_gpu()
    aq = mmq.quantize_q8_1(to_dev(x))
    return mmq, aq, to_dev(blk.reshape(-1))


def _full_check(x, blk, N, path):
    mmq, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N, path=path).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    ok = oracle.within_tolerance(C, C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance; worst at {np.unravel_index(np.argmax(np.abs(C - C_ref) - RTOL * T), C.shape)}"
    return C


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (1, 4, 256), (130, 260, 2816),
                                   (256, 128, 256)])
def test_block_dots_bit_exact(path_name, M, N, K):
    mmq = require_gpu()
    path = getattr(mmq, path_name)
    x = synthetic.activations(M, K, 31 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 41 + N)
    _, aq, w = _dev_inputs(x, blk)
    S = mmq.q4K_block_dots(aq, w, N, path=path).cpu().numpy()
    assert mmq.status() == 0
    q, _, _ = oracle.quantize_q8_1(x)
    assert (S == oracle.block_dots(q, blk, N)).all()


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR"])
@pytest.mark.parametrize("sign", [1, -1])
def test_block_dots_extremes(path_name, sign):
    # all quants at +-127 and all nibbles at 15: |S| reaches 32*127*15 = 60960
    mmq = require_gpu()
    M, N, K = 128, 128, 512
    x = np.full((M, K), 2.0 * sign, np.float32)
    blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.ones((N, 16)),
                            np.zeros((N, 16)), np.full((N, K), 15))
    _, aq, w = _dev_inputs(x, blk)
    S = mmq.q4K_block_dots(aq, w, N, path=getattr(mmq, path_name)).cpu().numpy()
    assert (S == sign * 60960).all()


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR",
                                       "MMQ_PATH_TC_SMALL"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (64, 128, 2816)])
def test_gemm_full_small(path_name, M, N, K):
    mmq = require_gpu()
    x = synthetic.activations(M, K, 51 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 61 + N)
    _full_check(x, blk, N, getattr(mmq, path_name))


@pytest.mark.parametrize("path_name", ["MMQ_PATH_SMALL_M", "MMQ_PATH_TC_SMALL"])
def test_gemm_small_m_full(path_name):
    mmq = require_gpu()
    for M in (1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64):
        x = synthetic.activations(M, 1024, 71 + M, 0.01)
        blk = synthetic.q4K_weights(260, 1024, 81)
        _full_check(x, blk, 260, getattr(mmq, path_name))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (64, 4096, 4096),
                                   (40, 4096, 11008), (16, 11008, 4096), (9, 388, 256)])
def test_tc_small_full_size_sampled(M, N, K):
    # the few-token tcgen05 kernel at full decode / sweep sizes (cluster split-K up to 4)
    mmq = require_gpu()
    x = synthetic.activations(M, K, 111 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 121 + K % 7)
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N, path=mmq.MMQ_PATH_TC_SMALL).cpu().numpy()
    assert mmq.status() == 0
    assert np.isfinite(C).all()
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 7)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    ok = oracle.within_tolerance(C[rows, cols], C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} sampled outputs outside tolerance"


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR",
                                       "MMQ_PATH_TC_SMALL"])
@pytest.mark.parametrize("name", ["q_proj", "down", "gate_up"])
def test_gemm_full_size_sampled(path_name, name):
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs(name)
    M = x.shape[0]
    mmq_, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N, path=getattr(mmq, path_name)).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 5)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    ok = oracle.within_tolerance(C[rows, cols], C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} sampled outputs outside tolerance"
    assert np.isfinite(C).all()


@pytest.mark.parametrize("M", synthetic.SWEEP_M)
def test_gemm_sweep_auto_sampled(M):
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs("sweep", M)
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 2000, 6)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    assert oracle.within_tolerance(C[rows, cols], C_ref, T, RTOL, ATOL).all()


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR",
                                       "MMQ_PATH_SMALL_M", "MMQ_PATH_TC_SMALL"])
def test_every_output_written_and_deterministic(path_name):
    import torch
    mmq = require_gpu()
    M, N, K = (37 if path_name in ("MMQ_PATH_SMALL_M", "MMQ_PATH_TC_SMALL") else 200), 516, 1024
    x = synthetic.activations(M, K, 91, 0.01)
    blk = synthetic.q4K_weights(N, K, 92)
    _, aq, w = _dev_inputs(x, blk)
    path = getattr(mmq, path_name)
    # guard bands around C must stay untouched; C itself starts as NaN
    buf = torch.full((M * N + 2 * 1024,), float("nan"), device="cuda")
    buf[:1024] = 7.0
    buf[-1024:] = 7.0
    C1 = buf[1024:1024 + M * N].view(M, N)
    mmq.q4K_gemm(aq, w, N, path=path, out=C1)
    C2 = mmq.q4K_gemm(aq, w, N, path=path)
    torch.cuda.synchronize()
    assert torch.isfinite(C1).all()
    assert (buf[:1024] == 7.0).all() and (buf[-1024:] == 7.0).all()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_TC_PAIR",
                                       "MMQ_PATH_SMALL_M", "MMQ_PATH_TC_SMALL"])
def test_worked_examples_exact(path_name):
    mmq = require_gpu()
    path = getattr(mmq, path_name)
    M, N, K = 4, 8, 512
    # E2: w == 0 through exact per-chunk cancellation of the two terms
    x = np.ones((M, K), np.float32)
    blk = q4k_layout.encode(np.ones((N, 2)), np.ones((N, 2)), np.ones((N, 16)), np.ones((N, 16)),
                            np.ones((N, K)))
    mmq_, aq, w = _dev_inputs(x, blk)
    assert (mmq.q4K_gemm(aq, w, N, path=path).cpu().numpy() == 0).all()
    # E4: v = 0 and m = 0 give C = 0 for any activations and scales
    rng = np.random.default_rng(3)
    x = rng.standard_normal((M, K)).astype(np.float32)
    blk = q4k_layout.encode(rng.uniform(1e-3, 1, (N, 2)), rng.uniform(1e-3, 1, (N, 2)),
                            rng.integers(0, 64, (N, 16)), np.zeros((N, 16)), np.zeros((N, K)))
    _, aq, w = _dev_inputs(x, blk)
    assert (mmq.q4K_gemm(aq, w, N, path=path).cpu().numpy() == 0).all()
    # E5: d = sc = 1, m = dmin = 0, integer activations with amax 127 per block
    x = rng.integers(-127, 128, (M, K)).astype(np.float32)
    x.reshape(M, K // 32, 32)[:, :, 0] = 127.0
    v = rng.integers(0, 16, (N, K))
    blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.ones((N, 16)), np.zeros((N, 16)), v)
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N, path=path).cpu().numpy()
    assert (C.astype(np.int64) == x.astype(np.int64) @ v.T).all()
