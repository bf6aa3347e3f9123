"""The q6_K tcgen05 kernel (mmq_q6K_gemm_path with MMQ_PATH_TC) and the
explicit q6_K kernel families vs the CPU oracle (oracle.q6k).

The tcgen05 kernel forms per 32-k chunk S' = sum a * sc * q exactly in f32
tensor memory (sc * q split into an fp16 hi part and an exact lo part) and
then C += da * d * S'.  C must satisfy |C - C_ref| <= 1e-4 * sum |a w| + 1e-6
element by element; where every operand and partial sum is an exact
integer (or an exact power-of-two multiple of one) C must be exact, which
pins the split of sc * q at its extremes (|sc * q| = 4096, and 3937, whose
fp16 rounding leaves lo = +-1).
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


def _setup(blk, N, K, x):
    mmq = require_gpu()
    w_dev = mmq.repack_q6K(to_dev(blk.reshape(-1)), N, K)
    aq = mmq.quantize_q8_1(to_dev(x))
    return mmq, w_dev, aq


def _paths(mmq, M):
    out = [mmq.MMQ_PATH_TC, mmq.MMQ_PATH_MMA_S8, mmq.MMQ_PATH_AUTO]
    if M <= 16:
        out.append(mmq.MMQ_PATH_SMALL_M)
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (17, 260, 2816), (130, 516, 256), (64, 128, 11008), (513, 132, 1024),
                                   (16, 68, 4096)])
def test_q6k_paths_within_tolerance(M, N, K):
    x = synthetic.activations(M, K, 700 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 710 + N)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    q, da, _ = oracle.quantize_q8_1(x)
    _, C64, T = q6k.gemm(q, da, blk, N)
    for path in _paths(mmq, M):
        C = mmq.q6K_gemm(aq, w_dev, N, path=path).cpu().numpy()
        assert mmq.status() == 0
        ok = np.abs(C.astype(np.float64) - C64) <= RTOL * T + ATOL
        assert ok.all(), f"path {path}: {(~ok).sum()} of {ok.size} outside tolerance"


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (130, 260, 2816)])
def test_q6k_tc_scaled_block_dots_bit_exact(M, N, K):
    # the kernel's own per-chunk S' = sc_2c * S16_2c + sc_2c+1 * S16_2c+1,
    # against the oracle's exact per-16 dots and the unpacked scales
    x = synthetic.activations(M, K, 790 + M, 0.01)
    blk = synthetic.q6K_weights(N, K, 795 + N)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    S = mmq.q6K_scaled_block_dots(aq, w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    q, _, _ = oracle.quantize_q8_1(x)
    S16 = q6k.block_dots16(q, blk, N).astype(np.int64)                      # [M][N][K/16]
    sc = q6k.unpack_q6K(blk, N, K)["sc"].astype(np.int64)                    # [N][K/16]
    ref = (S16 * sc[None]).reshape(M, N, K // 32, 2).sum(axis=3)
    assert (S.astype(np.int64) == ref).all()


def test_q6k_tc_scaled_block_dots_extremes():
    # |S'| = 32 * 127 * 4096 = 16,646,144 < 2^24 at sc = -128, q = -32, a = +-127
    M, N, K = 128, 128, 512
    x = np.full((M, K), 3.0, np.float32)
    x[::2] *= -1.0
    blk = q6k_layout.encode(np.full((N, K), -32), np.full((N, K // 16), -128), np.ones((N, K // 256)))
    mmq, w_dev, aq = _setup(blk, N, K, x)
    S = mmq.q6K_scaled_block_dots(aq, w_dev, N).cpu().numpy()
    assert mmq.status() == 0
    sign = np.where(np.arange(M) % 2 == 0, -1, 1)[:, None, None]
    assert (S == sign * 16646144).all()


@pytest.mark.parametrize("sc,q", [(-128, -32), (127, 31), (-127, 31), (-1, -32)])
def test_q6k_tc_exact_at_the_product_extremes(sc, q):
    # x = 127 everywhere: da = 1 and a = 127; every weight sc * q with d = 1, so
    # C = K * 127 * sc * q exactly (every partial sum below 2^24 or an exact
    # multiple of a power of two)
    M, N, K = 130, 132, 256
    x = np.full((M, K), 127.0, np.float32)
    blk = q6k_layout.encode(np.full((N, K), q), np.full((N, K // 16), sc), np.ones((N, K // 256)))
    mmq, w_dev, aq = _setup(blk, N, K, x)
    C = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0
    assert (C.astype(np.float64) == float(K * 127 * sc * q)).all()


@pytest.mark.parametrize("M,N,K", [(128, 132, 1024), (300, 260, 256)])
def test_q6k_tc_exact_with_mixed_scales(M, N, K):
    # integer activations with one +-127 per block (da = 1, a = x), small scales
    # and d = 2^-4: C = 2^-4 * sum_k a * sc * q exactly
    rng = np.random.default_rng(720 + M)
    x = rng.integers(-8, 9, (M, K)).astype(np.float32)
    x.reshape(M, K // 32, 32)[:, :, 3] = 127.0 * rng.choice([-1.0, 1.0], (M, K // 32))
    q = rng.integers(-32, 32, (N, K))
    sc = rng.integers(-8, 9, (N, K // 16))
    blk = q6k_layout.encode(q, sc, np.full((N, K // 256), 2.0 ** -4))
    mmq, w_dev, aq = _setup(blk, N, K, x)
    C = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0
    w = q * np.repeat(sc, 16, axis=1)
    exact = x.astype(np.int64) @ w.T.astype(np.int64)
    assert np.abs(exact).max() < 2 ** 24
    assert (C.astype(np.float64) == exact * 2.0 ** -4).all()


@pytest.mark.parametrize("name", ["q_proj", "down"])
def test_q6k_tc_full_size_sampled(name):
    M, K, N = synthetic.SHAPES[name]
    x = synthetic.activations(M, K, 730, 0.01)
    blk = synthetic.q6K_weights(N, K, 740)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    C = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0
    assert np.isfinite(C).all()
    q, da, _ = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 2000, 13)
    _, C64, T = q6k.gemm(q, da, blk, N, rows=rows, cols=cols)
    ok = np.abs(C[rows, cols].astype(np.float64) - C64) <= RTOL * T + ATOL
    assert ok.all(), f"{(~ok).sum()} sampled outputs outside tolerance"


@pytest.mark.parametrize("name", ["q_proj", "gate_up", "down"])
def test_q6k_tc_every_element(name):
    # every output of the 2048-token workloads against the oracle's
    # brute-force dequantized dot (float64 BLAS over the same a = da * q and
    # w = d * sc * q; pinned to the blockwise form in the oracle tests), with
    # T = |a| . |w|^T
    M, K, N = synthetic.SHAPES[name]
    x = synthetic.activations(M, K, 731 + K + N, 0.01)
    blk = synthetic.q6K_weights(N, K, 741 + N)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    C = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0
    q, da, _ = oracle.quantize_q8_1(x)
    D = q6k.dequant_dot(q, da, blk, N)
    a = np.repeat(da.astype(np.float64), 32, axis=1) * q.astype(np.float64)
    T = np.abs(a) @ np.abs(q6k.dequant_q6K(blk, N, K)).T
    ok = np.abs(C.astype(np.float64) - D) <= RTOL * T + ATOL
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outputs outside tolerance"


def test_q6k_tc_every_output_written_and_deterministic():
    import torch
    M, N, K = 300, 516, 1024
    x = synthetic.activations(M, K, 750, 0.01)
    blk = synthetic.q6K_weights(N, K, 760)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    buf = torch.full((M * N + 2048,), float("nan"), device="cuda")
    buf[:1024] = 7.0
    buf[-1024:] = 7.0
    C1 = buf[1024:1024 + M * N].view(M, N)
    mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC, out=C1)
    C2 = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC)
    torch.cuda.synchronize()
    assert torch.isfinite(C1).all()
    assert (buf[:1024] == 7.0).all() and (buf[-1024:] == 7.0).all()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


def test_q6k_launch_counts_and_argument_errors():
    import ctypes
    import torch
    mmq = require_gpu()
    assert mmq.mmq_q6K_gemm_launches(2048, 4096, 4096, mmq.MMQ_PATH_TC) == 2   # 512 tiles: rounds + tail
    assert mmq.mmq_q6K_gemm_launches(77, 4096, 4096, mmq.MMQ_PATH_TC) == 1
    assert mmq.mmq_q6K_gemm_launches(8, 4096, 4096, mmq.MMQ_PATH_AUTO) == 1
    assert mmq.mmq_q6K_gemm_launches(17, 4096, 4096, mmq.MMQ_PATH_SMALL_M) == mmq.MMQ_ERR_ARG
    M, N, K = 32, 128, 512
    aq = mmq.quantize_q8_1(torch.zeros((M, K), device="cuda"))
    w = torch.zeros((mmq.mmq_q6K_dev_bytes(N, K),), dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    sp = mmq._stream_ptr()
    q = mmq.q8_1_struct(*aq)
    assert mmq.mmq_q6K_gemm_path(q, P(w), P(C), M, N, K, mmq.MMQ_PATH_SMALL_M, sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q6K_gemm_path(q, P(w), P(C), M, N, K, 17, sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q6K_gemm_path(q, P(w), P(C), M, 6, K, mmq.MMQ_PATH_TC, sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q6K_gemm_path(q, P(w), P(C), M, N, K, mmq.MMQ_PATH_TC, sp) == 0
    assert mmq.status() == 0


@pytest.mark.parametrize("M", [128, 2048])
def test_q6k_tc_injected_timeout_is_reported_and_context_survives(M):
    mmq = require_gpu()
    N, K = 256, 512
    x = synthetic.activations(M, K, 770)
    blk = synthetic.q6K_weights(N, K, 780)
    mmq, w_dev, aq = _setup(blk, N, K, x)
    assert mmq.status() == 0
    mmq.mmq_debug_inject_timeout(True)
    mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC)
    assert mmq.status() == mmq.MMQ_ERR_DEVICE_TIMEOUT
    assert mmq.status() == 0
    C = mmq.q6K_gemm(aq, w_dev, N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0
    q, da, _ = oracle.quantize_q8_1(x)
    _, C64, T = q6k.gemm(q, da, blk, N)
    assert (np.abs(C.astype(np.float64) - C64) <= RTOL * T + ATOL).all()
