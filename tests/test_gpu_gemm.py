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
    return [mmq.MMQ_PATH_MMA_S8, mmq.MMQ_PATH_TC]


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


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC"])
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


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_SMALL_M"])
@pytest.mark.parametrize("sign", [1, -1])
def test_block_dots_extremes(path_name, sign):
    # all quants at +-127 and all nibbles at 15: |S| reaches 32*127*15 = 60960
    mmq = require_gpu()
    Ms = (1, 4, 64) if path_name == "MMQ_PATH_SMALL_M" else (128,)
    N, K = 128, 512
    for M in Ms:
        x = np.full((M, K), 2.0 * sign, np.float32)
        blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.ones((N, 16)),
                                np.zeros((N, 16)), np.full((N, K), 15))
        _, aq, w = _dev_inputs(x, blk)
        S = mmq.q4K_block_dots(aq, w, N, path=getattr(mmq, path_name)).cpu().numpy()
        assert (S == sign * 60960).all()


# The kernels mmq_q4K_gemm runs for few tokens: the dot-product kernel (M <= 4)
# and the mma.sync kernel (4 < M <= 64), each dumping S from its own unpack and
# dot-product code (page r15 section 2.1 for S, 2.3 for its bound).
SMALL_M_DOTS = [1, 2, 3, 4, 5, 16, 33, 64]


@pytest.mark.parametrize("M", SMALL_M_DOTS)
@pytest.mark.parametrize("N,K", [(260, 256), (132, 11008), (4096, 1024)])
def test_block_dots_small_m_bit_exact(M, N, K):
    mmq = require_gpu()
    x = synthetic.activations(M, K, 131 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 141 + N + K)
    _, aq, w = _dev_inputs(x, blk)
    q, _, _ = oracle.quantize_q8_1(x)
    S_ref = oracle.block_dots(q, blk, N)
    for path in (mmq.MMQ_PATH_SMALL_M, mmq.MMQ_PATH_AUTO):   # AUTO picks the same kernel here
        S = mmq.q4K_block_dots(aq, w, N, path=path).cpu().numpy()
        assert mmq.status() == 0
        assert (S == S_ref).all(), f"{(S != S_ref).sum()} dots differ"


@pytest.mark.parametrize("ks", [1, 2, 4])
@pytest.mark.parametrize("M,N,K", [(1, 260, 11008), (4, 4096, 4096), (2, 256, 11008)])
def test_block_dots_dot_product_every_split(ks, M, N, K):
    # the dot-product kernel with each K split forced: same exact dots
    mmq = require_gpu()
    x = synthetic.activations(M, K, 151 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 161 + N)
    _, aq, w = _dev_inputs(x, blk)
    q, _, _ = oracle.quantize_q8_1(x)
    mmq.force_gemv_split(ks)
    try:
        S = mmq.q4K_block_dots(aq, w, N, path=mmq.MMQ_PATH_SMALL_M).cpu().numpy()
    finally:
        mmq.force_gemv_split(0)
    assert mmq.status() == 0
    assert (S == oracle.block_dots(q, blk, N)).all()


def _sub_block_scales(blk, N, K):
    return q4k_layout.decode(blk, N, K)["sc"]   # [N][K/32]


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (130, 260, 2816), (300, 388, 1280)])
def test_scaled_block_dots_product_operand(M, N, K):
    # the tcgen05 kernel's own weight operand carries sc * v: its MMA gives
    # S' = sc * S exactly (|S'| < 2^22), compared with sc x the oracle's S
    mmq = require_gpu()
    x = synthetic.activations(M, K, 171 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 181 + N)
    _, aq, w = _dev_inputs(x, blk)
    S = mmq.q4K_scaled_block_dots(aq, w, N).cpu().numpy()
    assert mmq.status() == 0
    q, _, _ = oracle.quantize_q8_1(x)
    ref = oracle.block_dots(q, blk, N).astype(np.int64) * _sub_block_scales(blk, N, K)[None, :, :]
    assert (S.astype(np.int64) == ref).all()


@pytest.mark.parametrize("sign", [1, -1])
def test_scaled_block_dots_extremes(sign):
    # sc = 63, v = 15, quants +-127: S' = 63 * 60960 = 3840480, the largest the operand can hold
    mmq = require_gpu()
    M, N, K = 128, 128, 512
    x = np.full((M, K), 2.0 * sign, np.float32)
    blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.full((N, 16), 63),
                            np.zeros((N, 16)), np.full((N, K), 15))
    _, aq, w = _dev_inputs(x, blk)
    S = mmq.q4K_scaled_block_dots(aq, w, N).cpu().numpy()
    assert (S == sign * 63 * 60960).all()


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (64, 128, 2816)])
def test_gemm_full_small(path_name, M, N, K):
    mmq = require_gpu()
    x = synthetic.activations(M, K, 51 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 61 + N)
    _full_check(x, blk, N, getattr(mmq, path_name))


def test_gemm_small_m_full():
    mmq = require_gpu()
    for M in (1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64):
        x = synthetic.activations(M, 1024, 71 + M, 0.01)
        blk = synthetic.q4K_weights(260, 1024, 81)
        _full_check(x, blk, 260, mmq.MMQ_PATH_SMALL_M)


@pytest.mark.parametrize("ks", [1, 2, 4])
@pytest.mark.parametrize("M,N,K", [(1, 256, 11008), (3, 4096, 4096), (4, 4100, 1280)])
def test_gemm_dot_product_every_split(ks, M, N, K):
    # each K split of the dot-product kernel, forced, within tolerance
    mmq = require_gpu()
    x = synthetic.activations(M, K, 191 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 201 + N)
    mmq.force_gemv_split(ks)
    try:
        _full_check(x, blk, N, mmq.MMQ_PATH_SMALL_M)
    finally:
        mmq.force_gemv_split(0)


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC"])
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


def test_q_proj_every_element():
    # the headline workload, every one of its 8.4 M outputs against the oracle
    # (the oracle's full C and bound take a few seconds on the host's cores)
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs("q_proj")
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    ok = oracle.within_tolerance(C, C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outputs outside tolerance"


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


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_SMALL_M"])
def test_every_output_written_and_deterministic(path_name):
    import torch
    mmq = require_gpu()
    M, N, K = (37 if path_name == "MMQ_PATH_SMALL_M" else 200), 516, 1024
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


@pytest.mark.parametrize("path_name", ["MMQ_PATH_MMA_S8", "MMQ_PATH_TC", "MMQ_PATH_SMALL_M"])
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


@pytest.mark.parametrize("path_name,M", [("MMQ_PATH_MMA_S8", 128), ("MMQ_PATH_TC", 128), ("MMQ_PATH_TC", 77),
                                         ("MMQ_PATH_SMALL_M", 1), ("MMQ_PATH_SMALL_M", 2), ("MMQ_PATH_SMALL_M", 4),
                                         ("MMQ_PATH_SMALL_M", 5), ("MMQ_PATH_SMALL_M", 16),
                                         ("MMQ_PATH_SMALL_M", 33), ("MMQ_PATH_SMALL_M", 64)])
@pytest.mark.parametrize("N,K", [(132, 1024), (260, 256)])
def test_exact_c_with_sub_block_scales(path_name, M, N, K):
    # sc != 1 on every path: m = dmin = 0, d = 2^-4, integer activations with
    # one +-127 per block (so da = 1 and q = x) and the rest small, so that
    # every partial sum is an integer multiple of 2^-4 below 2^20 in any
    # order: C = d * sum_c sc_c * S_c holds exactly (page r15 section 2.1
    # with dmin = 0, the second term vanishes).
    mmq = require_gpu()
    rng = np.random.default_rng(211 + M + N)
    x = rng.integers(-8, 9, (M, K)).astype(np.float32)
    x.reshape(M, K // 32, 32)[:, :, 5] = 127.0 * rng.choice([-1.0, 1.0], (M, K // 32))
    sc = rng.integers(0, 64, (N, K // 32))
    v = rng.integers(0, 16, (N, K))
    blk = q4k_layout.encode(np.full((N, K // 256), 2.0 ** -4), np.zeros((N, K // 256)), sc,
                            np.zeros((N, K // 32)), v)
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N, path=getattr(mmq, path_name)).cpu().numpy()
    assert mmq.status() == 0
    xi = x.astype(np.int64).reshape(M, K // 32, 32)
    S = np.einsum("mcl,ncl->mnc", xi, v.reshape(N, K // 32, 32).astype(np.int64))
    total = (S * sc[None, :, :]).sum(axis=2)
    assert np.abs(S * sc[None]).sum(axis=2).max() < 2 ** 24   # the exactness premise
    assert (C.astype(np.float64) == total * 2.0 ** -4).all()


@pytest.mark.parametrize("M", [5, 16, 40, 64])
@pytest.mark.parametrize("N", [11008, 9792])
def test_small_m_partial_round_split(M, N):
    # 5-64 tokens over more 64-row tiles than one round of CTAs holds: the
    # partial last round runs as a second launch with K split over a cluster.
    # C within tolerance everywhere, S bit-exact, the same bits on a rerun.
    import torch
    mmq = require_gpu()
    K = 4096
    x = synthetic.activations(M, K, 611 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 621 + N)
    C = _full_check(x, blk, N, mmq.MMQ_PATH_SMALL_M)
    _, aq, w = _dev_inputs(x, blk)
    C2 = mmq.q4K_gemm(aq, w, N, path=mmq.MMQ_PATH_SMALL_M).cpu().numpy()
    assert mmq.status() == 0
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))
    n = mmq.mmq_q4K_gemm_launches(M, N, K, mmq.MMQ_PATH_SMALL_M)
    assert n in (1, 2)
    assert mmq.mmq_q4K_gemm_launches(M, N, K, mmq.MMQ_PATH_AUTO) == n
    if M == 16 and N == 11008 and torch.cuda.get_device_properties(0).multi_processor_count < 172:
        assert n == 2   # 172 tiles of one CTA per SM: a partial second round
    if M == 16:
        q, _, _ = oracle.quantize_q8_1(x)
        S = mmq.q4K_block_dots(aq, w, N, path=mmq.MMQ_PATH_SMALL_M).cpu().numpy()
        assert mmq.status() == 0
        assert (S == oracle.block_dots(q, blk, N)).all()


@pytest.mark.parametrize("name", ["gate_up", "down"])
def test_ffn_every_element(name):
    # the FFN workloads at 2048 tokens, every output against the oracle
    # (gate/up: 22.5 M outputs; down: K = 11008)
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs(name)
    _, aq, w = _dev_inputs(x, blk)
    C = mmq.q4K_gemm(aq, w, N).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    ok = oracle.within_tolerance(C, C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outputs outside tolerance"


@pytest.mark.parametrize("M", [4, 5, 64, 65])
@pytest.mark.parametrize("N,K", [(1100, 1280), (4100, 256)])
def test_auto_path_boundaries(M, N, K):
    # the automatic choice on both sides of each switch (dot product | mma.sync
    # at 4/5 tokens, mma.sync | tcgen05 at 64/65), every output, ragged N
    mmq = require_gpu()
    x = synthetic.activations(M, K, 731 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 741 + N)
    _full_check(x, blk, N, mmq.MMQ_PATH_AUTO)
