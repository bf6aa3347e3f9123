"""The tensor-core operand plane and the super-block GEMM that reads it
(mmq_quantize_q8_1_tcop, mmq_q4K_gemm_tcop) vs the CPU oracle.

The GEMM never forms the per-chunk integer dots S: each chunk's activation
scale rides in the activation operand (two fp16 parts per element, within
2^-14 of q*s) and a whole 256-k super-block accumulates on the tensor core.
Its contract is the GEMM tolerance |C - C_ref| <= 1e-4 * sum_k |a_k w_k| +
1e-6 element by element (web page "20 . r15 -- f32-accumulate mma probe
(dead end) + rank-1 term2 rescale", section 2.1 for the math), plus exact
results where every operand and partial sum is exactly representable.  The
plane itself is checked bit for bit against its encoding restated in numpy
(tests/tcop_layout.py), and the q8_1 values the same call writes against
the oracle.
"""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests import q4k_layout, tcop_layout
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _run(x, blk, N):
    mmq = require_gpu()
    M, K = x.shape
    _, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    C = mmq.q4K_gemm_tcop(tcop, to_dev(blk.reshape(-1)), M, N, K).cpu().numpy()
    assert mmq.status() == 0
    return C


def _check(x, blk, N):
    C = _run(x, blk, N)
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    ok = oracle.within_tolerance(C, C_ref, T, RTOL, ATOL)
    bad = np.argmax(np.abs(C - C_ref) - RTOL * T)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance; worst at {np.unravel_index(bad, C.shape)}"


@pytest.mark.parametrize("M,K", [(1, 256), (77, 768), (300, 4096), (128, 11008)])
def test_plane_bit_exact_and_q8_1_unchanged(M, K):
    mmq = require_gpu()
    x = synthetic.activations(M, K, 301 + M, 0.01)
    x[0, :32] = 0.0                 # a zero block (da = 0)
    x[-1, 256:288] *= 1e-30         # a block far below the rest of its super-block
    aq, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    q, da, sa = oracle.quantize_q8_1(x)
    assert (aq[0].cpu().numpy() == q).all()
    assert (aq[1].cpu().numpy().view(np.uint32) == da.view(np.uint32)).all()
    assert (aq[2].cpu().numpy() == sa).all()
    hi, lo, t2, g = tcop_layout.split(tcop.cpu().numpy(), M, K)
    e_hi, e_lo, e_t2, e_g = tcop_layout.encode(q, da, sa)
    assert (hi == e_hi).all() and (lo == e_lo).all()
    assert (t2 == e_t2).all()
    assert (g.view(np.uint32) == e_g.view(np.uint32)).all()


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (77, 132, 768), (300, 388, 1280), (1, 4, 256),
                                   (513, 260, 2816), (130, 516, 256), (64, 128, 11008)])
def test_full_small(M, N, K):
    x = synthetic.activations(M, K, 51 + M, 0.01)
    blk = synthetic.q4K_weights(N, K, 61 + N)
    _check(x, blk, N)


def test_more_tiles_than_ctas():
    # 18 x 9 tiles of 128 x 256: each CTA takes two tiles in turn
    M, N, K = 2304, 2304, 256
    x = synthetic.activations(M, K, 221, 0.01)
    blk = synthetic.q4K_weights(N, K, 222)
    _check(x, blk, N)


def test_chunk_scales_far_apart():
    # chunks of one super-block whose amax differ by up to 2^15 (the operand
    # is scaled per token row and super-block; each chunk keeps 2^-14)
    rng = np.random.default_rng(231)
    M, N, K = 256, 256, 1024
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-15, 1, (M, K // 32))).repeat(32, axis=1).astype(np.float32)
    blk = synthetic.q4K_weights(N, K, 232)
    _check(x, blk, N)


def test_zero_and_extreme_super_block_scales():
    # d = 0 (only the second term remains), the smallest fp16 d with dmin = 1
    # (dmin / d = 2^24), and a large d with a tiny dmin, mixed per row and
    # super-block
    rng = np.random.default_rng(241)
    M, N, K = 130, 260, 1280
    nsb = K // 256
    d = rng.uniform(1e-3, 1e-2, (N, nsb))
    dmin = rng.uniform(1e-3, 1e-2, (N, nsb))
    pick = rng.integers(0, 4, (N, nsb))
    d[pick == 0] = 0.0
    d[pick == 1], dmin[pick == 1] = 2.0 ** -24, 1.0
    d[pick == 2], dmin[pick == 2] = 60000.0, 2.0 ** -20
    blk = q4k_layout.encode(d, dmin, rng.integers(0, 64, (N, K // 32)), rng.integers(0, 64, (N, K // 32)),
                            rng.integers(0, 16, (N, K)))
    x = synthetic.activations(M, K, 242, 0.01)
    _check(x, blk, N)


def test_worked_examples_exact():
    M, N, K = 4, 8, 512
    # E2: w == 0 through exact per-chunk cancellation of the two terms
    x = np.ones((M, K), np.float32)
    blk = q4k_layout.encode(np.ones((N, 2)), np.ones((N, 2)), np.ones((N, 16)), np.ones((N, 16)),
                            np.ones((N, K)))
    assert (_run(x, blk, N) == 0).all()
    # E4: v = 0 and m = 0 give C = 0 for any activations and scales
    rng = np.random.default_rng(3)
    x = rng.standard_normal((M, K)).astype(np.float32)
    blk = q4k_layout.encode(rng.uniform(1e-3, 1, (N, 2)), rng.uniform(1e-3, 1, (N, 2)),
                            rng.integers(0, 64, (N, 16)), np.zeros((N, 16)), np.zeros((N, K)))
    assert (_run(x, blk, N) == 0).all()
    # E5: d = sc = 1, m = dmin = 0, integer activations with amax 127 per
    # block (da = 1: the scale splits exactly, lo = 0)
    x = rng.integers(-127, 128, (M, K)).astype(np.float32)
    x.reshape(M, K // 32, 32)[:, :, 0] = 127.0
    v = rng.integers(0, 16, (N, K))
    blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.ones((N, 16)), np.zeros((N, 16)), v)
    C = _run(x, blk, N)
    assert (C.astype(np.int64) == x.astype(np.int64) @ v.T).all()


@pytest.mark.parametrize("M,N,K", [(128, 132, 1024), (300, 260, 256)])
def test_exact_c_with_sub_block_scales(M, N, K):
    # sc != 1: m = dmin = 0, d = 2^-4, one +-127 per block (da = 1, q = x):
    # every partial sum is a multiple of 2^-17 below 2^7, so C = d * sum sc * S
    # holds exactly (page r15 section 2.1 with dmin = 0)
    rng = np.random.default_rng(211 + M + N)
    x = rng.integers(-8, 9, (M, K)).astype(np.float32)
    x.reshape(M, K // 32, 32)[:, :, 5] = 127.0 * rng.choice([-1.0, 1.0], (M, K // 32))
    sc = rng.integers(0, 64, (N, K // 32))
    v = rng.integers(0, 16, (N, K))
    blk = q4k_layout.encode(np.full((N, K // 256), 2.0 ** -4), np.zeros((N, K // 256)), sc,
                            np.zeros((N, K // 32)), v)
    C = _run(x, blk, N)
    xi = x.astype(np.int64).reshape(M, K // 32, 32)
    S = np.einsum("mcl,ncl->mnc", xi, v.reshape(N, K // 32, 32).astype(np.int64))
    total = (S * sc[None, :, :]).sum(axis=2)
    assert np.abs(S * sc[None]).sum(axis=2).max() < 2 ** 24   # the exactness premise
    assert (C.astype(np.float64) == total * 2.0 ** -4).all()


def test_every_output_written_and_deterministic():
    import torch
    mmq = require_gpu()
    M, N, K = 300, 516, 1024
    x = synthetic.activations(M, K, 91, 0.01)
    blk = synthetic.q4K_weights(N, K, 92)
    _, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    w = to_dev(blk.reshape(-1))
    # guard bands around C must stay untouched; C itself starts as NaN
    buf = torch.full((M * N + 2 * 1024,), float("nan"), device="cuda")
    buf[:1024] = 7.0
    buf[-1024:] = 7.0
    C1 = buf[1024:1024 + M * N].view(M, N)
    mmq.q4K_gemm_tcop(tcop, w, M, N, K, out=C1)
    C2 = mmq.q4K_gemm_tcop(tcop, w, M, N, K)
    torch.cuda.synchronize()
    assert torch.isfinite(C1).all()
    assert (buf[:1024] == 7.0).all() and (buf[-1024:] == 7.0).all()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


@pytest.mark.parametrize("name", ["q_proj", "down", "gate_up"])
def test_full_size_sampled(name):
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs(name)
    M, K = x.shape
    _, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    C = mmq.q4K_gemm_tcop(tcop, to_dev(blk.reshape(-1)), M, N, K).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 5)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    ok = oracle.within_tolerance(C[rows, cols], C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} sampled outputs outside tolerance"
    assert np.isfinite(C).all()


@pytest.mark.parametrize("name", ["q_proj", "gate_up", "down"])
def test_every_element(name):
    # every output of the 2048-token workloads through the operand plane
    mmq = require_gpu()
    x, blk, N = synthetic.config_inputs(name)
    M, K = x.shape
    _, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    C = mmq.q4K_gemm_tcop(tcop, to_dev(blk.reshape(-1)), M, N, K).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    ok = oracle.within_tolerance(C, C_ref, T, RTOL, ATOL)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outputs outside tolerance"


def test_argument_errors():
    import torch
    mmq = require_gpu()
    M, N, K = 64, 128, 512
    x = torch.zeros((M, K), device="cuda")
    aq, tcop = mmq.quantize_q8_1_tcop(x)
    w = torch.zeros((N * (K // 256) * 144,), dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), device="cuda")
    sp = mmq._stream_ptr()
    import ctypes
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    assert mmq.mmq_q4K_gemm_tcop(P(tcop, 16), P(w), P(C), M, N, K, sp) == mmq.MMQ_ERR_ALIGN
    assert mmq.mmq_q4K_gemm_tcop(P(tcop), P(w), P(C), M, N, 300, sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_tcop(P(tcop), P(w), P(C), M, 6, K, sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_quantize_q8_1_tcop(P(x), M, 96, mmq.q8_1_struct(*aq), P(tcop), sp) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q8_1_tcop_bytes(M, 300) == 0


@pytest.mark.parametrize("M", [128, 2048])
def test_injected_timeout_is_reported_and_context_survives(M):
    mmq = require_gpu()
    N, K = 256, 512
    x = synthetic.activations(M, K, 5)
    blk = synthetic.q4K_weights(N, K, 6)
    _, tcop = mmq.quantize_q8_1_tcop(to_dev(x))
    w = to_dev(blk.reshape(-1))
    assert mmq.status() == 0
    mmq.mmq_debug_inject_timeout(True)
    mmq.q4K_gemm_tcop(tcop, w, M, N, K)
    assert mmq.status() == mmq.MMQ_ERR_DEVICE_TIMEOUT
    assert mmq.status() == 0
    C = mmq.q4K_gemm_tcop(tcop, w, M, N, K).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    assert oracle.within_tolerance(C, C_ref, T).all()
