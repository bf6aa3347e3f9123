"""The dequantize-then-dense control path on the GPU vs the CPU oracle.

Dequantized weights and fp16 activations must match bit for bit; the dense
GEMM must satisfy |C - C_ref| <= 1e-4 * sum_k |a_k b_k| + 1e-6, where C_ref
sums the exact products in float64.  The kernel accumulates K/16 partial
sums of 16 exact products in float32, so its error is at most about
K * 2^-28 of sum |a b| (1.5e-5 at K = 4096); the bound holds for K up to
~26000.  (The control is the f16 GEMM path of web page "16 . r12 --
16-chain warp tile + ldmatrix", its dequantize step that of page "Round 31
Track C Audit: dq_f16 (dense_mm.metal) & DW<F> (mma.metal)", section 2.1.)
"""
import os

import numpy as np
import pytest

from oracle import dense
from q4_q8_int8_gb300 import synthetic
from tests import q4k_layout
from tests.gpu_util import require_gpu, sample_points, to_dev

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _bits(a):
    return np.asarray(a).view(np.uint16)


@pytest.mark.parametrize("N,K", [(4, 256), (260, 1024), (33, 11008), (4096, 4096)])
def test_dequant_bit_exact(N, K):
    mmq = require_gpu()
    blk = synthetic.q4K_weights(N, K, 300 + N)
    wh = mmq.dequantize_q4K_f16(to_dev(blk.reshape(-1)), N, K).cpu().numpy()
    assert mmq.status() == 0
    assert (_bits(wh) == _bits(dense.dequantize_q4K_f16(blk, N, K))).all()


def test_dequant_golden_and_extreme_fields():
    mmq = require_gpu()
    rows = []
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "dequant_f16_values.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            f = line.split()
            rows.append((int(f[0], 16), int(f[1], 16), int(f[2]), int(f[3]), int(f[4]), float(f[5])))
    N, K = len(rows) + 2, 512
    d = [[np.array(r[0], np.uint16).view(np.float16)] * 2 for r in rows]
    dmin = [[np.array(r[1], np.uint16).view(np.float16)] * 2 for r in rows]
    sc = [[r[2]] * 16 for r in rows]
    m = [[r[3]] * 16 for r in rows]
    v = [[r[4]] * K for r in rows]
    # largest fields: fp16 max d and dmin, sc = m = 63, v = 15 (difference of two huge products);
    # and a row of all-zero scales
    d += [[np.float16(65504.0)] * 2, [np.float16(0.0)] * 2]
    dmin += [[np.float16(65504.0)] * 2, [np.float16(0.0)] * 2]
    sc += [[63] * 16, [0] * 16]
    m += [[63] * 16, [0] * 16]
    rng = np.random.default_rng(5)
    v += [list(rng.integers(0, 16, K)), [15] * K]
    blk = q4k_layout.encode(np.array(d), np.array(dmin), np.array(sc), np.array(m), np.array(v))
    wh = mmq.dequantize_q4K_f16(to_dev(blk.reshape(-1)), N, K).cpu().numpy()
    ref = dense.dequantize_q4K_f16(blk, N, K)
    assert (_bits(wh) == _bits(ref)).all()
    for j, r in enumerate(rows):
        assert (wh[j] == np.float16(r[5])).all()
    assert (wh[-1] == 0).all()


def test_convert_bit_exact_with_edge_values():
    mmq = require_gpu()
    rng = np.random.default_rng(6)
    x = rng.standard_normal(4096).astype(np.float32) * 100
    edge = np.array([65504.0, 65519.0, 65520.0, -65536.0, 1e-8, -3e-8, 6.1e-5, 0.0, -0.0,
                     2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -12,
                     np.inf, -np.inf], np.float32)
    x[:edge.size] = edge
    xh = mmq.convert_f16(to_dev(x)).cpu().numpy()
    assert (_bits(xh) == _bits(dense.convert_f16(x))).all()


def _dense_inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal((M, K)) * 2).astype(np.float16)
    b = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    return a, b


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (77, 132, 320), (300, 516, 1024), (1, 4, 64),
                                   (129, 260, 4096), (256, 512, 11008)])
def test_gemm_f16_full(M, N, K):
    mmq = require_gpu()
    a, b = _dense_inputs(M, N, K, M + N + K)
    C = mmq.gemm_f16(to_dev(a), to_dev(b)).cpu().numpy()
    assert mmq.status() == 0
    C_ref, T = dense.gemm_f16(a, b)
    ok = np.abs(C.astype(np.float64) - C_ref) <= RTOL * T + ATOL
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance"


def test_gemm_f16_q_proj_sampled_and_deterministic():
    import torch
    mmq = require_gpu()
    M, N, K = 2048, 4096, 4096
    a, b = _dense_inputs(M, N, K, 7)
    da, db = to_dev(a), to_dev(b)
    C1 = mmq.gemm_f16(da, db)
    C2 = mmq.gemm_f16(da, db)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    C = C1.cpu().numpy()
    rows, cols = sample_points(M, N, 3000, 8)
    C_ref, T = dense.gemm_f16_sampled(a, b, rows, cols)
    assert (np.abs(C[rows, cols].astype(np.float64) - C_ref) <= RTOL * T + ATOL).all()
    assert np.isfinite(C).all()


def test_gemm_f16_guard_bands():
    import torch
    mmq = require_gpu()
    M, N, K = 200, 516, 512
    a, b = _dense_inputs(M, N, K, 9)
    buf = torch.full((M * N + 2048,), float("nan"), device="cuda")
    buf[:1024] = 7.0
    buf[-1024:] = 7.0
    C = buf[1024:1024 + M * N].view(M, N)
    mmq.gemm_f16(to_dev(a), to_dev(b), out=C)
    torch.cuda.synchronize()
    assert torch.isfinite(C).all()
    assert (buf[:1024] == 7.0).all() and (buf[-1024:] == 7.0).all()


def test_control_path_end_to_end():
    # x (f32) -> fp16, q4_K -> fp16, dense GEMM: against the oracle's chain
    mmq = require_gpu()
    M, N, K = 130, 388, 1280
    x = synthetic.activations(M, K, 17, 0.01)
    blk = synthetic.q4K_weights(N, K, 18)
    xh = mmq.convert_f16(to_dev(x))
    wh = mmq.dequantize_q4K_f16(to_dev(blk.reshape(-1)), N, K)
    C = mmq.gemm_f16(xh, wh).cpu().numpy()
    C_ref, T = dense.gemm_f16(dense.convert_f16(x), dense.dequantize_q4K_f16(blk, N, K))
    assert (np.abs(C.astype(np.float64) - C_ref) <= RTOL * T + ATOL).all()


def test_dense_argument_errors():
    import torch
    mmq = require_gpu()
    a = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((128, 256), device="cuda")
    P = lambda t: __import__("ctypes").c_void_p(t.data_ptr())
    assert mmq.mmq_gemm_f16(P(a), P(b), P(C), 128, 256, 48, None) == mmq.MMQ_ERR_ARG    # K % 64
    assert mmq.mmq_gemm_f16(P(a), P(b), P(C), 128, 254, 64, None) == mmq.MMQ_ERR_ARG    # N % 4
    assert mmq.mmq_gemm_f16(None, P(b), P(C), 128, 256, 64, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_dequantize_q4K_f16(P(a), P(b), 4, 250, None) == mmq.MMQ_ERR_ARG      # K % 256
    assert mmq.mmq_convert_f32_f16(P(C), P(a), 6, None) == mmq.MMQ_ERR_ARG            # n % 4
    assert mmq.status() == 0
