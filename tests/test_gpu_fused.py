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
                                   (1, 32, 256)])
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
    if M > 64:   # without the f32 result: the same q8_1 bits
        _, o2 = mmq.q4K_gemm_q8_1(aq, to_dev(blk.reshape(-1)), N, with_c=False)
        assert mmq.status() == 0
        for a, b in zip(o, o2):
            assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())


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
