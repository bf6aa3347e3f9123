"""Weights loaded from a GGUF file feed the GEMM: q4_K and q6_K tensors
written with mmq_gguf_write, read back with mmq_gguf_read, multiplied on
the GPU and checked against the oracle on the original weights."""
import numpy as np
import pytest

import oracle
from oracle import q6k
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_gemm_on_weights_from_gguf(tmp_path):
    mmq = require_gpu()
    M, N, K = 130, 260, 1024
    x = synthetic.activations(M, K, 701, 0.01)
    w4 = synthetic.q4K_weights(N, K, 702)
    w6 = synthetic.q6K_weights(N, K, 703)
    path = str(tmp_path / "w.gguf")
    mmq.gguf_write(path, [("blk.0.attn_q.weight", mmq.MMQ_GGUF_Q4_K, K, N, w4),
                          ("blk.0.attn_k.weight", mmq.MMQ_GGUF_Q6_K, K, N, w6)])
    got = mmq.gguf_read(path)
    aq = mmq.quantize_q8_1(to_dev(x))
    q, da, sa = oracle.quantize_q8_1(x)
    C4 = mmq.q4K_gemm(aq, to_dev(got["blk.0.attn_q.weight"][2]), N).cpu().numpy()
    C_ref, _, T = oracle.gemm(q, da, sa, w4, N)
    assert oracle.within_tolerance(C4, C_ref, T).all()
    C6 = mmq.q6K_gemm(aq, mmq.repack_q6K(to_dev(got["blk.0.attn_k.weight"][2]), N, K), N).cpu().numpy()
    _, C64, T6 = q6k.gemm(q, da, w6, N)
    assert (np.abs(C6.astype(np.float64) - C64) <= 1e-4 * T6 + 1e-6).all()
    assert mmq.status() == 0
