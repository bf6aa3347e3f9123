"""Failure detection without a GPU fault: a withheld producer arrival makes
the tcgen05 kernel's bounded waits run out; the kernel records
MMQ_ERR_DEVICE_TIMEOUT, unwinds and returns, and the context stays usable."""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path_name,M", [("MMQ_PATH_TC", 128), ("MMQ_PATH_TC", 77), ("MMQ_PATH_TC", 2048)])
def test_injected_timeout_is_reported_and_context_survives(path_name, M):
    mmq = require_gpu()
    path = getattr(mmq, path_name)
    N, K = 256, 512
    x = synthetic.activations(M, K, 5)
    blk = synthetic.q4K_weights(N, K, 6)
    aq = mmq.quantize_q8_1(to_dev(x))
    w = to_dev(blk.reshape(-1))
    assert mmq.status() == 0
    mmq.mmq_debug_inject_timeout(True)
    mmq.q4K_gemm(aq, w, N, path=path)
    assert mmq.status() == mmq.MMQ_ERR_DEVICE_TIMEOUT
    assert mmq.status() == 0   # read-and-clear
    # the next launch is unaffected and correct
    C = mmq.q4K_gemm(aq, w, N, path=path).cpu().numpy()
    assert mmq.status() == 0
    q, da, sa = oracle.quantize_q8_1(x)
    C_ref, _, T = oracle.gemm(q, da, sa, blk, N)
    assert oracle.within_tolerance(C, C_ref, T).all()


def test_injection_flag_is_one_shot():
    mmq = require_gpu()
    mmq.mmq_debug_inject_timeout(True)
    mmq.mmq_debug_inject_timeout(False)
    M, N, K = 130, 128, 256
    x = synthetic.activations(M, K, 7)
    blk = synthetic.q4K_weights(N, K, 8)
    aq = mmq.quantize_q8_1(to_dev(x))
    C = mmq.q4K_gemm(aq, to_dev(blk.reshape(-1)), N, path=mmq.MMQ_PATH_TC).cpu().numpy()
    assert mmq.status() == 0 and np.isfinite(C).all()
