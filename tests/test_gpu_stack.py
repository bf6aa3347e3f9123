"""The 7B-shaped prefill stack (32 layers x q, k, v, o, gate, up, down at
2048 tokens): its GEMMs are the q-proj / gate-up / down shapes with their
own seeded weights and activations.  Sampled outputs of the first and last
layer's q, gate and down GEMMs (prepass + GEMM through the C ABI, automatic
kernel choice) against the oracle, within the stated tolerance."""
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, sample_points

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


@pytest.mark.parametrize("layer", [0, synthetic.STACK_LAYERS - 1])
@pytest.mark.parametrize("g", [0, 4, 6])   # q, gate, down
def test_stack_gemm_sampled(layer, g):
    import torch
    mmq = require_gpu()
    dev = torch.device("cuda", 0)
    M = synthetic.STACK_TOKENS
    _, K, N = synthetic.STACK_GEMMS[g]
    wseed, xseed = synthetic.stack_seeds(layer, g)
    w = synthetic.torch_q4K_weights(N, K, wseed, dev)
    x = synthetic.torch_activations(M, K, xseed, dev, 0.01)
    aq = mmq.quantize_q8_1(x)
    C = mmq.q4K_gemm(aq, w.view(-1), N).cpu().numpy()
    assert mmq.status() == 0
    xh, blk = x.cpu().numpy(), w.cpu().numpy()
    q, da, sa = oracle.quantize_q8_1(xh)
    assert (q == aq[0].cpu().numpy()).all()
    rows, cols = sample_points(M, N, 1500, 17 + g)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    assert oracle.within_tolerance(C[rows, cols], C_ref, T, RTOL, ATOL).all()
