"""Programmatic dependent launch changes when kernels start, not what they
compute: a chain quantize -> GEMM -> quantize(its output) -> GEMM gives the
same bits with the launch mode on and off, launched directly and from a
CUDA graph, on the dp4a (M <= 4), mma.sync (M <= 64) and tcgen05 paths
(M = 700: K split over clusters for few tiles);
and the second GEMM matches the oracle on the first GEMM's output."""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _chain(mmq, x, w1, w2, K, N1, N2):
    aq1 = mmq.quantize_q8_1(x)
    c1 = mmq.q4K_gemm(aq1, w1, N1)
    aq2 = mmq.quantize_q8_1(c1)
    c2 = mmq.q4K_gemm(aq2, w2, N2)
    return c1, aq2, c2


@pytest.mark.parametrize("M", [1, 4, 9, 64, 200, 700])
def test_pdl_chain_same_bits_and_oracle(M):
    import torch
    mmq = require_gpu()
    K, N1, N2 = 1024, 512, 260
    x = to_dev(synthetic.activations(M, K, 800 + M, 0.01))
    b1 = synthetic.q4K_weights(N1, K, 801)
    b2 = synthetic.q4K_weights(N2, N1, 802)
    w1, w2 = to_dev(b1.reshape(-1)), to_dev(b2.reshape(-1))
    try:
        mmq.mmq_set_programmatic_launch(False)
        ref = _chain(mmq, x, w1, w2, K, N1, N2)
        torch.cuda.synchronize()
        mmq.mmq_set_programmatic_launch(True)
        for _ in range(3):
            got = _chain(mmq, x, w1, w2, K, N1, N2)
            torch.cuda.synchronize()
            assert torch.equal(got[0].view(torch.int32), ref[0].view(torch.int32))
            assert torch.equal(got[2].view(torch.int32), ref[2].view(torch.int32))
        # the same chain captured in a graph and replayed
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            _chain(mmq, x, w1, w2, K, N1, N2)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                gout = _chain(mmq, x, w1, w2, K, N1, N2)
            for _ in range(3):
                g.replay()
            s.synchronize()
        assert torch.equal(gout[2].view(torch.int32), ref[2].view(torch.int32))
        assert mmq.status() == 0
    finally:
        mmq.mmq_set_programmatic_launch(False)
    c1 = ref[0].cpu().numpy()
    q, da, sa = oracle.quantize_q8_1(c1)
    C_ref, _, T = oracle.gemm(q, da, sa, b2, N2)
    assert oracle.within_tolerance(ref[2].cpu().numpy(), C_ref, T).all()


def test_pdl_split_tail_same_bits():
    # more tiles than SMs: the GEMM runs as two launches (whole rounds, then
    # the last partial round with K split); with the launch mode on, each
    # starts while the previous kernel finishes.  Same bits either way, and
    # sampled outputs within the tolerance of the oracle.
    import torch
    from tests.gpu_util import sample_points
    mmq = require_gpu()
    M, K, N = 2048, 512, 4096
    x = synthetic.activations(M, K, 830, 0.01)
    blk = synthetic.q4K_weights(N, K, 831)
    xd, w = to_dev(x), to_dev(blk.reshape(-1))
    # 512 tiles on 152 SMs: three whole rounds, then 56 tiles split-K
    assert mmq.mmq_q4K_gemm_launches(M, N, K, mmq.MMQ_PATH_AUTO) == 2
    assert mmq.mmq_q4K_gemm_launches(700, 512, 1024, mmq.MMQ_PATH_AUTO) == 1   # 24 tiles, one split launch
    assert mmq.mmq_q4K_gemm_launches(64, N, K, mmq.MMQ_PATH_AUTO) == 1         # few tokens
    try:
        mmq.mmq_set_programmatic_launch(False)
        ref = mmq.q4K_gemm(mmq.quantize_q8_1(xd), w, N)
        torch.cuda.synchronize()
        mmq.mmq_set_programmatic_launch(True)
        for _ in range(2):
            got = mmq.q4K_gemm(mmq.quantize_q8_1(xd), w, N)
            torch.cuda.synchronize()
            assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
        assert mmq.status() == 0
    finally:
        mmq.mmq_set_programmatic_launch(False)
    q, da, sa = oracle.quantize_q8_1(x)
    rows, cols = sample_points(M, N, 3000, 31)
    C_ref, _, T = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
    assert oracle.within_tolerance(ref.cpu().numpy()[rows, cols], C_ref, T).all()
