"""The library called from several host threads at once, each on its own
stream: every kernel family, the thread-local K-split hook, and the
per-device caches (tensor-map encoder, occupancy, status word).  Every
result must be bit-identical to the same call made alone: no kernel uses
atomics, so concurrency may only change timing."""
import threading

import numpy as np
import pytest

from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _cases(mmq):
    # (name, M, K, N, weights, call(aq, w, N) -> tensor)
    q4 = lambda path: (lambda aq, w, N: mmq.q4K_gemm(aq, w, N, path=path))
    return [
        ("dot product", 1, 4096, 4096, "q4k", q4(mmq.MMQ_PATH_AUTO)),
        ("mma.sync two launches", 16, 4096, 11008, "q4k", q4(mmq.MMQ_PATH_AUTO)),
        ("tcgen05 split-K", 128, 1024, 1024, "q4k", q4(mmq.MMQ_PATH_AUTO)),
        ("tcgen05", 300, 512, 388, "q4k", q4(mmq.MMQ_PATH_TC)),
        ("q8_1 output", 4, 1024, 4096, "q4k", lambda aq, w, N: mmq.q4K_gemm_q8_1(aq, w, N)[1][0]),
        ("q6_K dot product", 2, 4096, 1024, "q6k", lambda aq, w, N: mmq.q6K_gemm(aq, w, N)),
        ("q6_K tcgen05", 130, 512, 260, "q6k", lambda aq, w, N: mmq.q6K_gemm(aq, w, N)),
    ]


def _inputs(mmq, M, K, N, kind, seed):
    x = to_dev(synthetic.activations(M, K, 900 + seed, 0.01))
    if kind == "q4k":
        w = to_dev(synthetic.q4K_weights(N, K, 910 + seed).reshape(-1))
    else:
        w = mmq.repack_q6K(to_dev(synthetic.q6K_weights(N, K, 910 + seed).reshape(-1)), N, K)
    return x, w


def test_threads_on_separate_streams_bit_identical():
    import torch
    mmq = require_gpu()
    cases = _cases(mmq)
    inputs = [_inputs(mmq, M, K, N, kind, i) for i, (_, M, K, N, kind, _) in enumerate(cases)]
    ref = []
    for (name, M, K, N, kind, call), (x, w) in zip(cases, inputs):
        out = call(mmq.quantize_q8_1(x), w, N)
        torch.cuda.synchronize()
        assert mmq.status() == 0, name
        ref.append(out.cpu().numpy().copy())
    # one case forced onto another K split in a thread of its own: the hook is per thread
    x1, w1 = inputs[0]
    mmq.force_gemv_split(4)
    try:
        forced_ref = mmq.q4K_gemm(mmq.quantize_q8_1(x1), w1, 4096).cpu().numpy().copy()
    finally:
        mmq.force_gemv_split(0)

    errors, results = [], {}

    def worker(tid):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                if tid == len(cases):   # the forced-split thread
                    mmq.force_gemv_split(4)
                    try:
                        outs = [mmq.q4K_gemm(mmq.quantize_q8_1(x1), w1, 4096) for _ in range(20)]
                    finally:
                        mmq.force_gemv_split(0)
                else:
                    name, M, K, N, kind, call = cases[tid]
                    x, w = inputs[tid]
                    outs = [call(mmq.quantize_q8_1(x), w, N) for _ in range(20)]
                s.synchronize()
            results[tid] = [o.cpu().numpy() for o in outs]
        except Exception as e:   # reported on the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(cases) + 1)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    assert mmq.status() == 0
    for tid, (name, *_rest) in enumerate(cases):
        for o in results[tid]:
            assert np.array_equal(o.view(np.uint8), ref[tid].view(np.uint8)), name
    for o in results[len(cases)]:
        assert np.array_equal(o.view(np.uint8), forced_ref.view(np.uint8))
