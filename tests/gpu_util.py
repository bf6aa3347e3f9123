"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q4_q8_int8_gb300 as mmq
    from q4_q8_int8_gb300 import build as mmq_build
    mmq_build.build()
    mmq.load_library()
    return mmq


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def oracle_q8(x):
    return oracle.quantize_q8_1(x)


def sample_points(M, N, n, seed):
    """Rows/cols to check at full size: first/last rows and columns in full
    plus n random points."""
    rng = np.random.default_rng(seed)
    rows = [np.full(N, r) for r in sorted({0, M - 1})]
    cols = [np.arange(N) for _ in rows]
    for c in sorted({0, N - 1}):
        rows.append(np.arange(M))
        cols.append(np.full(M, c))
    rows.append(rng.integers(0, M, n))
    cols.append(rng.integers(0, N, n))
    return np.concatenate(rows), np.concatenate(cols)
