"""The operand plane's encoding (tests/tcop_layout.py, the bytes the
tensor-core prepass writes) keeps each activation within 2^-14 of q * da /
g, g the power of two of its token row and super-block; checked in float64
on host data, including chunks whose scales differ by up to 2^12 within one
super-block."""
import numpy as np

import oracle
from tests import tcop_layout


def test_plane_error_bound():
    # hi + lo against q * s (s = da / g) in float64: within 2^-14 relative
    rng = np.random.default_rng(311)
    M, K = 64, 1024
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-12, 1, (M, K // 32))).repeat(32, axis=1).astype(np.float32)
    q, da, sa = oracle.quantize_q8_1(x)
    hi, lo, _, g = tcop_layout.encode(q, da, sa)
    perm = np.arange(K).reshape(-1, 4)[:, [0, 2, 1, 3]].reshape(-1)
    val = hi.view(np.float16).astype(np.float64) + lo.view(np.float16).astype(np.float64)
    exact = (q.astype(np.float64) * np.repeat(da.astype(np.float64) / np.repeat(g, 8, axis=1), 32, axis=1))[:, perm]
    assert (np.abs(val - exact) <= 2.0 ** -14 * np.abs(exact) + 1e-300).all()
