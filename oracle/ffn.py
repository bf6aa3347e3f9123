"""CPU oracle for the SwiGLU epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product library never calls it.

The fused neighbour of an MMQ GEMM in a SwiGLU FFN block (the next step
after the q8_1 prepass on web page "16 . r12 -- 16-chain warp tile +
ldmatrix", whose prepass/transpose work fed the following GEMM): with g, u
the gate and up projections of the same tokens, the down projection's input
is h = silu(g) * u, silu(g) = g * sigmoid(g) = g / (1 + exp(-g)), quantized
to q8_1 as the prepass would (oracle.quantize_q8_1).

Pins (tests/test_oracle_pins.py): silu(0) = 0, silu(ln 3) = 0.75 ln 3,
silu(x) - silu(-x) = x, silu of large |x| (x and 0).
"""
from __future__ import annotations

import numpy as np


def silu(g) -> np.ndarray:
    """g / (1 + exp(-g)) in float64 (overflow of exp gives 0 for g << 0)."""
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu(g, u) -> np.ndarray:
    """h = silu(g) * u in float64."""
    return silu(g) * np.asarray(u, np.float64)


def swiglu_bound(g, u, Eg, Eu) -> np.ndarray:
    """Bound on |h(g', u') - h(g, u)| for |g' - g| <= Eg, |u' - u| <= Eu, plus
    the f32 epilogue's own rounding (exp, add, divide, multiply: a few ulp):
    |silu'| <= 1.1 everywhere, so the first-order change is at most
    1.1 |u| Eg + |silu(g)| Eu, and the cross term 1.1 Eg Eu."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    h = swiglu(g, u)
    return 1.1 * np.abs(u) * Eg + (np.abs(silu(g)) + 1.1 * Eg) * Eu + 1e-6 * np.abs(h) + 1e-6
