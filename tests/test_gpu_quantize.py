"""q8_1 prepass on the GPU vs the oracle: quants, scale bits and block sums
must agree bit for bit (web page "20 . r15 -- f32-accumulate mma probe (dead
end) + rank-1 term2 rescale", section 2.1)."""
import numpy as np
import pytest

import oracle
from q4_q8_int8_gb300 import synthetic
from tests.gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _check(x):
    mmq = require_gpu()
    qs, da, sa = mmq.quantize_q8_1(to_dev(x))
    q_ref, da_ref, sa_ref = oracle.quantize_q8_1(x)
    assert (qs.cpu().numpy() == q_ref).all()
    assert (da.cpu().numpy().view(np.int32) == da_ref.view(np.int32)).all()
    assert (sa.cpu().numpy() == sa_ref).all()
    assert mmq.status() == 0


@pytest.mark.parametrize("name", ["tiny", "q_proj", "down"])
def test_named_workloads(name):
    x, _, _ = synthetic.config_inputs(name)
    _check(x)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (5, 4096), (77, 4096), (2047, 256), (8192, 4096)])
def test_shapes_and_ragged_tails(M, K):
    _check(synthetic.activations(M, K, 500 + M, 0.01))


def test_edge_blocks():
    blocks = []
    blocks.append(np.zeros(32))                                 # zero
    blocks.append(np.full(32, -0.0))                            # negative zero
    blocks.append(np.full(32, 3.0))                             # constant
    blocks.append(np.full(32, -0.75))
    oh = np.zeros(32); oh[7] = -254.0; blocks.append(oh)        # one-hot
    t = np.zeros(32); t[:7] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5]; blocks.append(t)   # exact ties
    blocks.append(np.tile([1.5, -1.5], 16))                    # alternating
    s = np.zeros(32); s[0] = 1e-40; s[1] = -3e-41; blocks.append(s)   # subnormal, not flushed
    u = np.zeros(32); u[3] = 1.4e-45; blocks.append(u)          # scale underflows to 0
    b = np.linspace(-3e37, 3e37, 32); blocks.append(b)          # huge magnitudes
    rng = np.random.default_rng(0)
    r = rng.standard_normal(32) * 1e-30; blocks.append(r)       # tiny normals
    x = np.concatenate(blocks).astype(np.float32).reshape(1, -1)
    _check(x)
    _check(x.reshape(len(blocks), 32).copy())


def test_near_tie_quotients():
    # Activations whose quotients x/da sit at or within a few ulps of
    # half-integers, for many scales: exercises both the reciprocal fast path
    # and the exact-division fallback, which must agree with IEEE division.
    rng = np.random.default_rng(42)
    rows = []
    for _ in range(256):
        amax = np.float32(rng.uniform(0.5, 2.0) * 2.0 ** int(rng.integers(-60, 60)))
        d = np.float32(amax) / np.float32(127.0)
        x = np.empty(31, np.float32)
        for i in range(31):
            k = int(rng.integers(-126, 127))
            v = np.float32((k + 0.5) * float(d))           # nearest float to the tie point
            for _ in range(abs(int(rng.integers(-3, 4)))):
                v = np.nextafter(v, np.float32(np.inf if rng.integers(0, 2) else -np.inf))
            x[i] = v
        rows.append(np.concatenate([[amax], x]).astype(np.float32))
    _check(np.stack(rows))
