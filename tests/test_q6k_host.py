"""q6_K host-side pieces without a GPU: the product's C packer against the
tests' independent encoder and the oracle's decoder."""
import numpy as np

from oracle import q6k
from tests import q6k_layout


def test_pack_q6K_matches_independent_encoder():
    import q4_q8_int8_gb300 as mmq
    from q4_q8_int8_gb300 import build
    build.build()
    mmq.load_library()
    rng = np.random.default_rng(31)
    N, K = 7, 768
    q = rng.integers(-32, 32, (N, K)).astype(np.int8)
    sc = rng.integers(-128, 128, (N, K // 16)).astype(np.int8)
    d = rng.uniform(-1, 1, (N, K // 256)).astype(np.float16)
    out = mmq.pack_q6K(q, sc, d.view(np.uint16))
    assert out.shape == (N, K // 256, 210)
    assert (out == q6k_layout.encode(q, sc, d)).all()
    u = q6k.unpack_q6K(out, N, K)
    assert (u["q"] == q).all() and (u["sc"] == sc).all()
    assert mmq.mmq_q6K_bytes(N, K) == N * (K // 256) * 210
    assert mmq.mmq_q6K_dev_bytes(N, K) == N * (K // 256) * 224


def test_pack_q6K_rejects_out_of_range_quants():
    import ctypes
    import q4_q8_int8_gb300 as mmq
    mmq.load_library()
    q = np.zeros((1, 256), np.int8)
    q[0, 3] = 32                                        # above 31
    sc = np.zeros((1, 16), np.int8)
    d = np.zeros((1, 1), np.uint16)
    out = np.empty((1, 1, 210), np.uint8)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert mmq.mmq_pack_q6K(p(q), p(sc), p(d), 1, 256, p(out)) == mmq.MMQ_ERR_ARG
