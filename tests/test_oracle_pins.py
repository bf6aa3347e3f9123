"""Pins for the CPU oracle: closed forms, hand-worked examples, invariants,
library reductions and brute force -- never the oracle's own formula retyped.

Sources: "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2
rescale" section 2.1 (formats, S, the two-term rescale) and 2.3 (|S| bound);
"21 . r16 -- Narrow kernel gets the rank-1 fold" section 2.1 (fold).
"""
import os

import numpy as np
import pytest

import oracle
from tests import q4k_layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _block(x):
    return np.asarray(x, np.float32).reshape(1, 32)


# ----------------------------------------------------------------- O1 quantize
class TestQuantize:
    def test_constant_positive(self):
        q, da, sa = oracle.quantize_q8_1(np.full((1, 32), 3.0, np.float32))
        assert (q == 127).all() and sa[0, 0] == 4064
        assert da[0, 0] == np.float32(3.0) / np.float32(127.0)

    def test_constant_negative(self):
        q, da, sa = oracle.quantize_q8_1(np.full((1, 32), -0.75, np.float32))
        assert (q == -127).all() and sa[0, 0] == -4064

    @pytest.mark.parametrize("z", [0.0, -0.0])
    def test_zero_block(self, z):
        q, da, sa = oracle.quantize_q8_1(np.full((1, 32), z, np.float32))
        assert (q == 0).all() and sa[0, 0] == 0 and da[0, 0] == 0.0
        assert not np.signbit(da[0, 0])

    def test_one_hot(self):
        x = np.zeros(32, np.float32)
        x[5] = 254.0                      # da = 254/127 = 2 exactly
        q, da, sa = oracle.quantize_q8_1(_block(x))
        expect = np.zeros(32, np.int8)
        expect[5] = 127
        assert (q[0] == expect).all() and sa[0, 0] == 127 and da[0, 0] == 2.0

    def test_alternating(self):
        x = np.array([1.5, -1.5] * 16, np.float32)
        q, da, sa = oracle.quantize_q8_1(_block(x))
        assert sa[0, 0] == 0 and (np.abs(q) == 127).all()

    def test_ties_round_half_away_from_zero(self):
        # amax = 127 -> da = 1 exactly, so x/da = x and the x.5 values are
        # exact ties; round-half-away-from-zero gives 3, -3, 1, -1, 2, -2.
        x = np.zeros(32, np.float32)
        x[:7] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5]
        q, da, sa = oracle.quantize_q8_1(_block(x))
        assert da[0, 0] == 1.0
        assert list(q[0, :7]) == [127, 3, -3, 1, -1, 2, -2]
        assert sa[0, 0] == 127 + 3 - 3 + 1 - 1 + 2 - 2

    def test_subnormal_input_not_flushed(self):
        x = np.zeros(32, np.float32)
        x[0] = np.float32(1e-40)          # subnormal amax, da is subnormal too
        q, da, sa = oracle.quantize_q8_1(_block(x))
        assert da[0, 0] > 0 and q[0, 0] == 127 and sa[0, 0] == 127

    def test_scale_underflow_gives_zero_block(self):
        x = np.zeros(32, np.float32)
        x[3] = np.float32(1.4e-45)        # smallest subnormal: amax/127 -> 0
        q, da, sa = oracle.quantize_q8_1(_block(x))
        assert da[0, 0] == 0.0 and (q == 0).all() and sa[0, 0] == 0

    def test_invariants_random(self):
        rng = np.random.default_rng(7)
        x = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
        q, da, sa = oracle.quantize_q8_1(x)
        qb = q.reshape(64, 16, 32).astype(np.int64)
        assert (np.abs(qb) <= 127).all()
        assert (np.abs(qb).max(axis=2) == 127).all()            # amax element -> 127
        assert (qb.sum(axis=2) == sa).all()                      # sa = in-block sum
        xb = x.reshape(64, 16, 32).astype(np.float64)
        dab = da.astype(np.float64)[:, :, None]
        err = np.abs(xb - dab * qb)
        assert (err <= dab * (0.5 + 128 * 2.0 ** -24)).all()    # half a step (+ f32 quotient rounding)
        amax = np.abs(xb).max(axis=2)
        assert np.allclose(da, amax / 127.0, rtol=2 ** -23, atol=0)


# ------------------------------------------------------------------- O2 unpack
def _read_golden_scales():
    vals = {}
    with open(os.path.join(GOLDEN, "q4k_scale_bytes.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split(":")
            vals[k.strip()] = [int(t) for t in v.split()]
    return vals


class TestUnpack:
    def test_hand_packed_scale_bytes(self):
        g = _read_golden_scales()
        blk = np.zeros((1, 1, 144), np.uint8)
        blk[0, 0, 4:16] = g["bytes"]
        out = oracle.unpack_q4K(blk, 1, 256)
        assert list(out["sc"][0]) == g["sc"]
        assert list(out["m"][0]) == g["m"]

    def test_fp16_decode(self):
        with open(os.path.join(GOLDEN, "fp16_bits.txt")) as f:
            rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
        for lo, hi, val in rows:
            blk = np.zeros((1, 1, 144), np.uint8)
            blk[0, 0, 0] = int(lo, 16)
            blk[0, 0, 1] = int(hi, 16)
            blk[0, 0, 2] = int(lo, 16)
            blk[0, 0, 3] = int(hi, 16)
            out = oracle.unpack_q4K(blk, 1, 256)
            assert out["d"][0, 0] == float(val) and out["dmin"][0, 0] == float(val)

    def test_nibble_order(self):
        blk = np.zeros((1, 1, 144), np.uint8)
        for p in range(4):
            for l in range(32):
                blk[0, 0, 16 + 32 * p + l] = ((l + p) % 16) | (((3 * l + p) % 16) << 4)
        v = oracle.unpack_q4K(blk, 1, 256)["v"][0]
        for p in range(4):
            for l in range(32):
                assert v[64 * p + l] == (l + p) % 16              # low nibble: sub-block 2p
                assert v[64 * p + 32 + l] == (3 * l + p) % 16     # high nibble: sub-block 2p+1

    def test_random_bytes_agree_with_numpy_reading(self):
        rng = np.random.default_rng(3)
        N, K = 9, 768
        blk = rng.integers(0, 256, (N, K // 256, 144), dtype=np.uint8)
        blk[:, :, 1] &= 0x3B                                      # keep d, dmin finite
        blk[:, :, 3] &= 0x3B
        o = oracle.unpack_q4K(blk, N, K)
        r = q4k_layout.decode(blk, N, K)
        for k in ("d", "dmin", "sc", "m", "v"):
            assert (np.asarray(o[k], np.float64) == np.asarray(r[k], np.float64)).all(), k

    def test_encode_decode_round_trip(self):
        rng = np.random.default_rng(4)
        N, K = 5, 512
        f = dict(d=rng.uniform(1e-3, 1e-2, (N, 2)).astype(np.float16),
                 dmin=rng.uniform(1e-3, 1e-2, (N, 2)).astype(np.float16),
                 sc=rng.integers(0, 64, (N, 16)), m=rng.integers(0, 64, (N, 16)),
                 v=rng.integers(0, 16, (N, K)))
        o = oracle.unpack_q4K(q4k_layout.encode(**f), N, K)
        assert (o["d"] == f["d"].astype(np.float64)).all()
        assert (o["dmin"] == f["dmin"].astype(np.float64)).all()
        assert (o["sc"] == f["sc"]).all() and (o["m"] == f["m"]).all() and (o["v"] == f["v"]).all()

    def test_dequant_closed_form(self):
        # d = 0.5, dmin = 0.25, sc = 3, m = 5, v = 7 everywhere: w = 0.5*3*7 - 0.25*5 = 9.25
        N, K = 2, 256
        blk = q4k_layout.encode(np.full((N, 1), 0.5), np.full((N, 1), 0.25),
                                np.full((N, 8), 3), np.full((N, 8), 5), np.full((N, K), 7))
        assert (oracle.dequant_q4K(blk, N, K) == 9.25).all()


# ------------------------------------------------------------- O3 block dots
class TestBlockDots:
    def test_against_numpy_einsum(self):
        rng = np.random.default_rng(5)
        M, N, K = 6, 7, 512
        q = rng.integers(-127, 128, (M, K), dtype=np.int8)
        blk = rng.integers(0, 256, (N, K // 256, 144), dtype=np.uint8)
        v = q4k_layout.decode(blk, N, K)["v"]
        ref = np.einsum("ick,jck->ijc", q.astype(np.int64).reshape(M, K // 32, 32),
                        v.astype(np.int64).reshape(N, K // 32, 32))
        assert (oracle.block_dots(q, blk, N) == ref).all()

    @pytest.mark.parametrize("sign", [1, -1])
    def test_extreme_bound(self, sign):
        # |S| <= 32*127*15 = 60960, reached with all-extreme blocks
        q = np.full((1, 256), 127 * sign, np.int8)
        blk = q4k_layout.encode([[1.0]], [[0.0]], np.ones((1, 8)), np.zeros((1, 8)), np.full((1, 256), 15))
        S = oracle.block_dots(q, blk, 1)
        assert (S == sign * 60960).all()


# ------------------------------------------------------- O4 GEMM, O5, O6
def _one_block_weights(d, dmin, sc, m, v, K=256):
    nsb = K // 256
    return q4k_layout.encode(np.full((1, nsb), d), np.full((1, nsb), dmin),
                             np.full((1, K // 32), sc), np.full((1, K // 32), m),
                             np.broadcast_to(np.asarray(v), (1, K)))


class TestGemmExamples:
    def test_E1(self):
        # x = 1, v = 1, sc = 1, m = 0, d = 1, dmin = 0: every chunk has
        # da = fl(1/127), q = 127, sa = S = 4064, so C = 8 * 4064 * fl(1/127).
        q, da, sa = oracle.quantize_q8_1(np.ones((1, 256), np.float32))
        C, C64, T = oracle.gemm(q, da, sa, _one_block_weights(1.0, 0.0, 1, 0, 1), 1, want_c64=True)
        expect = 32512.0 * float(np.float32(1.0) / np.float32(127.0))
        assert C64[0, 0] == expect and C[0, 0] == np.float32(expect)
        assert abs(C[0, 0] - 256.0) < 1e-4

    def test_E2_terms_cancel_exactly(self):
        # m = 1, dmin = 1 on top of E1: w = 1*1*1 - 1*1 = 0, term1 and term2
        # cancel exactly in every chunk.
        q, da, sa = oracle.quantize_q8_1(np.ones((1, 256), np.float32))
        C, C64, T = oracle.gemm(q, da, sa, _one_block_weights(1.0, 1.0, 1, 1, 1), 1, want_c64=True)
        assert C64[0, 0] == 0.0 and T[0, 0] == 0.0

    def test_E3_zero_block_sum_kills_term2(self):
        x = np.tile(np.array([1.0, -1.0], np.float32), 128).reshape(1, 256)
        v = np.tile(np.array([1, 0]), 128)                        # picks the +1 lanes
        q, da, sa = oracle.quantize_q8_1(x)
        assert (sa == 0).all()
        Ca, _, _ = oracle.gemm(q, da, sa, _one_block_weights(0.5, 1.0, 3, 7, v), 1)
        Cb, _, _ = oracle.gemm(q, da, sa, _one_block_weights(0.5, 0.0, 3, 0, v), 1)
        expect = 8 * 16 * 127 * float(np.float32(1.0) / np.float32(127.0)) * 0.5 * 3
        assert Ca[0, 0] == Cb[0, 0] == np.float32(expect)

    def test_E4_v0_m0_gives_zero(self):
        rng = np.random.default_rng(9)
        M, N, K = 4, 5, 512
        x = rng.standard_normal((M, K)).astype(np.float32)
        blk = q4k_layout.encode(rng.uniform(1e-3, 1, (N, 2)), rng.uniform(1e-3, 1, (N, 2)),
                                rng.integers(0, 64, (N, 16)), np.zeros((N, 16)), np.zeros((N, K)))
        q, da, sa = oracle.quantize_q8_1(x)
        C, _, T = oracle.gemm(q, da, sa, blk, N)
        assert (C == 0).all() and (T == 0).all()

    def test_E5_reduces_to_integer_matmul(self):
        # d = sc = 1, m = dmin = 0 and integer x with amax = 127 in each block:
        # da = 1 exactly, q = x, so C = x @ v^T exactly (|C| < 2^24).
        rng = np.random.default_rng(11)
        M, N, K = 6, 5, 512
        x = rng.integers(-127, 128, (M, K)).astype(np.float32)
        x.reshape(M, K // 32, 32)[:, :, 0] = 127.0
        v = rng.integers(0, 16, (N, K))
        blk = q4k_layout.encode(np.ones((N, 2)), np.zeros((N, 2)), np.ones((N, 16)),
                                np.zeros((N, 16)), v)
        q, da, sa = oracle.quantize_q8_1(x)
        assert (da == 1.0).all() and (q == x).all()
        C, _, _ = oracle.gemm(q, da, sa, blk, N)
        assert (C.astype(np.int64) == x.astype(np.int64) @ v.T).all()

    def test_identity_with_brute_force(self):
        # blockwise two-term result == dot(dequant(A), dequant(B))
        rng = np.random.default_rng(13)
        M, N, K = 5, 7, 512
        x = (rng.standard_normal((M, K)) * 3).astype(np.float32)
        from q4_q8_int8_gb300 import synthetic
        blk = synthetic.q4K_weights(N, K, 77)
        q, da, sa = oracle.quantize_q8_1(x)
        C, C64, T = oracle.gemm(q, da, sa, blk, N, want_c64=True)
        D = oracle.dequant_dot(q, da, blk, N)
        assert (np.abs(C64 - D) <= 1e-12 * T).all()
        # D again from numpy: test-side decode and a float64 matmul
        f = q4k_layout.decode(blk, N, K)
        w = (f["d"].repeat(256, 1) * f["sc"].repeat(32, 1) * f["v"]
             - f["dmin"].repeat(256, 1) * f["m"].repeat(32, 1))
        a = da.astype(np.float64).repeat(32, 1) * q
        assert np.allclose(a @ w.T, D, rtol=1e-12, atol=1e-12 * T.max())
        assert np.allclose(np.abs(a) @ np.abs(w).T, T, rtol=1e-12, atol=0)
        assert (np.abs(D) <= T * (1 + 1e-12)).all()

    def test_sampled_equals_full(self):
        rng = np.random.default_rng(17)
        M, N, K = 9, 11, 768
        x = rng.standard_normal((M, K)).astype(np.float32)
        from q4_q8_int8_gb300 import synthetic
        blk = synthetic.q4K_weights(N, K, 78)
        q, da, sa = oracle.quantize_q8_1(x)
        C, C64, T = oracle.gemm(q, da, sa, blk, N, want_c64=True)
        rows = rng.integers(0, M, 40)
        cols = rng.integers(0, N, 40)
        Cs, C64s, Ts = oracle.gemm_sampled(q, da, sa, blk, N, rows, cols)
        assert (Cs == C[rows, cols]).all() and (C64s == C64[rows, cols]).all() and (Ts == T[rows, cols]).all()


# ---------------------------------------------------------------------------
# Control path (dequantize to fp16, dense GEMM): oracle.dense
# ---------------------------------------------------------------------------
def _golden_dequant_rows():
    rows = []
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "dequant_f16_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        rows.append((int(f[0], 16), int(f[1], 16), int(f[2]), int(f[3]), int(f[4]), float(f[5])))
    return rows


def test_dense_dequant_golden_values():
    from oracle import dense
    rows = _golden_dequant_rows()
    assert len(rows) >= 5
    N, K = len(rows), 256
    d = np.array([[np.array(r[0], np.uint16).view(np.float16)] for r in rows])
    dmin = np.array([[np.array(r[1], np.uint16).view(np.float16)] for r in rows])
    sc = np.array([[r[2]] * 8 for r in rows])
    m = np.array([[r[3]] * 8 for r in rows])
    v = np.array([[r[4]] * K for r in rows])
    blk = q4k_layout.encode(d, dmin, sc, m, v)
    w = dense.dequantize_q4K_f16(blk, N, K)
    assert w.dtype == np.float16
    for j, r in enumerate(rows):
        assert (w[j] == np.float16(r[5])).all(), (r, w[j][:4])


def test_dense_dequant_matches_fraction_definition():
    # random fields: fp16(float32-rounded exact difference) computed with Fractions
    from fractions import Fraction
    from oracle import dense
    rng = np.random.default_rng(11)
    N, K = 6, 512
    d = rng.uniform(1e-3, 4.0, (N, 2)).astype(np.float16)
    dmin = rng.uniform(1e-3, 4.0, (N, 2)).astype(np.float16)
    sc = rng.integers(0, 64, (N, 16))
    m = rng.integers(0, 64, (N, 16))
    v = rng.integers(0, 16, (N, K))
    blk = q4k_layout.encode(d, dmin, sc, m, v)
    w = dense.dequantize_q4K_f16(blk, N, K)
    for j in range(N):
        for k in range(0, K, 7):
            sb, c = k // 256, k // 32
            exact = (Fraction(float(d[j, sb])) * int(sc[j, c]) * int(v[j, k])
                     - Fraction(float(dmin[j, sb])) * int(m[j, c]))
            f32 = np.float32(float(exact))      # exact fits a double; one rounding to float32
            assert w[j, k] == np.float16(f32), (j, k, exact)


def test_dense_gemm_integer_matrices_exact():
    # small integers are exact in fp16 and every sum is exact in float64
    from oracle import dense
    rng = np.random.default_rng(12)
    A = rng.integers(-8, 9, (5, 64))
    B = rng.integers(-8, 9, (3, 64))
    C, T = dense.gemm_f16(A.astype(np.float16), B.astype(np.float16))
    assert C.shape == (5, 3)
    assert (C == A @ B.T).all()
    assert (T == np.abs(A) @ np.abs(B).T).all()
    Cs, Ts = dense.gemm_f16_sampled(A.astype(np.float16), B.astype(np.float16), [4, 0, 2], [0, 2, 1])
    assert (Cs == np.array([C[4, 0], C[0, 2], C[2, 1]])).all()
    assert (Ts == np.array([T[4, 0], T[0, 2], T[2, 1]])).all()


# ---------------------------------------------------------------------------
# SwiGLU epilogue: oracle.ffn
# ---------------------------------------------------------------------------
def test_ffn_silu_closed_forms():
    from oracle import ffn
    assert ffn.silu(0.0) == 0.0
    assert abs(ffn.silu(np.log(3.0)) - 0.75 * np.log(3.0)) < 1e-15      # sigmoid(ln 3) = 3/4
    x = np.linspace(-20, 20, 81)
    assert np.allclose(ffn.silu(x) - ffn.silu(-x), x, rtol=0, atol=1e-13)  # x s(x) - (-x) s(-x) = x
    assert abs(ffn.silu(40.0) - 40.0) < 1e-15 * 40 * 1e3                  # sigmoid(40) = 1 - 4e-18
    assert ffn.silu(-800.0) == 0.0 or abs(ffn.silu(-800.0)) < 1e-300
    g = np.array([1.0, -2.0]); u = np.array([3.0, 0.5])
    assert np.allclose(ffn.swiglu(g, u), [3.0 / (1 + np.exp(-1.0)), 0.5 * -2.0 / (1 + np.exp(2.0))])


def test_ffn_swiglu_bound_lipschitz_constant():
    # the bound uses |silu'| <= 1.1: silu'(g) = s(g) (1 + g (1 - s(g))), s the
    # logistic function, peaks at 1.0998... near g = 2.40 and tends to 1 and 0
    from oracle import ffn
    g = np.linspace(-60.0, 60.0, 1_200_001)
    sg = 1.0 / (1.0 + np.exp(-g))
    d = sg * (1.0 + g * (1.0 - sg))
    assert d.max() < 1.1 and d.max() > 1.099
    assert d.min() > -0.1 - 1e-12 and d.min() < -0.099   # the negative lobe near g = -2.40
    # the closed-form derivative agrees with a difference quotient of ffn.silu
    h = 1e-6
    gs = np.linspace(-30.0, 30.0, 6001)
    fd = (ffn.silu(gs + h) - ffn.silu(gs - h)) / (2 * h)
    sgs = 1.0 / (1.0 + np.exp(-gs))
    assert np.allclose(fd, sgs * (1.0 + gs * (1.0 - sgs)), rtol=0, atol=1e-8)


def test_ffn_swiglu_bound_holds_for_perturbed_inputs():
    # |h(g', u') - h(g, u)| <= bound for every |g' - g| <= Eg, |u' - u| <= Eu
    # (the corners of the box and random points inside it), without the
    # rounding allowance: the Lipschitz part of the bound alone must hold
    from oracle import ffn
    rng = np.random.default_rng(901)
    n = 200_000
    g = rng.normal(0, 4, n) * np.where(rng.random(n) < 0.1, 10.0, 1.0)
    u = rng.normal(0, 4, n)
    Eg = np.abs(g) * 10.0 ** rng.uniform(-6, -1, n) + 1e-6
    Eu = np.abs(u) * 10.0 ** rng.uniform(-6, -1, n) + 1e-6
    h = ffn.swiglu(g, u)
    lip = 1.1 * np.abs(u) * Eg + (np.abs(ffn.silu(g)) + 1.1 * Eg) * Eu
    assert (ffn.swiglu_bound(g, u, Eg, Eu) >= lip).all()
    for sgn_g, sgn_u in ((1, 1), (1, -1), (-1, 1), (-1, -1)):
        dh = np.abs(ffn.swiglu(g + sgn_g * Eg, u + sgn_u * Eu) - h)
        assert (dh <= lip * (1 + 1e-12) + 1e-300).all()
    tg, tu = rng.uniform(-1, 1, n), rng.uniform(-1, 1, n)
    dh = np.abs(ffn.swiglu(g + tg * Eg, u + tu * Eu) - h)
    assert (dh <= lip * (1 + 1e-12) + 1e-300).all()
    # the constant is needed: with |silu'| taken as 1 the bound fails somewhere
    lip1 = np.abs(u) * Eg + (np.abs(ffn.silu(g)) + Eg) * Eu
    worst = np.abs(ffn.swiglu(g + Eg, u) - h) - lip1
    assert worst.max() > 0


def test_ffn_swiglu_bound_covers_f32_evaluation():
    # the rounding allowance 1e-6 |h| + 1e-6 covers h evaluated in f32 the way
    # the epilogue does it (exp, add, divide, multiply), against float64
    from oracle import ffn
    rng = np.random.default_rng(902)
    g = rng.normal(0, 6, 500_000).astype(np.float32)
    u = rng.normal(0, 6, 500_000).astype(np.float32)
    with np.errstate(over="ignore"):
        h32 = (g / (np.float32(1) + np.exp(-g))) * u
    h64 = ffn.swiglu(g.astype(np.float64), u.astype(np.float64))
    assert (np.abs(h32.astype(np.float64) - h64) <= 1e-6 * np.abs(h64) + 1e-6).all()
    assert (ffn.swiglu_bound(g, u, 0.0, 0.0) == 1e-6 * np.abs(h64) + 1e-6).all()


# ---------------------------------------------------------------------------
# q6_K x q8_1: oracle.q6k
# ---------------------------------------------------------------------------
def _q6k_golden():
    vals = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "q6k_bytes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            f = line.split()
            vals[int(f[0])] = int(f[1], 16)
    return vals


def _q6k_golden_fields():
    e = np.arange(256)
    q = (e % 64 - 32)[None, :]
    sc = (np.arange(16) - 8)[None, :]
    return q, sc, np.ones((1, 1))


def test_q6k_hand_packed_bytes():
    from oracle import q6k
    from tests import q6k_layout
    q, sc, d = _q6k_golden_fields()
    blk = q6k_layout.encode(q, sc, d).reshape(-1)
    for off, v in _q6k_golden().items():
        assert blk[off] == v, (off, hex(blk[off]), hex(v))
    u = q6k.unpack_q6K(blk, 1, 256)
    assert (u["q"] == q).all() and (u["sc"] == sc).all() and (u["d"] == 1.0).all()


def test_q6k_round_trip_random_fields():
    from oracle import q6k
    from tests import q6k_layout
    rng = np.random.default_rng(21)
    N, K = 5, 768
    q = rng.integers(-32, 32, (N, K))
    sc = rng.integers(-128, 128, (N, K // 16))
    d = rng.uniform(-2, 2, (N, K // 256)).astype(np.float16)
    u = q6k.unpack_q6K(q6k_layout.encode(q, sc, d), N, K)
    assert (u["q"] == q).all() and (u["sc"] == sc).all() and (u["d"] == d.astype(np.float64)).all()


def test_q6k_block_dots_brute_force():
    from oracle import q6k
    from tests import q6k_layout
    rng = np.random.default_rng(22)
    M, N, K = 3, 4, 512
    qa = rng.integers(-127, 128, (M, K)).astype(np.int8)
    q = rng.integers(-32, 32, (N, K))
    blk = q6k_layout.encode(q, rng.integers(-128, 128, (N, K // 16)), np.ones((N, 2)))
    S = q6k.block_dots16(qa, blk, N)
    for i in range(M):
        for j in range(N):
            for s in range(K // 16):
                assert S[i, j, s] == sum(int(qa[i, 16 * s + k]) * int(q[j, 16 * s + k]) for k in range(16))


def test_q6k_worked_examples():
    from oracle import q6k
    from tests import q6k_layout
    M, N, K = 1, 3, 256
    # x = 1 everywhere: q8_1 gives da = fl32(1/127), q = 127 in every block
    x = np.ones((M, K), np.float32)
    qa, da, _ = oracle.quantize_q8_1(x)
    assert (qa == 127).all() and (da == np.float32(1.0) / np.float32(127.0)).all()
    q = np.array([[31] * K, [0] * K, [-32] * K])          # stored u = 63, 32, 0
    sc = np.array([[1] * 16, [5] * 16, [-128] * 16])
    blk = q6k_layout.encode(q, sc, np.array([[1.0], [3.0], [0.5]]))
    C, C64, T = q6k.gemm(qa, da, blk, N)
    da64 = float(da[0, 0])
    assert C64[0, 0] == 256 * 127 * 31 * da64                # 8 blocks x 2 halves x 16 x 127 x 31 x 1
    assert C64[0, 1] == 0.0                                  # q = 0: no minimum term to leave behind
    assert C64[0, 2] == 256 * 127 * (-32) * (-128) * 0.5 * da64
    assert (T[0] == np.abs(C64[0])).all()                    # all products of one sign per row


def test_q6k_gemm_equals_dequantized_dot():
    from oracle import q6k
    from tests import q6k_layout
    rng = np.random.default_rng(23)
    M, N, K = 4, 5, 512
    x = rng.standard_normal((M, K)).astype(np.float32)
    qa, da, _ = oracle.quantize_q8_1(x)
    blk = q6k_layout.encode(rng.integers(-32, 32, (N, K)), rng.integers(-128, 128, (N, K // 16)),
                            rng.uniform(1e-3, 1e-2, (N, 2)))
    C, C64, T = q6k.gemm(qa, da, blk, N)
    D = q6k.dequant_dot(qa, da, blk, N)
    assert np.allclose(C64, D, rtol=1e-12, atol=1e-12 * np.abs(T).max())
    Cs, C64s, Ts = q6k.gemm(qa, da, blk, N, rows=[3, 0, 2], cols=[1, 4, 0])
    assert np.allclose(C64s, C64[[3, 0, 2], [1, 4, 0]], rtol=1e-14, atol=0)
    assert np.allclose(Ts, T[[3, 0, 2], [1, 4, 0]], rtol=1e-14, atol=0)
