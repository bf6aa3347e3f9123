"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol the header declares, packs q4_K exactly like the oracle reads
it, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import q4_q8_int8_gb300 as mmq
from q4_q8_int8_gb300 import build as mmq_build
from tests import q4k_layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mmq_build.build()
    return mmq.load_library()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(mmq_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(mmq.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_sizes(lib):
    assert mmq.mmq_q4K_bytes(4096, 4096) == 4096 * 16 * 144
    assert mmq.mmq_q4K_bytes(1, 100) == 0
    assert mmq.mmq_q8_1_bytes(2048, 4096) >= 2048 * 4096 + 2 * 2048 * 128 * 4
    assert mmq.mmq_q8_1_bytes(3, 48) == 0


def test_view_carves_aligned_planes(lib):
    M, K = 77, 512
    nbytes = mmq.mmq_q8_1_bytes(M, K)
    buf = (ctypes.c_uint8 * (nbytes + 256))()
    base = (ctypes.addressof(buf) + 255) & ~255
    v = mmq.mmq_q8_1_t()
    assert mmq.mmq_q8_1_view(base, M, K, v) == 0
    assert v.qs == base and v.da % 256 == 0 and v.sa % 256 == 0
    assert v.da >= v.qs + M * K and v.sa >= v.da + M * (K // 32) * 4
    assert v.sa + M * (K // 32) * 4 <= base + nbytes
    assert mmq.mmq_q8_1_view(base + 16, M, K, v) == mmq.MMQ_ERR_ALIGN


def _random_fields(rng, N, K):
    return dict(v=rng.integers(0, 16, (N, K), dtype=np.uint8),
                sc=rng.integers(0, 64, (N, K // 32), dtype=np.uint8),
                m=rng.integers(0, 64, (N, K // 32), dtype=np.uint8),
                d=rng.uniform(1e-3, 1e-2, (N, K // 256)).astype(np.float16),
                dmin=rng.uniform(1e-3, 1e-2, (N, K // 256)).astype(np.float16))


def test_packer_matches_oracle_unpack(lib):
    rng = np.random.default_rng(21)
    N, K = 37, 1024
    f = _random_fields(rng, N, K)
    blk = mmq.pack_q4K(f["v"], f["sc"], f["m"], f["d"].view(np.uint16), f["dmin"].view(np.uint16))
    o = oracle.unpack_q4K(blk, N, K)
    assert (o["v"] == f["v"]).all() and (o["sc"] == f["sc"]).all() and (o["m"] == f["m"]).all()
    assert (o["d"] == f["d"].astype(np.float64)).all()
    assert (o["dmin"] == f["dmin"].astype(np.float64)).all()
    # and byte-identical to the test-side encoder
    assert (blk == q4k_layout.encode(f["d"], f["dmin"], f["sc"], f["m"], f["v"])).all()


def test_packer_hand_bytes(lib):
    g = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "q4k_scale_bytes.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split(":")
            g[k.strip()] = [int(t) for t in v.split()]
    N, K = 1, 256
    blk = mmq.pack_q4K(np.zeros((N, K), np.uint8), np.array([g["sc"]], np.uint8),
                       np.array([g["m"]], np.uint8), np.zeros((1, 1), np.uint16),
                       np.zeros((1, 1), np.uint16))
    assert list(blk[0, 0, 4:16]) == g["bytes"]


@pytest.mark.parametrize("field,bad", [("v", 16), ("sc", 64), ("m", 255)])
def test_packer_rejects_out_of_range(lib, field, bad):
    rng = np.random.default_rng(1)
    f = _random_fields(rng, 2, 256)
    f[field][0, 0] = bad
    with pytest.raises(mmq.MMQError) as e:
        mmq.pack_q4K(f["v"], f["sc"], f["m"], f["d"].view(np.uint16), f["dmin"].view(np.uint16))
    assert e.value.code == mmq.MMQ_ERR_ARG


def test_argument_errors_before_device(lib):
    Q = mmq.mmq_q8_1_t
    good = Q(0x10000, 0x20000, 0x30000)
    w, C = ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000)
    # null pointers
    assert mmq.mmq_q4K_gemm(Q(0, 0x20000, 0x30000), w, C, 1, 4, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm(good, None, C, 1, 4, 256, None) == mmq.MMQ_ERR_ARG
    # sizes
    assert mmq.mmq_q4K_gemm(good, w, C, 0, 4, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm(good, w, C, 1, 4, 300, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm(good, w, C, 1, 6, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_path(good, w, C, 65, 4, 256, mmq.MMQ_PATH_SMALL_M, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_path(good, w, C, 1, 4, 256, 9, None) == mmq.MMQ_ERR_ARG
    # the launch-count query refuses what the GEMM refuses, before the device
    assert mmq.mmq_q4K_gemm_launches(0, 4, 256, mmq.MMQ_PATH_AUTO) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_launches(1, 6, 256, mmq.MMQ_PATH_AUTO) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_launches(1, 4, 300, mmq.MMQ_PATH_AUTO) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_launches(65, 4, 256, mmq.MMQ_PATH_SMALL_M) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_launches(1, 4, 256, 9) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_block_dots(good, w, C, 65, 4, 256, mmq.MMQ_PATH_SMALL_M, None) == mmq.MMQ_ERR_ARG
    for retired in (4, 5):   # two retired tensor-core paths are refused like unknown values
        assert mmq.mmq_q4K_block_dots(good, w, C, 1, 4, 256, retired, None) == mmq.MMQ_ERR_ARG
        assert mmq.mmq_q4K_gemm_path(good, w, C, 128, 4, 256, retired, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_scaled_block_dots(good, w, None, 1, 4, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_scaled_block_dots(good, w, C, 1, 6, 256, None) == mmq.MMQ_ERR_ARG
    # the split hook takes 0, 1, 2, 4 only
    for bad in (-1, 3, 8):
        assert mmq.mmq_debug_force_gemv_split(bad) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_debug_force_gemv_split(0) == mmq.MMQ_OK
    # alignment
    assert mmq.mmq_q4K_gemm(Q(0x10004, 0x20000, 0x30000), w, C, 1, 4, 256, None) == mmq.MMQ_ERR_ALIGN
    assert mmq.mmq_q4K_gemm(good, ctypes.c_void_p(0x40008), C, 1, 4, 256, None) == mmq.MMQ_ERR_ALIGN
    assert mmq.mmq_quantize_q8_1(ctypes.c_void_p(0x1004), 1, 32, good, None) == mmq.MMQ_ERR_ALIGN
    assert mmq.mmq_quantize_q8_1(ctypes.c_void_p(0x1000), 1, 40, good, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_quantize_q8_1(None, 1, 32, good, None) == mmq.MMQ_ERR_ARG
    # fused q8_1 output: N % 32, aligned output planes (C may be null at any M)
    assert mmq.mmq_q4K_gemm_q8_1(good, w, C, good, 128, 48, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_q8_1(good, w, C, Q(0, 0x20000, 0x30000), 128, 64, 256, None) == mmq.MMQ_ERR_ARG
    assert mmq.mmq_q4K_gemm_q8_1(good, w, C, Q(0x10000, 0x20004, 0x30000), 128, 64, 256, None) == mmq.MMQ_ERR_ALIGN


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert mmq.strerror(code) and mmq.strerror(code) != "unknown error code"
    assert mmq.strerror(-99) == "unknown error code"
