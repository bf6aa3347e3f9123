"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins in test_oracle_pins.py catch every one of them.

Each mutant is oracle.c with one textual change, built into a temporary
library and swapped in for the real one while the pins run.
"""
import ctypes
import inspect
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "dmv_sign": ("const double dmv = -(dmin * (double)m[c8]);",
                 "const double dmv = (dmin * (double)m[c8]);"),
    "nibble_order": ("v[e] = h ? (byte >> 4) : (byte & 15);",
                     "v[e] = h ? (byte & 15) : (byte >> 4);"),
    "scale_high_bits": ("sc[c] = (uint8_t)((s[c + 4] & 15) | ((s[c - 4] >> 6) << 4));",
                        "sc[c] = (uint8_t)((s[c + 4] & 15) | ((s[c] >> 6) << 4));"),
    "min_low_nibble": ("m[c] = (uint8_t)((s[c + 4] >> 4) | ((s[c] >> 6) << 4));",
                       "m[c] = (uint8_t)((s[c + 4] & 15) | ((s[c] >> 6) << 4));"),
    "bankers_rounding": ("const float r = roundf(xb[k] / d);",
                         "const float r = rintf(xb[k] / d);"),
    "scale_divisor": ("const float d = amax / 127.0f;", "const float d = amax / 128.0f;"),
    "term2_missing_da": ("acc += a_d * dsv * (double)S + dmv * (a_d * a_s);",
                         "acc += a_d * dsv * (double)S + dmv * a_s;"),
    "dsv_uses_dmin": ("const double dsv = d * (double)sc[c8];",
                      "const double dsv = dmin * (double)sc[c8];"),
    "sa_off_by_one_chunk": ("const double a_s = (double)sa[i * nb + c];",
                            "const double a_s = (double)sa[i * nb + (c + 1) % nb];"),
    "fp16_bias": ("v = ldexp((double)(1024 + f), e - 25);",
                  "v = ldexp((double)(1024 + f), e - 24);"),
    "block_dot_index": ("s += (int32_t)q[i * K + c * QK + l] * (int32_t)v[j * K + c * QK + l];",
                        "s += (int32_t)q[i * K + c * QK + l] * (int32_t)v[j * K + c * QK + (l ^ 1)];"),
}


def _all_pin_calls():
    """(name, zero-argument callable) for every pin, parametrized ones expanded."""
    calls = []
    for cname, cls in inspect.getmembers(pins, inspect.isclass):
        if not cname.startswith("Test"):
            continue
        for mname, fn in inspect.getmembers(cls, inspect.isfunction):
            if not mname.startswith("test_"):
                continue
            kwargs_list = [{}]
            for mark in getattr(fn, "pytestmark", []):
                if mark.name == "parametrize":
                    kwargs_list = [{mark.args[0]: val} for val in mark.args[1]]
            for kw in kwargs_list:
                calls.append((f"{cname}.{mname}{kw or ''}",
                              lambda fn=fn, cls=cls, kw=kw: fn(cls(), **kw)))
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(mpath), "-o", str(lib_path), "-lm"], check=True)
    real = oracle._load()
    mutant = ctypes.CDLL(str(lib_path))
    for fname in ("oracle_quantize_q8_1", "oracle_unpack_q4K", "oracle_dequant_q4K",
                  "oracle_block_dots", "oracle_gemm", "oracle_gemm_sampled",
                  "oracle_dequant_dot"):
        f, g = getattr(mutant, fname), getattr(real, fname)
        f.argtypes, f.restype = g.argtypes, g.restype
    caught = []
    oracle._lib = mutant
    try:
        for pname, call in _all_pin_calls():
            try:
                call()
            except AssertionError:
                caught.append(pname)
    finally:
        oracle._lib = real
    assert caught, f"no pin caught mutant {name}"
