"""Pins for the oracle's 16-bit storage decode (CPU only).

``oracle.cache.bits_to_f64`` and ``oracle.fp8.bits16_to_f32`` turn the
fp16 / bf16 bit patterns the caches and the query rows hold into the values
every other oracle function works on (the pages store K/V as 16-bit
elements, or as one-byte codes of the 16-bit values: m.lsln.cn article
§6.1–6.2).  Both sides of every other CPU pin go through them, so they are
pinned here to conversions outside the oracle, over all 65,536 patterns:

* torch's own bf16 / fp16 → float64 conversion (a library routine);
* a decode written here from the IEEE 754 field definitions (sign,
  biased exponent, fraction; subnormals, infinities and NaN);
* values worked by hand.

A planted shift error and a planted byte swap must each fail the check.
"""
import math

import numpy as np
import pytest
import torch

from oracle import cache, fp8

ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)

# (exponent bits, fraction bits) of the two 16-bit formats: binary16, and
# bfloat16 = the upper half of binary32.
FIELDS = {"f16": (5, 10), "bf16": (8, 7)}


def ieee_decode(pattern: int, dtype: str) -> float:
    """Value of one 16-bit pattern from the IEEE 754 field definitions."""
    e_bits, f_bits = FIELDS[dtype]
    bias = (1 << (e_bits - 1)) - 1
    sign = -1.0 if pattern >> 15 else 1.0
    e = (pattern >> f_bits) & ((1 << e_bits) - 1)
    f = pattern & ((1 << f_bits) - 1)
    if e == (1 << e_bits) - 1:
        return sign * math.inf if f == 0 else math.nan
    if e == 0:                                     # zero and subnormals
        return sign * math.ldexp(f, 1 - bias - f_bits)
    return sign * math.ldexp((1 << f_bits) + f, e - bias - f_bits)


def torch_decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    t = torch.from_numpy(bits.view(np.int16).copy()).view(tdt)
    return t.double().numpy()


def mismatches(got: np.ndarray, want: np.ndarray) -> int:
    """Count of patterns whose values differ (NaN equals NaN; -0 != +0)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    both_nan = np.isnan(got) & np.isnan(want)
    same = (got == want) & (np.signbit(got) == np.signbit(want))
    return int(np.count_nonzero(~(same | both_nan)))


IEEE = {d: np.array([ieee_decode(int(p), d) for p in ALL]) for d in FIELDS}


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ieee_decode_agrees_with_torch(dtype):
    # the two independent references agree with each other first
    assert mismatches(IEEE[dtype], torch_decode(ALL, dtype)) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_bits_to_f64_all_patterns(dtype):
    got = cache.bits_to_f64(ALL, dtype)
    assert got.dtype == np.float64
    assert mismatches(got, torch_decode(ALL, dtype)) == 0
    assert mismatches(got, IEEE[dtype]) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_bits16_to_f32_all_patterns(dtype):
    got = fp8.bits16_to_f32(ALL, dtype)
    assert got.dtype == np.float32
    # every 16-bit value is exact in binary32
    assert mismatches(got, IEEE[dtype]) == 0


@pytest.mark.parametrize("dtype,pattern,value", [
    ("bf16", 0x3F80, 1.0),
    ("bf16", 0xC000, -2.0),
    ("bf16", 0x0001, 2.0 ** -133),          # smallest subnormal
    ("bf16", 0x0080, 2.0 ** -126),          # smallest normal
    ("bf16", 0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127),
    ("bf16", 0x4049, 3.140625),
    ("bf16", 0x8000, -0.0),
    ("bf16", 0xFF80, -math.inf),
    ("f16", 0x3C00, 1.0),
    ("f16", 0xC000, -2.0),
    ("f16", 0x0001, 2.0 ** -24),
    ("f16", 0x0400, 2.0 ** -14),
    ("f16", 0x7BFF, 65504.0),
    ("f16", 0x3555, 0.333251953125),
    ("f16", 0x7C00, math.inf),
])
def test_hand_worked_values(dtype, pattern, value):
    bits = np.array([pattern], dtype=np.uint16)
    for got in (cache.bits_to_f64(bits, dtype)[0], fp8.bits16_to_f32(bits, dtype)[0]):
        assert float(got) == value and math.copysign(1, got) == math.copysign(1, value)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nan_patterns_decode_to_nan(dtype):
    e_bits, f_bits = FIELDS[dtype]
    top = ((1 << e_bits) - 1) << f_bits
    nans = np.array([top | 1, top | (1 << (f_bits - 1)), 0x8000 | top | 3], dtype=np.uint16)
    assert np.isnan(cache.bits_to_f64(nans, dtype)).all()
    assert np.isnan(fp8.bits16_to_f32(nans, dtype)).all()


# -- planted mistakes: each must fail the all-pattern check -----------------

def _wrong_shift(bits, dtype):
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (b.astype(np.uint32) << 15).view(np.float32).astype(np.float64)
    return b.view(np.float16).astype(np.float64)


def _byte_swapped(bits, dtype):
    b = np.asarray(bits, dtype=np.uint16).byteswap()
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return b.view(np.float16).astype(np.float64)


@pytest.mark.parametrize("planted,dtypes", [(_wrong_shift, ["bf16"]),
                                            (_byte_swapped, ["f16", "bf16"])])
def test_planted_decode_mistakes_are_caught(monkeypatch, planted, dtypes):
    monkeypatch.setattr(cache, "bits_to_f64", planted)
    for dtype in dtypes:
        assert mismatches(cache.bits_to_f64(ALL, dtype), torch_decode(ALL, dtype)) > 1000
        # the cache's value path goes through the planted function too
        assert mismatches(cache.values(ALL, dtype), IEEE[dtype]) > 1000
