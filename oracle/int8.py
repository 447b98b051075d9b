"""Symmetric 8-bit integer KV codes: encode / decode.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[P3] §6 names INT8 beside FP8 as a one-byte element type that halves the KV
cache, and §6.1 gives the rule for every 8-bit cache: the value is divided by
a scale before it is stored and multiplied by it on read.  The page gives no
integer format, so the plainest reading is taken:

* the code is a two's-complement int8 (stored as its byte);
* code = x / scale rounded to the nearest integer, ties to even, and
  saturated to the int8 range [-128, 127] (a value beyond the range is cut
  off, as §6.1 says of an unfit scale);
* a NaN input stores 0 (the integer format has no NaN);
* read value = code * scale.

As for FP8, the quotient x / scale is taken in IEEE float32: the device
computes it in float32 and the integer code must agree bit for bit.
"""

from __future__ import annotations

import math
from functools import lru_cache

import numpy as np

from .fp8 import bits16_to_f32

QMIN, QMAX = -128, 127


def encode_value(x: float) -> int:
    """Code (as a signed integer) of one already-divided value."""
    if math.isnan(x):
        return 0
    if math.isinf(x):
        return QMAX if x > 0 else QMIN
    r = round(x)                  # Python rounds half to even
    return max(QMIN, min(QMAX, int(r)))


def code_to_int(code: int) -> int:
    """Two's-complement value of a stored byte."""
    code &= 0xFF
    return code - 256 if code & 0x80 else code


def decode(codes: np.ndarray) -> np.ndarray:
    """float64 integer values of stored bytes (uint8 bit patterns)."""
    return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)


def quantize(values_f32: np.ndarray, scale: float) -> np.ndarray:
    """Stored byte of ``value / scale`` for every element ([P3] §6.1)."""
    v = np.asarray(values_f32, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        q = (v / np.float32(scale)).astype(np.float32)
    flat = q.reshape(-1)
    uniq, inv = np.unique(flat.view(np.uint32), return_inverse=True)
    codes = np.array([encode_value(float(u)) & 0xFF for u in uniq.view(np.float32)],
                     dtype=np.uint8)
    return codes[inv.reshape(-1)].reshape(q.shape)


@lru_cache(maxsize=64)
def _table16(src_dtype: str, scale: float) -> np.ndarray:
    """Byte of every 16-bit source pattern (same rule as ``quantize``)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore", over="ignore"):
        return quantize(bits16_to_f32(allbits, src_dtype), scale)


def quantize_bits16(bits: np.ndarray, src_dtype: str, scale: float) -> np.ndarray:
    """``quantize`` of fp16/bf16 values given as bit patterns, by table."""
    return _table16(src_dtype, float(scale))[np.asarray(bits, dtype=np.uint16)]
