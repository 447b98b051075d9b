"""OCP 8-bit floating point: E4M3 and E5M2 encode / decode.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages fix the use: [P3] §6.1 stores a KV value divided by a scale and
multiplies it back on read; §6.2 names e4m3 (1 sign, 4 exponent, 3 mantissa
bits, largest value 448, relative precision about 1/8) and e5m2 (one more
exponent bit, one fewer mantissa bit, wider range, coarser); §6.3 says the
default scale is 1.0, per tensor, optionally per head.

The bit formats are the OCP 8-bit floating point definitions:

* E4M3: exponent bias 7, no infinities, S.1111.111 is NaN; exponent field 0
  is subnormal with value 2^-6 * m/8; largest finite 2^8 * 1.75 = 448.
* E5M2: exponent bias 15, IEEE-style: exponent field 31 is inf (m == 0) or
  NaN (m != 0); exponent field 0 is subnormal 2^-14 * m/4; largest finite
  2^15 * 1.75 = 57344.

Encoding rounds to nearest, ties to even, and saturates values beyond the
largest finite number to it (``satfinite``): the pages only say that a
value outside the range is cut off ([P3] §6.1).
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from functools import lru_cache

import numpy as np


@dataclass(frozen=True)
class Fp8Format:
    name: str
    exp_bits: int
    man_bits: int
    bias: int
    has_inf: bool

    @property
    def emin(self) -> int:
        """Exponent of the smallest normal number."""
        return 1 - self.bias

    @property
    def max_finite(self) -> float:
        if self.has_inf:   # top exponent field reserved for inf / NaN
            top = (1 << self.exp_bits) - 2
            frac = 2.0 - 2.0 ** (-self.man_bits)
        else:              # E4M3: top field usable except the all-ones NaN
            top = (1 << self.exp_bits) - 1
            frac = 2.0 - 2.0 ** (1 - self.man_bits)
        return math.ldexp(frac, top - self.bias)


E4M3 = Fp8Format("e4m3", 4, 3, 7, has_inf=False)
E5M2 = Fp8Format("e5m2", 5, 2, 15, has_inf=True)
FORMATS = {"e4m3": E4M3, "e5m2": E5M2}


def decode_code(code: int, fmt: Fp8Format) -> float:
    """Value of one 8-bit code."""
    code &= 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> fmt.man_bits) & ((1 << fmt.exp_bits) - 1)
    m = code & ((1 << fmt.man_bits) - 1)
    e_all_ones = (1 << fmt.exp_bits) - 1
    if fmt.has_inf and e == e_all_ones:
        return sign * math.inf if m == 0 else math.nan
    if (not fmt.has_inf) and e == e_all_ones and m == (1 << fmt.man_bits) - 1:
        return math.nan
    if e == 0:
        return sign * math.ldexp(m, fmt.emin - fmt.man_bits)
    return sign * math.ldexp((1 << fmt.man_bits) + m, e - fmt.bias - fmt.man_bits)


def encode_value(x: float, fmt: Fp8Format) -> int:
    """Round ``x`` to the nearest code (ties to even), saturating to ±max."""
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a == 0.0:
        return sign
    if math.isinf(a):
        a = fmt.max_finite
    # floor(log2 a) exactly, via the binary exponent
    _, E = math.frexp(a)          # a = f * 2^E, f in [0.5, 1)
    e_eff = max(E - 1, fmt.emin)  # subnormals share the smallest normal's step
    quantum = math.ldexp(1.0, e_eff - fmt.man_bits)
    n = a / quantum               # exact: a and quantum are binary floats
    r = round(n)                  # Python rounds half to even
    value = r * quantum
    if value > fmt.max_finite:
        value = fmt.max_finite
    if value == 0.0:
        return sign
    if value < math.ldexp(1.0, fmt.emin):
        e_field = 0
        m = int(value / math.ldexp(1.0, fmt.emin - fmt.man_bits))
    else:
        _, E2 = math.frexp(value)
        exp = E2 - 1
        e_field = exp + fmt.bias
        m = int(value / math.ldexp(1.0, exp - fmt.man_bits)) - (1 << fmt.man_bits)
    return sign | (e_field << fmt.man_bits) | m


_DECODE_TABLES = {
    name: np.array([decode_code(c, f) for c in range(256)], dtype=np.float64)
    for name, f in FORMATS.items()
}


def decode(codes: np.ndarray, fmt_name: str) -> np.ndarray:
    """Vectorised decode of uint8 codes to float64."""
    return _DECODE_TABLES[fmt_name][np.asarray(codes, dtype=np.uint8)]


def quantize(values_f32: np.ndarray, scale: float, fmt_name: str) -> np.ndarray:
    """Stored code of ``value / scale`` ([P3] §6.1).

    The quotient is taken in IEEE float32 (the precision of the device
    path, whose integer outcome must agree bit for bit), then encoded.
    """
    fmt = FORMATS[fmt_name]
    v = np.asarray(values_f32, dtype=np.float32)
    q = (v / np.float32(scale)).astype(np.float32)
    flat = q.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    # encode each distinct float32 value once
    uniq, inv = np.unique(flat.view(np.uint32), return_inverse=True)
    codes = np.array([encode_value(float(u), fmt)
                      for u in uniq.view(np.float32)], dtype=np.uint8)
    out[:] = codes[inv.reshape(-1)]
    return out.reshape(q.shape)


def bits16_to_f32(bits: np.ndarray, src_dtype: str) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    if src_dtype == "f16":
        return b.view(np.float16).astype(np.float32)
    if src_dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(src_dtype)


@lru_cache(maxsize=64)
def _table16(src_dtype: str, scale: float, fmt_name: str) -> np.ndarray:
    """Code of every 16-bit source pattern (same rule as ``quantize``)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore", over="ignore"):   # NaN / inf patterns included
        return quantize(bits16_to_f32(allbits, src_dtype), scale, fmt_name)


def quantize_bits16(bits: np.ndarray, src_dtype: str, scale: float, fmt_name: str) -> np.ndarray:
    """``quantize`` of fp16/bf16 values given as bit patterns, by table."""
    return _table16(src_dtype, float(scale), fmt_name)[np.asarray(bits, dtype=np.uint16)]
