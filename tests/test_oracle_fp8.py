"""Pins for the oracle's FP8 encode/decode (CPU only).

Pinned to: the figures the page prints for e4m3 (max 448, 3 mantissa bits,
relative step about 1/8), the exact fact that e5m2 is the upper byte of an
IEEE binary16, torch's own float8 conversions (a library routine) on
in-range values, and hand-built rounding ties.
"""
import math

import numpy as np
import pytest
import torch

from oracle import fp8
from tests._golden import load

G = load("fp8_formats.json")


def test_e4m3_figures_from_the_page():
    g = G["e4m3"]
    assert fp8.E4M3.max_finite == g["max_finite"]
    assert fp8.E4M3.man_bits == g["man_bits"] and fp8.E4M3.exp_bits == g["exp_bits"]
    one = fp8.encode_value(1.0, fp8.E4M3)
    step = fp8.decode_code(one + 1, fp8.E4M3) - 1.0
    assert step == g["relative_step_near_one"]
    # largest code value and saturation to it
    assert fp8.decode_code(0x7E, fp8.E4M3) == 448.0
    assert math.isnan(fp8.decode_code(0x7F, fp8.E4M3))
    assert fp8.encode_value(1.0e4, fp8.E4M3) == 0x7E
    assert fp8.encode_value(-1.0e4, fp8.E4M3) == 0xFE
    assert fp8.encode_value(math.inf, fp8.E4M3) == 0x7E


def test_e5m2_wider_range_and_saturation():
    assert fp8.E5M2.max_finite == 57344.0 > fp8.E4M3.max_finite
    assert fp8.encode_value(-1.0e6, fp8.E5M2) == 0xFB
    assert fp8.encode_value(math.inf, fp8.E5M2) == 0x7B


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_every_code_round_trips(name):
    f = fp8.FORMATS[name]
    for c in range(256):
        v = fp8.decode_code(c, f)
        if math.isnan(v) or math.isinf(v):
            continue
        assert fp8.encode_value(v, f) == c, (name, c, v)


def test_e5m2_is_upper_byte_of_binary16():
    for c in range(256):
        half = np.array([c << 8], dtype=np.uint16).view(np.float16)[0]
        v = fp8.decode_code(c, fp8.E5M2)
        if math.isnan(float(half)):
            assert math.isnan(v)
        else:
            assert v == float(half)


def test_subnormals():
    assert fp8.decode_code(0x01, fp8.E4M3) == 2.0 ** -9
    assert fp8.decode_code(0x08, fp8.E4M3) == 2.0 ** -6
    assert fp8.decode_code(0x01, fp8.E5M2) == 2.0 ** -16


def test_ties_round_to_even():
    # 1.0625 lies halfway between 1.0 (m=0) and 1.125 (m=1): even -> 1.0
    assert fp8.encode_value(1.0625, fp8.E4M3) == fp8.encode_value(1.0, fp8.E4M3)
    # 1.1875 lies halfway between 1.125 (m=1) and 1.25 (m=2): even -> 1.25
    assert fp8.encode_value(1.1875, fp8.E4M3) == fp8.encode_value(1.25, fp8.E4M3)
    # half the smallest subnormal rounds to zero; 1.5x rounds up to 2x
    assert fp8.encode_value(2.0 ** -10, fp8.E4M3) == 0x00
    assert fp8.encode_value(3 * 2.0 ** -10, fp8.E4M3) == 0x02
    assert fp8.encode_value(-0.0, fp8.E4M3) == 0x80


@pytest.mark.parametrize("name,tdtype", [("e4m3", torch.float8_e4m3fn),
                                         ("e5m2", torch.float8_e5m2)])
def test_matches_torch_on_in_range_values(name, tdtype):
    f = fp8.FORMATS[name]
    g = torch.Generator().manual_seed(7)
    x = torch.cat([
        torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0)
    ])
    x = x[x.abs() <= f.max_finite]
    ref = x.to(tdtype).view(torch.uint8).numpy()
    ours = fp8.quantize(x.numpy(), 1.0, name)
    np.testing.assert_array_equal(ours, ref)


def test_quantize_divides_by_scale_in_float32():
    x = np.array([0.3, -1.7, 2.9, 100.0], dtype=np.float32)
    scale = np.float32(0.37)
    codes = fp8.quantize(x, float(scale), "e4m3")
    expect = [fp8.encode_value(float(np.float32(v / scale)), fp8.E4M3) for v in x]
    assert codes.tolist() == expect
    back = fp8.decode(codes, "e4m3") * float(scale)
    assert np.all(np.abs(back - x) <= np.abs(x) / 16 + 2.0 ** -9 * float(scale))


@pytest.mark.parametrize("src", ["f16", "bf16"])
@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_table_quantizer_equals_direct(src, name):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 65536, 4000).astype(np.uint16)
    vals = fp8.bits16_to_f32(bits, src)
    keep = np.isfinite(vals)
    for scale in (1.0, 0.37, 3.5):
        a = fp8.quantize_bits16(bits[keep], src, scale, name)
        b = fp8.quantize(vals[keep], scale, name)
        np.testing.assert_array_equal(a, b)
