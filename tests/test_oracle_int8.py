"""Pins for the oracle's int8 KV codes and per-head scales (CPU only).

Pinned to: closed forms of symmetric rounding (integers map to themselves,
ties go to the even integer, values past the range saturate, the round trip
error is at most half a scale step), numpy's own round-half-even and clip as
a library routine, exact power-of-two scalings, and attention on values that
the per-head scales represent exactly, compared with torch's SDPA.  A planted
mistake (one head's scale used for every head) must fail a pin.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import cache as C
from oracle import fp8
from oracle import int8


def test_integers_are_their_own_codes():
    for c in range(-128, 128):
        assert int8.encode_value(float(c)) == c
        assert int8.code_to_int(c & 0xFF) == c
    codes = np.arange(256, dtype=np.uint8)
    np.testing.assert_array_equal(int8.decode(codes),
                                  np.where(codes >= 128, codes.astype(int) - 256, codes))


@pytest.mark.parametrize("x,code", [(0.5, 0), (1.5, 2), (2.5, 2), (-0.5, 0), (-1.5, -2),
                                    (-2.5, -2), (126.5, 126), (127.49, 127), (127.5, 127),
                                    (-127.5, -128), (-128.5, -128), (0.49999997, 0),
                                    (3.5000002, 4)])
def test_ties_to_even_and_saturation(x, code):
    assert int8.encode_value(x) == code


def test_special_values():
    assert int8.encode_value(math.nan) == 0
    assert int8.encode_value(math.inf) == 127
    assert int8.encode_value(-math.inf) == -128
    assert int8.encode_value(1e30) == 127
    assert int8.encode_value(-1e30) == -128
    assert int8.encode_value(-0.0) == 0


def test_matches_numpy_rint_and_clip():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * 60).astype(np.float32)
    x[:1000] = np.round(x[:1000]) + 0.5          # many exact ties
    got = int8.quantize(x, 1.0).view(np.int8).astype(np.int64)
    want = np.clip(np.rint(x.astype(np.float64)), -128, 127).astype(np.int64)
    np.testing.assert_array_equal(got, want)


def test_round_trip_error_is_half_a_step():
    rng = np.random.default_rng(8)
    scale = 0.037
    x = rng.uniform(-127 * scale, 127 * scale, 100000).astype(np.float32)
    back = int8.decode(int8.quantize(x, scale)) * scale
    assert np.abs(back - x).max() <= scale / 2 * (1 + 1e-6)


@pytest.mark.parametrize("x,code", [(0.3499999940395355, 4), (0.45000001788139343, 4),
                                    (0.75, 8), (0.8500000238418579, 8)])
def test_quotient_is_taken_in_float32(x, code):
    # with scale 0.1 the float32 quotient of these float32 inputs lands
    # exactly on k + 0.5 (ties to even), while the float64 quotient falls on
    # the other side: 0.75 / 0.1 is 7.4999999 in float64 but 7.5 in float32
    x32 = np.array([x], dtype=np.float32)
    assert int8.quantize(x32, 0.1)[0].view(np.int8) == code
    assert int(np.rint(np.float64(x32[0]) / np.float64(np.float32(0.1)))) != code


def test_table_quantizer_equals_direct():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    for src in ("f16", "bf16"):
        vals = fp8.bits16_to_f32(bits, src)
        with np.errstate(invalid="ignore", over="ignore"):
            direct = int8.quantize(vals, 0.05)
        np.testing.assert_array_equal(int8.quantize_bits16(bits, src, 0.05), direct)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "int8"])
def test_power_of_two_scaling_leaves_codes_unchanged(fmt):
    # x * 2^k / (s * 2^k) == x / s exactly in float32 (no overflow or
    # underflow here), so the codes of a head depend on its own scale only
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(5000) * 3).astype(np.float32)
    q = (lambda v, s: int8.quantize(v, s)) if fmt == "int8" else \
        (lambda v, s: fp8.quantize(v, s, fmt))
    base = q(x, 0.25)
    for k in (-3, 2, 5):
        np.testing.assert_array_equal(q(x * np.float32(2.0 ** k), 0.25 * 2.0 ** k), base)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _exact_case(dtype, seed=3):
    """A workload whose per-head scaled values are exactly representable:
    head h holds integer codes times the power-of-two scale s_h."""
    rng = np.random.default_rng(seed)
    Hkv, d, bs = 4, 16, 8
    lens = [13, 29, 5]
    w = W.random_case(seed, len(lens), 8, Hkv, d, bs, dtype, "bf16", lens)
    ks = tuple(2.0 ** e for e in (-6, -4, -3, -1))
    vs = tuple(2.0 ** e for e in (-2, -5, -3, -4))
    hi = 100 if dtype == "int8" else 7      # small integers are exact in e4m3 / e5m2 too
    for t, sc in ((w.ctx_k, ks), (w.ctx_v, vs), (w.new_k, ks), (w.new_v, vs)):
        codes = rng.integers(-hi, hi + 1, tuple(t.shape))
        t.copy_(torch.from_numpy(codes * np.asarray(sc)[None, :, None]).to(t.dtype))
    w.k_scale, w.v_scale = ks, vs
    return w


def _fill(w, k_scale, v_scale):
    c = C.PagedKVCache(w.num_blocks, w.Hkv, w.bs, w.d, w.cache_dtype, k_scale, v_scale)
    c.reshape_and_cache(_bits(w.ctx_k), _bits(w.ctx_v), w.src_dtype, w.ctx_slots)
    c.reshape_and_cache(_bits(w.new_k), _bits(w.new_v), w.src_dtype, w.new_slots)
    return c


def _sdpa_on_inputs(w):
    """torch SDPA (float64) on the original, exactly representable values."""
    q = w.q.double()
    out = np.zeros((w.S, w.Hq, w.d))
    for s in range(w.S):
        rows = w.token_rows(s)
        K = torch.stack([(w.ctx_k if k == "ctx" else w.new_k)[i] for k, i in rows]).double()
        V = torch.stack([(w.ctx_v if k == "ctx" else w.new_v)[i] for k, i in rows]).double()
        Kq = K.repeat_interleave(w.G, dim=1).transpose(0, 1)
        Vq = V.repeat_interleave(w.G, dim=1).transpose(0, 1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[s][:, None, :], Kq, Vq, scale=w.scale)
        out[s] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("dtype", ["int8", "e4m3", "e5m2"])
def test_per_head_scales_reproduce_exact_values(dtype):
    w = _exact_case(dtype)
    c = _fill(w, w.k_scale, w.v_scale)
    # codes are the integers the values were built from
    kv = C.values(c.k, dtype, w.k_scale)
    for s in range(w.S):
        for p, (kind, i) in enumerate(w.token_rows(s)):
            blk, off = w.block_tables[s][p // w.bs], p % w.bs
            src = (w.ctx_k if kind == "ctx" else w.new_k)[i].double().numpy()
            np.testing.assert_array_equal(kv[blk, :, off, :], src)
    q = C.bits_to_f64(_bits(w.q), "bf16")
    out = A.paged_decode(q, c.k, c.v, dtype, w.block_tables, w.seq_lens, w.scale,
                         w.k_scale, w.v_scale)
    np.testing.assert_allclose(out, _sdpa_on_inputs(w), rtol=1e-10, atol=1e-12)


def test_uniform_per_head_scale_equals_per_tensor():
    w = W.random_case(4, 2, 4, 2, 16, 16, "int8", "bf16", [20, 45])
    a = _fill(w, 0.03, 0.05)
    b = _fill(w, (0.03, 0.03), (0.05, 0.05))
    np.testing.assert_array_equal(a.k, b.k)
    np.testing.assert_array_equal(a.v, b.v)
    q = C.bits_to_f64(_bits(w.q), "bf16")
    oa = A.paged_decode(q, a.k, a.v, "int8", w.block_tables, w.seq_lens, w.scale, 0.03, 0.05)
    ob = A.paged_decode(q, b.k, b.v, "int8", w.block_tables, w.seq_lens, w.scale,
                        (0.03, 0.03), (0.05, 0.05))
    np.testing.assert_array_equal(oa, ob)


def test_planted_single_scale_fails_the_pin(monkeypatch):
    w = _exact_case("int8")
    c = _fill(w, w.k_scale, w.v_scale)
    monkeypatch.setattr(A, "head_scale", lambda scale, h: C.head_scale(scale, 0))
    q = C.bits_to_f64(_bits(w.q), "bf16")
    out = A.paged_decode(q, c.k, c.v, "int8", w.block_tables, w.seq_lens, w.scale,
                         w.k_scale, w.v_scale)
    assert not np.allclose(out, _sdpa_on_inputs(w), rtol=1e-6, atol=1e-8)


def test_unwritten_int8_slots_hold_the_most_negative_code():
    c = C.PagedKVCache(2, 1, 4, 8, "int8")
    assert (c.k.view(np.int8) == -128).all()
