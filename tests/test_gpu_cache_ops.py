"""Cache write and block copy on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.cache import PagedKVCache
from tests import _gpu as G

pytestmark = pytest.mark.gpu

DTYPES = [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16"), ("e4m3", "f16"),
          ("e5m2", "f16"), ("e5m2", "bf16"), ("int8", "bf16"), ("int8", "f16")]
SCALES = {"e4m3": (0.37, 2.5), "e5m2": (0.37, 2.5), "int8": (0.021, 0.033)}


@pytest.mark.parametrize("cache_dtype,src", DTYPES)
@pytest.mark.parametrize("d,bs", [(64, 16), (128, 8), (128, 32)])
def test_reshape_and_cache_bit_exact(cache_dtype, src, d, bs):
    scales = SCALES.get(cache_dtype, (1.0, 1.0))
    w = W.random_case(5, 5, 4, 2, d, bs, cache_dtype, src, [1, bs - 1, bs, bs + 1, 77],
                      device=G.DEV, k_scale=scales[0], v_scale=scales[1])
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    np.testing.assert_array_equal(G.bits(run.kc), c.k)
    np.testing.assert_array_equal(G.bits(run.vc), c.v)


@pytest.mark.parametrize("cache_dtype", ["f16", "e4m3", "int8"])
def test_reshape_and_cache_large_values_saturate(cache_dtype):
    w = W.random_case(6, 2, 2, 2, 128, 16, cache_dtype, "f16" if cache_dtype == "f16" else "bf16",
                      [40, 33], device=G.DEV, k_scale=0.01, v_scale=0.02)
    w.ctx_k.mul_(100)   # many values beyond the largest code * scale: saturate
    w.new_v.mul_(300)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    c = G.oracle_cache(w)
    np.testing.assert_array_equal(G.bits(run.kc), c.k)
    np.testing.assert_array_equal(G.bits(run.vc), c.v)


@pytest.mark.parametrize("cache_dtype,src", [("e4m3", "bf16"), ("e5m2", "f16"), ("int8", "bf16"),
                                             ("int8", "f16")])
def test_reshape_and_cache_per_head_scales(cache_dtype, src):
    Hkv = 4
    base = 0.02 if cache_dtype == "int8" else 0.5
    ks = tuple(base * f for f in (1.0, 0.37, 2.9, 1.61))
    vs = tuple(base * f for f in (0.8, 3.3, 0.51, 1.0))
    w = W.random_case(17, 4, 8, Hkv, 128, 16, cache_dtype, src, [5, 16, 40, 131],
                      device=G.DEV, k_scale=ks, v_scale=vs)
    w.ctx_k[:, 2].mul_(50)   # head 2 also saturates
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    np.testing.assert_array_equal(G.bits(run.kc), c.k)
    np.testing.assert_array_equal(G.bits(run.vc), c.v)


def test_int8_nan_and_inf_inputs():
    w = W.random_case(18, 2, 2, 2, 64, 16, "int8", "f16", [9, 20], device=G.DEV,
                      k_scale=0.05, v_scale=0.05)
    w.ctx_k[0, 0, :4] = torch.tensor([float("nan"), float("inf"), -float("inf"), -0.0])
    w.ctx_v[3, 1, 7] = float("nan")
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    kc = G.bits(run.kc)
    blk, off = divmod(int(w.ctx_slots[0]), w.bs)
    assert kc[blk, 0, off, :4].view(np.int8).tolist() == [0, 127, -128, 0]
    np.testing.assert_array_equal(kc, c.k)
    np.testing.assert_array_equal(G.bits(run.vc), c.v)


def test_padding_slots_are_skipped():
    import paged_kv_cache_54_gb300 as pa
    kc = torch.zeros((8, 2, 16, 64), dtype=torch.float16, device=G.DEV)
    vc = torch.zeros_like(kc)
    key = torch.randn((4, 2, 64), device=G.DEV).half()
    val = torch.randn((4, 2, 64), device=G.DEV).half()
    slots = torch.tensor([3, -1, 17, -1], dtype=torch.int64, device=G.DEV)
    pa.pa_reshape_and_cache(key, val, slots, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(kc[0, :, 3], key[0]) and torch.equal(vc[1, :, 1], val[2])
    assert int((kc != 0).sum()) == int((key[0] != 0).sum() + (key[2] != 0).sum())


@pytest.mark.parametrize("cache_dtype", ["f16", "bf16", "e4m3", "int8"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_copy_blocks_bit_exact(cache_dtype, bs):
    import paged_kv_cache_54_gb300 as pa
    nb, H, d = 40, 3, 128
    g = torch.Generator(device=G.DEV).manual_seed(bs)
    if cache_dtype in ("e4m3", "int8"):
        kc = torch.randint(0, 256, (nb, H, bs, d), generator=g, device=G.DEV, dtype=torch.int32).to(torch.uint8)
        vc = torch.randint(0, 256, (nb, H, bs, d), generator=g, device=G.DEV, dtype=torch.int32).to(torch.uint8)
    else:
        dt = torch.float16 if cache_dtype == "f16" else torch.bfloat16
        kc = torch.randn((nb, H, bs, d), generator=g, device=G.DEV).to(dt)
        vc = torch.randn((nb, H, bs, d), generator=g, device=G.DEV).to(dt)
    rng = np.random.default_rng(bs)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1)      # dst never a src
    ref = PagedKVCache(nb, H, bs, d, cache_dtype, fill_nan=False)   # the oracle's copy
    ref.k[:], ref.v[:] = G.bits(kc), G.bits(vc)
    ref.copy_blocks(pairs)
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(G.DEV), cache_dtype=cache_dtype)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(G.bits(kc), ref.k)
    np.testing.assert_array_equal(G.bits(vc), ref.v)


def test_out_of_range_slot_and_pair_are_reported():
    import paged_kv_cache_54_gb300 as pa
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.float16, device=G.DEV)
    vc = torch.zeros_like(kc)
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    key = torch.ones((2, 1, 64), dtype=torch.float16, device=G.DEV)
    pa.pa_reshape_and_cache(key, key, torch.tensor([5, 64], device=G.DEV), kc, vc, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2
    assert float(kc.sum()) == 64.0          # the valid row was still written
    err.zero_()
    pa.pa_copy_blocks(kc, vc, torch.tensor([[0, 9]], device=G.DEV), device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
