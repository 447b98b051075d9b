"""Block swap between the device caches and a pool in page-locked host
memory (GPU): bit-exact against the oracle's pool-to-pool moves."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from oracle.cache import PagedKVCache
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def _pool(nb, H, bs, d, elt, gen, device):
    shape = (nb, H, bs, d)
    if elt == 1:
        t = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    else:
        t = torch.randint(-32768, 32768, shape, generator=gen, dtype=torch.int32).to(torch.int16)
    return t.pin_memory() if device == "pinned" else t.to(device)


def _oracle_pools(dev_k, dev_v, host_k, host_v, dtype):
    dev = PagedKVCache(dev_k.shape[0], *dev_k.shape[1:], dtype, fill_nan=False)
    host = PagedKVCache(host_k.shape[0], *host_k.shape[1:], dtype, fill_nan=False)
    dev.k[:], dev.v[:] = G.bits(dev_k), G.bits(dev_v)
    host.k[:], host.v[:] = G.bits(host_k), G.bits(host_v)
    return dev, host


@pytest.mark.parametrize("dtype", ["f16", "e4m3", "int8"])
@pytest.mark.parametrize("bs,d,H", [(8, 64, 3), (16, 128, 8), (32, 128, 2)])
@pytest.mark.parametrize("where", ["pinned", "cuda"])
def test_swap_out_then_in_is_bit_exact(dtype, bs, d, H, where):
    elt = 1 if dtype in W.BYTE_DTYPES else 2
    gen = torch.Generator().manual_seed(bs * 100 + d + H)
    nb, hb = 50, 20
    kc = _pool(nb, H, bs, d, elt, gen, G.DEV)
    vc = _pool(nb, H, bs, d, elt, gen, G.DEV)
    hk = _pool(hb, H, bs, d, elt, gen, "pinned" if where == "pinned" else G.DEV)
    hv = _pool(hb, H, bs, d, elt, gen, "pinned" if where == "pinned" else G.DEV)
    dev, host = _oracle_pools(kc, vc, hk, hv, dtype)
    rng = np.random.default_rng(bs + d)
    out_pairs = np.stack([rng.permutation(nb)[:13], rng.permutation(hb)[:13]], axis=1)
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    pa.pa_swap_blocks(kc, vc, hk, hv, torch.from_numpy(out_pairs).to(G.DEV), "out",
                      cache_dtype=dtype, device_error=err)
    torch.cuda.synchronize()
    dev.swap_blocks(host, out_pairs, "out")
    np.testing.assert_array_equal(G.bits(hk), host.k)
    np.testing.assert_array_equal(G.bits(hv), host.v)
    np.testing.assert_array_equal(G.bits(kc), dev.k)
    in_pairs = np.stack([rng.permutation(hb)[:9], rng.permutation(nb)[:9]], axis=1)
    pa.pa_swap_blocks(kc, vc, hk, hv, torch.from_numpy(in_pairs).to(G.DEV), "in",
                      cache_dtype=dtype, device_error=err)
    torch.cuda.synchronize()
    dev.swap_blocks(host, in_pairs, "in")
    np.testing.assert_array_equal(G.bits(kc), dev.k)
    np.testing.assert_array_equal(G.bits(vc), dev.v)
    assert int(err.item()) == 0


def test_out_of_range_pairs_are_skipped_and_reported():
    gen = torch.Generator().manual_seed(5)
    kc = _pool(10, 2, 16, 64, 2, gen, G.DEV)
    vc = _pool(10, 2, 16, 64, 2, gen, G.DEV)
    hk = _pool(4, 2, 16, 64, 2, gen, "pinned")
    hv = _pool(4, 2, 16, 64, 2, gen, "pinned")
    dev, host = _oracle_pools(kc, vc, hk, hv, "f16")
    pairs = np.array([[1, 0], [2, 4], [-1, 1], [3, 3]])      # host has blocks 0..3
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    pa.pa_swap_blocks(kc, vc, hk, hv, torch.from_numpy(pairs).to(G.DEV), "out", cache_dtype="f16",
                      device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    dev.swap_blocks(host, [(1, 0), (3, 3)], "out")
    np.testing.assert_array_equal(G.bits(hk), host.k)
    np.testing.assert_array_equal(G.bits(hv), host.v)


def test_decode_after_swap_round_trip_is_unchanged():
    """Swap a sequence's blocks out, back into other free blocks, rewrite its
    table: the decode output is bit-identical."""
    lens = [300, 517, 64, 1000]
    w = W.random_case(21, len(lens), 8, 2, 128, 16, "e4m3", "bf16", lens, device=G.DEV,
                      pool_factor=2.0, k_scale=0.5)
    run = G.GpuRun(w, partition_size=256).setup()
    run.step()
    torch.cuda.synchronize()
    before = run.out.clone()
    s = 1
    nblk = -(-lens[s] // w.bs)
    blocks = w.block_tables[s, :nblk].tolist()
    used = {int(b) for r in range(w.S) for b in w.block_tables[r, :-(-lens[r] // w.bs)]}
    free = [b for b in range(w.num_blocks) if b not in used][:nblk]
    assert len(free) == nblk
    hk = torch.zeros((nblk, w.Hkv, w.bs, w.d), dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], device=G.DEV)
    in_pairs = torch.tensor([[i, f] for i, f in enumerate(free)], device=G.DEV)
    pa.pa_swap_blocks(run.kc, run.vc, hk, hv, out_pairs, "out", cache_dtype="e4m3",
                      device_error=run.err)
    run.kc[blocks] = 0          # the swapped-out blocks are reused by others
    run.vc[blocks] = 0
    pa.pa_swap_blocks(run.kc, run.vc, hk, hv, in_pairs, "in", cache_dtype="e4m3",
                      device_error=run.err)
    run.bt[s, :nblk] = torch.tensor(free, dtype=torch.int32, device=G.DEV)
    run.decode()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    assert torch.equal(before, run.out)


def test_unregistered_host_memory_is_refused_before_any_launch():
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=G.DEV)
    host = np.zeros((4, 2, 16, 64), dtype=np.float16)      # pageable, not registered
    pairs = torch.tensor([[0, 0]], device=G.DEV)
    lib = pa.load_library()
    desc = pa.cache_desc(kc)
    ptr = host.ctypes.data
    st = lib.pa_swap_blocks(kc.data_ptr(), kc.data_ptr(), ctypes.byref(desc), ptr, ptr, 4,
                            pairs.data_ptr(), 1, pa.PA_SWAP_OUT, None, None)
    assert st == 2        # PA_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(kc, kc, torch.zeros(4, 2, 16, 64, dtype=torch.float16),
                          torch.zeros(4, 2, 16, 64, dtype=torch.float16), pairs, "out")
