"""pa_prefill against the float64 oracle (GPU): small seeded cases over the
supported shapes with ragged new-token counts, the shared-prefix workload at
full size on sampled rows, and the device checks."""
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from oracle import attention as A
from tests import _gpu as G

pytestmark = pytest.mark.gpu

# (L_s, n_s): whole prompts, suffixes after a cached prefix, single tokens,
# lengths around the 64-key stage and the query tiles
# (520 new tokens: three query ranges of 256 rows even at group size 1, the
# last with one tile)
CASES = [(1, 1), (17, 17), (100, 37), (64, 64), (65, 1), (300, 129), (700, 5), (129, 128),
         (250, 250), (33, 9), (600, 520)]


def _seed(*key):
    return zlib.crc32(repr(key).encode()) % 1000


def _run(w, q, q_lens, err=None):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32, device=G.DEV)
    out = torch.empty_like(q)
    run = G.GpuRun(w).setup()
    run.step()
    err = run.err if err is None else err
    pa.pa_prefill(out, q, cu, run.kc, run.vc, run.bt, run.sl, max(q_lens), w.scale, device_error=err,
                  **run.kw)
    torch.cuda.synchronize()
    return out, run


def _check(w, got, ref):
    tol = G.tolerance(w)
    got = got.float().cpu().numpy().astype(np.float64)
    bound = np.maximum(tol, G.ulp(ref, w.q_dtype))
    err = np.abs(got - ref)
    assert not (err > bound).any(), (f"max |err| {err.max():.3e} at "
                                     f"{np.argwhere(err > bound)[:5].tolist()}")
    return float(err.max())


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_prefill_matches_oracle(dtype, d, bs, group):
    Hkv = 2
    lens = [L for L, _ in CASES]
    q_lens = [n for _, n in CASES]
    w = W.random_case(_seed(dtype, d, bs, group), len(lens), Hkv * group, Hkv, d, bs, dtype, dtype,
                      lens, device=G.DEV)
    gen = torch.Generator(device=G.DEV).manual_seed(_seed("q", dtype, d, bs, group))
    q = torch.randn((sum(q_lens), Hkv * group, d), generator=gen, device=G.DEV).to(w.q.dtype)
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), dtype), q_lens, c.k, c.v, dtype,
                          w.block_tables, w.seq_lens, w.scale)
    _check(w, out, ref)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefill_long_block_tables(bs):
    """The producer reads block-table entries from 32-entry windows, the next
    fetched while the current one is in use: tables of up to 263 entries
    (several window moves at every block size), ranges that start deep in
    the table, and one-token and whole-tile ranges."""
    Hkv, group, d = 2, 2, 128
    lens, q_lens = [2100, 700, 1025, 64], [70, 3, 130, 64]
    w = W.random_case(_seed("long", bs), len(lens), Hkv * group, Hkv, d, bs, "bf16", "bf16", lens,
                      device=G.DEV)
    gen = torch.Generator(device=G.DEV).manual_seed(_seed("qlong", bs))
    q = torch.randn((sum(q_lens), Hkv * group, d), generator=gen, device=G.DEV).bfloat16()
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), "bf16"), q_lens, c.k, c.v, "bf16",
                          w.block_tables, w.seq_lens, w.scale)
    _check(w, out, ref)


@pytest.mark.parametrize("lens,q_lens", [([512, 300], [100, 5]), ([1024, 20], [129, 20])])
def test_prefill_tables_exactly_one_or_two_windows_wide(lens, q_lens):
    """Block tables 32 and 64 entries wide (block size 16): the windows' last
    entries are the table's last, and the fetch of the window after them is
    skipped."""
    Hkv, group, d = 2, 4, 128
    w = W.random_case(_seed("win", lens), len(lens), Hkv * group, Hkv, d, 16, "f16", "f16", lens, device=G.DEV)
    assert w.block_tables.shape[1] == max(lens) // 16
    gen = torch.Generator(device=G.DEV).manual_seed(_seed("qwin", lens))
    q = torch.randn((sum(q_lens), Hkv * group, d), generator=gen, device=G.DEV).half()
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), "f16"), q_lens, c.k, c.v, "f16",
                          w.block_tables, w.seq_lens, w.scale)
    _check(w, out, ref)


BYTE_CASES = [("e4m3", "bf16"), ("e5m2", "f16"), ("int8", "bf16"), ("int8", "f16"), ("e4m3", "f16")]


@pytest.mark.parametrize("cache_dtype,q_dtype", BYTE_CASES)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 8])
@pytest.mark.parametrize("per_head", [False, True])
def test_prefill_byte_cache_matches_oracle(cache_dtype, q_dtype, d, group, per_head):
    """FP8 and INT8 caches: codes widened to fp16 for the products, a bf16 q
    rewritten as fp16, the K scale in the scores and the V scale in the
    output; against the oracle on the dequantised values."""
    Hkv = 2
    lens = [L for L, _ in CASES]
    q_lens = [n for _, n in CASES]
    ks, vs = ((0.03, 0.07), (0.05, 0.02)) if per_head else (0.04, 0.06)
    if cache_dtype != "int8" and not per_head:
        ks, vs = 1.0, 0.5
    w = W.random_case(_seed(cache_dtype, q_dtype, d, group, per_head), len(lens), Hkv * group, Hkv, d, 16,
                      cache_dtype, q_dtype, lens, device=G.DEV, k_scale=ks, v_scale=vs)
    gen = torch.Generator(device=G.DEV).manual_seed(_seed("qb", cache_dtype, d, group))
    q = torch.randn((sum(q_lens), Hkv * group, d), generator=gen, device=G.DEV).to(w.q.dtype)
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), q_dtype), q_lens, c.k, c.v, cache_dtype,
                          w.block_tables, w.seq_lens, w.scale, w.k_scale, w.v_scale)
    _check(w, out, ref)


@pytest.mark.parametrize("cache_dtype,q_dtype", [("e4m3", "bf16"), ("int8", "f16")])
@pytest.mark.parametrize("bs", [8, 32])
def test_prefill_byte_cache_block_sizes(cache_dtype, q_dtype, bs):
    """One-byte caches at block sizes 8 and 32: eight or two code tiles a
    stage, whole blocks widened."""
    Hkv, group = 2, 2
    lens = [L for L, _ in CASES]
    q_lens = [n for _, n in CASES]
    w = W.random_case(_seed("bs", cache_dtype, bs), len(lens), Hkv * group, Hkv, 128, bs, cache_dtype,
                      q_dtype, lens, device=G.DEV, k_scale=0.05, v_scale=0.04)
    gen = torch.Generator(device=G.DEV).manual_seed(_seed("qbs", cache_dtype, bs))
    q = torch.randn((sum(q_lens), Hkv * group, 128), generator=gen, device=G.DEV).to(w.q.dtype)
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), q_dtype), q_lens, c.k, c.v, cache_dtype,
                          w.block_tables, w.seq_lens, w.scale, w.k_scale, w.v_scale)
    _check(w, out, ref)


def test_prefill_byte_cache_large_bf16_queries():
    """bf16 q beyond fp16's range: the query tile is scaled by a power of two
    before it is rounded to fp16, and the factor undone on the scores."""
    lens, q_lens = [300, 90], [200, 90]
    w = W.random_case(4, 2, 4, 2, 128, 16, "e4m3", "bf16", lens, device=G.DEV, k_scale=0.02, v_scale=1.0)
    gen = torch.Generator(device=G.DEV).manual_seed(12)
    q = (torch.randn((sum(q_lens), 4, 128), generator=gen, device=G.DEV) * 2e5).bfloat16()
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), "bf16"), q_lens, c.k, c.v, "e4m3",
                          w.block_tables, w.seq_lens, w.scale, w.k_scale, w.v_scale)
    assert np.isfinite(out.float().cpu().numpy()).all()
    _check(w, out, ref)


@pytest.mark.parametrize("cache_dtype,q_dtype", [("f16", "f16"), ("e4m3", "bf16")])
def test_sequences_without_new_tokens(cache_dtype, q_dtype):
    """cu_q_lens may repeat: sequences with no new token produce no rows and
    leave the others' rows intact."""
    lens = [40, 300, 17, 129, 64]
    q_lens = [0, 120, 0, 129, 1]
    w = W.random_case(21, len(lens), 4, 2, 128, 16, cache_dtype, q_dtype, lens, device=G.DEV)
    gen = torch.Generator(device=G.DEV).manual_seed(22)
    q = torch.randn((sum(q_lens), 4, 128), generator=gen, device=G.DEV).to(w.q.dtype)
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), q_dtype), q_lens, c.k, c.v, cache_dtype,
                          w.block_tables, w.seq_lens, w.scale, w.k_scale, w.v_scale)
    _check(w, out, ref)


def test_many_short_sequences():
    """3000 sequences of 1-3 new tokens (a decode-sized prefill): a grid of
    3000 sequences by 2 KV heads, most CTAs holding a few rows."""
    rng = np.random.default_rng(8)
    lens = rng.integers(3, 200, 3000).tolist()
    q_lens = [int(min(L, n)) for L, n in zip(lens, rng.integers(1, 4, 3000))]
    w = W.random_case(23, len(lens), 4, 2, 64, 16, "bf16", "bf16", lens, device=G.DEV)
    gen = torch.Generator(device=G.DEV).manual_seed(24)
    q = torch.randn((sum(q_lens), 4, 64), generator=gen, device=G.DEV).bfloat16()
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    ref = A.paged_prefill(G.bits_to_f64(G.bits(q), "bf16"), q_lens, c.k, c.v, "bf16",
                          w.block_tables, w.seq_lens, w.scale)
    _check(w, out, ref)


def test_prefill_last_rows_agree_with_decode():
    lens = [300, 77, 1024]
    q_lens = [40, 77, 3]
    w = W.random_case(8, len(lens), 8, 2, 128, 16, "bf16", "bf16", lens, device=G.DEV)
    gen = torch.Generator(device=G.DEV).manual_seed(9)
    q = torch.randn((sum(q_lens), 8, 128), generator=gen, device=G.DEV).bfloat16()
    out, run = _run(w, q, q_lens)
    last = np.cumsum(q_lens) - 1
    dec = torch.empty((len(lens), 8, 128), dtype=torch.bfloat16, device=G.DEV)
    pa.pa_decode(dec, q[torch.from_numpy(last).to(G.DEV)].contiguous(), run.kc, run.vc, run.bt,
                 run.sl, max(lens), w.scale)
    torch.cuda.synchronize()
    diff = (out[torch.from_numpy(last).to(G.DEV)].float() - dec.float()).abs().max().item()
    assert diff <= 2e-2


def test_shared_prefix_suffix_prefill_full_size():
    """The shared-prefix workload (256 sequences, one 1024-token prefix):
    prefill each sequence's own tokens after the cached prefix; sampled rows
    against the oracle computed one row at a time."""
    w = W.make_workload("qwen3-prefix", W.config_seed("qwen3-prefix"), device=G.DEV)
    q_lens = [int(L) - 1024 for L in w.seq_lens]
    gen = torch.Generator(device=G.DEV).manual_seed(31)
    q = torch.randn((sum(q_lens), w.Hq, w.d), generator=gen, device=G.DEV).bfloat16()
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    got = out.float().cpu().numpy()
    qv = G.bits_to_f64(G.bits(q), "bf16")
    rng = np.random.default_rng(4)
    starts = np.concatenate([[0], np.cumsum(q_lens)])
    worst = 0.0
    for _ in range(24):
        s = int(rng.integers(w.S))
        j = int(rng.integers(q_lens[s]))
        hq = int(rng.integers(w.Hq))
        p = int(w.seq_lens[s]) - q_lens[s] + j
        K, V = G.logical_kv(w, s, hq // w.G)
        ref = A.attend(qv[starts[s] + j, hq], K[:p + 1], V[:p + 1], w.scale)[0]
        e = float(np.abs(got[starts[s] + j, hq] - ref).max())
        worst = max(worst, e)
        assert e <= G.TOL["bf16"], (s, j, hq, e)
    print(f"sampled rows, max |err| {worst:.2e}")


@pytest.mark.parametrize("cache_dtype,k_scale,v_scale", [
    ("e4m3", 1.0, 1.0),
    ("int8", tuple(0.02 + 0.004 * h for h in range(8)), tuple(0.035 - 0.003 * h for h in range(8)))])
def test_shared_prefix_suffix_prefill_full_size_one_byte(cache_dtype, k_scale, v_scale):
    """The same full-size launch over a one-byte cache (e4m3 with one scale,
    INT8 with one scale per KV head): the widening warpgroup's path at the
    size the bench times; sampled rows against the oracle on the
    dequantised cache."""
    w = W.make_workload("qwen3-prefix", W.config_seed("qwen3-prefix"), device=G.DEV,
                        overrides=dict(cache_dtype=cache_dtype, k_scale=k_scale, v_scale=v_scale))
    q_lens = [int(L) - 1024 for L in w.seq_lens]
    gen = torch.Generator(device=G.DEV).manual_seed(37)
    q = torch.randn((sum(q_lens), w.Hq, w.d), generator=gen, device=G.DEV).to(w.q.dtype)
    out, run = _run(w, q, q_lens)
    assert int(run.err.item()) == 0
    got = out.float().cpu().numpy()
    qv = G.bits_to_f64(G.bits(q), w.q_dtype)
    rng = np.random.default_rng(5)
    starts = np.concatenate([[0], np.cumsum(q_lens)])
    tol = G.tolerance(w)
    worst = 0.0
    for _ in range(24):
        s = int(rng.integers(w.S))
        j = int(rng.integers(q_lens[s]))
        hq = int(rng.integers(w.Hq))
        p = int(w.seq_lens[s]) - q_lens[s] + j
        K, V = G.logical_kv(w, s, hq // w.G)
        ref = A.attend(qv[starts[s] + j, hq], K[:p + 1], V[:p + 1], w.scale)[0]
        e = np.abs(got[starts[s] + j, hq] - ref)
        worst = max(worst, float(e.max()))
        assert not (e > np.maximum(tol, G.ulp(ref, w.q_dtype))).any(), (s, j, hq, float(e.max()))
    print(f"{cache_dtype}: sampled rows, max |err| {worst:.2e}")


def test_bad_lengths_and_blocks_are_reported():
    lens = [40, 50]
    w = W.random_case(3, 2, 2, 2, 64, 16, "f16", "f16", lens, device=G.DEV)
    q = torch.randn((60, 2, 64), device=G.DEV).half()
    # n_s > L_s for the second sequence: skipped, error 3
    cu = torch.tensor([0, 10, 60], dtype=torch.int32, device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    out = torch.zeros_like(q)
    pa.pa_prefill(out, q, cu, run.kc, run.vc, run.bt,
                  torch.tensor([40, 45], dtype=torch.int32, device=G.DEV), 50, w.scale,
                  device_error=run.err)
    torch.cuda.synchronize()
    assert int(run.err.item()) == 3
    assert torch.all(out[10:] == 0) and torch.isfinite(out[:10].float()).all()
    # a block id past the pool: error 1
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    bt = run.bt.clone()
    bt[0, 1] = w.num_blocks + 5
    pa.pa_prefill(out[:20], q[:20].contiguous(), torch.tensor([0, 10, 20], dtype=torch.int32, device=G.DEV),
                  run.kc, run.vc, bt, run.sl, 10, w.scale, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1


def test_rows_outside_q_are_refused_and_out_is_not_overrun():
    """cu_q_lens entries that name rows outside q/out, or a sequence with more
    new tokens than max_q_len, skip that sequence with error 3; nothing past
    ``out`` is written (a guard region follows it in the same buffer)."""
    lens = [40, 50]
    w = W.random_case(4, 2, 2, 2, 64, 16, "f16", "f16", lens, device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    q = torch.randn((60, 2, 64), device=G.DEV).half()
    buf = torch.full((60 + 300, 2, 64), 7.0, dtype=torch.float16, device=G.DEV)
    out = buf[:60]
    out.zero_()
    sl = torch.tensor([40, 50], dtype=torch.int32, device=G.DEV)

    def call(cu, max_q_len):
        err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
        pa.pa_prefill(out, q, torch.tensor(cu, dtype=torch.int32, device=G.DEV), run.kc, run.vc,
                      run.bt, sl, max_q_len, w.scale, device_error=err)
        torch.cuda.synchronize()
        return int(err.item())

    # the second sequence's rows 10..309 run 250 rows past the end of q and out
    assert call([0, 10, 310], 300) == 3
    assert torch.isfinite(out[:10].float()).all() and torch.all(out[10:] == 0)
    assert torch.all(buf[60:] == 7.0)
    # a negative start
    out.zero_()
    assert call([-20, 10, 60], 50) == 3
    assert torch.all(out[:10] == 0) and torch.isfinite(out[10:].float()).all()
    assert torch.all(buf[60:] == 7.0)
    # 50 new tokens against a declared max_q_len of 20 (the grid still covers
    # them: its CTAs take 256 / G tokens each)
    out.zero_()
    assert call([0, 10, 60], 20) == 3
    assert torch.isfinite(out[:10].float()).all() and torch.all(out[10:] == 0)
    # and the same call within bounds reports nothing
    assert call([0, 10, 60], 50) == 0


def test_unsupported_inputs_are_refused_on_the_host():
    import ctypes
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=G.DEV)
    q = torch.zeros((3, 2, 64), dtype=torch.float16, device=G.DEV)
    cu = torch.tensor([0, 3], dtype=torch.int32, device=G.DEV)
    bt = torch.zeros((1, 4), dtype=torch.int32, device=G.DEV)
    sl = torch.tensor([3], dtype=torch.int32, device=G.DEV)
    lib = pa.load_library()

    def call(desc, q_dtype, heads=2):
        return lib.pa_prefill(q.data_ptr(), q.data_ptr(), q_dtype, 3, cu.data_ptr(), 1, heads, 3,
                              kc.data_ptr(), kc.data_ptr(), ctypes.byref(desc), bt.data_ptr(), 4,
                              sl.data_ptr(), 0.125, None, None)
    assert call(pa.cache_desc(kc, "f16"), pa.PA_BF16) == 2    # a 16-bit cache takes its own q dtype
    assert call(pa.cache_desc(kc, "f16"), pa.PA_F16, heads=6) == 2   # group size 3
    kb = kc.view(torch.uint8)[..., :64]
    assert call(pa.cache_desc(kb.contiguous(), "e4m3"), 7) == 2      # q neither fp16 nor bf16
