"""pa_decode against the float64 oracle on small seeded cases (GPU)."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu

DTYPES = [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16"), ("e4m3", "f16"),
          ("e5m2", "f16"), ("e5m2", "bf16"), ("int8", "bf16"), ("int8", "f16")]


def _seed(*key):
    """A seed fixed by the test's parameters (str hashes vary between runs)."""
    return zlib.crc32(repr(key).encode()) % 1000


def _check(w, got, ref, extra_ulp=True):
    tol = G.tolerance(w)
    got = got.float().cpu().numpy().astype(np.float64)
    bound = np.maximum(tol, G.ulp(ref, w.q_dtype)) if extra_ulp else tol
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (f"max |err| {err.max():.3e} at {np.argwhere(bad)[:5].tolist()}, "
                           f"tol {tol}")
    return float(err.max())


def _lens(bs, P):
    return [0, 1, bs - 1, bs, bs + 1, 63, 64, 65, P - 1, P, P + 1, 2 * P + 17, 700]


@pytest.mark.parametrize("cache_dtype,q_dtype", DTYPES)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_matches_oracle(cache_dtype, q_dtype, d, bs, group):
    Hkv = 2
    P = 128
    lens = _lens(bs, P)
    scales = {"e4m3": (0.5, 1.5), "e5m2": (0.5, 1.5), "int8": (0.03, 0.045)}
    ks, vs = scales.get(cache_dtype, (1.0, 1.0))
    w = W.random_case(_seed(cache_dtype, q_dtype, d, bs, group), len(lens), Hkv * group,
                      Hkv, d, bs, cache_dtype, q_dtype, lens, device=G.DEV,
                      k_scale=ks, v_scale=vs)
    run = G.GpuRun(w, partition_size=P).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    ref = G.oracle_decode(w, G.oracle_cache(w))
    _check(w, run.out, ref)
    assert torch.all(run.out[0] == 0)          # length 0 gives zeros


@pytest.mark.parametrize("cache_dtype,q_dtype", [("e4m3", "bf16"), ("e5m2", "f16"),
                                                 ("int8", "bf16"), ("int8", "f16")])
@pytest.mark.parametrize("group", [1, 2, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_per_head_scales(cache_dtype, q_dtype, group, d):
    Hkv = 4
    base = 0.03 if cache_dtype == "int8" else 0.5
    ks = tuple(base * f for f in (1.0, 0.37, 2.9, 1.61))
    vs = tuple(base * f for f in (0.8, 3.3, 0.51, 1.0))
    lens = [1, 17, 64, 200, 513, 1100]
    w = W.random_case(_seed("per-head", cache_dtype, q_dtype, group, d), len(lens),
                      Hkv * group, Hkv, d, 16, cache_dtype, q_dtype, lens, device=G.DEV,
                      k_scale=ks, v_scale=vs, partition_size=256)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    ref = G.oracle_decode(w, G.oracle_cache(w))
    _check(w, run.out, ref)


@pytest.mark.parametrize("cache_dtype,q_dtype,group", [("f16", "f16", 1), ("bf16", "bf16", 2),
                                                       ("e4m3", "bf16", 8), ("f16", "f16", 4),
                                                       ("int8", "bf16", 8), ("int8", "f16", 1)])
def test_partition_size_does_not_change_the_result(cache_dtype, q_dtype, group):
    lens = [1, 100, 511, 512, 513, 1500, 2049]
    w = W.random_case(9, len(lens), 2 * group, 2, 128, 16, cache_dtype, q_dtype, lens,
                      device=G.DEV)
    c = G.oracle_cache(w)
    ref = G.oracle_decode(w, c)
    outs = []
    for P in (64, 192, 512, 1024, 0):
        run = G.GpuRun(w, partition_size=P).setup()
        run.step()
        torch.cuda.synchronize()
        assert int(run.err.item()) == 0
        _check(w, run.out, ref)
        outs.append(run.out.float())
    tol = G.tolerance(w)
    for o in outs[1:]:
        assert float((o - outs[0]).abs().max()) <= 2 * tol


def test_equal_keys_give_mean_of_values():
    lens = [1, 37, 300, 1000]
    w = W.random_case(3, len(lens), 2, 2, 128, 16, "f16", "f16", lens, device=G.DEV)
    w.ctx_k.copy_(w.ctx_k[:1].expand_as(w.ctx_k))
    w.new_k.copy_(w.ctx_k[:1].expand_as(w.new_k))
    run = G.GpuRun(w, partition_size=128).setup()
    run.step()
    torch.cuda.synchronize()
    for s in range(w.S):
        for hq in range(w.Hq):
            _, V = G.logical_kv(w, s, hq)
            np.testing.assert_allclose(run.out[s, hq].float().cpu().numpy(), V.mean(axis=0),
                                       atol=2e-3)


def test_repeated_calls_are_deterministic():
    lens = [5, 900, 1700, 3]
    w = W.random_case(4, len(lens), 8, 1, 128, 16, "e4m3", "bf16", lens, device=G.DEV)
    run = G.GpuRun(w, partition_size=256).setup()
    run.step()
    a = run.out.clone()
    for _ in range(3):
        run.decode()
    torch.cuda.synchronize()
    assert torch.equal(a, run.out)


@pytest.mark.parametrize("cache_dtype", ["e4m3", "int8"])
def test_large_query_values_with_byte_cache(cache_dtype):
    lens = [50, 300]
    w = W.random_case(8, 2, 8, 1, 128, 16, cache_dtype, "bf16", lens, device=G.DEV)
    # entries beyond fp16's range (the fp16 tensor-core path rescales q by a
    # power of two); the softmax scale shrinks by the same factor so that the
    # scores, and the conditioning of the problem, stay as before
    w.q.mul_(3.0e4)
    w.scale /= 3.0e4
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    ref = G.oracle_decode(w, G.oracle_cache(w))
    _check(w, run.out, ref)


def test_bad_block_id_and_length_are_reported():
    lens = [40, 20]
    w = W.random_case(1, 2, 2, 2, 64, 16, "f16", "f16", lens, device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    run.bt[0, 1] = w.num_blocks + 5
    run.decode()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 1
    run.err.zero_()
    run.bt.copy_(torch.from_numpy(w.block_tables).to(G.DEV))
    run.sl[1] = w.block_tables.shape[1] * w.bs + 1
    run.decode()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 3


SHARED_DTYPES = [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "bf16"), ("int8", "f16")]


@pytest.mark.parametrize("cache_dtype,q_dtype", SHARED_DTYPES)
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_shared_prefix_matches_oracle(cache_dtype, q_dtype, group, bs):
    """Sequences whose tables name the same blocks over whole partitions are
    decoded together; every output still equals the oracle's.  13 sequences
    leave a ragged last group at every group size."""
    Hkv = 2
    w = W.make_workload("qwen3-prefix", 31 + group + bs, device=G.DEV, overrides=dict(
        S=13, prefix=256, suffix_lo=1, suffix_hi=300, Hq=Hkv * group, Hkv=Hkv, d=128, bs=bs,
        cache_dtype=cache_dtype, q_dtype=q_dtype, src_dtype=q_dtype))
    for P in (64, 128):
        run = G.GpuRun(w, partition_size=P).setup()
        run.step()
        torch.cuda.synchronize()
        assert int(run.err.item()) == 0
        ref = G.oracle_decode(w, G.oracle_cache(w))
        _check(w, run.out, ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [2, 4, 8])
@pytest.mark.parametrize("bs,d", [(8, 128), (16, 128), (32, 128), (16, 64)])
def test_wide_shared_prefix_matches_oracle(dtype, group, bs, d):
    """Many sequences sharing a prefix: runs of 256 / G sequences (from a
    multiple of that count) whose tables agree over a whole partition are
    decoded on the tensor cores as wide items, the rest as usual.  Two full
    runs and a short third one; the prefix (300 tokens) ends inside a
    partition, so its last partition is only partly shared; partitions of
    64 tokens and the automatic size."""
    Hkv = 2
    W_seqs = 256 // group
    S = 2 * W_seqs + 7
    w = W.make_workload("qwen3-prefix", 101 + group + bs + d, device=G.DEV, overrides=dict(
        S=S, prefix=304 if bs == 16 else 320, suffix_lo=1, suffix_hi=200, Hq=Hkv * group, Hkv=Hkv, d=d,
        bs=bs, cache_dtype=dtype, q_dtype=dtype, src_dtype=dtype))
    ref = G.oracle_decode(w, G.oracle_cache(w))
    for P in (64, 0):
        run = G.GpuRun(w, partition_size=P).setup()
        run.step()
        torch.cuda.synchronize()
        assert int(run.err.item()) == 0
        _check(w, run.out, ref)


@pytest.mark.parametrize("group", [2, 8])
def test_wide_chunk_broken_by_a_copied_block(group):
    """One sequence in the middle of a would-be wide chunk reads one shared
    block through a copy (same contents, another physical block): the plan
    must find the rows differ, so that partition of the chunk is decoded as
    ordinary items, and every output still equals the oracle's."""
    import paged_kv_cache_54_gb300 as pa
    from oracle.cache import PagedKVCache
    Hkv, bs, d = 2, 16, 128
    W_seqs = 256 // group
    S = 2 * W_seqs
    w = W.make_workload("qwen3-prefix", 211 + group, device=G.DEV, overrides=dict(
        S=S, prefix=256, suffix_lo=1, suffix_hi=100, Hq=Hkv * group, Hkv=Hkv, d=d, bs=bs,
        cache_dtype="bf16", q_dtype="bf16", src_dtype="bf16"))
    run = G.GpuRun(w, partition_size=64).setup()
    run.step()
    torch.cuda.synchronize()
    # a free physical block, and the sequence and entry that will use it
    used = {int(b) for srow, L in zip(w.block_tables, w.seq_lens) for b in srow[:-(-int(L) // bs)]}
    free = next(b for b in range(w.num_blocks) if b not in used)
    s_star, entry = W_seqs // 2 + 1, 5          # partition 1 (entries 4..7) of chunk 0
    old = int(w.block_tables[s_star, entry])
    pa.pa_copy_blocks(run.kc, run.vc, torch.tensor([[old, free]], dtype=torch.int64, device=G.DEV),
                      cache_dtype="bf16", device_error=run.err)
    w.block_tables = w.block_tables.copy()
    w.block_tables[s_star, entry] = free
    run.bt = torch.from_numpy(w.block_tables).to(G.DEV)
    run.decode()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    c = G.oracle_cache(w)
    c.copy_blocks([(old, free)])
    ref = G.oracle_decode(w, c)
    _check(w, run.out, ref)


@pytest.mark.parametrize("cache_dtype,q_dtype", SHARED_DTYPES)
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (8, 1)])
def test_beam_fork_matches_oracle(cache_dtype, q_dtype, bs, heads):
    Hq, Hkv = heads
    w = W.make_workload("opt13b-beam", 7 + bs + Hq, device=G.DEV, overrides=dict(
        prompts=5, len_lo=100, len_hi=700, Hq=Hq, Hkv=Hkv, d=64 if Hq == 8 else 128, bs=bs,
        cache_dtype=cache_dtype, q_dtype=q_dtype, src_dtype=q_dtype))
    for P in (64, 256):
        run = G.GpuRun(w, partition_size=P).setup()
        run.step()
        torch.cuda.synchronize()
        assert int(run.err.item()) == 0
        ref = G.oracle_decode(w, G.oracle_cache(w))
        _check(w, run.out, ref)


@pytest.mark.parametrize("cache_dtype,q_dtype,heads", [("f16", "f16", (1, 1)),
                                                       ("bf16", "bf16", (2, 1))])
def test_many_sequences(cache_dtype, q_dtype, heads):
    """5000 sequences of 1..329 tokens in partitions of 64 (a table width that
    is not a multiple of four entries, so the plan reads the rows in place)."""
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 330, 5000).tolist()
    Hq, Hkv = heads
    w = W.random_case(12, len(lens), Hq, Hkv, 64, 16, cache_dtype, q_dtype, lens, device=G.DEV)
    run = G.GpuRun(w, partition_size=64).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    ref = G.oracle_decode(w, G.oracle_cache(w))
    _check(w, run.out, ref)


def test_plan_tables_beyond_shared_memory():
    """17 000 sequences sharing a 384-token prefix, each with 1..128 tokens of
    its own, in partitions of 64: each of the plan's eight CTAs owns more
    than 2048 sequences and 16 384 (sequence, partition) slots, so its
    lengths and join flags live in the workspace and its block-table rows
    are read in place; the shared partitions also form wide chunks across
    the CTAs' runs.  Sampled rows (the sequences around every CTA's first and
    last, and a spread between) against the oracle."""
    w = W.make_workload("qwen3-prefix", 91, device=G.DEV, overrides=dict(
        S=17000, prefix=384, suffix_lo=1, suffix_hi=128, Hq=2, Hkv=1, d=64, bs=16,
        cache_dtype="bf16", q_dtype="bf16", src_dtype="bf16"))
    run = G.GpuRun(w, partition_size=64).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    groups = -(-w.S // 4)                      # kmax = 4 sequences at G = 2
    edges = {min(w.S, (r * groups // 8) * 4) for r in range(9)}
    seqs = {x for e in edges for x in range(e - 2, e + 3) if 0 <= x < w.S}
    seqs |= set(range(0, w.S, 97))
    rows = [(s, hq) for s in sorted(seqs) for hq in range(w.Hq)]
    ref = G.oracle_rows(w, rows)
    got = run.out.float().cpu().numpy().astype(np.float64)
    tol = G.tolerance(w)
    worst = 0.0
    for (s, hq), r in ref.items():
        err = np.abs(got[s, hq] - r)
        bound = np.maximum(tol, G.ulp(r, w.q_dtype))
        assert not (err > bound).any(), (s, hq, float(err.max()))
        worst = max(worst, float(err.max()))
    print(f"{len(rows)} sampled rows of {w.S * w.Hq}, max |err| {worst:.2e}")


def test_shared_prefix_across_plan_chunks():
    """Sharing runs that cross the plan kernel's 1024-sequence chunks."""
    w = W.make_workload("qwen3-prefix", 77, device=G.DEV, overrides=dict(
        S=2100, prefix=128, suffix_lo=1, suffix_hi=40, Hq=2, Hkv=1, d=64, bs=16,
        cache_dtype="bf16", q_dtype="bf16", src_dtype="bf16"))
    run = G.GpuRun(w, partition_size=64).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    ref = G.oracle_decode(w, G.oracle_cache(w))
    _check(w, run.out, ref)
