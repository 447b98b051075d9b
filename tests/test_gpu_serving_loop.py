"""A serving loop through the library (GPU): the native prefix cache admits
requests with shared prompts, every step appends one token per sequence,
writes its K/V and decodes all live sequences; halfway through one sequence
is swapped out to page-locked host memory, its blocks are freed, and it is
later re-admitted (its prompt blocks hit the cache) and swapped back in to
the blocks the cache hands out.  Each token's K/V row is a function of the
tokens up to it, so every output is checked against the oracle's attention
over the sequence's own tokens.  The partition is 64 tokens, so sequences
cross partition boundaries as they grow and the split-K merge runs."""
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
from oracle import attention as A
from tests import _gpu as G

pytestmark = pytest.mark.gpu

HKV, GROUP, D, BS, P = 2, 2, 64, 16, 64


def _kv_row(prefix):
    seed = zlib.crc32(np.asarray(prefix, dtype=np.int32).tobytes())
    return np.random.default_rng(seed).standard_normal((2, HKV, D)).astype(np.float16)


def _write(kc, vc, rows, slots, err):
    k = torch.from_numpy(np.stack([r[0] for r in rows])).to(G.DEV)
    v = torch.from_numpy(np.stack([r[1] for r in rows])).to(G.DEV)
    pa.pa_reshape_and_cache(k, v, torch.tensor(slots, dtype=torch.int64, device=G.DEV), kc, vc,
                            device_error=err)


def _check(out, q, live, tokens):
    got = out.float().cpu().numpy()
    qv = q.double().cpu().numpy()
    for i, s in enumerate(live):
        rows = np.stack([_kv_row(tokens[s][:p + 1]) for p in range(len(tokens[s]))]).astype(np.float64)
        for h in range(HKV):
            heads = slice(h * GROUP, (h + 1) * GROUP)
            ref = A.attend(qv[i, heads], rows[:, 0, h], rows[:, 1, h], 1.0 / np.sqrt(D))
            e = np.abs(got[i, heads] - ref)
            assert not (e > np.maximum(2e-3, G.ulp(ref, "f16"))).any(), (s, h, float(e.max()))


def test_serving_loop_with_swap():
    rng = np.random.default_rng(17)
    nb = 160
    cache = pa.PrefixCache(nb, BS, rng.permutation(nb))
    kc = torch.full((nb, HKV, BS, D), float("nan"), dtype=torch.float16, device=G.DEV)
    vc = torch.full_like(kc, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    prompts = [rng.integers(0, 500, n).tolist() for n in (40, 100)]
    tokens = {}
    for s in range(6):
        toks = prompts[s % 2] + rng.integers(0, 500, int(rng.integers(1, 30))).tolist()
        cached = cache.add_sequence(s, toks)
        table = cache.table(s)
        _write(kc, vc, [_kv_row(toks[:p + 1]) for p in range(cached, len(toks))],
               [table[p // BS] * BS + p % BS for p in range(cached, len(toks))], err)
        tokens[s] = toks
    assert cache.stats()["hit_tokens"] > 0
    live = list(range(6))
    host_k = host_v = None
    swapped = None
    max_len = 256
    ws = torch.empty(max(256, pa.pa_decode_workspace_size(8, HKV * GROUP, HKV, D, max_len, P)),
                     dtype=torch.uint8, device=G.DEV)
    gen = torch.Generator().manual_seed(23)
    for step in range(48):
        if step == 16:    # swap sequence 3 out: every block of its table to host, then free them
            swapped = 3
            table = cache.table(swapped)
            host_k = torch.empty((len(table), HKV, BS, D), dtype=torch.float16).pin_memory()
            host_v = torch.empty_like(host_k).pin_memory()
            pairs = torch.tensor([[b, i] for i, b in enumerate(table)], dtype=torch.int64, device=G.DEV)
            pa.pa_swap_blocks(kc, vc, host_k, host_v, pairs, "out", device_error=err)
            torch.cuda.synchronize()
            cache.free_sequence(swapped)
            live.remove(swapped)
        if step == 28:    # swap it back in: re-admit (the prompt hits), restore the blocks that missed
            cached = cache.add_sequence(swapped, tokens[swapped])
            table = cache.table(swapped)
            pairs = torch.tensor([[i, table[i]] for i in range(cached // BS, len(table))],
                                 dtype=torch.int64, device=G.DEV)
            pa.pa_swap_blocks(kc, vc, host_k, host_v, pairs, "in", device_error=err)
            live = sorted(live + [swapped])
        rows, slots = [], []
        for s in live:
            tokens[s].append(int(rng.integers(0, 500)))
            slots.append(cache.append_token(s, tokens[s][-1]))
            rows.append(_kv_row(tokens[s]))
        _write(kc, vc, rows, slots, err)
        width = max(len(cache.table(s)) for s in live)
        tables, lens = cache.block_tables(live, width)
        q = torch.randn((len(live), HKV * GROUP, D), generator=gen).half()
        out = torch.empty_like(q).to(G.DEV)
        pa.pa_decode(out, q.to(G.DEV), kc, vc, torch.from_numpy(tables).to(G.DEV),
                     torch.from_numpy(lens).to(G.DEV), int(lens.max()), 1.0 / np.sqrt(D),
                     partition_size=P, workspace=ws, device_error=err)
        if step % 6 == 5 or step in (16, 28, 29, 47):
            torch.cuda.synchronize()
            assert int(err.item()) == 0, step
            _check(out, q, live, tokens)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max(len(t) for t in tokens.values()) > 2 * P   # several partitions by the end
