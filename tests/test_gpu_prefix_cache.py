"""Prefix cache -> cache writes of the missed tokens only -> paged prefill of
those tokens and paged decode (GPU), against the oracle's attention over
each sequence's logical K/V.

Every token's K/V row is a function of the token ids up to and including
it (seeded by their bytes), the way a model's K/V depend on the prefix.
So a block the cache shares holds the right values for every sequence
that maps it exactly when the sharing is right, and the expected output
of a sequence depends on its own tokens only."""
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
from oracle import attention as A
from tests import _gpu as G

pytestmark = pytest.mark.gpu

HKV, GROUP, D, BS = 2, 4, 64, 16


def _kv_row(prefix):
    seed = zlib.crc32(np.asarray(prefix, dtype=np.int32).tobytes())
    r = np.random.default_rng(seed).standard_normal((2, HKV, D))
    return r.astype(np.float16)                      # K and V rows [Hkv, d]


def _write(c, s, toks, start, kc, vc, err):
    if start >= len(toks):
        return
    rows = np.stack([_kv_row(toks[:p + 1]) for p in range(start, len(toks))])
    table = c.table(s)
    slots = [table[p // BS] * BS + p % BS for p in range(start, len(toks))]
    k = torch.from_numpy(rows[:, 0].copy()).to(G.DEV)
    v = torch.from_numpy(rows[:, 1].copy()).to(G.DEV)
    pa.pa_reshape_and_cache(k, v, torch.tensor(slots, dtype=torch.int64, device=G.DEV), kc, vc,
                            device_error=err)


def test_prefix_cached_tables_decode_like_the_oracle():
    rng = np.random.default_rng(11)
    nb = 150
    c = pa.PrefixCache(nb, BS, rng.permutation(nb))
    kc = torch.full((nb, HKV, BS, D), float("nan"), dtype=torch.float16, device=G.DEV)
    vc = torch.full_like(kc, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    prompts = [rng.integers(0, 1000, n).tolist() for n in (0, 70, 160, 333)]
    tokens, live, hits = {}, [], 0

    def with_room(fn):
        """Run fn; when the pool is out of blocks, finish the ten oldest
        requests (their blocks stay cached) and retry."""
        nonlocal live
        while True:
            try:
                return fn()
            except pa.OutOfBlocks:
                assert live, "pool too small for one request"
                for old in live[:10]:
                    c.free_sequence(old)
                live = live[10:]

    for s in range(60):
        toks = prompts[int(rng.integers(len(prompts)))] + \
            rng.integers(0, 1000, int(rng.integers(1, 90))).tolist()
        cached = with_room(lambda: c.add_sequence(s, toks))
        hits += cached
        _write(c, s, toks, cached, kc, vc, err)
        for _ in range(int(rng.integers(0, 20))):    # a few decoded tokens
            toks.append(int(rng.integers(0, 1000)))
            slot = with_room(lambda: c.append_token(s, toks[-1]))
            row = _kv_row(toks)
            pa.pa_reshape_and_cache(torch.from_numpy(row[0][None].copy()).to(G.DEV),
                                    torch.from_numpy(row[1][None].copy()).to(G.DEV),
                                    torch.tensor([slot], device=G.DEV), kc, vc, device_error=err)
        tokens[s] = toks
        live.append(s)
    assert hits > 0 and c.stats()["evictions"] > 0
    width = max(len(c.table(s)) for s in live)
    tables, lens = c.block_tables(live, width)
    S = len(live)
    q = torch.randn((S, HKV * GROUP, D), generator=torch.Generator().manual_seed(5)).half()
    out = torch.empty_like(q).to(G.DEV)
    pa.pa_decode(out, q.to(G.DEV), kc, vc, torch.from_numpy(tables).to(G.DEV),
                 torch.from_numpy(lens).to(G.DEV), int(lens.max()), 1.0 / np.sqrt(D),
                 partition_size=128, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.float().cpu().numpy()
    qv = q.double().numpy()
    worst = 0.0
    for i, s in enumerate(live):
        toks = tokens[s]
        rows = np.stack([_kv_row(toks[:p + 1]) for p in range(len(toks))]).astype(np.float64)
        for hq in range(HKV * GROUP):
            h = hq // GROUP
            ref = A.attend(qv[i, hq], rows[:, 0, h], rows[:, 1, h], 1.0 / np.sqrt(D))[0]
            e = float(np.abs(got[i, hq] - ref).max())
            worst = max(worst, e)
            assert e <= max(2e-3, float(G.ulp(ref, "f16").max())), (s, hq, e)
    print(f"{S} sequences, {hits} prompt tokens hit, max |err| {worst:.2e}")


def test_prefix_hit_prefill_then_decode():
    """A request's whole flow: the prefix cache maps the prompt's cached
    blocks; only the missed tokens' K/V are written, and only those tokens
    are prefilled, over the shared blocks; then one decoded token per
    request attends to its whole sequence.  A prompt that hits in full
    prefills its last token again (its logits are still needed)."""
    rng = np.random.default_rng(23)
    nb = 600
    c = pa.PrefixCache(nb, BS, rng.permutation(nb))
    kc = torch.full((nb, HKV, BS, D), float("nan"), dtype=torch.float16, device=G.DEV)
    vc = torch.full_like(kc, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    prompts = [rng.integers(0, 1000, n).tolist() for n in (48, 130, 257)]
    seqs, tokens, q_lens = list(range(24)), {}, []
    for s in seqs:
        own = int(rng.integers(0, 40)) if s % 4 else 0
        toks = prompts[s % 3] + rng.integers(0, 1000, own).tolist()
        cached = c.add_sequence(s, toks)
        n = max(1, len(toks) - cached)
        _write(c, s, toks, len(toks) - n, kc, vc, err)
        tokens[s], q_lens = toks, q_lens + [n]
    assert c.stats()["hit_tokens"] > 0 and min(q_lens) == 1
    Hq, scale = HKV * GROUP, 1.0 / np.sqrt(D)
    gen = torch.Generator().manual_seed(8)
    q = torch.randn((sum(q_lens), Hq, D), generator=gen).half()
    width = max(len(c.table(s)) + 1 for s in seqs)
    tables, lens = c.block_tables(seqs, width)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32, device=G.DEV)
    out = torch.empty_like(q).to(G.DEV)
    pa.pa_prefill(out, q.to(G.DEV), cu, kc, vc, torch.from_numpy(tables).to(G.DEV),
                  torch.from_numpy(lens).to(G.DEV), max(q_lens), scale, device_error=err)
    # one decoded token per request
    for s in seqs:
        tokens[s].append(int(rng.integers(0, 1000)))
        slot = c.append_token(s, tokens[s][-1])
        row = _kv_row(tokens[s])
        pa.pa_reshape_and_cache(torch.from_numpy(row[0][None].copy()).to(G.DEV),
                                torch.from_numpy(row[1][None].copy()).to(G.DEV),
                                torch.tensor([slot], device=G.DEV), kc, vc, device_error=err)
    tables2, lens2 = c.block_tables(seqs, width)
    q2 = torch.randn((len(seqs), Hq, D), generator=gen).half()
    out2 = torch.empty_like(q2).to(G.DEV)
    pa.pa_decode(out2, q2.to(G.DEV), kc, vc, torch.from_numpy(tables2).to(G.DEV),
                 torch.from_numpy(lens2).to(G.DEV), int(lens2.max()), scale, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, got2 = out.float().cpu().numpy(), out2.float().cpu().numpy()
    qv, qv2 = q.double().numpy(), q2.double().numpy()
    worst, row0 = 0.0, 0
    for i, s in enumerate(seqs):
        toks = tokens[s]
        rows = np.stack([_kv_row(toks[:p + 1]) for p in range(len(toks))]).astype(np.float64)
        L, n = len(toks) - 1, q_lens[i]          # length at prefill time
        for h in range(HKV):
            heads = slice(h * GROUP, (h + 1) * GROUP)
            K, V = rows[:, 0, h], rows[:, 1, h]
            for j in range(n):
                p = L - n + j
                ref = A.attend(qv[row0 + j, heads], K[:p + 1], V[:p + 1], scale)
                e = np.abs(got[row0 + j, heads] - ref)
                assert not (e > np.maximum(G.TOL["f16"], G.ulp(ref, "f16"))).any(), ("prefill", s, j, h)
                worst = max(worst, float(e.max()))
            ref = A.attend(qv2[i, heads], K, V, scale)
            e = np.abs(got2[i, heads] - ref)
            assert not (e > np.maximum(G.TOL["f16"], G.ulp(ref, "f16"))).any(), ("decode", s, h)
            worst = max(worst, float(e.max()))
        row0 += n
    print(f"{len(seqs)} requests, {sum(q_lens)} tokens prefilled, max |err| {worst:.2e}")
