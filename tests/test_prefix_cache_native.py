"""The native prefix cache (libpa's pa_prefix_cache_*, host code) against the
oracle on the same operation sequences: tables, cached-token counts, slots,
reference counts, free order and counters equal after every operation
(CPU only; no GPU needed for host code)."""
import random

import numpy as np
import pytest

from oracle import prefix_cache as O


def _native():
    import paged_kv_cache_54_gb300 as pa
    return pa


def _same_state(a, b, live, nb):
    assert a.stats() == b.stats()
    assert a.free_order() == b.free_order()
    for s in live:
        assert a.table(s) == b.table(s), s
    for blk in range(nb):
        assert a.ref_count(blk) == b.ref[blk]


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_the_oracle(seed):
    pa = _native()
    rng = random.Random(100 + seed)
    bs = rng.choice([1, 2, 4, 16])
    nb = rng.randrange(8, 200)
    order = rng.sample(range(nb), nb)
    vocab = rng.choice([2, 3, 50])
    nat, orc = pa.PrefixCache(nb, bs, order), O.PrefixCache(nb, bs, order)
    prefixes = [[rng.randrange(vocab) for _ in range(rng.randrange(0, 8 * bs))] for _ in range(4)]
    live, next_id = [], 0
    for step in range(400):
        op = rng.random()
        if op < 0.35 or not live:
            toks = rng.choice(prefixes) + [rng.randrange(vocab) for _ in range(rng.randrange(0, 3 * bs))]
            res = []
            for c in (nat, orc):
                try:
                    res.append(c.add_sequence(next_id, toks))
                except (O.OutOfBlocks, pa.OutOfBlocks):
                    res.append("oob")
            assert res[0] == res[1], (step, res)
            if res[0] != "oob":
                live.append(next_id)
            next_id += 1
        elif op < 0.75:
            s = rng.choice(live)
            tok = rng.randrange(vocab)
            res = []
            for c in (nat, orc):
                try:
                    res.append(c.append_token(s, tok))
                except (O.OutOfBlocks, pa.OutOfBlocks):
                    res.append("oob")
            assert res[0] == res[1], (step, res)
        else:
            s = live.pop(rng.randrange(len(live)))
            nat.free_sequence(s)
            orc.free_sequence(s)
        _same_state(nat, orc, live, nb)
    nat.close()


def test_shared_prompt_tables_for_decode():
    """256 requests with one 1024-token prompt and their own suffixes (the
    shared-prefix decode workload's structure): one copy of the prompt's 64
    blocks, referenced 256 times; padded tables and lengths as pa_decode
    reads them."""
    pa = _native()
    rng = np.random.default_rng(3)
    bs, S = 16, 256
    prompt = rng.integers(0, 32000, 1024).tolist()
    c = pa.PrefixCache(20000, bs, rng.permutation(20000))
    cached = []
    for s in range(S):
        suffix = rng.integers(0, 32000, int(rng.integers(16, 513))).tolist()
        cached.append(c.add_sequence(s, prompt + suffix))
    assert cached[0] == 0 and all(x == 1024 for x in cached[1:])
    width = max(len(c.table(s)) for s in range(S))
    tables, lens = c.block_tables(range(S), width)
    assert (tables[:, :64] == tables[0, :64]).all()
    for b in tables[0, :64]:
        assert c.ref_count(int(b)) == S
    st = c.stats()
    assert st["hit_tokens"] == 1024 * (S - 1)
    assert st["used_blocks"] == 64 + sum(-(-(int(L) - 1024) // bs) for L in lens)


def test_invalid_calls_are_refused():
    pa = _native()
    with pytest.raises(ValueError):
        pa.PrefixCache(4, 2, [0, 1, 1, 3])          # not a permutation
    c = pa.PrefixCache(4, 2)
    c.add_sequence(0, [1, 2, 3])
    with pytest.raises(pa.PaError):
        c.add_sequence(0, [1])                      # exists
    with pytest.raises(pa.PaError):
        c.free_sequence(7)                          # unknown
    with pytest.raises(pa.OutOfBlocks):
        c.add_sequence(1, list(range(10)))          # 5 blocks, 2 free
    with pytest.raises(pa.PaError):
        c.block_tables([0], 1)                      # 2 blocks > width 1
    assert c.stats()["used_blocks"] == 2
