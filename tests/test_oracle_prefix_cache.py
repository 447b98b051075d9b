"""Pins for the oracle's prefix cache (CPU only).

Pinned to: what the pages state about prefix caching (a shared system
prompt is stored once and hit by every later request; blocks are shared
through reference counts and return to the pool only at zero; a hit needs
the whole prefix to match), the hit-rate arithmetic of the two-request
experiment in [P3] §5 (first request 0%, second the whole shared prefix,
about half overall), closed forms for block counts, brute-force content
checks over random operation sequences, and planted mistakes.
"""
import random

import pytest

from oracle.prefix_cache import OutOfBlocks, PrefixCache


def _toks(rng, n, vocab=50):
    return [rng.randrange(vocab) for _ in range(n)]


def test_shared_system_prompt_is_stored_once():
    bs = 16
    c = PrefixCache(64, bs)
    system = list(range(1000, 1000 + 10 * bs))          # 10 full blocks
    got = [c.add_sequence(s, system + [s] * 7) for s in range(4)]
    assert got == [0, 10 * bs, 10 * bs, 10 * bs]
    t = [c.table(s) for s in range(4)]
    assert all(x[:10] == t[0][:10] for x in t)           # one copy of the prompt
    assert len({x[10] for x in t}) == 4                   # private partial blocks
    for b in t[0][:10]:
        assert c.ref[b] == 4
    assert c.stats()["used_blocks"] == 10 + 4


def test_two_request_experiment_hit_rate():
    """[P3] §5: two requests with one long system prompt; the first hits
    nothing, the second hits the whole prompt; the log's overall rate is
    about half.  With a prompt of P full blocks and questions of q tokens
    the rate is exactly P*bs / (2*(P*bs + q))."""
    bs, P, q = 16, 50, 12
    c = PrefixCache(256, bs)
    system = list(range(P * bs))
    assert c.add_sequence(0, system + [7] * q) == 0
    c.free_sequence(0)                                  # the first request finished
    assert c.add_sequence(1, system + [9] * q) == P * bs
    assert c.hit_rate() == pytest.approx(P * bs / (2 * (P * bs + q)))
    assert 0.45 < c.hit_rate() < 0.5


def test_hit_needs_the_whole_prefix():
    bs = 4
    c = PrefixCache(32, bs)
    c.add_sequence(0, [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12])
    # same second and third blocks, different first block: no hit at all
    assert c.add_sequence(1, [0, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12]) == 0
    # same first block, different second: only the first block hits
    assert c.add_sequence(2, [1, 2, 3, 4, 5, 6, 7, 0, 9, 10, 11, 12]) == 4
    assert c.table(2)[0] == c.table(0)[0] and c.table(2)[1] != c.table(0)[1]


def test_same_tokens_after_a_different_prefix_are_a_different_block():
    bs = 4
    A, B, C = [1, 2, 3, 4], [5, 6, 7, 8], [9, 9, 9, 9]
    c = PrefixCache(32, bs)
    c.add_sequence(0, A + B)
    c.add_sequence(1, C + B)
    assert c.add_sequence(2, C + B + [1]) == 8
    assert c.table(2)[:2] == c.table(1)[:2]
    assert c.table(2)[1] != c.table(0)[1]      # B after C was computed with C before it


def test_partial_blocks_are_never_shared_until_full():
    bs = 4
    c = PrefixCache(16, bs)
    c.add_sequence(0, [1, 2, 3, 4, 5, 6])             # 1 full + partial
    assert c.add_sequence(1, [1, 2, 3, 4, 5, 6]) == 4  # the partial block is private
    assert c.table(0)[1] != c.table(1)[1]
    c.append_token(0, 7)
    c.append_token(0, 8)                              # seq 0's second block is now full
    assert c.add_sequence(2, [1, 2, 3, 4, 5, 6, 7, 8, 9]) == 8
    assert c.table(2)[:2] == c.table(0)[:2]


def test_reference_counts_and_return_to_pool():
    bs = 4
    c = PrefixCache(8, bs, pool_order=[3, 1, 4, 0, 5, 2, 6, 7])
    c.add_sequence(0, list(range(8)))                 # blocks 3, 1
    c.add_sequence(1, list(range(8)) + [99])          # hits 3, 1; fresh 4
    assert c.table(1) == [3, 1, 4]
    assert (c.ref[3], c.ref[1], c.ref[4]) == (2, 2, 1)
    c.free_sequence(0)
    assert (c.ref[3], c.ref[1]) == (1, 1) and c.free_order() == [0, 5, 2, 6, 7]
    c.free_sequence(1)                                # returned last block first
    assert c.free_order() == [0, 5, 2, 6, 7, 4, 1, 3]
    # the freed prompt blocks keep their content and are hit again
    assert c.add_sequence(2, list(range(8)) + [5]) == 8
    assert c.table(2)[:2] == [3, 1] and c.table(2)[2] == 0


def test_least_recently_freed_block_is_evicted_first():
    bs = 2
    c = PrefixCache(4, bs)
    c.add_sequence(0, [1, 1])          # block 0
    c.add_sequence(1, [2, 2])          # block 1
    c.add_sequence(2, [3, 3])          # block 2
    c.free_sequence(1)                 # free: 3, 1
    c.free_sequence(0)                 # free: 3, 1, 0
    c.add_sequence(3, [4, 4])          # takes 3 (never used)
    c.add_sequence(4, [5, 5])          # takes 1, evicting [2, 2]
    assert c.stats()["evictions"] == 1
    assert c.add_sequence(5, [1, 1]) == 2   # block 0 was kept: hit
    c.free_sequence(5)
    assert c.add_sequence(6, [2, 2]) == 0   # evicted: miss (takes block 0)
    assert c.table(6) == [0] and c.stats()["evictions"] == 2


def test_out_of_blocks_changes_nothing():
    bs = 4
    c = PrefixCache(3, bs)
    c.add_sequence(0, list(range(8)))
    before = (c.free_order(), dict(c.tables), list(c.ref), c.stats())
    with pytest.raises(OutOfBlocks):
        c.add_sequence(1, list(range(100, 112)))     # 3 fresh blocks, 1 free
    assert (c.free_order(), dict(c.tables), list(c.ref), c.stats()) == before
    assert c.add_sequence(1, list(range(8)) + [1, 2, 3]) == 8


def test_block_counts_closed_form():
    for bs in (1, 2, 4, 16):
        for n in range(1, 5 * bs + 2):
            c = PrefixCache(64, bs)
            c.add_sequence(0, list(range(n)))
            assert len(c.table(0)) == -(-n // bs)
            assert c.stats()["cached_blocks"] == n // bs


def _content(c, seq):
    return c.tokens[seq]


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_only_share_equal_content(seed):
    """Brute force: after every operation, each block's content (the tokens
    of every sequence that maps it, at its positions, and everything before
    it) is the same for all its users; counts and the free list agree."""
    rng = random.Random(seed)
    bs = rng.choice([2, 4, 8])
    nb = rng.randrange(40, 120)
    c = PrefixCache(nb, bs, pool_order=rng.sample(range(nb), nb))
    prefixes = [_toks(rng, rng.randrange(0, 6 * bs), vocab=4) for _ in range(3)]
    live, next_id = [], 0
    for _ in range(300):
        op = rng.random()
        try:
            if op < 0.4 or not live:
                p = rng.choice(prefixes)
                c.add_sequence(next_id, p + _toks(rng, rng.randrange(1, 3 * bs), vocab=4))
                live.append(next_id)
                next_id += 1
            elif op < 0.75:
                c.append_token(rng.choice(live), rng.randrange(4))
            else:
                s = live.pop(rng.randrange(len(live)))
                c.free_sequence(s)
        except OutOfBlocks:
            pass
        ok, why = c.check_invariants()
        assert ok, why
        owner = {}
        for s in live:
            toks = _content(c, s)
            for j, b in enumerate(c.table(s)):
                end = min(len(toks), (j + 1) * bs)
                full = end == (j + 1) * bs
                if full:
                    pre = tuple(toks[:end])
                    if b in owner:
                        assert owner[b] == pre, (b, owner[b], pre)
                    owner[b] = pre
                else:
                    # a partial block belongs to one sequence only
                    assert sum(b in c.table(o) for o in live) == 1


def test_planted_key_without_prefix_fails_a_pin(monkeypatch):
    """A key of the block's own tokens only (prefix dropped) would share
    blocks of different prefixes: the whole-prefix pin catches it."""
    monkeypatch.setattr(PrefixCache, "_block_key", lambda self, parent, toks: (None, tuple(toks)))
    with pytest.raises(AssertionError):
        test_same_tokens_after_a_different_prefix_are_a_different_block()
