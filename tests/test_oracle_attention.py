"""Pins for the oracle's paged decode attention and cache ops (CPU only).

Pinned to: torch's scaled_dot_product_attention in float64 on the
contiguous (unpaged) sequence, a library routine; closed forms (equal keys
give the mean of V; a single token gives v_0; length 0 gives 0); brute force
with explicit Python loops on tiny inputs; and the allocator's own block
tables.  A few tests plant a mistake in the oracle and check a pin catches it.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle.allocator import BlockAllocator
from oracle.cache import PagedKVCache, bits_to_f64


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _fill(w):
    """Host cache after set-up and one step of workload ``w``."""
    c = PagedKVCache(w.num_blocks, w.Hkv, w.bs, w.d, w.cache_dtype, w.k_scale, w.v_scale)
    c.reshape_and_cache(_bits(w.ctx_k), _bits(w.ctx_v), w.src_dtype, w.ctx_slots)
    c.copy_blocks(w.cow_pairs)
    c.reshape_and_cache(_bits(w.new_k), _bits(w.new_v), w.src_dtype, w.new_slots)
    return c


def _qvals(w):
    return bits_to_f64(_bits(w.q), w.q_dtype)


def _logical(w, s, which):
    """[L, Hkv, d] source values of sequence s in logical order."""
    src = {"ctx": (w.ctx_k, w.ctx_v), "new": (w.new_k, w.new_v)}
    rows = []
    for kind, i in w.token_rows(s):
        t = src[kind][0 if which == "k" else 1][i]
        rows.append(bits_to_f64(_bits(t), w.src_dtype))
    return np.stack(rows) if rows else np.zeros((0, w.Hkv, w.d))


def _sdpa(q, K, V, scale, G):
    """torch SDPA in float64: q [Hq, d], K/V [L, Hkv, d] -> [Hq, d]."""
    qt = torch.from_numpy(q)[:, None, :]                      # [Hq, 1, d]
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    return torch.nn.functional.scaled_dot_product_attention(
        qt, Kt, Vt, scale=scale)[:, 0, :].numpy()


CASES = [
    # S, Hq, Hkv, d, bs, dtype, lens
    (3, 4, 4, 16, 16, "f16", [1, 17, 40]),
    (2, 4, 2, 8, 4, "bf16", [13, 30]),
    (4, 8, 1, 8, 8, "f16", [7, 8, 9, 64]),
    (2, 6, 3, 16, 2, "bf16", [5, 33]),
]


@pytest.mark.parametrize("case", CASES)
def test_paged_equals_contiguous_sdpa(case):
    S, Hq, Hkv, d, bs, dt, lens = case
    w = W.random_case(11, S, Hq, Hkv, d, bs, dt, dt, lens)
    c = _fill(w)
    out = A.paged_decode(_qvals(w), c.k, c.v, w.cache_dtype, w.block_tables,
                         w.seq_lens, w.scale)
    q = _qvals(w)
    for s in range(S):
        ref = _sdpa(q[s], _logical(w, s, "k"), _logical(w, s, "v"), w.scale, w.G)
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-12)


def test_permuting_physical_blocks_changes_nothing():
    w = W.random_case(3, 3, 4, 2, 16, 4, "f16", "f16", [9, 22, 31])
    c = _fill(w)
    base = A.paged_decode(_qvals(w), c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    rng = np.random.default_rng(5)
    for _ in range(3):
        perm = rng.permutation(w.num_blocks)           # old block b -> perm[b]
        k2, v2 = np.empty_like(c.k), np.empty_like(c.v)
        k2[perm], v2[perm] = c.k, c.v
        bt2 = perm[w.block_tables]
        out = A.paged_decode(_qvals(w), k2, v2, "f16", bt2, w.seq_lens, w.scale)
        np.testing.assert_array_equal(out, base)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(0)
    L, d = 37, 8
    K = np.tile(rng.standard_normal(d), (L, 1))
    V = rng.standard_normal((L, d))
    out = A.attend(rng.standard_normal((3, d)), K, V, 0.7)
    np.testing.assert_allclose(out, np.tile(V.mean(axis=0), (3, 1)), rtol=1e-13)


def test_single_token_gives_v0_and_empty_gives_zero():
    rng = np.random.default_rng(1)
    K, V = rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    np.testing.assert_allclose(A.attend(rng.standard_normal(8), K, V, 1.0)[0], V[0], rtol=1e-15)
    z = A.attend(rng.standard_normal(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert np.all(z == 0)


def _brute(q, K, V, scale):
    L = len(K)
    scores = [scale * sum(q[j] * K[i][j] for j in range(len(q))) for i in range(L)]
    m = max(scores)
    e = [math.exp(x - m) for x in scores]
    tot = sum(e)
    return [sum(e[i] * V[i][j] for i in range(L)) / tot for j in range(len(V[0]))]


@pytest.mark.parametrize("bs", [1, 2, 4, 16])
def test_brute_force_tiny(bs):
    rng = np.random.default_rng(bs)
    S, Hkv, G, d = 3, 2, 2, 4
    lens = [1, bs + 1, 40 if bs > 1 else 23]
    w = W.random_case(bs, S, Hkv * G, Hkv, d, bs, "f16", "f16", lens)
    c = _fill(w)
    out = A.paged_decode(_qvals(w), c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    q = _qvals(w)
    for s in range(S):
        K, V = _logical(w, s, "k"), _logical(w, s, "v")
        for hq in range(Hkv * G):
            h = hq // G
            ref = _brute(list(q[s, hq]), K[:, h].tolist(), V[:, h].tolist(), w.scale)
            np.testing.assert_allclose(out[s, hq], ref, rtol=1e-12, atol=1e-14)
    assert rng is not None


def test_stale_slots_are_never_read():
    w = W.random_case(2, 2, 2, 2, 8, 16, "f16", "f16", [3, 17])
    c = _fill(w)          # every unwritten slot holds NaN
    out = A.paged_decode(_qvals(w), c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    assert np.isfinite(out).all()


def test_fp8_cache_dequantises_with_scale():
    w = W.random_case(4, 2, 4, 2, 16, 16, "e4m3", "bf16", [20, 45],
                      k_scale=0.5, v_scale=2.0)
    c = _fill(w)
    out = A.paged_decode(_qvals(w), c.k, c.v, "e4m3", w.block_tables, w.seq_lens,
                         w.scale, w.k_scale, w.v_scale)
    from oracle import fp8
    q = _qvals(w)
    for s in range(2):
        Kraw, Vraw = _logical(w, s, "k"), _logical(w, s, "v")
        K = fp8.decode(fp8.quantize(Kraw.astype(np.float32), 0.5, "e4m3"), "e4m3") * 0.5
        V = fp8.decode(fp8.quantize(Vraw.astype(np.float32), 2.0, "e4m3"), "e4m3") * 2.0
        np.testing.assert_allclose(out[s], _sdpa(q[s], K, V, w.scale, w.G), rtol=1e-12)


@pytest.mark.parametrize("name", ["tiny"])
def test_workload_tables_match_allocator_replay(name):
    w = W.make_workload(name, 1, values=False)
    m = BlockAllocator(w.num_blocks, w.bs, pool_order=w.pool_order.tolist())
    for s in range(w.S):
        m.allocate(s, int(w.seq_lens[s]))
    for s in range(w.S):
        t = m.tables[s]
        assert list(w.block_tables[s, :len(t)]) == t
        assert w.new_slots[s] == m.slot(s, int(w.seq_lens[s]) - 1)


def test_prefix_workload_matches_allocator_replay():
    w = W.make_workload("qwen3-prefix", 2, values=False,
                        overrides=dict(S=12, prefix=64, suffix_lo=1, suffix_hi=40))
    m = BlockAllocator(w.num_blocks, w.bs, pool_order=w.pool_order.tolist())
    m.allocate(0, 64)
    for s in range(1, w.S):
        m.share_prefix(0, 64 // w.bs, s)
    for s in range(w.S):
        assert m.append(s, int(w.seq_lens[s]) - 64) == []
    for s in range(w.S):
        t = m.tables[s]
        assert list(w.block_tables[s, :len(t)]) == t
        assert w.new_slots[s] == m.slot(s, int(w.seq_lens[s]) - 1)
    for b in m.tables[0][:64 // w.bs]:
        assert m.refcount[b] == w.S


def test_beam_workload_matches_allocator_replay():
    w = W.make_workload("opt13b-beam", 3, values=False,
                        overrides=dict(prompts=6, len_lo=30, len_hi=200, bs=8))
    m = BlockAllocator(w.num_blocks, w.bs, pool_order=w.pool_order.tolist())
    B = 4
    P = w.S // B
    for i in range(P):
        m.allocate((i, 0), int(w.seq_lens[i * B]) - 1)
    for i in range(P):
        for b in range(1, B):
            m.fork((i, 0), (i, b))
    pairs = []
    for i in range(P):
        for b in range(B):
            pairs += m.append((i, b))
    assert [tuple(p) for p in w.cow_pairs.tolist()] == pairs
    for i in range(P):
        for b in range(B):
            t = m.tables[(i, b)]
            s = i * B + b
            assert list(w.block_tables[s, :len(t)]) == t
            assert w.new_slots[s] == m.slot((i, b), int(w.seq_lens[s]) - 1)


def test_beam_step_matches_logical_sequences():
    w = W.make_workload("opt13b-beam", 4, overrides=dict(
        prompts=3, len_lo=20, len_hi=70, bs=8, Hq=2, Hkv=2, d=16))
    c = _fill(w)
    q = _qvals(w)
    out = A.paged_decode(q, c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    for s in range(w.S):
        ref = _sdpa(q[s], _logical(w, s, "k"), _logical(w, s, "v"), w.scale, w.G)
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-12)


def test_reshape_and_cache_skips_padding_and_copy_blocks_copies():
    c = PagedKVCache(4, 2, 4, 8, "f16", fill_nan=False)
    rows = (np.arange(3 * 2 * 8, dtype=np.uint16).reshape(3, 2, 8) + 1)
    c.reshape_and_cache(rows, rows + 100, "f16", np.array([5, -1, 14]))
    assert (c.k[1, :, 1, :] == rows[0]).all() and (c.v[3, :, 2, :] == rows[2] + 100).all()
    assert int((c.k != 0).sum()) == 2 * 2 * 8
    c.copy_blocks([(1, 0)])
    assert (c.k[0] == c.k[1]).all() and (c.v[0] == c.v[1]).all()


# -- planted mistakes: each must be caught by a pin above ------------------

def _run_sdpa_pin():
    test_paged_equals_contiguous_sdpa(CASES[1])


def test_planted_wrong_head_mapping_is_caught(monkeypatch):
    orig = A.paged_decode

    def wrong(q, k, v, dtype, bt, lens, scale, ks=1.0, vs=1.0, rows=None):
        # KV head taken as hq % Hkv instead of hq // G
        S, Hq, d = q.shape
        Hkv = k.shape[1]
        out = np.empty((S, Hq, d))
        for s in range(S):
            for hq in range(Hq):
                K = A.gather(k, dtype, ks, bt[s], int(lens[s]), hq % Hkv, k.shape[2])
                V = A.gather(v, dtype, vs, bt[s], int(lens[s]), hq % Hkv, k.shape[2])
                out[s, hq] = A.attend(q[s, hq], K, V, scale)[0]
        return out

    monkeypatch.setattr(A, "paged_decode", wrong)
    with pytest.raises(AssertionError):
        _run_sdpa_pin()
    monkeypatch.setattr(A, "paged_decode", orig)


def test_planted_missing_max_subtraction_sign_is_caught(monkeypatch):
    def wrong_attend(q, K, V, scale):
        q = np.atleast_2d(q)
        s = scale * (K @ q.T)
        p = np.exp(s + s.max(axis=0))      # wrong sign: still finite here
        p = p / p.sum(axis=0)
        return (p.T @ V) * 0.999           # and a dropped normalisation term
    monkeypatch.setattr(A, "attend", wrong_attend)
    with pytest.raises(AssertionError):
        _run_sdpa_pin()


def test_planted_offset_error_in_gather_is_caught(monkeypatch):
    orig = A.gather

    def wrong_gather(codes, dtype, scale, row, length, h, bs):
        pos = np.arange(length)
        blocks = np.asarray(row)[pos // bs]
        from oracle.cache import values
        return values(codes[blocks, h, (pos + 1) % bs, :], dtype, scale)

    monkeypatch.setattr(A, "gather", wrong_gather)
    with pytest.raises(AssertionError):
        _run_sdpa_pin()
    monkeypatch.setattr(A, "gather", orig)


def test_swap_out_and_in_round_trip():
    """Blocks swapped out to a second pool and back into other device blocks
    hold the same codes; decoding through the remapped tables gives the same
    result; every block no pair names is untouched."""
    w = W.random_case(12, 3, 4, 2, 16, 8, "e4m3", "bf16", [13, 30, 7], k_scale=0.5)
    c = _fill(w)
    before_k, before_v = c.k.copy(), c.v.copy()
    host = PagedKVCache(10, w.Hkv, w.bs, w.d, w.cache_dtype, fill_nan=False)
    seq1 = [int(b) for b in w.block_tables[1, :-(-30 // w.bs)]]
    out_pairs = [(b, i) for i, b in enumerate(seq1)]
    c.swap_blocks(host, out_pairs, "out")
    for b, i in out_pairs:
        assert (host.k[i] == c.k[b]).all() and (host.v[i] == c.v[b]).all()
    assert (host.k[len(seq1):] == 0).all()
    used = {int(b) for s in range(w.S) for b in w.block_tables[s, :-(-int(w.seq_lens[s]) // w.bs)]}
    free = [b for b in range(w.num_blocks) if b not in used][:len(seq1)]
    c.swap_blocks(host, [(i, f) for i, f in enumerate(free)], "in")
    for (b, i), f in zip(out_pairs, free):
        assert (c.k[f] == before_k[b]).all() and (c.v[f] == before_v[b]).all()
    untouched = [b for b in range(w.num_blocks) if b not in free]
    assert (c.k[untouched] == before_k[untouched]).all()
    tables = w.block_tables.copy()
    tables[1, :len(free)] = free
    q = _qvals(w)
    a = A.paged_decode(q, before_k, before_v, "e4m3", w.block_tables, w.seq_lens, w.scale, 0.5)
    b = A.paged_decode(q, c.k, c.v, "e4m3", tables, w.seq_lens, w.scale, 0.5)
    np.testing.assert_array_equal(a, b)
    with pytest.raises(ValueError):
        c.swap_blocks(PagedKVCache(4, w.Hkv, 16, w.d, w.cache_dtype), [(0, 0)], "out")


def _prefill_case(seed, lens, q_lens, Hq=4, Hkv=2, d=16, bs=4, dtype="f16"):
    w = W.random_case(seed, len(lens), Hq, Hkv, d, bs, dtype, dtype, lens)
    c = _fill(w)
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((sum(q_lens), Hq, d))
    return w, c, q


def test_prefill_whole_sequence_equals_causal_sdpa():
    lens = [9, 23, 1]
    w, c, q = _prefill_case(40, lens, lens)
    out = A.paged_prefill(q, lens, c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    row = 0
    for s, L in enumerate(lens):
        K = torch.from_numpy(np.stack([_logical(w, s, "k")[:, h] for h in range(w.Hkv)]))
        V = torch.from_numpy(np.stack([_logical(w, s, "v")[:, h] for h in range(w.Hkv)]))
        Kq, Vq = K.repeat_interleave(w.G, 0), V.repeat_interleave(w.G, 0)
        Q = torch.from_numpy(q[row:row + L]).transpose(0, 1)          # [Hq, L, d]
        mask = torch.ones(L, L, dtype=torch.bool).tril()
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kq, Vq, attn_mask=mask,
                                                               scale=w.scale)
        np.testing.assert_allclose(out[row:row + L], ref.transpose(0, 1).numpy(), rtol=1e-12,
                                   atol=1e-14)
        row += L


def test_prefill_last_row_is_the_decode():
    lens, q_lens = [30, 17, 5], [7, 17, 1]
    w, c, q = _prefill_case(41, lens, q_lens, Hq=8, Hkv=2)
    out = A.paged_prefill(q, q_lens, c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    last = np.cumsum(q_lens) - 1
    dec = A.paged_decode(q[last], c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    np.testing.assert_allclose(out[last], dec, rtol=1e-13, atol=1e-15)


def test_prefill_of_the_missed_suffix_equals_the_full_prefill():
    """[P3] §4.2: with the prefix cached, computing only the new tokens gives
    the rows a prefill of the whole sequence gives them."""
    lens = [26, 40]
    w, c, q_full = _prefill_case(42, lens, lens)
    full = A.paged_prefill(q_full, lens, c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    cached = [16, 36]
    q_lens = [L - k for L, k in zip(lens, cached)]
    sel = np.concatenate([np.arange(k, L) + off for k, L, off in
                          zip(cached, lens, np.cumsum([0] + lens[:-1]))])
    part = A.paged_prefill(q_full[sel], q_lens, c.k, c.v, "f16", w.block_tables, w.seq_lens,
                           w.scale)
    np.testing.assert_allclose(part, full[sel], rtol=1e-13, atol=1e-15)


def test_prefill_brute_force_tiny():
    lens, q_lens = [6, 3], [4, 3]
    w, c, q = _prefill_case(43, lens, q_lens, Hq=2, Hkv=1, d=3, bs=2)
    out = A.paged_prefill(q, q_lens, c.k, c.v, "f16", w.block_tables, w.seq_lens, w.scale)
    row = 0
    for s, (L, n) in enumerate(zip(lens, q_lens)):
        K, V = _logical(w, s, "k")[:, 0], _logical(w, s, "v")[:, 0]
        for j in range(n):
            p = L - n + j
            for hq in range(2):
                sc = [w.scale * sum(q[row + j, hq, e] * K[i, e] for e in range(3)) for i in range(p + 1)]
                mx = max(sc)
                ws = [math.exp(x - mx) for x in sc]
                ref = [sum(ws[i] * V[i, e] for i in range(p + 1)) / sum(ws) for e in range(3)]
                np.testing.assert_allclose(out[row + j, hq], ref, rtol=1e-12)
        row += n


def test_planted_off_by_one_causal_mask_fails(monkeypatch):
    real = A.attend
    monkeypatch.setattr(A, "attend", lambda q, K, V, scale: real(q, K[:-1] if len(K) > 1 else K,
                                                                 V[:-1] if len(V) > 1 else V, scale))
    with pytest.raises(AssertionError):
        test_prefill_whole_sequence_equals_causal_sdpa()


def test_prefill_int8_per_head_scales_equal_dequantised_sdpa():
    """Prefill over an INT8 cache with one scale per KV head ([P3] §6.3) is
    causal attention over code x scale of the head: the codes are read here
    as two's-complement bytes and gathered through the tables with NumPy,
    and the attention is torch's."""
    lens, q_lens = [21, 9], [13, 9]
    ks, vs = (0.05, 0.11), (0.07, 0.03)
    w = W.random_case(44, 2, 4, 2, 16, 4, "int8", "f16", lens, k_scale=ks, v_scale=vs)
    c = _fill(w)
    q = np.random.default_rng(44).standard_normal((sum(q_lens), 4, 16))
    out = A.paged_prefill(q, q_lens, c.k, c.v, "int8", w.block_tables, w.seq_lens, w.scale, ks, vs)
    kf, vf = c.k.view(np.int8).astype(np.float64), c.v.view(np.int8).astype(np.float64)
    row = 0
    for s, (L, n) in enumerate(zip(lens, q_lens)):
        blocks = w.block_tables[s, :-(-L // w.bs)]
        K = kf[blocks].transpose(1, 0, 2, 3).reshape(w.Hkv, -1, w.d)[:, :L] * np.array(ks)[:, None, None]
        V = vf[blocks].transpose(1, 0, 2, 3).reshape(w.Hkv, -1, w.d)[:, :L] * np.array(vs)[:, None, None]
        Kq = torch.from_numpy(K).repeat_interleave(w.G, 0)
        Vq = torch.from_numpy(V).repeat_interleave(w.G, 0)
        Q = torch.from_numpy(q[row:row + n]).transpose(0, 1)
        mask = torch.arange(L)[None, :] <= torch.arange(L - n, L)[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kq, Vq, attn_mask=mask, scale=w.scale)
        np.testing.assert_allclose(out[row:row + n], ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-14)
        row += n
