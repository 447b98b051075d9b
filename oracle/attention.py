"""Single-query decode attention over a paged KV cache, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

For sequence s with length L_s and query head hq, whose KV head is
h = hq // G (G = query heads / KV heads, the query group sharing one KV
head), the output is the plain definition of scaled dot-product attention
over the sequence's tokens 0..L_s-1:

    o[s, hq] = sum_i softmax_i(scale * <q[s, hq], k_i>) * v_i

where k_i and v_i are read through the block table: token i lives in
physical block ``block_tables[s][i // block_size]`` at offset
``i % block_size`` ([P1] §2.1, [P2] §2.2, [P3] §3.2: logical blocks map to
scattered physical blocks through a per-sequence table).  The pages never
write the attention formula down; this is the textbook definition the
paged layout exists to serve.  The softmax subtracts the maximum score
before exponentiating (an exact identity, used for range only).

Readings where the pages are silent: a sequence of length 0 yields zeros;
the output is the float64 value here, the device rounds it to the query's
dtype.
"""

from __future__ import annotations

import numpy as np

from .cache import head_scale, values


def gather(codes: np.ndarray, dtype: str, scale: float, table_row, length: int,
           kv_head: int, block_size: int) -> np.ndarray:
    """[length, head_dim] float64 rows of one KV head of one sequence
    (``scale``: that head's scale)."""
    pos = np.arange(length)
    blocks = np.asarray(table_row, dtype=np.int64)[pos // block_size]
    return values(codes[blocks, kv_head, pos % block_size, :], dtype, scale)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for query rows q [G, d]; K, V [L, d]."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]), dtype=np.float64)
    s = scale * (K @ q.T)                  # [L, G]
    p = np.exp(s - s.max(axis=0))          # [L, G]
    return (p.T @ V) / p.sum(axis=0)[:, None]


def paged_decode(q: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray,
                 dtype: str, block_tables, seq_lens, scale: float,
                 k_scale=1.0, v_scale=1.0, rows=None) -> np.ndarray:
    """Decode attention for every (s, hq), or only for the (s, hq) in ``rows``.

    q: [S, Hq, d] float64 query values; k_codes/v_codes: the cache codes
    [num_blocks, Hkv, block_size, d]; k_scale / v_scale: one number, or one
    per KV head ([P3] §6.3).  Returns float64 [S, Hq, d] (rows not requested
    are left as NaN).
    """
    S, Hq, d = q.shape
    Hkv, bs = k_codes.shape[1], k_codes.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    out = np.full((S, Hq, d), np.nan)
    wanted = None if rows is None else {(int(s), int(h)) for s, h in rows}
    for s in range(S):
        L = int(seq_lens[s])
        for h in range(Hkv):
            heads = [h * G + g for g in range(G)
                     if wanted is None or (s, h * G + g) in wanted]
            if not heads:
                continue
            K = gather(k_codes, dtype, head_scale(k_scale, h), block_tables[s], L, h, bs)
            V = gather(v_codes, dtype, head_scale(v_scale, h), block_tables[s], L, h, bs)
            out[s, heads] = attend(q[s, heads], K, V, scale)
    return out


def paged_prefill(q: np.ndarray, q_lens, k_codes: np.ndarray, v_codes: np.ndarray,
                  dtype: str, block_tables, seq_lens, scale: float,
                  k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """Causal attention of several new tokens per sequence over the paged cache.

    [P3] §4.2: after a prefix hit only the part that missed is computed.
    Sequence s holds L_s = seq_lens[s] tokens in the cache, of which the
    last n_s = q_lens[s] are new; new token j sits at position
    p = L_s - n_s + j and attends to the tokens at positions 0..p (itself
    included), read through the block table like the decode's:

        o[j, hq] = sum_{i <= p} softmax_i(scale * <q[j, hq], k_i>) * v_i

    q: [sum_s n_s, Hq, d] float64, the sequences' new tokens one after the
    other.  Returns float64 [sum_s n_s, Hq, d].
    """
    T, Hq, d = q.shape
    Hkv, bs = k_codes.shape[1], k_codes.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    q_lens = [int(n) for n in q_lens]
    if sum(q_lens) != T:
        raise ValueError("q rows must equal the sum of q_lens")
    out = np.zeros((T, Hq, d))
    row = 0
    for s, n in enumerate(q_lens):
        L = int(seq_lens[s])
        if n > L:
            raise ValueError("more new tokens than the sequence holds")
        for h in range(Hkv):
            K = gather(k_codes, dtype, head_scale(k_scale, h), block_tables[s], L, h, bs)
            V = gather(v_codes, dtype, head_scale(v_scale, h), block_tables[s], L, h, bs)
            for j in range(n):
                p = L - n + j
                heads = [h * G + g for g in range(G)]
                out[row + j, heads] = attend(q[row + j, heads], K[:p + 1], V[:p + 1], scale)
        row += n
    return out
