"""Seeded synthetic workloads for the paged decode path.

This module only draws inputs and lays out their structure; it holds none of
the attention or quantisation arithmetic.  It feeds both the device path
(tests, ``bench.py``, ``smoke``) and the CPU oracle, which receive the same
arrays.

Structure (all integer draws from numpy PCG64 with the given seed; K/V/q
values from ``torch.randn`` with a generator seeded the same way on the
device the tensors live on, float32 N(0, 1) rounded to the storage dtype):

* ``seq_lens[s]`` is the length of sequence s *including* the token being
  decoded, which sits at position ``L - 1``.
* The physical pool is a seeded shuffle of ``0..num_blocks-1``.  Blocks are
  taken from its front in the order the operations below name them, the way
  a FIFO free pool hands them out:

  independent  (tiny, llama2-7b, gqa-fp8):
      for s in order: allocate(s, L_s)
  prefix       (qwen3-prefix):
      allocate(0, prefix); share_prefix(0, prefix_blocks, s) for s >= 1;
      then for s in order: append(s, L_s - prefix)
  beam         (opt13b-beam):
      for each prompt i: allocate(i, L_i - 1); fork it into beams 1..3;
      then for prompt i, beam b = 0..3 in order: append one token.  When the
      prompt's last block is partial and shared by 4 beams, beams 0..2 take a
      new block and copy the old one (copy-on-write); beam 3 finds the old
      block exclusively held and writes in place.  When the last block is
      full every beam takes a fresh block.  Decode row 4*i + b is beam b.

* Context tokens (every position before the decoded one) are written once at
  set-up; a *step* is: copy the copy-on-write pairs, write the decoded
  tokens, decode.

* ``token_rows(s)`` names, for each position of sequence s, the input row
  that supplies its K/V: ``("ctx", index)`` or ``("new", index)``.  It is
  the logical sequence, independent of the block tables.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

try:  # torch is only needed for the value tensors
    import torch
except ImportError:  # pragma: no cover
    torch = None

TORCH_DTYPES = {}
if torch is not None:
    TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


# ---------------------------------------------------------------------------
# The five named workloads (sizes as stated for each; pool factor 1.25 where
# the size is not stated).
# ---------------------------------------------------------------------------
CONFIGS: Dict[str, dict] = {
    "tiny": dict(
        kind="independent", S=4, len_lo=1, len_hi=100, Hq=4, Hkv=4, d=64,
        bs=16, num_blocks=64, cache_dtype="f16", q_dtype="f16",
        scale=1.0 / 8.0, partition_size=0, layers_of_model=None),
    "llama2-7b": dict(
        kind="independent", S=64, len_lo=512, len_hi=4096, Hq=32, Hkv=32,
        d=128, bs=16, pool_factor=1.25, cache_dtype="f16", q_dtype="f16",
        partition_size=0, layers_of_model=32),
    "qwen3-prefix": dict(
        kind="prefix", S=256, prefix=1024, suffix_lo=16, suffix_hi=512,
        Hq=16, Hkv=8, d=128, bs=16, pool_factor=1.25, cache_dtype="bf16",
        q_dtype="bf16", partition_size=0, layers_of_model=28),
    "opt13b-beam": dict(
        kind="beam", prompts=32, beams=4, len_lo=2048, len_hi=8192, Hq=40,
        Hkv=40, d=128, bs=32, pool_factor=1.25, cache_dtype="f16",
        q_dtype="f16", partition_size=0, layers_of_model=40),
    "gqa-fp8": dict(
        kind="independent", S=128, len_lo=256, len_hi=32768, log_uniform=True,
        Hq=64, Hkv=8, d=128, bs=16, pool_factor=1.25, cache_dtype="e4m3",
        q_dtype="bf16", src_dtype="bf16", k_scale=1.0, v_scale=1.0,
        partition_size=512, layers_of_model=80),
    # The gqa-fp8 shapes with an int8 cache and one scale per KV head: 127
    # codes span about 5 standard deviations of the N(0, 1) values, a little
    # more for each further head.
    "gqa-int8": dict(
        kind="independent", S=128, len_lo=256, len_hi=32768, log_uniform=True,
        Hq=64, Hkv=8, d=128, bs=16, pool_factor=1.25, cache_dtype="int8",
        q_dtype="bf16", src_dtype="bf16",
        k_scale=tuple(0.04 + 0.0025 * h for h in range(8)),
        v_scale=tuple(0.045 - 0.0025 * h for h in range(8)),
        partition_size=512, layers_of_model=80),
}
CONFIG_ORDER = ["tiny", "llama2-7b", "qwen3-prefix", "opt13b-beam", "gqa-fp8"]
EXTRA_CONFIGS = ["gqa-int8"]
ALL_CONFIGS = CONFIG_ORDER + EXTRA_CONFIGS


def config_seed(name: str) -> int:
    """Default seed of a named workload (its position, from 1)."""
    return ALL_CONFIGS.index(name) + 1
BYTE_DTYPES = ("e4m3", "e5m2", "int8")


def _scale(x):
    """A scale as given: one number, or a tuple of one per KV head."""
    if np.ndim(x) == 0:
        return float(x)
    return tuple(float(v) for v in x)


@dataclass
class Workload:
    name: str
    S: int
    Hq: int
    Hkv: int
    d: int
    bs: int
    num_blocks: int
    cache_dtype: str
    q_dtype: str
    src_dtype: str
    scale: float
    k_scale: object               # float, or a tuple of one per KV head
    v_scale: object
    partition_size: int
    seq_lens: np.ndarray          # int32 [S]
    block_tables: np.ndarray      # int32 [S, width]
    pool_order: np.ndarray        # int64 [num_blocks]
    ctx_slots: np.ndarray         # int64 [Tc]
    new_slots: np.ndarray         # int64 [S]
    cow_pairs: np.ndarray         # int64 [n, 2]
    rows: List[List[Tuple[str, int]]] = field(repr=False, default=None)
    ctx_k: object = None          # torch [Tc, Hkv, d] in src_dtype
    ctx_v: object = None
    new_k: object = None          # torch [S, Hkv, d]
    new_v: object = None
    q: object = None              # torch [S, Hq, d] in q_dtype
    kind: str = "independent"

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.S else 0

    def token_rows(self, s: int) -> List[Tuple[str, int]]:
        return self.rows[s]

    # -- byte counts for the measurement ---------------------------------
    def elt_bytes(self) -> int:
        return 1 if self.cache_dtype in BYTE_DTYPES else 2

    def kv_logical_bytes(self) -> int:
        """Bytes of K and V the definition reads: sum_s L_s * Hkv * d * elt * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * self.d * self.elt_bytes() * 2

    def kv_unique_bytes(self) -> int:
        """Bytes of K and V in the distinct (block, token) slots that are read."""
        used = set()
        for s in range(self.S):
            L = int(self.seq_lens[s])
            nb = (L + self.bs - 1) // self.bs
            for j in range(nb):
                toks = min(self.bs, L - j * self.bs)
                blk = int(self.block_tables[s, j])
                used.add((blk, toks))
        per_block_tokens: Dict[int, int] = {}
        for blk, toks in used:
            per_block_tokens[blk] = max(per_block_tokens.get(blk, 0), toks)
        tokens = sum(per_block_tokens.values())
        return tokens * self.Hkv * self.d * self.elt_bytes() * 2


def _lens(rng, cfg, n):
    if cfg.get("log_uniform"):
        u = rng.uniform(math.log(cfg["len_lo"]), math.log(cfg["len_hi"]), n)
        return np.clip(np.rint(np.exp(u)), cfg["len_lo"], cfg["len_hi"]).astype(np.int64)
    return rng.integers(cfg["len_lo"], cfg["len_hi"] + 1, n).astype(np.int64)


def _ceil(a, b):
    return (a + b - 1) // b


def build_structure(name: str, seed: int, overrides: Optional[dict] = None,
                    lens=None) -> dict:
    """Integer structure of a workload: lengths, pool, tables, slots, pairs.

    ``name`` selects a named workload (``overrides`` replaces some of its
    keys) or, with ``name=None``, ``overrides`` is the whole configuration.
    ``lens`` gives the lengths explicitly instead of drawing them.
    """
    cfg = dict(CONFIGS[name]) if name is not None else {}
    if overrides:
        cfg.update(overrides)
    rng = np.random.Generator(np.random.PCG64(seed))
    bs = cfg["bs"]
    kind = cfg["kind"]
    if kind == "independent":
        S = cfg["S"]
        lens = _lens(rng, cfg, S) if lens is None else np.asarray(lens, dtype=np.int64)
        need = int(sum(_ceil(int(L), bs) for L in lens))
    elif kind == "prefix":
        S = cfg["S"]
        suffix = rng.integers(cfg["suffix_lo"], cfg["suffix_hi"] + 1, S).astype(np.int64)
        lens = cfg["prefix"] + suffix
        if cfg["prefix"] % bs:
            raise ValueError("prefix must fill whole blocks")
        need = cfg["prefix"] // bs + int(sum(_ceil(int(x), bs) for x in suffix))
    elif kind == "beam":
        P, B = cfg["prompts"], cfg["beams"]
        S = P * B
        plen = _lens(rng, cfg, P)          # decode length of every beam of prompt i
        lens = np.repeat(plen, B)
        need = int(sum(_ceil(int(L) - 1, bs) + B for L in plen))
    else:
        raise ValueError(kind)
    nb = cfg.get("num_blocks") or int(math.ceil(cfg["pool_factor"] * need))
    if nb < need:
        raise ValueError("pool too small")
    pool = rng.permutation(nb).astype(np.int64)
    cursor = 0

    def take(n):
        nonlocal cursor
        out = pool[cursor:cursor + n].tolist()
        if len(out) < n:
            raise MemoryError("pool exhausted")
        cursor += n
        return out

    tables: List[List[int]] = []
    ctx_slots: List[int] = []
    new_slots: List[int] = []
    rows: List[List[Tuple[str, int]]] = []
    pairs: List[Tuple[int, int]] = []

    def slot(table, p):
        return table[p // bs] * bs + p % bs

    if kind == "independent":
        for s in range(S):
            L = int(lens[s])
            t = take(_ceil(L, bs))
            tables.append(t)
            r = []
            for p in range(L - 1):
                r.append(("ctx", len(ctx_slots)))
                ctx_slots.append(slot(t, p))
            if L > 0:
                r.append(("new", s))
            new_slots.append(slot(t, L - 1) if L > 0 else -1)
            rows.append(r)
    elif kind == "prefix":
        prefix = cfg["prefix"]
        pre = take(prefix // bs)
        for p in range(prefix):
            ctx_slots.append(slot(pre, p))
        for s in range(S):
            tables.append(list(pre))
        for s in range(S):
            L = int(lens[s])
            tables[s] = tables[s] + take(_ceil(L - prefix, bs))
        for s in range(S):
            L = int(lens[s])
            t = tables[s]
            r = [("ctx", p) for p in range(prefix)]
            for p in range(prefix, L - 1):
                r.append(("ctx", len(ctx_slots)))
                ctx_slots.append(slot(t, p))
            r.append(("new", s))
            new_slots.append(slot(t, L - 1))
            rows.append(r)
    else:  # beam
        P, B = cfg["prompts"], cfg["beams"]
        prompt_tables, prompt_rows = [], []
        for i in range(P):
            C = int(plen[i]) - 1
            t = take(_ceil(C, bs))
            prompt_tables.append(t)
            pr = []
            for p in range(C):
                pr.append(("ctx", len(ctx_slots)))
                ctx_slots.append(slot(t, p))
            prompt_rows.append(pr)
        for i in range(P):
            C = int(plen[i]) - 1
            base = prompt_tables[i]
            for b in range(B):
                if C % bs:                      # partial, shared last block
                    if b < B - 1:
                        (new,) = take(1)
                        pairs.append((base[-1], new))
                        t = base[:-1] + [new]
                    else:
                        t = list(base)
                else:                           # full last block: fresh block
                    t = base + take(1)
                tables.append(t)
                new_slots.append(slot(t, C))
                rows.append(prompt_rows[i] + [("new", i * B + b)])

    width = max(1, max(len(t) for t in tables))
    bt = np.zeros((S, width), dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    return dict(
        cfg=cfg, S=S, seq_lens=np.asarray(lens, dtype=np.int32), block_tables=bt,
        num_blocks=nb, pool_order=pool, ctx_slots=np.asarray(ctx_slots, dtype=np.int64),
        new_slots=np.asarray(new_slots, dtype=np.int64),
        cow_pairs=np.asarray(pairs, dtype=np.int64).reshape(-1, 2), rows=rows)


def make_workload(name: Optional[str], seed: int, device: str = "cpu",
                  overrides: Optional[dict] = None, values: bool = True,
                  lens=None) -> Workload:
    st = build_structure(name, seed, overrides, lens)
    cfg = st["cfg"]
    d, Hkv, Hq = cfg["d"], cfg["Hkv"], cfg["Hq"]
    cache_dtype = cfg["cache_dtype"]
    src_dtype = cfg.get("src_dtype", cache_dtype if cache_dtype in ("f16", "bf16") else "bf16")
    w = Workload(
        name=name or "case", S=st["S"], Hq=Hq, Hkv=Hkv, d=d, bs=cfg["bs"],
        num_blocks=st["num_blocks"], cache_dtype=cache_dtype,
        q_dtype=cfg["q_dtype"], src_dtype=src_dtype,
        scale=float(cfg.get("scale") or 1.0 / math.sqrt(d)),
        k_scale=_scale(cfg.get("k_scale", 1.0)), v_scale=_scale(cfg.get("v_scale", 1.0)),
        partition_size=int(cfg.get("partition_size", 0)),
        seq_lens=st["seq_lens"], block_tables=st["block_tables"],
        pool_order=st["pool_order"], ctx_slots=st["ctx_slots"],
        new_slots=st["new_slots"], cow_pairs=st["cow_pairs"], rows=st["rows"],
        kind=cfg["kind"])
    if values:
        if torch is None:
            raise RuntimeError("torch is required for value tensors")
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        Tc = len(w.ctx_slots)
        sd, qd = TORCH_DTYPES[src_dtype], TORCH_DTYPES[w.q_dtype]

        def randn(*shape, dtype):
            return torch.randn(*shape, generator=g, device=device,
                               dtype=torch.float32).to(dtype)

        w.ctx_k = randn(Tc, Hkv, d, dtype=sd)
        w.ctx_v = randn(Tc, Hkv, d, dtype=sd)
        w.new_k = randn(w.S, Hkv, d, dtype=sd)
        w.new_v = randn(w.S, Hkv, d, dtype=sd)
        w.q = randn(w.S, Hq, d, dtype=qd)
    return w


def random_case(seed: int, S: int, Hq: int, Hkv: int, d: int, bs: int,
                cache_dtype: str, q_dtype: str, lens, device: str = "cpu",
                pool_factor: float = 1.5, scale: Optional[float] = None,
                k_scale=1.0, v_scale=1.0,
                partition_size: int = 0) -> Workload:
    """A small independent-sequence workload with the given lengths."""
    cfg = dict(kind="independent", S=S, Hq=Hq, Hkv=Hkv, d=d, bs=bs,
               cache_dtype=cache_dtype, q_dtype=q_dtype, pool_factor=pool_factor,
               scale=scale, k_scale=k_scale, v_scale=v_scale,
               partition_size=partition_size)
    if cache_dtype in BYTE_DTYPES:
        cfg["src_dtype"] = q_dtype
    return make_workload(None, seed, device=device, overrides=cfg, lens=lens)


def subset(w: Workload, seqs, seed: int, device: str = "cpu") -> Workload:
    """The sequences ``seqs`` of ``w`` on their own: their blocks renumbered
    into a compact pool (same block-table structure and sharing), and fresh
    seeded values for just their tokens.  Used for bounded CPU samples."""
    seqs = list(seqs)
    bs = w.bs
    used = []
    for s in seqs:
        used += w.block_tables[s, :-(-int(w.seq_lens[s]) // bs)].tolist()
    remap = {b: i for i, b in enumerate(dict.fromkeys(used))}
    width = max(1, max(-(-int(w.seq_lens[s]) // bs) for s in seqs))
    bt = np.zeros((len(seqs), width), dtype=np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(w.seq_lens[s]) // bs)
        bt[i, :n] = [remap[b] for b in w.block_tables[s, :n]]
    ctx_map: Dict[int, int] = {}
    rows, ctx_slots, new_slots = [], [], []
    for i, s in enumerate(seqs):
        r = []
        for p, (kind, idx) in enumerate(w.token_rows(s)):
            slot = int(bt[i, p // bs]) * bs + p % bs
            if kind == "ctx":
                if idx not in ctx_map:
                    ctx_map[idx] = len(ctx_slots)
                    ctx_slots.append(slot)
                r.append(("ctx", ctx_map[idx]))
            else:
                r.append(("new", i))
        L = int(w.seq_lens[s])
        new_slots.append(int(bt[i, (L - 1) // bs]) * bs + (L - 1) % bs if L > 0 else -1)
        rows.append(r)
    sub = Workload(
        name=f"{w.name}[{len(seqs)} seqs]", S=len(seqs), Hq=w.Hq, Hkv=w.Hkv, d=w.d, bs=bs,
        num_blocks=max(1, len(remap)), cache_dtype=w.cache_dtype, q_dtype=w.q_dtype,
        src_dtype=w.src_dtype, scale=w.scale, k_scale=w.k_scale, v_scale=w.v_scale,
        partition_size=w.partition_size, seq_lens=w.seq_lens[seqs].copy(), block_tables=bt,
        pool_order=np.arange(max(1, len(remap))), ctx_slots=np.asarray(ctx_slots, np.int64),
        new_slots=np.asarray(new_slots, np.int64), cow_pairs=np.zeros((0, 2), np.int64),
        rows=rows, kind=w.kind)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    sd, qd = TORCH_DTYPES[w.src_dtype], TORCH_DTYPES[w.q_dtype]

    def randn(*shape, dtype):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    sub.ctx_k = randn(len(ctx_slots), w.Hkv, w.d, dtype=sd)
    sub.ctx_v = randn(len(ctx_slots), w.Hkv, w.d, dtype=sd)
    sub.new_k = randn(sub.S, w.Hkv, w.d, dtype=sd)
    sub.new_v = randn(sub.S, w.Hkv, w.d, dtype=sd)
    sub.q = randn(sub.S, w.Hq, w.d, dtype=qd)
    return sub
