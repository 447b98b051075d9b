"""Prefix cache over the block pool: content-keyed full blocks, reference
counts, least-recently-freed eviction.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the pages fix ([P3] §4.2–§4.3, [P1] §3.2):

* Each block's content gets a key that covers the token ids in the block
  and everything before it in the sequence (§4.2).  Here the key is the
  exact content: the tuple of the parent block's key and the block's own
  token ids, so two keys are equal exactly when the whole prefix up to the
  end of the block is equal.
* A new request looks its blocks up in order; a hit maps the existing
  physical block into its own block table, and only the part that missed is
  computed (§4.2).  Lookup stops at the first miss: a later block cannot be
  reused without every block before it.
* A shared block counts its users; a finished request decrements, and a
  block whose count reaches zero goes to the free pool, where it waits to be
  reused or reclaimed (§4.3).  While it waits it keeps its content and key,
  so a later request can still hit it.

Where the pages are silent, the plainest reading is taken:

* Only full blocks have a key.  The last, partial block of a prompt is
  private; when decoding fills it, it gets its key then.
* A fresh block is taken from the front of the free list, which is kept in
  the order blocks became free (least recently freed first; the initial
  pool comes first, in pool order).  Taking a block that still holds a key
  evicts the key.  [P3] §4.4 names least-recently-used eviction for the
  tree-shaped cache; the same order is used here.
* A finished request returns its blocks last block first, so that a
  prefix's tail is evicted before its head (a tail cannot be hit without
  its head).
* When a block's content is already cached in another block, the key keeps
  pointing at the cached one and the new block stays without a key.
* A request whose blocks cannot all be had is refused before anything
  changes ([P1] §2.3 raises before popping any block).
"""

from __future__ import annotations

from collections import OrderedDict
from typing import Dict, List, Optional, Tuple


class OutOfBlocks(RuntimeError):
    pass


class PrefixCache:
    def __init__(self, num_blocks: int, block_size: int, pool_order=None):
        self.num_blocks, self.block_size = num_blocks, block_size
        order = list(range(num_blocks)) if pool_order is None else [int(b) for b in pool_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("pool_order must be a permutation of the block ids")
        self.free: "OrderedDict[int, None]" = OrderedDict((b, None) for b in order)
        self.ref = [0] * num_blocks
        self.key_of: List[Optional[tuple]] = [None] * num_blocks
        self.block_of: Dict[tuple, int] = {}
        self.tables: Dict[int, List[int]] = {}
        self.tokens: Dict[int, List[int]] = {}
        self.queried_tokens = 0
        self.hit_tokens = 0
        self.evictions = 0

    # -- helpers --------------------------------------------------------
    def _block_key(self, parent: Optional[tuple], toks) -> tuple:
        return (parent, tuple(int(t) for t in toks))

    def _take_fresh(self) -> int:
        b, _ = self.free.popitem(last=False)
        if self.key_of[b] is not None:
            del self.block_of[self.key_of[b]]
            self.key_of[b] = None
            self.evictions += 1
        self.ref[b] = 1
        return b

    def _register(self, b: int, key: tuple) -> None:
        if key not in self.block_of:
            self.block_of[key] = b
            self.key_of[b] = key

    def _key_of_prefix(self, toks, nblocks: int) -> List[tuple]:
        keys, parent = [], None
        for j in range(nblocks):
            parent = self._block_key(parent, toks[j * self.block_size:(j + 1) * self.block_size])
            keys.append(parent)
        return keys

    # -- operations -----------------------------------------------------
    def add_sequence(self, seq: int, tokens) -> int:
        """Blocks for a new request's prompt; returns the number of prompt
        tokens whose KV is already cached (whole hit blocks)."""
        if seq in self.tables:
            raise ValueError("sequence exists")
        toks = [int(t) for t in tokens]
        bs = self.block_size
        nfull = len(toks) // bs
        nblocks = -(-len(toks) // bs)
        keys = self._key_of_prefix(toks, nfull)
        hits: List[int] = []
        for k in keys:
            b = self.block_of.get(k)
            if b is None:
                break
            hits.append(b)
        # blocks that will come off the free list: fresh ones, and hits on
        # blocks that are free (kept content, count 0)
        need_fresh = nblocks - len(hits)
        free_hits = sum(1 for b in hits if self.ref[b] == 0)
        if need_fresh + free_hits > len(self.free):
            raise OutOfBlocks(f"need {need_fresh + free_hits} free blocks, {len(self.free)} free")
        table: List[int] = []
        for b in hits:
            if self.ref[b] == 0:
                del self.free[b]
            self.ref[b] += 1
            table.append(b)
        for j in range(len(hits), nblocks):
            b = self._take_fresh()
            table.append(b)
            if j < nfull:
                self._register(b, keys[j])
        self.tables[seq] = table
        self.tokens[seq] = toks
        self.queried_tokens += len(toks)
        self.hit_tokens += len(hits) * bs
        return len(hits) * bs

    def append_token(self, seq: int, token: int) -> int:
        """One decoded token; returns its flat slot."""
        toks, table = self.tokens[seq], self.tables[seq]
        bs = self.block_size
        pos = len(toks)
        if pos % bs == 0:
            if not self.free:
                raise OutOfBlocks("no free block")
            table.append(self._take_fresh())
        toks.append(int(token))
        if len(toks) % bs == 0:              # the last block just filled
            j = len(toks) // bs - 1
            self._register(table[j], self._key_of_prefix(toks, j + 1)[j])
        return table[pos // bs] * bs + pos % bs

    def free_sequence(self, seq: int) -> None:
        for b in reversed(self.tables.pop(seq)):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free[b] = None          # most recently freed at the back
        del self.tokens[seq]

    # -- views ----------------------------------------------------------
    def table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def slot(self, seq: int, pos: int) -> int:
        return self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size

    def stats(self) -> Dict[str, int]:
        cached_free = sum(1 for b in self.free if self.key_of[b] is not None)
        return {"free_blocks": len(self.free), "cached_free_blocks": cached_free,
                "used_blocks": self.num_blocks - len(self.free),
                "cached_blocks": len(self.block_of), "queried_tokens": self.queried_tokens,
                "hit_tokens": self.hit_tokens, "evictions": self.evictions}

    def free_order(self) -> List[int]:
        return list(self.free)

    def hit_rate(self) -> float:
        return self.hit_tokens / self.queried_tokens if self.queried_tokens else 0.0

    def check_invariants(self) -> Tuple[bool, str]:
        users = [0] * self.num_blocks
        for t in self.tables.values():
            for b in t:
                users[b] += 1
        for b in range(self.num_blocks):
            if users[b] != self.ref[b]:
                return False, f"block {b}: {users[b]} tables, count {self.ref[b]}"
            if (self.ref[b] == 0) != (b in self.free):
                return False, f"block {b}: count {self.ref[b]}, free {b in self.free}"
        for k, b in self.block_of.items():
            if self.key_of[b] != k:
                return False, f"block {b}: key mismatch"
        return True, ""
