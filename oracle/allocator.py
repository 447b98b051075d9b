"""Block allocator: free pool, block tables, reference counts, copy-on-write.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the pages fix, and where:

* Fixed-size physical blocks holding ``block_size`` tokens of K and V, the
  default being 16 ([P3] §3.2; [P4] §3.1; [P1] §2.1 "关键设计").
* A per-sequence block table mapping logical block j to a physical block,
  like a page table ([P1] §2.1 figure: L0→P7, L1→P1, L2→P3; [P3] §3.2).
* Blocks needed for n tokens is ceil(n / block_size), so at most
  ``block_size - 1`` token slots are wasted, all in the last block
  ([P1] §2.3 ``_calc_needed_blocks``; [P2] §三 ``allocate_request``;
  [P3] §3.3 "最多浪费 15 个 token").
* A FIFO free pool: take from the front, return to the back ([P1] §2.3
  ``free_pool.pop(0)`` / ``extend``; [P2] §三 ``VecDeque`` ``pop_front`` /
  ``push_back``).
* Pool exhaustion is an error raised before anything is taken ([P1] §2.3
  ``_pop_blocks`` raises ``MemoryError``; [P2] §三 returns ``Err``).
* Appending a token takes a new block only when the last block is full
  ([P2] §三 ``append_token``; [P4] §3.2 first paragraph).
* Reference counts: sharing increments, freeing decrements, a block whose
  count reaches zero returns to the pool ([P2] §三 ``share_prefix`` /
  ``free_request``; [P3] §4.3; [P4] §3.2 B1–B6 walk-through).
* Copy-on-write: writing into a shared block first takes a new block, copies
  the old block into it, writes there, and decrements the old block's count
  ([P4] §3.3 last paragraph; [P1] §3.2).

Readings where the pages are silent or in error:

* [P1]'s ``handle_append`` takes a single block even when ``new_tokens``
  needs more; here ``append`` takes as many as the new token count needs.
* [P2]'s ``test_prefix_sharing`` asserts 96 free blocks after freeing the
  source request, but under its own ``free_request`` the two unshared blocks
  reach count zero and return, leaving 98; the tests assert 98.
* A ``fork`` shares every block of the source, partial last block included
  (beam search and parallel sampling in [P4] §3.2 and [P1] §6.1).
"""

from __future__ import annotations

from collections import deque
from typing import Dict, Iterable, List, Optional, Tuple


class OutOfBlocks(MemoryError):
    """The free pool cannot supply the blocks a request needs."""


class BlockAllocator:
    """Refcounted block pool with per-sequence block tables."""

    def __init__(self, num_blocks: int, block_size: int,
                 pool_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if pool_order is None else list(pool_order)
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("pool_order must be a permutation of 0..num_blocks-1")
        self.free: deque = deque(order)
        self.refcount: Dict[int, int] = {}
        self.tables: Dict[object, List[int]] = {}
        self.num_tokens: Dict[object, int] = {}

    # -- sizes ---------------------------------------------------------
    def blocks_needed(self, n_tokens: int) -> int:
        """ceil(n_tokens / block_size)."""
        return (n_tokens + self.block_size - 1) // self.block_size

    def available_blocks(self) -> int:
        return len(self.free)

    def utilization(self) -> float:
        """Fraction of physical blocks not in the free pool ([P2] §三)."""
        return (self.num_blocks - len(self.free)) / self.num_blocks

    def stats(self) -> dict:
        """Snapshot in the shape of [P1] §2.3 ``stats``."""
        return {
            "free_blocks": len(self.free),
            "active_requests": len(self.tables),
            "utilization_pct": round(self.utilization() * 100, 2),
        }

    # -- internal ------------------------------------------------------
    def _take(self, count: int) -> List[int]:
        if len(self.free) < count:
            raise OutOfBlocks(f"need {count} blocks, pool has {len(self.free)}")
        out = [self.free.popleft() for _ in range(count)]
        for b in out:
            self.refcount[b] = 1
        return out

    def _release(self, block: int) -> None:
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            del self.refcount[block]
            self.free.append(block)

    # -- operations ----------------------------------------------------
    def allocate(self, seq, n_tokens: int) -> List[int]:
        """First allocation of a sequence holding ``n_tokens`` tokens."""
        if seq in self.tables:
            raise ValueError(f"sequence {seq!r} already allocated")
        if n_tokens < 0:
            raise ValueError("n_tokens must be >= 0")
        self.tables[seq] = self._take(self.blocks_needed(n_tokens))
        self.num_tokens[seq] = n_tokens
        return self.tables[seq]

    def append(self, seq, n_new: int = 1) -> List[Tuple[int, int]]:
        """Append ``n_new`` tokens, one at a time.

        A token that lands in a block with room is written there; if that
        block is shared the copy-on-write step runs first.  A token that finds
        the last block full (or no block) takes a new block from the pool.
        Returns the (src, dst) copy pairs emitted by copy-on-write.
        """
        if seq not in self.tables:
            raise ValueError(f"sequence {seq!r} not allocated")
        pairs: List[Tuple[int, int]] = []
        for _ in range(n_new):
            pos = self.num_tokens[seq]
            table = self.tables[seq]
            if pos // self.block_size >= len(table):
                table.extend(self._take(1))
            else:
                cow = self.prepare_write(seq, pos)
                if cow is not None:
                    pairs.append(cow)
            self.num_tokens[seq] = pos + 1
        return pairs

    def prepare_write(self, seq, pos: int) -> Optional[Tuple[int, int]]:
        """Copy-on-write before writing token position ``pos`` of ``seq``.

        If the block holding ``pos`` is shared, take a new block, record the
        copy (old → new), point the table at the new block and drop one
        reference to the old block.  Returns the pair, or None when the block
        is exclusively owned.
        """
        table = self.tables[seq]
        j = pos // self.block_size
        old = table[j]
        if self.refcount[old] == 1:
            return None
        (new,) = self._take(1)
        table[j] = new
        self.refcount[old] -= 1  # stays >= 1: another holder remains
        return (old, new)

    def share_prefix(self, src, n_blocks: int, dst) -> List[int]:
        """``dst`` starts with the first ``n_blocks`` blocks of ``src``."""
        if src not in self.tables:
            raise ValueError(f"source {src!r} not allocated")
        if dst in self.tables:
            raise ValueError(f"sequence {dst!r} already allocated")
        src_table = self.tables[src]
        if n_blocks > len(src_table):
            raise ValueError("cannot share more blocks than the source holds")
        shared = list(src_table[:n_blocks])
        for b in shared:
            self.refcount[b] += 1
        self.tables[dst] = shared
        self.num_tokens[dst] = min(n_blocks * self.block_size, self.num_tokens[src])
        return shared

    def fork(self, src, dst) -> List[int]:
        """``dst`` shares every block of ``src`` (beam / parallel sampling)."""
        return self.share_prefix(src, len(self.tables[src]), dst)

    def free_seq(self, seq) -> None:
        """Drop the sequence; blocks whose count reaches zero return to the pool."""
        if seq not in self.tables:
            raise ValueError(f"sequence {seq!r} not allocated")
        for b in self.tables.pop(seq):
            self._release(b)
        del self.num_tokens[seq]

    # -- derived views -------------------------------------------------
    def slot(self, seq, pos: int) -> int:
        """Flat cache slot of token ``pos``: physical block * block_size + offset."""
        table = self.tables[seq]
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def block_table_array(self, seqs, width: int, pad: int = 0) -> List[List[int]]:
        """Rows of the block tables of ``seqs``, right-padded to ``width``."""
        rows = []
        for s in seqs:
            t = self.tables[s]
            if len(t) > width:
                raise ValueError("table wider than requested width")
            rows.append(list(t) + [pad] * (width - len(t)))
        return rows
