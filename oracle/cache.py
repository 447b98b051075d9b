"""Host paged KV cache: cache write through a slot mapping, whole-block copy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Layout: ``[num_blocks, kv_heads, block_size, head_dim]`` per cache (one for
K, one for V); the physical block is the page of [P1] §2.1 / [P3] §3.2 and
each block holds ``block_size`` tokens of every KV head.

The cache holds *storage codes*: uint16 bit patterns for fp16 / bf16, uint8
codes for e4m3 / e5m2 / int8.  Values are recovered with :func:`values`.

* ``reshape_and_cache``: token t of the new K/V rows goes to flat slot
  ``slot_mapping[t]`` = physical block * block_size + offset, the block being
  the one the block table names for the token's logical block ([P1] §2.1,
  [P2] §2.2).  A slot of -1 marks a padding row and is skipped (the pages are
  silent; this is the usual padding convention).  With an 8-bit cache each
  value is stored as value / scale ([P3] §6.1), see ``oracle.fp8`` and
  ``oracle.int8``; the scale is one per tensor or one per KV head ([P3]
  §6.3).
* ``copy_blocks``: the copy step of copy-on-write ([P4] §3.3): every element
  of block ``src`` (all heads, all token slots) is copied to block ``dst``,
  in K and in V.
* ``swap_blocks``: swapping a preempted request's blocks out to CPU memory
  and back ([P1] §5.1–5.2: on preemption the KV cache is copied to CPU
  memory instead of being dropped; [P4] §3.5: inactive blocks go to the
  CPU swap space; [P3] §7.2: reusable blocks are offloaded to CPU memory).
  A second pool of the same block shape stands for the CPU memory; each
  (src, dst) pair copies one whole block from one pool to the other, bit
  for bit.
"""

from __future__ import annotations

import numpy as np

from . import fp8 as _fp8
from . import int8 as _int8

STORAGE_DTYPES = ("f16", "bf16", "e4m3", "e5m2", "int8")
BYTE_DTYPES = ("e4m3", "e5m2", "int8")

# Patterns used to fill never-written slots, so that a read beyond a
# sequence's length shows up in the result: NaN for the float formats, the
# most negative code for int8 (which has no NaN).
NAN_CODE = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F, "e5m2": 0x7F, "int8": 0x80}


def code_dtype(dtype: str):
    return np.uint8 if dtype in BYTE_DTYPES else np.uint16


def head_scale(scale, h: int) -> float:
    """Scale of KV head h: one number for the tensor, or one per head.

    [P3] §6.3: the scale is per tensor by default and may be refined to one
    per attention head.
    """
    if np.ndim(scale) == 0:
        return float(scale)
    return float(np.asarray(scale, dtype=np.float64)[h])


def _scale_grid(scale, shape):
    """Scale broadcast over a [..., kv_heads, block_size, head_dim] array."""
    if np.ndim(scale) == 0:
        return float(scale)
    return np.asarray(scale, dtype=np.float64).reshape((shape[-3], 1, 1))


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of 16-bit storage bit patterns.

    fp16 is IEEE binary16 (numpy's float16); bf16 is the upper half of an
    IEEE binary32, so its value is the binary32 with 16 zero bits appended.
    """
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def values(codes: np.ndarray, dtype: str, scale=1.0) -> np.ndarray:
    """float64 values the cache codes stand for (8-bit: code value * scale).

    ``scale`` is one number, or one per KV head when ``codes`` keeps the
    ``[kv_heads, block_size, head_dim]`` trailing axes.
    """
    if dtype in ("f16", "bf16"):
        return bits_to_f64(codes, dtype)
    base = _int8.decode(codes) if dtype == "int8" else _fp8.decode(codes, dtype)
    return base * _scale_grid(scale, np.shape(codes))


class PagedKVCache:
    def __init__(self, num_blocks: int, kv_heads: int, block_size: int,
                 head_dim: int, dtype: str, k_scale=1.0, v_scale=1.0,
                 fill_nan: bool = True):
        if dtype not in STORAGE_DTYPES:
            raise ValueError(dtype)
        self.num_blocks, self.kv_heads = num_blocks, kv_heads
        self.block_size, self.head_dim = block_size, head_dim
        self.dtype, self.k_scale, self.v_scale = dtype, k_scale, v_scale
        shape = (num_blocks, kv_heads, block_size, head_dim)
        fill = NAN_CODE[dtype] if fill_nan else 0
        self.k = np.full(shape, fill, dtype=code_dtype(dtype))
        self.v = np.full(shape, fill, dtype=code_dtype(dtype))

    def _encode(self, src_bits: np.ndarray, src_dtype: str, scale):
        """Storage code of source rows [T, kv_heads, head_dim] given as
        16-bit bit patterns; each head is divided by its own scale."""
        if self.dtype in ("f16", "bf16"):
            if src_dtype != self.dtype:
                raise ValueError("16-bit caches take rows of their own dtype")
            return np.asarray(src_bits, dtype=np.uint16)
        src_bits = np.asarray(src_bits, dtype=np.uint16)
        out = np.empty(src_bits.shape, dtype=np.uint8)
        for h in range(src_bits.shape[1]):
            s_h = head_scale(scale, h)
            if self.dtype == "int8":
                out[:, h] = _int8.quantize_bits16(src_bits[:, h], src_dtype, s_h)
            else:
                out[:, h] = _fp8.quantize_bits16(src_bits[:, h], src_dtype, s_h, self.dtype)
        return out

    def reshape_and_cache(self, key_bits: np.ndarray, value_bits: np.ndarray,
                          src_dtype: str, slot_mapping: np.ndarray) -> None:
        """key/value: [T, kv_heads, head_dim] 16-bit patterns; slots: [T]."""
        T = len(slot_mapping)
        kc = self._encode(key_bits, src_dtype, self.k_scale)
        vc = self._encode(value_bits, src_dtype, self.v_scale)
        for t in range(T):
            slot = int(slot_mapping[t])
            if slot < 0:
                continue
            blk, off = divmod(slot, self.block_size)
            self.k[blk, :, off, :] = kc[t]
            self.v[blk, :, off, :] = vc[t]

    def copy_blocks(self, pairs) -> None:
        """For each (src, dst): block dst of K and of V becomes block src."""
        for src, dst in pairs:
            self.k[int(dst)] = self.k[int(src)]
            self.v[int(dst)] = self.v[int(src)]

    def swap_blocks(self, other: "PagedKVCache", pairs, direction: str) -> None:
        """Whole-block moves between this pool and ``other`` (same kv_heads,
        block_size, head_dim and dtype; any number of blocks).

        direction "out": block src of this pool -> block dst of ``other``;
        direction "in":  block src of ``other`` -> block dst of this pool.
        """
        if (other.kv_heads, other.block_size, other.head_dim, other.dtype) != \
                (self.kv_heads, self.block_size, self.head_dim, self.dtype):
            raise ValueError("pools differ in block shape")
        if direction == "out":
            src, dst = self, other
        elif direction == "in":
            src, dst = other, self
        else:
            raise ValueError(direction)
        for s, d in pairs:
            dst.k[int(d)] = src.k[int(s)]
            dst.v[int(d)] = src.v[int(s)]

    def k_values(self) -> np.ndarray:
        return values(self.k, self.dtype, self.k_scale)

    def v_values(self) -> np.ndarray:
        return values(self.v, self.dtype, self.v_scale)
