"""Python binding of libpa, the sm_103a paged KV-cache decode path.

Argument marshalling only: every step runs in the CUDA kernels of
``libpa.so`` (built in-tree by ``paged_kv_cache_54_gb300.build``).  The
functions carry the C ABI's names:

    pa_reshape_and_cache   write new tokens' K/V into the paged caches
    pa_decode              paged single-query decode attention
    pa_prefill             paged causal attention of several new tokens per
                           sequence (the part a prefix hit did not cover)
    pa_copy_blocks         whole-block copies (copy-on-write)
    pa_swap_blocks         whole-block moves between the device caches and
                           a pool in page-locked host memory
    pa_decode_workspace_size
    PrefixCache            the host block pool with prefix caching
                           (pa_prefix_cache_*)

PyTorch supplies the device memory and the stream; there is no CPU or
PyTorch fallback: if ``libpa.so`` is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_F16, PA_BF16, PA_FP8_E4M3, PA_FP8_E5M2, PA_INT8 = 0, 1, 2, 3, 4
DTYPE_CODES = {"f16": PA_F16, "bf16": PA_BF16, "e4m3": PA_FP8_E4M3, "e5m2": PA_FP8_E5M2,
               "int8": PA_INT8}
_TORCH_CODES = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.int8: PA_INT8}
if hasattr(torch, "float8_e4m3fn"):
    _TORCH_CODES[torch.float8_e4m3fn] = PA_FP8_E4M3
if hasattr(torch, "float8_e5m2"):
    _TORCH_CODES[torch.float8_e5m2] = PA_FP8_E5M2

EXPORTED = ("pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode", "pa_prefill",
            "pa_decode_static_scratch", "pa_copy_blocks", "pa_swap_blocks",
            "pa_status_string", "pa_last_cuda_error", "pa_selftest_wait_timeout",
            "pa_prefix_cache_create", "pa_prefix_cache_destroy", "pa_prefix_cache_add_sequence",
            "pa_prefix_cache_append_token", "pa_prefix_cache_free_sequence",
            "pa_prefix_cache_block_table", "pa_prefix_cache_block_tables",
            "pa_prefix_cache_get_stats", "pa_prefix_cache_free_order", "pa_prefix_cache_ref_count")
PA_ERR_OUT_OF_BLOCKS = 5
PA_SWAP_OUT, PA_SWAP_IN = 0, 1
STATIC_SCRATCH_BYTES = 16 << 20   # PA_DECODE_STATIC_SCRATCH_BYTES


class PaCacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("k_head_scales", ctypes.c_void_p),
                ("v_head_scales", ctypes.c_void_p)]


class PaError(RuntimeError):
    pass


class OutOfBlocks(PaError):
    pass


class PaPrefixCacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "free_blocks", "cached_free_blocks", "used_blocks", "cached_blocks",
        "queried_tokens", "hit_tokens", "evictions")]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpa.so and declare its C signatures (raises if it is absent)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run paged_kv_cache_54_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
    lib.pa_reshape_and_cache.argtypes = [vp, vp, i32, i64p, i32, vp, vp,
                                         ctypes.POINTER(PaCacheDesc), vp, vp]
    lib.pa_reshape_and_cache.restype = ctypes.c_int
    lib.pa_decode_workspace_size.argtypes = [i32] * 6
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode.argtypes = [vp, vp, i32, i32, i32, vp, vp, ctypes.POINTER(PaCacheDesc),
                              vp, i32, vp, i32, ctypes.c_float, i32, vp, ctypes.c_size_t,
                              vp, vp]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_decode_static_scratch.argtypes = [vp, vp, i32, i32, i32, vp, vp,
                                             ctypes.POINTER(PaCacheDesc), vp, i32, vp, i32,
                                             ctypes.c_float, i32, vp, vp]
    lib.pa_decode_static_scratch.restype = ctypes.c_int
    lib.pa_copy_blocks.argtypes = [vp, vp, ctypes.POINTER(PaCacheDesc), vp, i32, vp, vp]
    lib.pa_copy_blocks.restype = ctypes.c_int
    lib.pa_prefill.argtypes = [vp, vp, i32, i32, vp, i32, i32, i32, vp, vp, ctypes.POINTER(PaCacheDesc),
                               vp, i32, vp, ctypes.c_float, vp, vp]
    lib.pa_prefill.restype = ctypes.c_int
    lib.pa_swap_blocks.argtypes = [vp, vp, ctypes.POINTER(PaCacheDesc), vp, vp, ctypes.c_int64,
                                   vp, i32, i32, vp, vp]
    lib.pa_swap_blocks.restype = ctypes.c_int
    i64, i32p = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32)
    lib.pa_prefix_cache_create.argtypes = [i32, i32, vp]
    lib.pa_prefix_cache_create.restype = vp
    lib.pa_prefix_cache_destroy.argtypes = [vp]
    lib.pa_prefix_cache_destroy.restype = None
    lib.pa_prefix_cache_add_sequence.argtypes = [vp, i64, vp, i32, i32p]
    lib.pa_prefix_cache_append_token.argtypes = [vp, i64, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.pa_prefix_cache_free_sequence.argtypes = [vp, i64]
    lib.pa_prefix_cache_block_table.argtypes = [vp, i64, vp, i32, i32p]
    lib.pa_prefix_cache_block_table.restype = i32
    lib.pa_prefix_cache_block_tables.argtypes = [vp, vp, i32, vp, i32, vp]
    lib.pa_prefix_cache_get_stats.argtypes = [vp, ctypes.POINTER(PaPrefixCacheStats)]
    lib.pa_prefix_cache_free_order.argtypes = [vp, vp, i32]
    lib.pa_prefix_cache_free_order.restype = i32
    lib.pa_prefix_cache_ref_count.argtypes = [vp, i32]
    lib.pa_prefix_cache_ref_count.restype = i32
    for name in ("pa_prefix_cache_add_sequence", "pa_prefix_cache_append_token",
                 "pa_prefix_cache_free_sequence", "pa_prefix_cache_block_tables",
                 "pa_prefix_cache_get_stats"):
        getattr(lib, name).restype = ctypes.c_int
    lib.pa_selftest_wait_timeout.argtypes = [vp, vp]
    lib.pa_selftest_wait_timeout.restype = ctypes.c_int
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_cuda_error.argtypes = []
    lib.pa_last_cuda_error.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def pa_status_string(status: int) -> str:
    return load_library().pa_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        lib = load_library()
        msg = lib.pa_status_string(status).decode()
        if status == 3:
            msg += ": " + lib.pa_last_cuda_error().decode()
        cls = OutOfBlocks if status == PA_ERR_OUT_OF_BLOCKS else PaError
        raise cls(f"{what} failed: {msg} (status {status})")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _cache_code(k_cache: torch.Tensor, cache_dtype) -> int:
    if cache_dtype is not None:
        return DTYPE_CODES[cache_dtype] if isinstance(cache_dtype, str) else int(cache_dtype)
    if k_cache.dtype in _TORCH_CODES:
        return _TORCH_CODES[k_cache.dtype]
    raise ValueError("cache_dtype is required for a byte-typed FP8 cache")


def _scale_arg(scale, kv_heads: int, name: str):
    """(per-tensor value, per-head device pointer) of a scale argument: a
    number, or a contiguous float32 CUDA tensor of one scale per KV head."""
    if isinstance(scale, torch.Tensor):
        if (not scale.is_cuda or scale.dtype != torch.float32 or not scale.is_contiguous()
                or scale.numel() != kv_heads):
            raise ValueError(f"{name}: per-head scales must be a contiguous float32 CUDA "
                             f"tensor of {kv_heads} elements")
        return 1.0, scale.data_ptr()
    return float(scale), None


def cache_desc(k_cache: torch.Tensor, cache_dtype=None, k_scale=1.0,
               v_scale=1.0) -> PaCacheDesc:
    """Descriptor of a cache pair; k_scale / v_scale are numbers (per tensor)
    or float32 CUDA tensors [kv_heads] (per head; the tensors must outlive
    the calls that use the descriptor)."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, kv_heads, block_size, head_dim]")
    nb, h, bs, d = k_cache.shape
    ks, kp = _scale_arg(k_scale, h, "k_scale")
    vs, vp = _scale_arg(v_scale, h, "v_scale")
    return PaCacheDesc(nb, h, bs, d, _cache_code(k_cache, cache_dtype), ks, vs, kp, vp)


def _require(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def pa_reshape_and_cache(key, value, slot_mapping, k_cache, v_cache, cache_dtype=None,
                         k_scale=1.0, v_scale=1.0, device_error=None,
                         stream=None) -> None:
    """Write rows ``key/value [T, kv_heads, head_dim]`` into the caches."""
    for t, n in ((key, "key"), (value, "value"), (slot_mapping, "slot_mapping"),
                 (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    desc = cache_desc(k_cache, cache_dtype, k_scale, v_scale)
    src = _TORCH_CODES.get(key.dtype)
    if src is None or key.dtype != value.dtype:
        raise ValueError("key/value must be float16 or bfloat16 of one dtype")
    lib = load_library()
    _check(lib.pa_reshape_and_cache(key.data_ptr(), value.data_ptr(), src,
                                    slot_mapping.data_ptr(), slot_mapping.numel(),
                                    k_cache.data_ptr(), v_cache.data_ptr(),
                                    ctypes.byref(desc), _ptr(device_error), _stream(stream)),
           "pa_reshape_and_cache")


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                             head_dim: int, max_seq_len: int, partition_size: int = 0) -> int:
    return int(load_library().pa_decode_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, partition_size))


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len: int,
              scale: float, cache_dtype=None, k_scale=1.0, v_scale=1.0,
              partition_size: int = 0, workspace=None, device_error=None,
              stream=None) -> torch.Tensor:
    """Paged decode attention; writes ``out [S, Hq, head_dim]`` (q's dtype)."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _require(t, n)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    desc = cache_desc(k_cache, cache_dtype, k_scale, v_scale)
    S, Hq, D = q.shape
    qcode = _TORCH_CODES.get(q.dtype)
    if qcode not in (PA_F16, PA_BF16) or out.dtype != q.dtype or tuple(out.shape) != (S, Hq, D):
        raise ValueError("q/out must be float16 or bfloat16 [S, Hq, head_dim] of one dtype")
    need = pa_decode_workspace_size(S, Hq, desc.kv_heads, D, max_seq_len, partition_size)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.pa_decode(out.data_ptr(), q.data_ptr(), qcode, S, Hq, k_cache.data_ptr(),
                         v_cache.data_ptr(), ctypes.byref(desc), block_tables.data_ptr(),
                         block_tables.shape[1], seq_lens.data_ptr(), max_seq_len, scale,
                         partition_size, workspace.data_ptr(), workspace.numel(),
                         _ptr(device_error), _stream(stream)),
           "pa_decode")
    return out


def pa_prefill(out, q, cu_q_lens, k_cache, v_cache, block_tables, seq_lens, max_q_len: int,
               scale: float, cache_dtype=None, k_scale=1.0, v_scale=1.0, device_error=None,
               stream=None) -> torch.Tensor:
    """Causal attention of the new tokens ``q [T, Hq, head_dim]`` (sequence
    s's are rows cu_q_lens[s]..cu_q_lens[s+1]-1, its last tokens) over the
    paged cache; writes ``out`` like ``q``.  One-byte caches take their
    ``cache_dtype`` and scales as in ``pa_decode``."""
    for t, n in ((out, "out"), (q, "q"), (cu_q_lens, "cu_q_lens"), (k_cache, "k_cache"),
                 (v_cache, "v_cache"), (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _require(t, n)
    if cu_q_lens.dtype != torch.int32 or block_tables.dtype != torch.int32 or \
            seq_lens.dtype != torch.int32:
        raise ValueError("cu_q_lens, block_tables and seq_lens must be int32")
    desc = cache_desc(k_cache, cache_dtype, k_scale, v_scale)
    qcode = _TORCH_CODES.get(q.dtype)
    if out.dtype != q.dtype or out.shape != q.shape or q.dim() != 3:
        raise ValueError("q/out must be [T, Hq, head_dim] of one dtype")
    lib = load_library()
    _check(lib.pa_prefill(out.data_ptr(), q.data_ptr(), -1 if qcode is None else qcode, q.shape[0],
                          cu_q_lens.data_ptr(), cu_q_lens.numel() - 1, q.shape[1], int(max_q_len),
                          k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                          block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
                          scale, _ptr(device_error), _stream(stream)),
           "pa_prefill")
    return out


def pa_decode_static_scratch(out, q, k_cache, v_cache, block_tables, seq_lens,
                             max_seq_len: int, scale: float, cache_dtype=None,
                             k_scale=1.0, v_scale=1.0,
                             partition_size: int = 0, device_error=None,
                             stream=None) -> torch.Tensor:
    """``pa_decode`` for callers that cannot allocate device memory.

    Uses the library's own fixed 16 MiB device scratch instead of a
    workspace, so nothing is allocated here either; shapes that need more
    scratch than that are rejected (use ``pa_decode`` with a workspace).
    Calls that overlap on the GPU race on the shared scratch.
    """
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _require(t, n)
    desc = cache_desc(k_cache, cache_dtype, k_scale, v_scale)
    S, Hq, D = q.shape
    need = pa_decode_workspace_size(S, Hq, desc.kv_heads, D, max_seq_len, partition_size)
    if need > STATIC_SCRATCH_BYTES:
        raise PaError(f"pa_decode_static_scratch: these sizes need {need} bytes of scratch, "
                      f"more than its fixed {STATIC_SCRATCH_BYTES}; use pa_decode")
    lib = load_library()
    _check(lib.pa_decode_static_scratch(
        out.data_ptr(), q.data_ptr(), _TORCH_CODES.get(q.dtype, -1), S, Hq,
        k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), max_seq_len, scale, partition_size,
        _ptr(device_error), _stream(stream)), "pa_decode_static_scratch")
    return out


def pa_selftest_wait_timeout(device_error, stream=None) -> None:
    """Run the bounded-wait failure path once: after about 2 s the kernel
    writes device error 4 to ``device_error`` (a CUDA int32 tensor)."""
    _require(device_error, "device_error")
    _check(load_library().pa_selftest_wait_timeout(device_error.data_ptr(), _stream(stream)),
           "pa_selftest_wait_timeout")


def pa_copy_blocks(k_cache, v_cache, block_mapping, cache_dtype=None, device_error=None,
                   stream=None) -> None:
    """For each (src, dst) row of ``block_mapping [n, 2]`` copy block src to dst."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (block_mapping, "block_mapping")):
        _require(t, n)
    if block_mapping.dtype != torch.int64:
        raise ValueError("block_mapping must be int64")
    desc = cache_desc(k_cache, cache_dtype)
    lib = load_library()
    _check(lib.pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                              block_mapping.data_ptr(), block_mapping.shape[0],
                              _ptr(device_error), _stream(stream)),
           "pa_copy_blocks")


def pa_swap_blocks(k_cache, v_cache, host_k, host_v, block_mapping, direction: str,
                   cache_dtype=None, device_error=None, stream=None) -> None:
    """Whole-block moves between the device caches and a second pool.

    ``host_k`` / ``host_v``: ``[host_blocks, kv_heads, block_size, head_dim]``
    in page-locked CPU memory (``pin_memory()``) or on the caches' device.
    ``direction`` "out": for each (src, dst) row of ``block_mapping [n, 2]``
    device block src -> host block dst; "in": host block src -> device
    block dst.
    """
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (block_mapping, "block_mapping")):
        _require(t, n)
    for t, n in ((host_k, "host_k"), (host_v, "host_v")):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be contiguous, in page-locked host memory or on the device")
        if t.shape[1:] != k_cache.shape[1:] or t.element_size() != k_cache.element_size():
            raise ValueError(f"{n} must have the caches' block shape and element size")
    if host_k.shape != host_v.shape:
        raise ValueError("host_k and host_v must have one shape")
    if block_mapping.dtype != torch.int64:
        raise ValueError("block_mapping must be int64")
    codes = {"out": PA_SWAP_OUT, "in": PA_SWAP_IN}
    if direction not in codes:
        raise ValueError('direction must be "out" or "in"')
    desc = cache_desc(k_cache, cache_dtype)
    lib = load_library()
    _check(lib.pa_swap_blocks(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                              host_k.data_ptr(), host_v.data_ptr(), host_k.shape[0],
                              block_mapping.data_ptr(), block_mapping.shape[0], codes[direction],
                              _ptr(device_error), _stream(stream)),
           "pa_swap_blocks")


class PrefixCache:
    """The host block pool with prefix caching (``pa_prefix_cache_*``).

    Sequences are named by integer ids; token ids are int32.  Raises
    ``OutOfBlocks`` when the free list cannot supply a request (nothing is
    changed then)."""

    def __init__(self, num_blocks: int, block_size: int, pool_order=None):
        import numpy as np
        self._lib = load_library()
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        order = None
        if pool_order is not None:
            self._order = np.ascontiguousarray(pool_order, dtype=np.int32)
            order = self._order.ctypes.data
        self._h = self._lib.pa_prefix_cache_create(self.num_blocks, self.block_size, order)
        if not self._h:
            raise ValueError("invalid prefix cache arguments")

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pa_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_sequence(self, seq: int, tokens) -> int:
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(self._lib.pa_prefix_cache_add_sequence(self._h, int(seq), t.ctypes.data, t.size,
                                                      ctypes.byref(n)), "add_sequence")
        return n.value

    def append_token(self, seq: int, token: int) -> int:
        slot = ctypes.c_int64(0)
        _check(self._lib.pa_prefix_cache_append_token(self._h, int(seq), int(token),
                                                      ctypes.byref(slot)), "append_token")
        return slot.value

    def free_sequence(self, seq: int) -> None:
        _check(self._lib.pa_prefix_cache_free_sequence(self._h, int(seq)), "free_sequence")

    def table(self, seq: int):
        import numpy as np
        n = self._lib.pa_prefix_cache_block_table(self._h, int(seq), None, 0, None)
        if n < 0:
            raise KeyError(seq)
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_prefix_cache_block_table(self._h, int(seq), out.ctypes.data, n, None)
        return out[:n].tolist()

    def block_tables(self, seqs, width: int):
        """(int32 [len(seqs), width] tables, int32 [len(seqs)] lengths)."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        tables = np.zeros((len(ids), width), dtype=np.int32)
        lens = np.zeros(len(ids), dtype=np.int32)
        _check(self._lib.pa_prefix_cache_block_tables(self._h, ids.ctypes.data, len(ids),
                                                      tables.ctypes.data, width, lens.ctypes.data),
               "block_tables")
        return tables, lens

    def stats(self) -> dict:
        st = PaPrefixCacheStats()
        _check(self._lib.pa_prefix_cache_get_stats(self._h, ctypes.byref(st)), "get_stats")
        return {n: getattr(st, n) for n, _ in PaPrefixCacheStats._fields_}

    def free_order(self):
        import numpy as np
        n = self._lib.pa_prefix_cache_free_order(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_prefix_cache_free_order(self._h, out.ctypes.data, n)
        return out[:n].tolist()

    def ref_count(self, block: int) -> int:
        return int(self._lib.pa_prefix_cache_ref_count(self._h, int(block)))
