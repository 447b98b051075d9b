"""CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the pages on PagedAttention describe, written so that a
reader can check each step against them by eye.  It is imported only by
``tests/``, by ``__graft_entry__.smoke()`` (to check one small GPU result) and
by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  The
product path (``paged_kv_cache_54_gb300``) never imports it, and the two
share no code: no kernels, helpers, tables or constant generators.

Modules
-------
allocator   Block pool with FIFO free list and reference counts, block tables,
            slot mapping, copy-on-write decisions.
fp8         OCP 8-bit floating point (E4M3 / E5M2) encode and decode, written
            from the format definition (sign, biased exponent, mantissa).
int8        Symmetric int8 KV codes (round half to even, saturate), the
            integer one-byte format the pages name beside FP8.
cache       Host paged KV cache: the cache write through a slot mapping and
            the whole-block copy used by copy-on-write.
attention   Single-query decode attention over the paged cache in float64.
prefix_cache  Content-keyed full blocks with reference counts and a
            least-recently-freed free list (prefix caching).

Pages cited (by title and section):
  [P1] "【性能飞跃】从 OOM 到丝滑推理:深度工程化 RAG 架构下的内存管理艺术"
  [P2] "大模型推理引擎显存优化：从 KV Cache 管理到连续批处理的工程实践"
  [P3] the m.lsln.cn/news/213354 article on KV-cache memory (paging, prefix
       caching, FP8 quantisation, offload); its title is not preserved
  [P4] "第3章 vLLM架构与显存使用：PagedAttention、KV Cache管理与显存池化技术"

Every function here is pinned by ``-m "not gpu"`` tests in ``tests/`` to
values the pages print, closed forms, library routines or brute force.
"""

from . import allocator, attention, cache, fp8, int8, prefix_cache  # noqa: F401
