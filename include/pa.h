/*
 * pa.h — C ABI of libpa, the GB300 (sm_103a) paged KV-cache decode path.
 *
 * Three device operations, each asynchronous on the caller's stream:
 *
 *   pa_reshape_and_cache  write new tokens' K and V into fixed-size physical
 *                         blocks through a slot mapping (optionally as FP8
 *                         or INT8 with a scale per tensor or per KV head);
 *   pa_decode             single-query decode attention over the paged cache,
 *                         reached through per-sequence block tables;
 *   pa_prefill            causal attention of several new tokens per sequence
 *                         over the paged cache (the part of a prompt a
 *                         prefix-cache hit did not cover);
 *   pa_copy_blocks        whole-block copies, the copy step of copy-on-write;
 *   pa_swap_blocks        whole-block moves between the device caches and a
 *                         pool in host memory (swap-out / swap-in).
 *
 * and one host-side structure that hands out the blocks:
 *
 *   pa_prefix_cache_*     the block pool with prefix caching: full blocks
 *                         keyed by their content and everything before it,
 *                         shared through reference counts, kept after their
 *                         last user until needed again.
 *
 * Pages that state the problem (cited by title and section):
 *   [P1] "【性能飞跃】从 OOM 到丝滑推理:深度工程化 RAG 架构下的内存管理艺术"
 *        §2.1 (logical blocks mapped to scattered physical blocks through a
 *        block table; fixed block size, default 16), §3.2 (prefix sharing and
 *        copy-on-write), §6.1 (beam search shares blocks, copies only the
 *        last one).
 *   [P2] "大模型推理引擎显存优化：从 KV Cache 管理到连续批处理的工程实践"
 *        §2.2 (block table per request, blocks from a global pool), §三
 *        (refcounted block manager).
 *   [P3] m.lsln.cn/news/213354 (KV-cache memory article; title not
 *        preserved) §3.2 (paging), §4.3 (reference counts), §6 (FP8 or INT8
 *        halve the cache), §6.1–§6.3 (store value / scale, read back
 *        × scale; e4m3 and e5m2; default scale 1.0 per tensor, optionally
 *        one per attention head).
 *   [P4] "第3章 vLLM架构与显存使用：PagedAttention、KV Cache管理与显存池化技术"
 *        §3.2 (block life cycle, shared blocks), §3.3 (copy-on-write: take a
 *        new block, copy the old one, write the new one).
 * The pages do not write the attention formula or any kernel down; the
 * attention computed here is the textbook scaled dot-product attention of
 * one query row over the sequence's tokens.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Ownership: the caller owns every buffer, including the decode workspace.
 *   The library allocates no device or host memory and never synchronises.
 * - Pointers: every array argument is a DEVICE pointer except `cache`
 *   (a host struct read during the call).  Device arrays must be 16-byte
 *   aligned and densely packed in the layouts stated below.
 * - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Work is only enqueued; results are ready when the stream reaches them.
 * - Errors: invalid arguments are rejected on the host before anything is
 *   launched (PA_ERR_INVALID / PA_ERR_UNSUPPORTED).  A failed launch returns
 *   PA_ERR_CUDA.  Data that only the device can see (a block id outside the
 *   pool, a slot outside the cache, a length beyond the table width) is
 *   checked in the kernels: the bad access is skipped and a nonzero code is
 *   written to *device_error (when the pointer is not NULL; the first error
 *   wins), which the caller reads after synchronising.  Kernels never trap.
 * - Device error codes: 1 block id out of range, 2 slot out of range,
 *   3 sequence length out of range, 4 a pipeline wait exceeded its time
 *   limit, 5 copy pair out of range, 6 shared memory not aligned as the
 *   swizzled tile layout needs (nothing computed).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,      /* null pointer, negative size, misalignment, ... */
  PA_ERR_UNSUPPORTED = 2,  /* valid but outside the supported set below */
  PA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  PA_ERR_DEVICE_CHECK = 4, /* for callers that map a nonzero *device_error */
  PA_ERR_OUT_OF_BLOCKS = 5 /* the block pool cannot supply the request */
} pa_status;

typedef enum {
  PA_F16 = 0,       /* IEEE binary16 */
  PA_BF16 = 1,      /* bfloat16 */
  PA_FP8_E4M3 = 2,  /* OCP E4M3 (max 448, no inf), one byte */
  PA_FP8_E5M2 = 3,  /* OCP E5M2 (max 57344), one byte */
  PA_INT8 = 4       /* two's-complement int8 code, one byte */
} pa_dtype;

/*
 * Description of one paged cache pair (K and V).
 * Layout of k_cache and v_cache: [num_blocks, kv_heads, block_size, head_dim]
 * elements of `dtype`, row-major.  Physical block b holds block_size token
 * slots of every KV head; flat slot = b * block_size + offset.
 * For the one-byte caches (FP8, INT8) a stored code c of KV head h means
 * c * sk(h) in K and c * sv(h) in V: values are stored as value / scale
 * ([P3] §6.1; default 1.0 per tensor, one per head optionally, §6.3).
 * sk(h) is k_head_scales[h] when that pointer is not NULL, else k_scale
 * (likewise for V).
 * Supported set: block_size in {8, 16, 32}; head_dim in {64, 128}.
 */
typedef struct {
  int32_t num_blocks;
  int32_t kv_heads;
  int32_t block_size;
  int32_t head_dim;
  int32_t dtype;     /* pa_dtype */
  float k_scale;     /* one-byte caches only; must be > 0 and finite */
  float v_scale;
  /* One-byte caches only, else must be NULL: DEVICE float32 [kv_heads],
   * one scale per KV head (each > 0 and finite; not checked), or NULL for
   * the per-tensor scales above.  Read by the kernels, so they must stay
   * valid until the calls that use them have run. */
  const float *k_head_scales;
  const float *v_head_scales;
} pa_cache_desc;

/*
 * pa_reshape_and_cache — write T new tokens into the paged caches.
 * ([P1] §2.1 / [P2] §2.2 block tables; [P3] §6.1 FP8 with a scale.)
 *
 *   key, value     device, [num_tokens, kv_heads, head_dim] of src_dtype
 *                  (PA_F16 or PA_BF16), row-major.
 *   slot_mapping   device int64 [num_tokens]: flat slot of token t;
 *                  -1 marks a padding row that is skipped.
 *   k_cache/v_cache  device caches described by *cache.
 * For every token t with slot >= 0 and every head h:
 *   cache[slot / block_size, h, slot % block_size, :] = enc(row[t, h, :])
 * where enc is a bit copy for 16-bit caches (src_dtype must equal
 * cache->dtype); for FP8 caches, round-to-nearest-even with saturation to
 * the largest finite value of (float)x / scale computed in IEEE float32;
 * for INT8 caches, the same quotient rounded to the nearest integer (ties
 * to even) and saturated to [-128, 127], with NaN stored as 0.  The scale
 * is head h's (see pa_cache_desc).
 * Slots must be distinct among the call's tokens.  A slot >= num_blocks *
 * block_size is skipped and reported as device error 2.
 */
PA_API pa_status pa_reshape_and_cache(const void *key, const void *value,
                               int32_t src_dtype, const int64_t *slot_mapping,
                               int32_t num_tokens, void *k_cache, void *v_cache,
                               const pa_cache_desc *cache, int *device_error,
                               pa_stream_t stream);

/*
 * pa_decode_workspace_size — bytes of device workspace pa_decode needs for
 * these sizes (same arguments as pa_decode; 0 partition_size = automatic).
 * Returns 0 for arguments pa_decode would reject.
 */
PA_API size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_seq_len, int32_t partition_size);

/*
 * pa_decode — single-query decode attention over the paged cache.
 *
 * For every sequence s < num_seqs and query head hq < num_q_heads, with
 * G = num_q_heads / kv_heads and KV head h = hq / G (a group of G query heads
 * shares one KV head):
 *   out[s, hq, :] = sum_{i < L_s} softmax_i(scale * <q[s, hq, :], k_i>) v_i
 * where L_s = seq_lens[s] and token i of sequence s is read from physical
 * block block_tables[s, i / block_size] at offset i % block_size
 * ([P1] §2.1, [P2] §2.2, [P3] §3.2; one-byte codes are multiplied by
 * their head's scales of *cache, [P3] §6.1 and §6.3).  L_s = 0 gives zeros.
 *
 *   out            device [num_seqs, num_q_heads, head_dim], q_dtype.
 *   q              device [num_seqs, num_q_heads, head_dim], q_dtype
 *                  (PA_F16 or PA_BF16; for 16-bit caches it must equal the
 *                  cache dtype).
 *   block_tables   device int32 [num_seqs, max_blocks_per_seq]; only the
 *                  first ceil(L_s / block_size) entries of a row are read.
 *   seq_lens       device int32 [num_seqs]; each must satisfy
 *                  0 <= L_s <= min(max_seq_len, max_blocks_per_seq * block_size).
 *   max_seq_len    host upper bound of seq_lens, used to size the work.
 *   scale          softmax scale (e.g. 1/sqrt(head_dim)).
 *   partition_size 0 = automatic; else the number of tokens one work item
 *                  covers (multiple of 64 and of block_size, <= 1024).
 *                  Sequences longer than one partition are split and merged
 *                  exactly (flash-decoding), so the result does not depend
 *                  on it beyond rounding.
 *   workspace      device scratch of at least pa_decode_workspace_size(...)
 *                  bytes, 256-byte aligned; contents need no initialisation.
 *                  Calls sharing one workspace must be stream-ordered.
 * Supported set: num_q_heads / kv_heads in {1, 2, 4, 8}; cache dtypes of
 * pa_cache_desc; one-byte caches accept q in PA_F16 or PA_BF16.
 * Stream order: the call's first kernel may begin reading block_tables and
 * seq_lens while the kernel before it on the stream is still running, if
 * that kernel has signalled programmatic completion early
 * (griddepcontrol.launch_dependents).  pa_reshape_and_cache and
 * pa_copy_blocks do so; they never write those arrays.  A caller's kernel
 * that writes block_tables or seq_lens must not signal before its writes.
 * Everything else the call reads (q, the caches) is read only after all
 * earlier work on the stream has completed.
 */
PA_API pa_status pa_decode(void *out, const void *q, int32_t q_dtype,
                    int32_t num_seqs, int32_t num_q_heads,
                    const void *k_cache, const void *v_cache,
                    const pa_cache_desc *cache, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *seq_lens,
                    int32_t max_seq_len, float scale, int32_t partition_size,
                    void *workspace, size_t workspace_bytes, int *device_error,
                    pa_stream_t stream);

/*
 * pa_prefill — causal attention of each sequence's new tokens over all of
 * its tokens in the paged cache ([P3] §4.2: after a prefix hit only the part
 * that missed is computed; their K and V are written with
 * pa_reshape_and_cache first).
 *
 * Sequence s holds L_s = seq_lens[s] tokens, of which the last
 * n_s = cu_q_lens[s + 1] - cu_q_lens[s] are new.  New token j of sequence s
 * sits at position p = L_s - n_s + j; for each query head hq, with KV head
 * h = hq / G as in pa_decode:
 *   out[cu_q_lens[s] + j, hq, :] =
 *       sum_{i <= p} softmax_i(scale * <q[cu_q_lens[s] + j, hq, :], k_i>) v_i
 * with token i read from block block_tables[s, i / block_size] at offset
 * i % block_size, and one-byte codes dequantised with the cache's scales as
 * in pa_decode.
 *
 *   out, q         device [num_q_tokens, num_q_heads, head_dim] of q_dtype:
 *                  the cache dtype for 16-bit caches, PA_F16 or PA_BF16 for
 *                  one-byte ones; num_q_tokens = cu_q_lens[num_seqs].
 *   cu_q_lens      device int32 [num_seqs + 1], non-decreasing, from 0;
 *                  every sequence's rows must lie in [0, num_q_tokens).
 *   max_q_len      host upper bound of n_s, used to size the grid.
 *   block_tables, max_blocks_per_seq, seq_lens  as in pa_decode; each
 *                  n_s <= L_s <= max_blocks_per_seq * block_size.
 * Device checks: a length that breaks these bounds, n_s > max_q_len, or
 * rows of a sequence outside [0, num_q_tokens) skip that sequence (nothing
 * of its output is written) and report error 3; a block id out of range reads
 * block 0 instead and reports error 1; a stalled pipeline reports error 4.
 * Supported set: num_q_heads / kv_heads in {1, 2, 4, 8}; block_size and
 * head_dim as in pa_cache_desc; num_seqs and kv_heads <= 65535.  Needs no
 * workspace and allocates nothing.  With a one-byte cache the products run
 * on fp16 operands: a bf16 q is rounded to fp16 after scaling each 128-row
 * query tile by a power of two that brings its largest |q| within 2^15.
 */
PA_API pa_status pa_prefill(void *out, const void *q, int32_t q_dtype, int32_t num_q_tokens,
                            const int32_t *cu_q_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t max_q_len,
                            const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *seq_lens, float scale, int *device_error,
                            pa_stream_t stream);

/*
 * pa_decode_static_scratch — pa_decode for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for callers of this
 * library that may not allocate device memory at decode time: a plugin whose
 * host framework owns all GPU memory through its own pool (an allocation
 * outside the pool escapes its accounting and can fail once the KV pool has
 * been sized to fill the device), or a serving loop that allows no
 * allocation after start-up because cudaMalloc may synchronise the device.
 *
 * Same arguments and result as pa_decode, without `workspace`.  Its scratch
 * is a fixed device array of PA_DECODE_STATIC_SCRATCH_BYTES (16 MiB) inside
 * the library, held by every GPU that loads the library until the process
 * exits.  The call allocates nothing (no cudaMalloc / cudaFree, no library
 * routine that allocates).
 * - Limit: a call whose pa_decode_workspace_size(...) exceeds
 *   PA_DECODE_STATIC_SCRATCH_BYTES returns PA_ERR_UNSUPPORTED and launches
 *   nothing; pass a caller-owned workspace to pa_decode instead.
 * - First call on each device: it looks up the array's device address with
 *   cudaGetSymbolAddress (with that device current) and caches it, so make
 *   that first call before any stream capture begins.
 * - Sharing: every call uses the same array and it keeps the last call's
 *   contents; nothing in it needs to start at zero (each call rewrites its
 *   work list and claim counter first).  Calls whose execution overlaps on
 *   the GPU (different streams, or different threads without ordering) race
 *   on the array; order them on one stream.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
PA_API pa_status pa_decode_static_scratch(
    void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, float scale, int32_t partition_size, int *device_error,
    pa_stream_t stream);

/*
 * pa_copy_blocks — copy-on-write block copies ([P4] §3.3; [P1] §6.1: a
 * forked beam copies only the shared last block).
 *
 *   block_mapping  device int64 [num_pairs, 2]: (src, dst) physical blocks.
 * For each pair, block dst of k_cache and of v_cache becomes a bit-exact copy
 * of block src (all kv_heads * block_size * head_dim elements).
 * Destinations must be distinct and never also a source, so the result does
 * not depend on the order of the copies.  Out-of-range ids are skipped and
 * reported as device error 5.
 */
PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache,
                         const int64_t *block_mapping, int32_t num_pairs,
                         int *device_error, pa_stream_t stream);

typedef enum {
  PA_SWAP_OUT = 0, /* device cache block src -> second-pool block dst */
  PA_SWAP_IN = 1   /* second-pool block src -> device cache block dst */
} pa_swap_direction;

/*
 * pa_swap_blocks — move whole blocks between the device caches and a second
 * pool of the same block shape, normally in CPU memory: the swap-out of a
 * preempted request and its swap-in ([P1] §5.1–§5.2: the KV cache is copied
 * to CPU memory instead of being dropped; [P4] §3.5: inactive blocks go to
 * the CPU swap space; [P3] §7.2: reusable blocks are offloaded to CPU
 * memory).  One launch moves every pair, so small blocks cost no more
 * launches or copy commands than large ones ([P1] §5.2 names the per-block
 * copy count as what makes swapping slow for small blocks).
 *
 *   k_cache/v_cache  device caches described by *cache.
 *   host_k/host_v    the second pool, [host_num_blocks, kv_heads, block_size,
 *                    head_dim] of cache->dtype in the caches' layout.  It
 *                    must be memory the current device can address:
 *                    page-locked host memory (cudaHostAlloc / cudaMallocHost,
 *                    or registered with cudaHostRegister) or memory of the
 *                    current device, 16-byte aligned.  Any other memory
 *                    returns PA_ERR_UNSUPPORTED (checked with
 *                    cudaPointerGetAttributes before any launch).  The
 *                    caller guarantees that it holds host_num_blocks blocks.
 *   block_mapping    device int64 [num_pairs, 2]: (src, dst).  PA_SWAP_OUT:
 *                    src is a device block, dst a second-pool block;
 *                    PA_SWAP_IN: src is a second-pool block, dst a device
 *                    block.
 *   direction        pa_swap_direction.
 * For each pair, block dst of the destination pool (K and V) becomes a
 * bit-exact copy of block src of the source pool.  Destinations must be
 * distinct.  A pair with an id out of its pool's range is skipped and
 * reported as device error 5.  The host pool is read or written by the
 * kernel directly (over NVLink-C2C on a Grace system), so it must stay
 * allocated and page-locked until the stream has passed the call.
 */
PA_API pa_status pa_swap_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache,
                                void *host_k, void *host_v, int64_t host_num_blocks,
                                const int64_t *block_mapping, int32_t num_pairs,
                                int32_t direction, int *device_error, pa_stream_t stream);

/*
 * Prefix cache (host) — the block pool behind the block tables, with
 * prefix caching ([P3] §4.2–§4.3; [P1] §3.2).
 *
 * - A full block's key covers its token ids and everything before it: the
 *   64-bit FNV-1a hash of the parent block's key (8 bytes little-endian, 0
 *   for the first block) followed by the block's token ids (4 bytes each,
 *   little-endian).  A hit also requires the stored parent key and token
 *   ids to equal the request's.
 * - pa_prefix_cache_add_sequence maps the longest run of cached full blocks
 *   from the start of the prompt into the new table (reference count + 1)
 *   and takes fresh blocks for the rest; only the part that missed needs
 *   its KV computed and written.  Fresh full blocks are keyed at once (the
 *   caller writes their KV before any later request attends to them); the
 *   last, partial block stays private until decoding fills it.
 * - pa_prefix_cache_free_sequence decrements the sequence's blocks, last
 *   block first; a block at zero joins the back of the free list and keeps
 *   its content and key until it is taken again.
 * - Fresh blocks are taken from the front of the free list (least recently
 *   freed first; initially the pool order), which evicts a kept key.
 * - A request the free list cannot supply returns PA_ERR_OUT_OF_BLOCKS and
 *   changes nothing.
 * Ownership: the handle owns its memory (host only; no CUDA calls).  Calls
 * on one handle must not overlap (no internal lock).  Block ids are
 * 0..num_blocks-1, the physical blocks of the caches; slot = block *
 * block_size + offset as everywhere in this header.
 */
typedef struct pa_prefix_cache pa_prefix_cache;

typedef struct {
  int64_t free_blocks;         /* blocks on the free list */
  int64_t cached_free_blocks;  /* of which still keyed (hittable) */
  int64_t used_blocks;         /* blocks with a nonzero reference count */
  int64_t cached_blocks;       /* keyed blocks, used or free */
  int64_t queried_tokens;      /* prompt tokens passed to add_sequence */
  int64_t hit_tokens;          /* of which found cached */
  int64_t evictions;           /* keyed free blocks taken for new content */
} pa_prefix_cache_stats;

/* pool_order: host int32 [num_blocks], a permutation giving the initial free
 * order, or NULL for 0..num_blocks-1.  Returns NULL on invalid arguments
 * (or out of host memory). */
PA_API pa_prefix_cache *pa_prefix_cache_create(int32_t num_blocks, int32_t block_size,
                                               const int32_t *pool_order);
PA_API void pa_prefix_cache_destroy(pa_prefix_cache *cache);

/* New sequence seq_id (must not exist) with its prompt tokens (host int32
 * [num_tokens]); *num_cached_tokens (nullable) = prompt tokens found
 * cached, a multiple of block_size. */
PA_API pa_status pa_prefix_cache_add_sequence(pa_prefix_cache *cache, int64_t seq_id,
                                              const int32_t *tokens, int32_t num_tokens,
                                              int32_t *num_cached_tokens);

/* One decoded token: takes a block when the last one is full; *slot
 * (nullable) = the token's flat slot, for pa_reshape_and_cache. */
PA_API pa_status pa_prefix_cache_append_token(pa_prefix_cache *cache, int64_t seq_id,
                                              int32_t token, int64_t *slot);

PA_API pa_status pa_prefix_cache_free_sequence(pa_prefix_cache *cache, int64_t seq_id);

/* Block table of one sequence: returns its length (or -1 for an unknown
 * sequence) and copies up to `capacity` entries to `table` (nullable);
 * *num_tokens (nullable) = the sequence's length in tokens. */
PA_API int32_t pa_prefix_cache_block_table(const pa_prefix_cache *cache, int64_t seq_id,
                                           int32_t *table, int32_t capacity, int32_t *num_tokens);

/* Block tables of several sequences as the host int32 [num_seqs, width]
 * array pa_decode reads (rows zero-padded), and their lengths (host int32
 * [num_seqs], nullable).  PA_ERR_INVALID if a sequence is unknown or has
 * more than `width` blocks (nothing is written then). */
PA_API pa_status pa_prefix_cache_block_tables(const pa_prefix_cache *cache, const int64_t *seq_ids,
                                              int32_t num_seqs, int32_t *tables, int32_t width,
                                              int32_t *seq_lens);

PA_API pa_status pa_prefix_cache_get_stats(const pa_prefix_cache *cache, pa_prefix_cache_stats *out);

/* The free list front to back: returns its length and copies up to
 * `capacity` block ids (out nullable). */
PA_API int32_t pa_prefix_cache_free_order(const pa_prefix_cache *cache, int32_t *out, int32_t capacity);

/* Reference count of a block (-1 for an id out of range). */
PA_API int32_t pa_prefix_cache_ref_count(const pa_prefix_cache *cache, int32_t block);

/*
 * pa_selftest_wait_timeout — exercise the failure path every pipeline wait
 * of this library shares, without faulting the GPU.
 *
 * Launches one CTA that waits, with the same bounded wait the kernels use,
 * on an mbarrier phase that nothing completes.  After the wait's time limit
 * (2 s) the kernel writes device error 4 to *device_error (device int,
 * required) and returns normally: the context stays usable.  Asynchronous
 * on `stream`; allocates nothing.
 */
PA_API pa_status pa_selftest_wait_timeout(int *device_error, pa_stream_t stream);

/* Static description of a status code. */
PA_API const char *pa_status_string(pa_status status);

/* Last CUDA error text seen by a call that returned PA_ERR_CUDA on this
 * thread (static storage; empty if none). */
PA_API const char *pa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
