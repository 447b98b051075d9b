"""Helpers for the GPU parity tests: run a workload through the C ABI and
build the oracle's view of the same inputs."""
import numpy as np
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from oracle import attention as A
from oracle import fp8 as F
from oracle import int8 as I8
from oracle.cache import NAN_CODE, PagedKVCache, bits_to_f64, head_scale

DEV = "cuda:0"
TOL = {"f16": 2e-3, "bf16": 1e-2}
FP8_TOL = 1e-2    # one-byte caches (FP8, INT8) against the oracle on the dequantised values


def bits(t):
    t = t.detach().cpu().contiguous()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def new_caches(w):
    shape = (w.num_blocks, w.Hkv, w.bs, w.d)
    if w.cache_dtype in W.BYTE_DTYPES:
        kc = torch.full(shape, NAN_CODE[w.cache_dtype], dtype=torch.uint8, device=DEV)
        vc = torch.full(shape, NAN_CODE[w.cache_dtype], dtype=torch.uint8, device=DEV)
    else:
        dt = torch.float16 if w.cache_dtype == "f16" else torch.bfloat16
        kc = torch.full(shape, float("nan"), dtype=dt, device=DEV)
        vc = torch.full(shape, float("nan"), dtype=dt, device=DEV)
    return kc, vc


def scale_arg(scale):
    """A workload's scale as the binding takes it: a number, or a float32
    device tensor of one scale per KV head."""
    if np.ndim(scale) == 0:
        return float(scale)
    return torch.tensor(scale, dtype=torch.float32, device=DEV)


class GpuRun:
    """Set-up (context write) and one step (copies, new tokens, decode)."""

    def __init__(self, w, partition_size=None):
        self.w = w
        self.P = w.partition_size if partition_size is None else partition_size
        self.kc, self.vc = new_caches(w)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.bt = torch.from_numpy(w.block_tables).to(DEV)
        self.sl = torch.from_numpy(w.seq_lens).to(DEV)
        self.new_slots = torch.from_numpy(w.new_slots).to(DEV)
        self.pairs = torch.from_numpy(w.cow_pairs).to(DEV)
        self.out = torch.empty_like(w.q)
        self.kw = dict(cache_dtype=w.cache_dtype, k_scale=scale_arg(w.k_scale),
                       v_scale=scale_arg(w.v_scale))
        self.ws = torch.empty(max(256, pa.pa_decode_workspace_size(
            w.S, w.Hq, w.Hkv, w.d, w.max_seq_len, self.P)), dtype=torch.uint8, device=DEV)

    def setup(self):
        w = self.w
        if len(w.ctx_slots):
            slots = torch.from_numpy(w.ctx_slots).to(DEV)
            pa.pa_reshape_and_cache(w.ctx_k, w.ctx_v, slots, self.kc, self.vc,
                                    device_error=self.err, **self.kw)
        return self

    def step(self):
        w = self.w
        if len(w.cow_pairs):
            pa.pa_copy_blocks(self.kc, self.vc, self.pairs, cache_dtype=w.cache_dtype,
                              device_error=self.err)
        pa.pa_reshape_and_cache(w.new_k, w.new_v, self.new_slots, self.kc, self.vc,
                                device_error=self.err, **self.kw)
        self.decode()
        return self

    def decode(self):
        w = self.w
        pa.pa_decode(self.out, w.q, self.kc, self.vc, self.bt, self.sl, w.max_seq_len,
                     w.scale, partition_size=self.P, workspace=self.ws,
                     device_error=self.err, **self.kw)
        return self.out


def oracle_cache(w):
    """The oracle's own cache after set-up and one step (small workloads)."""
    c = PagedKVCache(w.num_blocks, w.Hkv, w.bs, w.d, w.cache_dtype, w.k_scale, w.v_scale)
    c.reshape_and_cache(bits(w.ctx_k), bits(w.ctx_v), w.src_dtype, w.ctx_slots)
    c.copy_blocks(w.cow_pairs)
    c.reshape_and_cache(bits(w.new_k), bits(w.new_v), w.src_dtype, w.new_slots)
    return c


def encode_rows(w, raw, which):
    """Oracle storage codes of source rows [n, Hkv, d] (16-bit patterns) for
    the K (which="k") or V cache: each head with its own scale."""
    if w.cache_dtype not in W.BYTE_DTYPES:
        return raw
    scales = w.k_scale if which == "k" else w.v_scale
    out = np.empty(raw.shape, dtype=np.uint8)
    for h in range(raw.shape[1]):
        sc = head_scale(scales, h)
        if w.cache_dtype == "int8":
            out[:, h] = I8.quantize_bits16(raw[:, h], w.src_dtype, sc)
        else:
            out[:, h] = F.quantize_bits16(raw[:, h], w.src_dtype, sc, w.cache_dtype)
    return out


def q_values(w):
    return bits_to_f64(bits(w.q), w.q_dtype)


def oracle_decode(w, c, rows=None):
    return A.paged_decode(q_values(w), c.k, c.v, w.cache_dtype, w.block_tables, w.seq_lens,
                          w.scale, w.k_scale, w.v_scale, rows=rows)


def logical_kv(w, s, h):
    """float64 [L, d] K and V of sequence s, KV head h, from the input rows."""
    rows = w.token_rows(s)
    ctx_idx = [i for k, i in rows if k == "ctx"]
    new_idx = [i for k, i in rows if k == "new"]
    out = []
    for src_ctx, src_new, scales in ((w.ctx_k, w.new_k, w.k_scale), (w.ctx_v, w.new_v, w.v_scale)):
        scale = head_scale(scales, h)
        parts = []
        if ctx_idx:
            parts.append(bits(src_ctx[torch.tensor(ctx_idx, device=src_ctx.device), h]))
        if new_idx:
            parts.append(bits(src_new[torch.tensor(new_idx, device=src_new.device), h]))
        raw = np.concatenate(parts) if parts else np.zeros((0, w.d), np.uint16)
        if w.cache_dtype == "int8":
            vals = I8.decode(I8.quantize_bits16(raw, w.src_dtype, scale)) * scale
        elif w.cache_dtype in ("e4m3", "e5m2"):
            vals = F.decode(F.quantize_bits16(raw, w.src_dtype, scale, w.cache_dtype),
                            w.cache_dtype) * scale
        else:
            vals = bits_to_f64(raw, w.src_dtype)
        out.append(vals)
    return out


def oracle_rows(w, rows):
    """Oracle output for sampled (s, hq) rows, from the logical sequences."""
    q = q_values(w)
    res = {}
    for s, hq in rows:
        h = hq // w.G
        K, V = logical_kv(w, s, h)
        res[(s, hq)] = A.attend(q[s, hq], K, V, w.scale)[0]
    return res


def ulp(x, dtype):
    """Spacing of the output dtype at |x| (fp16: 11 significant bits, bf16: 8)."""
    mant = 10 if dtype == "f16" else 7
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 2.0 ** (e - mant)


def tolerance(w):
    return FP8_TOL if w.cache_dtype in W.BYTE_DTYPES else TOL[w.q_dtype]


def _head_values(raw_h, w, scale):
    """float64 values of one KV head's source rows [L, d] (16-bit patterns) as
    the cache holds them: encoded with the head's scale and decoded for
    one-byte caches."""
    if w.cache_dtype not in W.BYTE_DTYPES:
        return bits_to_f64(raw_h, w.src_dtype)
    if w.cache_dtype == "int8":
        return I8.decode(I8.quantize_bits16(raw_h, w.src_dtype, scale)) * scale
    return F.decode(F.quantize_bits16(raw_h, w.src_dtype, scale, w.cache_dtype), w.cache_dtype) * scale


def _logical_raw(w, s):
    """16-bit patterns [Hkv, L, d] of sequence s's K and V input rows in
    position order."""
    rows = w.token_rows(s)
    ctx_idx = [i for k, i in rows if k == "ctx"]
    new_idx = [i for k, i in rows if k == "new"]
    out = []
    for src_ctx, src_new in ((w.ctx_k, w.new_k), (w.ctx_v, w.new_v)):
        parts = []
        if ctx_idx:
            parts.append(src_ctx[torch.tensor(ctx_idx, device=src_ctx.device)])
        if new_idx:
            parts.append(src_new[torch.tensor(new_idx, device=src_new.device)])
        if parts:
            out.append(bits(torch.cat(parts).transpose(0, 1)))
        else:
            out.append(np.zeros((w.Hkv, 0, w.d), np.uint16))
    return out


def oracle_all_rows(w, threads=None):
    """Oracle output for every (s, hq), float64 [S, Hq, d], from each
    sequence's logical tokens (its input rows in position order: independent
    of the block tables and of the device caches).  Sequences run on a thread
    pool; each one is the plain ``attend`` of its query group over its
    tokens."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    q = q_values(w)
    res = np.empty((w.S, w.Hq, w.d), dtype=np.float64)

    def one(s):
        rk, rv = _logical_raw(w, s)
        for h in range(w.Hkv):
            K = _head_values(rk[h], w, head_scale(w.k_scale, h))
            V = _head_values(rv[h], w, head_scale(w.v_scale, h))
            hs = slice(h * w.G, (h + 1) * w.G)
            res[s, hs] = A.attend(q[s, hs], K, V, w.scale)

    n = threads or min(16, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(one, range(w.S)))
    return res


def check_written_slots(w, kc, vc, chunk=8192):
    """Every slot the set-up and the step wrote holds the oracle's code of its
    source row, bit for bit (rows taken in chunks to bound host memory).
    Returns the number of slots checked."""
    new_set = set(int(x) for x in w.new_slots)
    checked = 0
    for src_k, src_v, slots, skip in ((w.ctx_k, w.ctx_v, w.ctx_slots, new_set),
                                      (w.new_k, w.new_v, w.new_slots, set())):
        for a in range(0, len(slots), chunk):
            sl = np.asarray(slots[a:a + chunk], dtype=np.int64)
            keep = np.array([x >= 0 and int(x) not in skip for x in sl], dtype=bool)
            if not keep.any():
                continue
            idx = torch.from_numpy(np.arange(a, a + len(sl))[keep]).to(src_k.device)
            blk = torch.from_numpy(sl[keep] // w.bs).to(kc.device)
            off = torch.from_numpy(sl[keep] % w.bs).to(kc.device)
            for src, cache, which in ((src_k, kc, "k"), (src_v, vc, "v")):
                want = encode_rows(w, bits(src[idx]), which)
                got = bits(cache[blk, :, off, :])
                np.testing.assert_array_equal(got, want)
            checked += int(keep.sum())
    return checked


def permuted_caches(kc, vc, block_tables, seed):
    """The same cache contents under a seeded permutation pi of the physical
    blocks: block b moves to pi[b] and every table entry follows it."""
    nb = kc.shape[0]
    pi = np.random.default_rng(seed).permutation(nb)
    pi_t = torch.from_numpy(pi).to(kc.device)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[pi_t] = kc
    vc2[pi_t] = vc
    bt = np.asarray(block_tables)
    bt2 = np.where((bt >= 0) & (bt < nb), pi[np.clip(bt, 0, nb - 1)], bt).astype(np.int32)
    return kc2, vc2, bt2
