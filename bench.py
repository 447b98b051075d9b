"""Benchmark of the paged decode path (one JSON line on stdout).

A step is one pass of the whole hot path over one batch: the copy-on-write
block copies (when the workload has any), the cache write of the new tokens,
and paged decode attention.  The default workload is the largest one that
fits one GPU: the OPT-13B-shaped long-context beam decode (32 prompts of
2048..8192 tokens forked into 4 beams = 128 decode rows, 40/40 heads,
head_dim 128, fp16, block size 32, copy-on-write of each shared partial last
block); ``--config`` selects another named workload.

Metric: KV bytes read per step (every K and V element of every sequence's
tokens, counted once per distinct slot: the unique bytes HBM must supply) /
step time, in GB/s; also sequence·layer/s and, for the workloads that share
blocks, the logical bytes the definition reads (``kv_logical_gbs``).  Inputs
are resident in HBM before timing starts; the KV working set (3.8 GB unique
for the default workload) is far larger than L2, so no flush is needed
between steps.

Timing: K steps back to back between two CUDA events give ``value`` (the
calls' kernels overlap as they do in use: the decode's plan may start while
the cache write is still running); K more steps with an event pair around
each ``pa_decode`` call give the decode launch group's duration for
``roofline``.

``--impl reference`` times the CPU oracle (float64 NumPy) on a bounded
sample of the same workload on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention: KV-read HBM GB/s vs GB300 peak; seq·layer/s"
DEFAULT_CONFIG = "opt13b-beam"
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
DECODE_SOURCES = [os.path.join(ROOT, "paged_kv_cache_54_gb300", "csrc", f)
                  for f in ("pa_decode.cuh", "pa_decode_params.h", "pa_common.cuh",
                            "pa_decode_api.cu", "pa_host.cu")]
PREFILL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_traffic.txt")
PREFILL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_54_gb300", "csrc", f)
                   for f in ("pa_prefill.cuh", "pa_prefill.cu", "pa_common.cuh")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=W.ALL_CONFIGS)
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seqs", type=int, default=None,
                    help="a smaller copy of the workload for profiling captures: this many "
                         "sequences (beam workloads: this many prompts); the line then names "
                         "the reduced workload and is not a bench result")
    ap.add_argument("--op", default="step", choices=["step", "swap", "prefix-cache", "prefill"],
                    help="step: the decode step (default); swap: pa_swap_blocks of "
                         "preempted sequences' blocks out to pinned host memory and back; "
                         "prefix-cache: the host prefix cache building shared-prefix tables; "
                         "prefill: causal prefill of each sequence's tokens after the shared "
                         "prefix (qwen3-prefix)")
    ap.add_argument("--swap-seqs", type=int, default=16)
    ap.add_argument("--prefill-cache", default="bf16", choices=["bf16", "e4m3", "e5m2", "int8"],
                    help="cache type of the prefill bench (one-byte caches: codes of N(0,1) K/V "
                         "with scale 1, or 1/32 for int8)")
    return ap.parse_args()


def seqs_override(args):
    """Workload override for --seqs (None: the named workload as it is)."""
    if args.seqs is None:
        return None
    key = "prompts" if W.CONFIGS[args.config]["kind"] == "beam" else "S"
    return {key: int(args.seqs)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def source_hash(paths=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str, path: str = TRAFFIC_FILE, sources=DECODE_SOURCES):
    """DRAM bytes per launch of a kernel from a committed ncu summary, if it
    was taken on the kernel's current source; else None."""
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    src, val = None, None
    for ln in lines:
        if ln.startswith("source_sha:"):
            src = ln.split(":", 1)[1].strip()
        if ln.startswith(f"bytes_per_launch[{key}]:"):
            val = float(ln.split(":", 1)[1].strip())
    if src != source_hash(sources):
        return None
    return val


class ClockSampler:
    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t_on = self.t_off = None

    def mark_start(self):
        self.t_on = time.time()

    def mark_end(self):
        self.t_off = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        # samples inside the timed region (second resolution, so widen by 1 s)
        inside = [r for r in rows if self.t_on - 1 <= r[0] <= self.t_off + 1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v == "Active"})
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in rows) if rows else None,
                "reasons": reasons, "samples": len(inside)}


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of the ranks' values (every rank gets it): the job's time
    is its slowest rank's.  Uses the process group already initialised."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput with the same work on every rank (weak scaling):
    all ranks' units over the slowest rank's time."""
    return world * units_per_rank / seconds


def workload_bytes(w):
    kv = w.kv_unique_bytes()
    qo = 2 * w.S * w.Hq * w.d * 2
    tables = int(sum(-(-int(L) // w.bs) for L in w.seq_lens)) * 4 + w.S * 4
    return kv, kv + qo + tables


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_54_gb300 as pa
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    seed = args.seed if args.seed is not None else W.config_seed(args.config)
    w = W.make_workload(args.config, seed, device=dev, overrides=seqs_override(args))
    shape = (w.num_blocks, w.Hkv, w.bs, w.d)
    if w.cache_dtype in W.BYTE_DTYPES:
        kc = torch.zeros(shape, dtype=torch.uint8, device=dev)
        vc = torch.zeros(shape, dtype=torch.uint8, device=dev)
    else:
        dt = torch.float16 if w.cache_dtype == "f16" else torch.bfloat16
        kc = torch.zeros(shape, dtype=dt, device=dev)
        vc = torch.zeros(shape, dtype=dt, device=dev)

    def scale_arg(x):   # a number, or one float32 scale per KV head on the device
        return float(x) if np.ndim(x) == 0 else torch.tensor(x, dtype=torch.float32, device=dev)

    kw = dict(cache_dtype=w.cache_dtype, k_scale=scale_arg(w.k_scale), v_scale=scale_arg(w.v_scale))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_reshape_and_cache(w.ctx_k, w.ctx_v, torch.from_numpy(w.ctx_slots).to(dev), kc, vc,
                            device_error=err, **kw)
    w.ctx_k = w.ctx_v = None
    torch.cuda.synchronize()
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    slots = torch.from_numpy(w.new_slots).to(dev)
    pairs = torch.from_numpy(w.cow_pairs).to(dev)
    out = torch.empty_like(w.q)
    P = w.partition_size
    ws = torch.empty(pa.pa_decode_workspace_size(w.S, w.Hq, w.Hkv, w.d, w.max_seq_len, P),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    n_pairs = len(w.cow_pairs)
    max_parts_gt1 = w.max_seq_len > (P or _auto_partition(w))
    launches_per_step = (1 if n_pairs else 0) + 1 + 2 + (1 if max_parts_gt1 else 0)

    def step(dec_events=None):
        if n_pairs:
            pa.pa_copy_blocks(kc, vc, pairs, cache_dtype=w.cache_dtype, device_error=err)
        pa.pa_reshape_and_cache(w.new_k, w.new_v, slots, kc, vc, device_error=err, **kw)
        if dec_events is not None:
            dec_events[0].record(stream)
        pa.pa_decode(out, w.q, kc, vc, bt, sl, w.max_seq_len, w.scale, partition_size=P,
                     workspace=ws, device_error=err, **kw)
        if dec_events is not None:
            dec_events[1].record(stream)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    torch.cuda.synchronize()
    # the steps, with nothing between their launches (value)
    t0.record(stream)
    for i in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed = t0.elapsed_time(t1) / 1e3
    # the same K steps again with events around each pa_decode call (the
    # roofline's launch duration); an event between the cache write and the
    # decode keeps the decode's first kernel from overlapping the write, so
    # this loop is not the one `value` comes from
    torch.cuda.synchronize()
    for i in range(K):
        step(ev[i])
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    dec_avg = statistics.mean(dec_ms) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    derr = int(err.item())
    graph_t = graph_step_time(step, K, stream)

    # End to end through the C ABI with host buffers (pinned), every step's
    # copies inside the timed region: the step's inputs are packed in one
    # pinned staging buffer and cross in one copy; the output comes back in
    # one copy.  The copies run on two copy streams, double-buffered, so
    # step i+1's inputs cross while step i computes and step i's output
    # returns while step i+1 computes (as a serving loop pipelines them).
    inputs = [("q", w.q), ("k", w.new_k), ("v", w.new_v), ("slots", slots), ("bt", bt), ("sl", sl)]
    if n_pairs:
        inputs.append(("pairs", pairs))
    offs, total = {}, 0
    for name, t in inputs:
        offs[name] = total
        total += -(-t.numel() * t.element_size() // 256) * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [{}, {}]
    for name, t in inputs:
        n = t.numel() * t.element_size()
        host_buf[offs[name]:offs[name] + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        for j in range(2):
            views[j][name] = dev_bufs[j][offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
    outs = [out, torch.empty_like(out)]
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for _, t in inputs)
    d2h = out.numel() * out.element_size()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_copied = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    for j in range(2):
        ev_free[j].record(stream)

    def e2e_step(i):
        j = i % 2
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(ev_free[j])        # step i-2 is done with buffer j
            dev_bufs[j].copy_(host_buf, non_blocking=True)
            ev_copied[j].record(h2d_stream)
        stream.wait_event(ev_copied[j])
        v = views[j]
        if n_pairs:
            pa.pa_copy_blocks(kc, vc, v["pairs"], cache_dtype=w.cache_dtype, device_error=err)
        pa.pa_reshape_and_cache(v["k"], v["v"], v["slots"], kc, vc, device_error=err, **kw)
        pa.pa_decode(outs[j], v["q"], kc, vc, v["bt"], v["sl"], w.max_seq_len, w.scale, partition_size=P,
                     workspace=ws, device_error=err, **kw)
        ev_done[j].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(ev_done[j])
            out_host.copy_(outs[j], non_blocking=True)
            ev_free[j].record(d2h_stream)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    KE = max(10, K // 5)
    e0.record(stream)
    h2d_stream.wait_stream(stream)  # the first input copy starts after e0
    for i in range(KE):
        e2e_step(i)
    stream.wait_stream(d2h_stream)  # the last output is back
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_t = e0.elapsed_time(e1) / 1e3 / KE
    clocks = sampler.finish() if sampler else None
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    kv_bytes, alg_bytes = workload_bytes(w)
    step_t = elapsed / K
    peaks, peak_kind = measured_peaks()
    achieved = alg_bytes / dec_avg / 1e9
    traffic = recorded_traffic(args.config)
    line = {
        "metric": METRIC,
        "value": round(job_rate(kv_bytes, world, step_t) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_t * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.cache_dtype,
        "data": "synthetic (seeded N(0,1) K/V/q, seeded lengths and shuffled block pool)",
        "config": decode_config(w, args.config, seed, world),
        "seq_layer_per_s": round(world * w.S / step_t, 1),
        "kv_logical_gbs": round(job_rate(w.kv_logical_bytes(), world, step_t) / 1e9, 2),
        "gpu_launches": launches_per_step * 2 * K,  # both timed loops
        "device_error": derr,
        "roofline": {
            "kernel": "pa_decode (plan + persistent decode + merge, CUDA events)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_kind": f"{peak_kind} (copy, burst)",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_bytes,
            "avg_launch_ms": round(dec_avg * 1e3, 4),
            "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
        },
        "e2e": {"value": round(kv_bytes / e2e_t / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "copies": "one packed pinned input copy and one output copy per step, on two copy "
                          "streams, double-buffered (step i+1's inputs cross while step i computes)",
                "ms_per_step": round(e2e_t * 1e3, 4)},
        "clocks": clocks,
        "graph": ({"ms_per_step": round(graph_t * 1e3, 4), "value": round(kv_bytes / graph_t / 1e9, 2),
                   "unit": "GB/s", "note": "the same step captured once in a CUDA graph and replayed"}
                  if isinstance(graph_t, float) else {"error": graph_t}),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config, seed, budget_s=12.0)
    print(json.dumps(line), flush=True)


def _named_seqs(config: str) -> int:
    cfg = W.CONFIGS[config]
    return cfg["prompts"] * cfg["beams"] if cfg["kind"] == "beam" else cfg["S"]


def decode_config(w, config: str, seed: int, world: int) -> dict:
    """The workload description of a decode bench line (both arms)."""
    kv_bytes, _ = workload_bytes(w)
    return {
        "workload": f"{config}{'' if w.S == _named_seqs(config) else ' (reduced)'}: {_describe(w)}",
        "num_seqs": w.S, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.d,
        "block_size": w.bs, "cache_dtype": w.cache_dtype, "q_dtype": w.q_dtype,
        "partition_size": w.partition_size or _auto_partition(w),
        "kv_bytes_per_step": kv_bytes, "seed": seed,
        "l2": "inputs larger than L2 (KV working set %.2f GB vs 129 MB L2)" % (kv_bytes / 1e9),
        "parallelism": f"replicas x{world}",
    }


def graph_step_time(step, K: int, stream):
    """Seconds per step when the step's launches are captured once in a CUDA
    graph and replayed K times (no host launch work between kernels); the
    error text if capture fails."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / K
    except RuntimeError as e:
        return str(e).splitlines()[0][:200]


def _auto_partition(w):
    P = 512
    while P > 64 and w.S * w.Hkv * (-(-w.max_seq_len // P)) < 1024:
        P //= 2
    return P


def _describe(w):
    lens = w.seq_lens
    return (f"{w.S} seqs, L {int(lens.min())}..{int(lens.max())} (mean {float(lens.mean()):.0f}), "
            f"{w.Hq}q/{w.Hkv}kv heads, d {w.d}, bs {w.bs}, {w.cache_dtype} KV"
            f"{', per-head scales' if np.ndim(w.k_scale) else ''}, {w.num_blocks} blocks")


# ---------------------------------------------------------------------------
# the CPU oracle, timed on a bounded sample
# ---------------------------------------------------------------------------
def _oracle_sample(config: str, seed: int, n_seqs: int):
    """Oracle paged cache holding the first n_seqs sequences of the workload
    (their blocks renumbered into a compact pool, fresh seeded values)."""
    import torch
    from oracle.cache import PagedKVCache, bits_to_f64
    full = W.make_workload(config, seed, values=False)
    w = W.subset(full, range(min(n_seqs, full.S)), seed)

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    c = PagedKVCache(w.num_blocks, w.Hkv, w.bs, w.d, w.cache_dtype, w.k_scale, w.v_scale)
    c.reshape_and_cache(bits(w.ctx_k), bits(w.ctx_v), w.src_dtype, w.ctx_slots)
    c.reshape_and_cache(bits(w.new_k), bits(w.new_v), w.src_dtype, w.new_slots)
    qv = bits_to_f64(bits(w.q), w.q_dtype)
    kv = int(w.seq_lens.astype(np.int64).sum()) * w.Hkv * w.d * w.elt_bytes() * 2
    return w, c, w.block_tables, w.seq_lens, qv, kv


def _oracle_rate(config: str, seed: int, budget_s: float, n_seqs: int = 4) -> dict:
    """The oracle's decode of a bounded sample, repeated for about budget_s."""
    from oracle import attention as A
    w, c, tables, lens, qv, kv = _oracle_sample(config, seed, n_seqs)
    t0 = time.perf_counter()
    reps = 0
    while True:
        A.paged_decode(qv, c.k, c.v, w.cache_dtype, tables, lens, w.scale, w.k_scale, w.v_scale)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"gbs": kv / dt / 1e9, "seq_per_s": len(lens) / dt, "reps": reps, "tokens": int(lens.sum()),
            "seqs": len(lens), "q_heads": w.Hq}


def _single_core_rate(config: str, seed: int, budget_s: float) -> dict | None:
    """_oracle_rate in a child process pinned to one core, with one BLAS
    thread; None if the child fails."""
    cpu = min(os.sched_getaffinity(0))
    code = ("import json, os, sys; os.sched_setaffinity(0, {%d}); sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_rate(%r, %d, %r)))" % (cpu, ROOT, config, seed, budget_s))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    env.pop("CUDA_VISIBLE_DEVICES", None)
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           timeout=budget_s + 240)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (subprocess.TimeoutExpired, ValueError, IndexError):
        return None


def cpu_baseline(config: str, seed: int, budget_s: float = 12.0, n_seqs: int = 4,
                 single_budget_s: float = 8.0):
    r = _oracle_rate(config, seed, budget_s, n_seqs)
    out = {"value": round(r["gbs"], 4), "unit": "GB/s", "cores": _cores(), "kind": "oracle",
           "sample": f"first {r['seqs']} sequences of {config} (all {r['q_heads']} query heads, "
                     f"{r['tokens']} tokens), float64 NumPy oracle, {r['reps']} passes in {budget_s:.0f} s",
           "seq_layer_per_s": round(r["seq_per_s"], 3)}
    one = _single_core_rate(config, seed, single_budget_s) if single_budget_s > 0 else None
    if one is not None:
        out["single_core"] = {"value": round(one["gbs"], 4), "unit": "GB/s", "cores": 1,
                              "seq_layer_per_s": round(one["seq_per_s"], 3),
                              "sample": f"the same sample in a process pinned to one core with one BLAS "
                                        f"thread, {one['reps']} passes in {single_budget_s:.0f} s"}
    return out


def _cores() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return len(os.sched_getaffinity(0))


def run_reference(args, rank, world):
    if rank != 0:
        return
    seed = args.seed if args.seed is not None else W.config_seed(args.config)
    from oracle import attention as A
    w, c, tables, lens, qv, kv = _oracle_sample(args.config, seed, 2)
    for _ in range(args.warmup):
        A.paged_decode(qv, c.k, c.v, w.cache_dtype, tables, lens, w.scale, w.k_scale, w.v_scale)
    steps = min(args.steps, 20)
    t0 = time.perf_counter()
    for _ in range(steps):
        A.paged_decode(qv, c.k, c.v, w.cache_dtype, tables, lens, w.scale, w.k_scale, w.v_scale)
    dt = (time.perf_counter() - t0) / steps
    val = round(kv / dt / 1e9, 4)
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": decode_config(W.make_workload(args.config, seed, values=False), args.config,
                                                   seed, world),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": _cores(), "kind": "oracle",
                         "sample": f"first 2 sequences of {args.config}, all query heads"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# block swap between the device caches and page-locked host memory
# ---------------------------------------------------------------------------
SWAP_METRIC = "KV block swap device<->host GB/s (pa_swap_blocks, out + in)"


def _swap_pairs(w, n_seqs):
    """Swap-out pairs (device block, host slot) of the first n_seqs sequences'
    blocks, and swap-in pairs (host slot, free device block)."""
    seqs = range(min(n_seqs, w.S))
    blocks = [int(b) for s in seqs for b in w.block_tables[s, :-(-int(w.seq_lens[s]) // w.bs)]]
    used = {int(b) for s in range(w.S) for b in w.block_tables[s, :-(-int(w.seq_lens[s]) // w.bs)]}
    free = [b for b in range(w.num_blocks) if b not in used]
    n = min(len(blocks), len(free))
    out_pairs = np.array([[b, i] for i, b in enumerate(blocks[:n])], dtype=np.int64)
    in_pairs = np.array([[i, f] for i, f in enumerate(free[:n])], dtype=np.int64)
    return out_pairs, in_pairs


def run_swap(args, rank, world, local):
    import torch
    import paged_kv_cache_54_gb300 as pa
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    seed = args.seed if args.seed is not None else W.config_seed(args.config)
    w = W.make_workload(args.config, seed, values=False)
    out_np, in_np = _swap_pairs(w, args.swap_seqs)
    n = len(out_np)
    elt = w.elt_bytes()
    shape = (w.num_blocks, w.Hkv, w.bs, w.d)
    cdt = torch.uint8 if elt == 1 else torch.int16
    gen = torch.Generator(device=dev).manual_seed(seed)
    kc = torch.randint(0, 255, shape, generator=gen, device=dev, dtype=torch.int32).to(cdt)
    vc = torch.randint(0, 255, shape, generator=gen, device=dev, dtype=torch.int32).to(cdt)
    hk = torch.empty((n,) + shape[1:], dtype=cdt).pin_memory()
    hv = torch.empty((n,) + shape[1:], dtype=cdt).pin_memory()
    out_pairs = torch.from_numpy(out_np).to(dev)
    in_pairs = torch.from_numpy(in_np).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kw = dict(cache_dtype=w.cache_dtype, device_error=err)
    block_bytes = w.Hkv * w.bs * w.d * elt
    moved = 2 * n * block_bytes                       # K and V, per direction
    stream = torch.cuda.current_stream()

    def swap_step(evs=None):
        if evs:
            evs[0].record(stream)
        pa.pa_swap_blocks(kc, vc, hk, hv, out_pairs, "out", **kw)
        if evs:
            evs[1].record(stream)
        pa.pa_swap_blocks(kc, vc, hk, hv, in_pairs, "in", **kw)
        if evs:
            evs[2].record(stream)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        swap_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if sampler:
        sampler.mark_start()
    torch.cuda.synchronize()
    for i in range(K):
        swap_step(evs[i])
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    t_out = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_in = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    elapsed = evs[0][0].elapsed_time(evs[-1][2]) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    # the link's copy-engine rate for the same bytes: one contiguous pinned
    # copy per direction (the denominator of the roofline)
    flat_d = torch.empty(moved, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(moved, dtype=torch.uint8).pin_memory()

    def ce_time(dst, src, reps=10):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / reps

    ce_d2h = ce_time(flat_h, flat_d)
    ce_h2d = ce_time(flat_d, flat_h)
    # end to end through the public call: the pairs are uploaded from pinned
    # host memory each step, the error flag read back
    hp_out, hp_in = out_pairs.cpu().pin_memory(), in_pairs.cpu().pin_memory()
    err_host = torch.empty(1, dtype=torch.int32).pin_memory()

    def e2e_step():
        out_pairs.copy_(hp_out, non_blocking=True)
        in_pairs.copy_(hp_in, non_blocking=True)
        swap_step()
        err_host.copy_(err, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KE = max(5, K // 4)
    e0.record(stream)
    for _ in range(KE):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_t = e0.elapsed_time(e1) / 1e3 / KE
    clocks = sampler.finish() if sampler else None
    derr = int(err.item())
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    step_t = elapsed / K
    achieved = 2 * moved / (t_out + t_in) / 1e9
    peak = 2 * moved / (ce_d2h + ce_h2d) / 1e9 if ce_d2h > 0 and ce_h2d > 0 else None
    line = {
        "metric": SWAP_METRIC, "value": round(job_rate(2 * moved, world, step_t) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(step_t * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (random cache bytes; block ids of the workload's first sequences)",
        "config": {
            "workload": f"swap of {min(args.swap_seqs, w.S)} sequences of {args.config} "
                        f"({n} blocks of {block_bytes // 1024} KiB per K or V) out to pinned host "
                        f"memory and back into free device blocks",
            "blocks": n, "bytes_per_direction": moved, "block_bytes": block_bytes,
            "l2": "inputs larger than L2 (%.0f MB per direction vs 129 MB L2)" % (moved / 1e6),
            "parallelism": f"replicas x{world}",
        },
        "gpu_launches": 2 * K,
        "device_error": derr,
        "swap_out_gbs": round(moved / t_out / 1e9, 2),
        "swap_in_gbs": round(moved / t_in / 1e9, 2),
        "roofline": {
            "kernel": "swap_blocks_kernel (out + in, CUDA events)", "bound": "c2c",
            "achieved": round(achieved, 2), "peak": None if peak is None else round(peak, 2),
            "unit": "GB/s", "frac": None if peak is None else round(achieved / peak, 4),
            "peak_kind": "measured in this run: one contiguous pinned copy-engine transfer of "
                         "the same bytes per direction (no host-link figure in the driver's peaks)",
            "copy_engine_d2h_gbs": round(moved / ce_d2h / 1e9, 2),
            "copy_engine_h2d_gbs": round(moved / ce_h2d / 1e9, 2),
            "traffic": None,
        },
        "e2e": {"value": round(2 * moved / e2e_t / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(2 * n * 16), "d2h_bytes_per_step": 4,
                "ms_per_step": round(e2e_t * 1e3, 4)},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = swap_cpu_baseline(w, out_np)
    print(json.dumps(line), flush=True)


def swap_cpu_baseline(w, out_np, budget_s: float = 5.0):
    """The oracle's pool-to-pool block moves on the host cores (a bounded
    sample: the first 64 swap-out pairs)."""
    from oracle.cache import PagedKVCache
    pairs = out_np[:64]
    nb = int(pairs[:, 0].max()) + 1
    dev = PagedKVCache(nb, w.Hkv, w.bs, w.d, w.cache_dtype, fill_nan=False)
    host = PagedKVCache(len(pairs), w.Hkv, w.bs, w.d, w.cache_dtype, fill_nan=False)
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s:
        dev.swap_blocks(host, pairs, "out")
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    nbytes = 2 * len(pairs) * dev.k[0].nbytes
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(pairs)} block pairs swapped out by the NumPy oracle, {reps} passes"}


# ---------------------------------------------------------------------------
# the host prefix cache (native C++ behind the C ABI)
# ---------------------------------------------------------------------------
PREFIX_METRIC = "prefix cache: prompt tokens looked up and placed per second (host, native)"


def _prefix_requests(seed, n=256, prompt_len=1024, lo=16, hi=512):
    rng = np.random.default_rng(seed)
    prompt = rng.integers(0, 32000, prompt_len).astype(np.int32)
    return [np.concatenate([prompt, rng.integers(0, 32000, int(rng.integers(lo, hi + 1)))
                            .astype(np.int32)]) for _ in range(n)]


def _prefix_pass(c, reqs):
    for s, t in enumerate(reqs):
        c.add_sequence(s, t)
    for s in range(len(reqs)):
        c.free_sequence(s)


def run_prefix_cache(args, rank, world):
    """A step: 256 requests sharing one 1024-token prompt (the shared-prefix
    decode workload's structure) are admitted, then all finish; the first
    step computes the prompt, every later one hits it in the kept blocks."""
    if rank != 0:
        return
    import paged_kv_cache_54_gb300 as pa
    seed = args.seed if args.seed is not None else 3
    reqs = _prefix_requests(seed)
    nb = 64 + sum(-(-(len(t) - 1024) // 16) for t in reqs) + 64
    c = pa.PrefixCache(nb, 16)
    for _ in range(max(3, args.warmup)):
        _prefix_pass(c, reqs)
    K = min(args.steps, 200)
    t0 = time.perf_counter()
    for _ in range(K):
        _prefix_pass(c, reqs)
    dt = (time.perf_counter() - t0) / K
    st = c.stats()
    ntok = int(sum(len(t) for t in reqs))
    line = {
        "metric": PREFIX_METRIC, "value": round(ntok / dt, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded token ids)",
        "config": {"workload": f"256 requests = one 1024-token prompt + U[16,512] own tokens, "
                               f"block size 16, {nb} blocks; admit all, then free all",
                   "tokens_per_step": ntok, "hit_rate": round(st["hit_tokens"] / st["queried_tokens"], 4)},
        "gpu_launches": 0,
        "roofline": None,
        "note": "host code: no GPU kernel runs in this operation",
    }
    if not args.no_cpu_baseline:
        from oracle.prefix_cache import PrefixCache
        o = PrefixCache(nb, 16)
        _prefix_pass(o, reqs)
        t0, reps = time.perf_counter(), 0
        while time.perf_counter() - t0 < 5.0:
            _prefix_pass(o, reqs)
            reps += 1
        odt = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": round(ntok / odt, 1), "unit": "tokens/s", "cores": 1,
                                "kind": "oracle", "sample": f"the same step in the Python oracle, {reps} passes"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# causal prefill of the part a prefix hit did not cover
# ---------------------------------------------------------------------------
PREFILL_METRIC = "paged causal prefill after a prefix hit: TFLOP/s (QK^T + PV) and new tokens/s"


def prefill_flops(w, q_lens):
    """Algorithmic flops: each new token j of sequence s (position p) does
    2*d multiply-adds per key for QK^T and for PV over p + 1 keys, per
    query head."""
    total = 0
    for s, n in enumerate(q_lens):
        L = int(w.seq_lens[s])
        keys = sum(range(L - n + 1, L + 1))          # sum over j of (p_j + 1)
        total += 4 * w.d * w.Hq * keys
    return total


def run_prefill(args, rank, world, local):
    import torch
    import paged_kv_cache_54_gb300 as pa
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    config = "qwen3-prefix"
    seed = args.seed if args.seed is not None else W.config_seed(config)
    w = W.make_workload(config, seed, device=dev)
    prefix = W.CONFIGS[config]["prefix"]
    q_lens = [int(L) - prefix for L in w.seq_lens]
    T = sum(q_lens)
    shape = (w.num_blocks, w.Hkv, w.bs, w.d)
    cdt = args.prefill_cache
    byte = cdt != "bf16"
    kc = torch.zeros(shape, dtype=torch.uint8 if byte else torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kw = dict(cache_dtype=cdt, k_scale=1 / 32 if cdt == "int8" else 1.0,
              v_scale=1 / 32 if cdt == "int8" else 1.0)
    # the cached prefix is written once (it was computed by an earlier
    # request); each step writes the new tokens' K/V and prefills them
    pa.pa_reshape_and_cache(w.ctx_k[:prefix].contiguous(), w.ctx_v[:prefix].contiguous(),
                            torch.from_numpy(w.ctx_slots[:prefix]).to(dev), kc, vc, **kw)
    gen = torch.Generator(device=dev).manual_seed(seed)
    k_new = torch.randn((T, w.Hkv, w.d), generator=gen, device=dev).bfloat16()
    v_new = torch.randn((T, w.Hkv, w.d), generator=gen, device=dev).bfloat16()
    q = torch.randn((T, w.Hq, w.d), generator=gen, device=dev).bfloat16()
    slots_np = np.concatenate([
        [int(w.block_tables[s, p // w.bs]) * w.bs + p % w.bs for p in range(prefix, int(w.seq_lens[s]))]
        for s in range(w.S)]).astype(np.int64)
    slots = torch.from_numpy(slots_np).to(dev)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32, device=dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    maxq = max(q_lens)

    def step(evs=None):
        pa.pa_reshape_and_cache(k_new, v_new, slots, kc, vc, device_error=err, **kw)
        if evs:
            evs[0].record(stream)
        pa.pa_prefill(out, q, cu, kc, vc, bt, sl, maxq, w.scale, device_error=err, **kw)
        if evs:
            evs[1].record(stream)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    elapsed = t0.elapsed_time(t1) / 1e3
    pf = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    # end to end: q and the new K/V from pinned host memory, the output back
    hq_, hk_, hv_ = q.cpu().pin_memory(), k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        q.copy_(hq_, non_blocking=True)
        k_new.copy_(hk_, non_blocking=True)
        v_new.copy_(hv_, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KE = max(5, K // 4)
    e0.record(stream)
    for _ in range(KE):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_t = e0.elapsed_time(e1) / 1e3 / KE
    clocks = sampler.finish() if sampler else None
    derr = int(err.item())
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    flops = prefill_flops(w, q_lens)
    peaks, kind = measured_peaks()
    peak = peaks.get("bf16_tflops")
    achieved = flops / pf / 1e12
    step_t = elapsed / K
    line = {
        "metric": PREFILL_METRIC, "value": round(job_rate(flops, world, step_t) / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(step_t * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if byte else "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V; the shared-prefix workload's tables and lengths)",
        "config": {"workload": f"{config}: {w.S} seqs, cached prefix {prefix} tokens, new tokens "
                               f"{min(q_lens)}..{max(q_lens)} (total {T}), {w.Hq}q/{w.Hkv}kv heads, "
                               f"d {w.d}, bs {w.bs}, q bf16, cache {cdt}",
                   "new_tokens_per_step": T, "flops_per_step": flops,
                   "l2": "K/V of the suffixes %.0f MB + the shared prefix; outputs %.0f MB"
                         % (T * w.Hkv * w.d * (2 if byte else 4) / 1e6, T * w.Hq * w.d * 2 / 1e6),
                   "parallelism": f"replicas x{world}"},
        "new_tokens_per_s": round(world * T / step_t, 1),
        "gpu_launches": 2 * K,
        "device_error": derr,
        "roofline": {"kernel": "prefill_kernel (CUDA events)", "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4) if peak else None,
                     "peak_kind": f"{kind} dense bf16 (cuBLAS, burst)",
                     "traffic": recorded_traffic(cdt, PREFILL_TRAFFIC_FILE, PREFILL_SOURCES),
                     "avg_launch_ms": round(pf * 1e3, 4),
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": round(flops / e2e_t / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(q.numel() * 2 + k_new.numel() * 4),
                "d2h_bytes_per_step": int(out.numel() * 2), "ms_per_step": round(e2e_t * 1e3, 4)},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w, q_lens, prefix, cdt)
    print(json.dumps(line), flush=True)


def prefill_cpu_baseline(w, q_lens, prefix, cache_dtype="bf16", budget_s: float = 10.0):
    """The oracle's prefill on a bounded sample: the first sequence's first
    16 new tokens, all query heads, over random finite codes of the cache
    type."""
    import torch
    from oracle import attention as A
    from oracle.cache import PagedKVCache
    sub = W.subset(w, [0], 1)
    n = min(16, q_lens[0])
    L = prefix + n
    c = PagedKVCache(sub.num_blocks, sub.Hkv, sub.bs, sub.d, cache_dtype, fill_nan=False)
    rng = np.random.default_rng(0)
    if cache_dtype == "bf16":
        c.k[:] = rng.integers(0, 1 << 15, c.k.shape, dtype=np.uint16) & 0x3BFF
        c.v[:] = rng.integers(0, 1 << 15, c.v.shape, dtype=np.uint16) & 0x3BFF
    else:  # finite codes (no FP8 NaN or infinity)
        c.k[:] = rng.integers(0, 256, c.k.shape, dtype=np.uint8) & 0xF6
        c.v[:] = rng.integers(0, 256, c.v.shape, dtype=np.uint8) & 0xF6
    q = rng.standard_normal((n, w.Hq, w.d))
    t0, reps = time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s:
        A.paged_prefill(q, [n], c.k, c.v, cache_dtype, sub.block_tables, np.array([L]), w.scale)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    flops = 4 * w.d * w.Hq * sum(range(L - n + 1, L + 1))
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{n} new tokens after a {prefix}-token prefix, all {w.Hq} query heads, "
                      f"float64 NumPy oracle, {reps} passes"}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.op == "prefill":
        run_prefill(args, rank, world, local)
    elif args.op == "prefix-cache":
        run_prefix_cache(args, rank, world)
    elif args.op == "swap":
        run_swap(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
