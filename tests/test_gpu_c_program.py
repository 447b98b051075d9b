"""A C99 program drives the device calls of include/pa.h with no Python in
between: it allocates the caches and inputs with the CUDA runtime, writes a
workload's context and new tokens with pa_reshape_and_cache, runs its
copy-on-write pairs with pa_copy_blocks and decodes with pa_decode into a
workspace sized by pa_decode_workspace_size, on a stream it created.  The
test compares what the program wrote back with the oracle: the caches bit
for bit, the decode within the dtype's tolerance."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads as W
from oracle import attention as A
from oracle.cache import PagedKVCache, bits_to_f64
from tests import _gpu as G

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "pa.h"

static char dir[4096];

static void *load(const char *name, size_t bytes) {
  char path[4200];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void *h = malloc(bytes ? bytes : 1);
  FILE *f = fopen(path, "rb");
  if (!h || !f || fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "read %s\n", name); exit(2); }
  fclose(f);
  return h;
}

static void save(const char *name, const void *h, size_t bytes) {
  char path[4200];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f || fwrite(h, 1, bytes, f) != bytes) { fprintf(stderr, "write %s\n", name); exit(2); }
  fclose(f);
}

static void *to_device(const char *name, size_t bytes) {
  void *h = load(name, bytes), *d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 256) != cudaSuccess ||
      cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) { fprintf(stderr, "h2d %s\n", name); exit(3); }
  free(h);
  return d;
}

#define CHECK(call) do { pa_status st_ = (call); if (st_ != PA_OK) { \
  fprintf(stderr, "%s: %s (%s)\n", #call, pa_status_string(st_), pa_last_cuda_error()); return 4; } } while (0)

int main(int argc, char **argv) {
  if (argc != 2) return 1;
  snprintf(dir, sizeof dir, "%s", argv[1]);
  char path[4200];
  snprintf(path, sizeof path, "%s/meta.txt", dir);
  FILE *m = fopen(path, "r");
  int S, Hq, Hkv, d, bs, nb, cdt, qdt, tc, tn, npairs, maxb, max_len;
  float scale, ks, vs;
  if (!m || fscanf(m, "%d %d %d %d %d %d %d %d %d %d %d %d %d %f %f %f", &S, &Hq, &Hkv, &d, &bs, &nb,
                   &cdt, &qdt, &tc, &tn, &npairs, &maxb, &max_len, &scale, &ks, &vs) != 16) return 1;
  fclose(m);
  const size_t elt = cdt >= PA_FP8_E4M3 ? 1 : 2;
  const size_t row = (size_t)Hkv * d * 2;  /* a source row is 16-bit */
  const size_t cache_bytes = (size_t)nb * Hkv * bs * d * elt;
  pa_cache_desc desc;
  memset(&desc, 0, sizeof desc);
  desc.num_blocks = nb; desc.kv_heads = Hkv; desc.block_size = bs; desc.head_dim = d;
  desc.dtype = cdt; desc.k_scale = ks; desc.v_scale = vs;

  cudaStream_t stream;
  if (cudaStreamCreate(&stream) != cudaSuccess) return 3;
  void *kc = NULL, *vc = NULL;
  int *err = NULL;
  if (cudaMalloc(&kc, cache_bytes) != cudaSuccess || cudaMalloc(&vc, cache_bytes) != cudaSuccess ||
      cudaMalloc((void **)&err, sizeof(int)) != cudaSuccess) return 3;
  /* never-written slots read as NaN (0xFF bytes: NaN in fp16, bf16 and e4m3) */
  cudaMemset(kc, 0xFF, cache_bytes);
  cudaMemset(vc, 0xFF, cache_bytes);
  cudaMemset(err, 0, sizeof(int));

  void *ck = to_device("ctx_k.bin", (size_t)tc * row), *cv = to_device("ctx_v.bin", (size_t)tc * row);
  void *cs = to_device("ctx_slots.bin", (size_t)tc * 8);
  void *nk = to_device("new_k.bin", (size_t)tn * row), *nv = to_device("new_v.bin", (size_t)tn * row);
  void *ns = to_device("new_slots.bin", (size_t)tn * 8);
  void *pairs = to_device("pairs.bin", (size_t)npairs * 16);
  void *q = to_device("q.bin", (size_t)S * Hq * d * 2);
  void *bt = to_device("bt.bin", (size_t)S * maxb * 4);
  void *sl = to_device("sl.bin", (size_t)S * 4);
  void *out = NULL;
  if (cudaMalloc(&out, (size_t)S * Hq * d * 2) != cudaSuccess) return 3;
  const size_t ws_bytes = pa_decode_workspace_size(S, Hq, Hkv, d, max_len, 0);
  void *ws = NULL;
  if (ws_bytes == 0 || cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 3;
  const int src = cdt >= PA_FP8_E4M3 ? qdt : cdt;

  /* set-up: the context; one step: copy-on-write, new tokens, decode */
  if (tc) CHECK(pa_reshape_and_cache(ck, cv, src, (const int64_t *)cs, tc, kc, vc, &desc, err, stream));
  if (npairs) CHECK(pa_copy_blocks(kc, vc, &desc, (const int64_t *)pairs, npairs, err, stream));
  CHECK(pa_reshape_and_cache(nk, nv, src, (const int64_t *)ns, tn, kc, vc, &desc, err, stream));
  CHECK(pa_decode(out, q, qdt, S, Hq, kc, vc, &desc, (const int32_t *)bt, maxb, (const int32_t *)sl,
                  max_len, scale, 0, ws, ws_bytes, err, stream));
  if (cudaStreamSynchronize(stream) != cudaSuccess) return 3;

  void *h = malloc(cache_bytes);
  int herr = -1;
  if (!h) return 2;
  cudaMemcpy(h, out, (size_t)S * Hq * d * 2, cudaMemcpyDeviceToHost);
  save("out.bin", h, (size_t)S * Hq * d * 2);
  cudaMemcpy(h, kc, cache_bytes, cudaMemcpyDeviceToHost);
  save("kc.bin", h, cache_bytes);
  cudaMemcpy(h, vc, cache_bytes, cudaMemcpyDeviceToHost);
  save("vc.bin", h, cache_bytes);
  cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost);
  printf("device_error %d\n", herr);
  return 0;
}
"""

CASES = {
    # beam forks with copy-on-write of the shared partial last blocks, fp16
    "beam-f16": ("opt13b-beam", dict(prompts=3, len_lo=40, len_hi=300)),
    # G = 8 over an e4m3 cache with bf16 queries
    "gqa-e4m3": ("gqa-fp8", dict(S=5, len_lo=20, len_hi=1500)),
}


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from paged_kv_cache_54_gb300 import build as B
    if not os.path.exists(B.LIB):
        B.build()
    d = tmp_path_factory.mktemp("cprog")
    (d / "prog.c").write_text(PROGRAM)
    exe = d / "prog"
    libdir = os.path.dirname(B.LIB)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), str(d / "prog.c"), "-o", str(exe),
                    "-L", libdir, "-l:" + os.path.basename(B.LIB), "-Wl,-rpath," + libdir,
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                   check=True)
    return exe


@pytest.mark.parametrize("case", sorted(CASES))
def test_c_program_drives_the_device_calls(program, case, tmp_path):
    name, ov = CASES[case]
    w = W.make_workload(name, 5, device="cpu", overrides=ov)
    codes = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3, "int8": 4}
    files = {"ctx_k.bin": G.bits(w.ctx_k), "ctx_v.bin": G.bits(w.ctx_v),
             "ctx_slots.bin": np.asarray(w.ctx_slots, np.int64),
             "new_k.bin": G.bits(w.new_k), "new_v.bin": G.bits(w.new_v),
             "new_slots.bin": np.asarray(w.new_slots, np.int64),
             "pairs.bin": np.asarray(w.cow_pairs, np.int64).reshape(-1, 2),
             "q.bin": G.bits(w.q), "bt.bin": np.asarray(w.block_tables, np.int32),
             "sl.bin": np.asarray(w.seq_lens, np.int32)}
    for f, a in files.items():
        np.ascontiguousarray(a).tofile(tmp_path / f)
    meta = [w.S, w.Hq, w.Hkv, w.d, w.bs, w.num_blocks, codes[w.cache_dtype], codes[w.q_dtype],
            len(w.ctx_slots), len(w.new_slots), len(w.cow_pairs), w.block_tables.shape[1],
            w.max_seq_len, repr(float(w.scale)), repr(float(w.k_scale)), repr(float(w.v_scale))]
    (tmp_path / "meta.txt").write_text(" ".join(str(x) for x in meta))
    r = subprocess.run([str(program), str(tmp_path)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "device_error 0", r.stdout

    # the oracle's cache after the same calls, from the same 0xFF fill
    c = PagedKVCache(w.num_blocks, w.Hkv, w.bs, w.d, w.cache_dtype, w.k_scale, w.v_scale, fill_nan=False)
    c.k[:] = np.iinfo(c.k.dtype).max
    c.v[:] = np.iinfo(c.v.dtype).max
    c.reshape_and_cache(G.bits(w.ctx_k), G.bits(w.ctx_v), w.src_dtype, w.ctx_slots)
    c.copy_blocks(w.cow_pairs)
    c.reshape_and_cache(G.bits(w.new_k), G.bits(w.new_v), w.src_dtype, w.new_slots)
    kc = np.fromfile(tmp_path / "kc.bin", dtype=c.k.dtype).reshape(c.k.shape)
    vc = np.fromfile(tmp_path / "vc.bin", dtype=c.v.dtype).reshape(c.v.shape)
    np.testing.assert_array_equal(kc, c.k)
    np.testing.assert_array_equal(vc, c.v)

    got = bits_to_f64(np.fromfile(tmp_path / "out.bin", dtype=np.uint16), w.q_dtype).reshape(w.S, w.Hq, w.d)
    ref = A.paged_decode(bits_to_f64(G.bits(w.q), w.q_dtype), c.k, c.v, w.cache_dtype, w.block_tables,
                         w.seq_lens, w.scale, w.k_scale, w.v_scale)
    err = np.abs(got - ref)
    bound = np.maximum(G.tolerance(w), G.ulp(ref, w.q_dtype))
    assert not (err > bound).any(), err.max()
    print(f"{case}: {len(w.cow_pairs)} copy-on-write pairs, max |err| {err.max():.2e}")
