"""include/pa.h is a C header: a C99 program compiles against it with
warnings as errors, links against libpa.so and runs the host-side calls
(status strings, workspace sizing, the prefix cache) through the ABI
alone, with no Python in between (CPU only; no device call)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pa.h"

static int fail(const char *what) { fprintf(stderr, "FAIL %s\n", what); return 1; }

int main(void) {
  if (strcmp(pa_status_string(PA_OK), "ok") != 0) return fail("status string");
  if (pa_decode_workspace_size(64, 32, 32, 128, 4096, 0) == 0) return fail("workspace size");
  if (pa_decode_workspace_size(4, 4, 4, 64, 100, 100) != 0) return fail("bad partition accepted");

  /* two prompts sharing 32 tokens (two blocks of 16) */
  pa_prefix_cache *c = pa_prefix_cache_create(16, 16, NULL);
  if (!c) return fail("create");
  int32_t a[35], b[40], cached = -1;
  for (int i = 0; i < 35; ++i) a[i] = i < 32 ? 100 + i : 7;
  for (int i = 0; i < 40; ++i) b[i] = i < 32 ? 100 + i : 200 + i;
  if (pa_prefix_cache_add_sequence(c, 1, a, 35, &cached) != PA_OK || cached != 0) return fail("add a");
  if (pa_prefix_cache_add_sequence(c, 2, b, 40, &cached) != PA_OK || cached != 32) return fail("add b");
  int64_t ids[2] = {1, 2};
  int32_t tables[2 * 3], lens[2];
  if (pa_prefix_cache_block_tables(c, ids, 2, tables, 3, lens) != PA_OK) return fail("tables");
  if (lens[0] != 35 || lens[1] != 40) return fail("lengths");
  if (tables[0] != tables[3] || tables[1] != tables[4] || tables[2] == tables[5]) return fail("sharing");
  if (pa_prefix_cache_ref_count(c, tables[0]) != 2) return fail("ref count");
  int64_t slot = -1;
  if (pa_prefix_cache_append_token(c, 1, 9, &slot) != PA_OK || slot != (int64_t)tables[2] * 16 + 3)
    return fail("append slot");
  pa_prefix_cache_stats st;
  if (pa_prefix_cache_get_stats(c, &st) != PA_OK || st.hit_tokens != 32) return fail("stats");
  if (pa_prefix_cache_free_sequence(c, 2) != PA_OK || pa_prefix_cache_ref_count(c, tables[0]) != 1)
    return fail("free");
  if (pa_prefix_cache_add_sequence(c, 1, a, 35, &cached) == PA_OK) return fail("duplicate id accepted");
  pa_prefix_cache_destroy(c);
  puts("c abi ok");
  return 0;
}
"""


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from paged_kv_cache_54_gb300 import build as B
    if not os.path.exists(B.LIB):
        B.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(B.LIB)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(B.LIB),
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "c abi ok"
