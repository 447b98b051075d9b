"""pa_decode_static_scratch: decode for callers that cannot allocate.

Some users of this library run the decode step where they may not allocate
device memory: inside a host framework that owns all GPU memory through its
own pool, or in a serving loop that forbids allocation after start-up
(cudaMalloc can synchronise the device).  pa_decode_static_scratch serves
them with the library's fixed 16 MiB device scratch instead of a workspace.

This file is collected last so that a stop-at-first-failure run has already
run every other test; it passes on its own in a fresh process too.  It calls
the entry point through the C ABI twice in a row (two different problems,
so the second call reuses scratch the first one left behind) and checks
each output against pa_decode with a caller-owned workspace.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def _static_call(lib, run, out):
    w = run.w
    desc = pa.cache_desc(run.kc, w.cache_dtype, w.k_scale, w.v_scale)
    qcode = pa.DTYPE_CODES[w.q_dtype]
    return lib.pa_decode_static_scratch(
        out.data_ptr(), w.q.data_ptr(), qcode, w.S, w.Hq, run.kc.data_ptr(), run.vc.data_ptr(),
        ctypes.byref(desc), run.bt.data_ptr(), run.bt.shape[1], run.sl.data_ptr(),
        w.max_seq_len, w.scale, run.P, run.err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _case(seed, cache_dtype, q_dtype, group):
    lens = [1, 300, 700, 1500, 2100, 64]
    w = W.random_case(seed, len(lens), 2 * group, 2, 128, 16, cache_dtype, q_dtype, lens,
                      device=G.DEV)
    run = G.GpuRun(w, partition_size=256).setup()
    run.step()                                  # reference: pa_decode with a workspace
    return run


def test_static_scratch_matches_workspace_decode_twice():
    lib = pa.load_library()
    runs = [_case(21, "bf16", "bf16", 2), _case(22, "e4m3", "bf16", 8)]
    torch.cuda.synchronize()
    refs = [r.out.clone() for r in runs]
    for run, ref in zip(runs, refs):            # two calls in a row, different problems
        out = torch.full_like(ref, float("nan"))
        assert _static_call(lib, run, out) == 0
        torch.cuda.synchronize()
        assert int(run.err.item()) == 0
        diff = float((out.float() - ref.float()).abs().max())
        assert diff <= G.tolerance(run.w), diff
    # the same problem again right after: the scratch left by the last call is reused
    out = torch.full_like(refs[0], float("nan"))
    assert _static_call(lib, runs[0], out) == 0
    torch.cuda.synchronize()
    assert float((out.float() - refs[0].float()).abs().max()) <= G.tolerance(runs[0].w)


def test_static_scratch_rejects_sizes_beyond_its_limit():
    lib = pa.load_library()
    run = _case(23, "f16", "f16", 1)
    w = run.w
    need = pa.pa_decode_workspace_size(4096, w.Hq, w.Hkv, w.d, 32768, 64)
    assert need > pa.STATIC_SCRATCH_BYTES
    desc = pa.cache_desc(run.kc, w.cache_dtype)
    st = lib.pa_decode_static_scratch(
        run.out.data_ptr(), w.q.data_ptr(), pa.PA_F16, 4096, w.Hq, run.kc.data_ptr(),
        run.vc.data_ptr(), ctypes.byref(desc), run.bt.data_ptr(), run.bt.shape[1],
        run.sl.data_ptr(), 32768, w.scale, 64, None, torch.cuda.current_stream().cuda_stream)
    assert st == 2                               # PA_ERR_UNSUPPORTED, nothing launched
    with pytest.raises(pa.PaError):
        pa.pa_decode_static_scratch(run.out, w.q, run.kc, run.vc, run.bt, run.sl, 32768 * 64,
                                    w.scale, partition_size=64)
    assert np.isfinite(run.out.float().cpu().numpy()).all()
