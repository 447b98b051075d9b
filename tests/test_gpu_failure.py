"""The failure path of the kernels' bounded waits, on the GPU without a
fault: a wait that nothing completes gives up after its limit, the kernel
reports device error 4 and returns, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def test_wait_timeout_reports_and_the_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    t0 = time.perf_counter()
    pa.pa_selftest_wait_timeout(err)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == 4
    assert 1.5 < elapsed < 30.0
    # the same process goes on to decode correctly
    w = W.random_case(2, 3, 4, 2, 64, 16, "f16", "f16", [5, 70, 200], device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    ref = G.oracle_decode(w, G.oracle_cache(w))
    got = run.out.float().cpu().numpy()
    assert np.abs(got - ref).max() <= max(G.TOL["f16"], float(G.ulp(ref, "f16").max()))
