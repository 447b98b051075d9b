"""The named workloads at full size, in the launch configuration the
benchmark times: every output row against the oracle (computed from each
sequence's logical tokens, not through the block tables), every written
cache slot bit-exact, the copy-on-write blocks against the oracle's
``copy_blocks``, and the decode unchanged under seeded permutations of the
physical blocks (block tables map logical blocks to scattered physical ones,
so where the blocks sit must not matter)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from oracle.cache import PagedKVCache
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=W.ALL_CONFIGS)
def ran(request):
    """A named workload after set-up and one step, with a snapshot of the
    copy-on-write blocks taken between the two."""
    name = request.param
    w = W.make_workload(name, W.config_seed(name), device=G.DEV)
    run = G.GpuRun(w).setup()
    torch.cuda.synchronize()
    involved = sorted({int(b) for pair in w.cow_pairs.tolist() for b in pair})
    snap = None
    if involved:
        idx = torch.tensor(involved, device=G.DEV)
        snap = (involved, G.bits(run.kc[idx]), G.bits(run.vc[idx]))
    run.step()
    torch.cuda.synchronize()
    yield name, w, run, snap
    del run


def test_every_row_matches_oracle(ran):
    name, w, run, _ = ran
    assert int(run.err.item()) == 0
    got = run.out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    ref = G.oracle_all_rows(w)
    err = np.abs(got - ref)
    tol = G.tolerance(w)
    assert err.max() <= tol, (f"{name}: max |err| {err.max():.3e} at "
                              f"{np.argwhere(err > tol)[:5].tolist()}")
    print(f"{name}: all {w.S * w.Hq} rows, max |err| {err.max():.2e}")


def test_every_written_slot_is_bit_exact(ran):
    name, w, run, _ = ran
    n = G.check_written_slots(w, run.kc, run.vc)
    assert n >= w.S
    print(f"{name}: {n} slots bit-exact")


def test_copy_on_write_blocks_match_oracle(ran):
    """The blocks the step's copy-on-write pairs touch, after the step, equal
    the oracle's: its copy_blocks applied to their state before the step,
    then the step's new tokens written into them."""
    name, w, run, snap = ran
    if snap is None:
        pytest.skip(f"{name} has no copy-on-write pairs")
    involved, k0, v0 = snap
    remap = {b: i for i, b in enumerate(involved)}
    c = PagedKVCache(len(involved), w.Hkv, w.bs, w.d, w.cache_dtype, w.k_scale, w.v_scale,
                     fill_nan=False)
    c.k[:], c.v[:] = k0, v0
    c.copy_blocks([(remap[int(a)], remap[int(b)]) for a, b in w.cow_pairs.tolist()])
    slots = np.array([remap[int(x) // w.bs] * w.bs + int(x) % w.bs if int(x) // w.bs in remap else -1
                      for x in w.new_slots], dtype=np.int64)
    c.reshape_and_cache(G.bits(w.new_k), G.bits(w.new_v), w.src_dtype, slots)
    idx = torch.tensor(involved, device=G.DEV)
    np.testing.assert_array_equal(G.bits(run.kc[idx]), c.k)
    np.testing.assert_array_equal(G.bits(run.vc[idx]), c.v)
    print(f"{name}: {len(w.cow_pairs)} copy-on-write pairs, {len(involved)} blocks bit-exact")


@pytest.mark.parametrize("perm_seed", [11, 12, 13])
def test_block_permutation_leaves_decode_unchanged(ran, perm_seed):
    name, w, run, _ = ran
    kc2, vc2, bt2 = G.permuted_caches(run.kc, run.vc, w.block_tables, perm_seed)
    out2 = torch.empty_like(run.out)
    err = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    pa.pa_decode(out2, w.q, kc2, vc2, torch.from_numpy(bt2).to(G.DEV), run.sl, w.max_seq_len,
                 w.scale, partition_size=run.P, workspace=run.ws, device_error=err, **run.kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    d = (out2.float() - run.out.float()).abs().max().item()
    assert d <= G.tolerance(w), d
    del kc2, vc2
    print(f"{name}: permutation {perm_seed}, max |diff| {d:.2e}")
