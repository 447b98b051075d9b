"""The named workloads at full size, in the launch configuration the
benchmark times: sampled outputs against the oracle (computed one by one
from the logical sequences), sampled cache slots bit-exact, invariants on
every output."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def _sample_rows(w, n, seed):
    rng = np.random.default_rng(seed)
    rows = {(int(rng.integers(w.S)), int(rng.integers(w.Hq))) for _ in range(n)}
    order = np.argsort(w.seq_lens)
    for s in (int(order[0]), int(order[-1])):        # shortest and longest sequence
        rows.add((s, 0))
        rows.add((s, w.Hq - 1))
    return sorted(rows)


@pytest.mark.parametrize("name", W.ALL_CONFIGS)
def test_named_config(name):
    w = W.make_workload(name, W.config_seed(name), device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    torch.cuda.synchronize()
    assert int(run.err.item()) == 0
    out = run.out.float()
    assert torch.isfinite(out).all()
    tol = G.tolerance(w)
    if name == "tiny":
        ref = G.oracle_decode(w, G.oracle_cache(w))
        err = np.abs(out.cpu().numpy() - ref).max()
        assert err <= tol, err
        return
    rows = _sample_rows(w, 40, 7)
    ref = G.oracle_rows(w, rows)
    got = out.cpu().numpy()
    worst = 0.0
    for (s, hq), r in ref.items():
        e = float(np.abs(got[s, hq] - r).max())
        worst = max(worst, e)
        assert e <= tol, (s, hq, e)
    # sampled cache slots: the written codes equal the oracle's encoding
    rng = np.random.default_rng(3)
    t_idx = np.unique(rng.integers(0, len(w.ctx_slots), 256))
    kc, vc = G.bits(run.kc), G.bits(run.vc)
    new_set = set(w.new_slots.tolist())
    for src, slots, idx in (("ctx", w.ctx_slots, t_idx), ("new", w.new_slots, np.arange(w.S))):
        ksrc = w.ctx_k if src == "ctx" else w.new_k
        vsrc = w.ctx_v if src == "ctx" else w.new_v
        sel = torch.from_numpy(idx).to(G.DEV)
        kb = G.encode_rows(w, G.bits(ksrc[sel]), "k")
        vb = G.encode_rows(w, G.bits(vsrc[sel]), "v")
        for j, t in enumerate(idx):
            slot = int(slots[t])
            blk, off = divmod(slot, w.bs)
            if src == "ctx" and slot in new_set:
                continue
            np.testing.assert_array_equal(kc[blk, :, off, :], kb[j])
            np.testing.assert_array_equal(vc[blk, :, off, :], vb[j])
    # copy-on-write: every copied block equals its source outside the written slot
    for src_b, dst_b in w.cow_pairs.tolist():
        written = {int(x) % w.bs for x in w.new_slots if int(x) // w.bs == dst_b}
        keep = [o for o in range(w.bs) if o not in written]
        np.testing.assert_array_equal(kc[dst_b][:, keep], kc[src_b][:, keep])
        np.testing.assert_array_equal(vc[dst_b][:, keep], vc[src_b][:, keep])
    print(f"{name}: {len(rows)} sampled rows, max |err| {worst:.2e}")
