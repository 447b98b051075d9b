"""The device operations capture into a CUDA graph and replay correctly
(GPU): the host side of every call only encodes arguments and launches on
the caller's stream, with no synchronisation or allocation, so a serving
loop can replay a captured step.  New inputs are copied into the captured
buffers before each replay; the replay's output must equal an eager call's
on the same inputs, bit for bit (the kernels are deterministic)."""
import pytest
import torch

import paged_kv_cache_54_gb300 as pa
import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


def _replay_matches_eager(w, fn, outs, inputs):
    """fn() runs the step on the buffers; inputs are (buffer, [new values...])."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the side stream (first-call host set-up stays outside the capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    for k in range(len(inputs[0][1])):
        for buf, vals in inputs:
            buf.copy_(vals[k])
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outs]
        fn()  # eager on the same inputs
        torch.cuda.synchronize()
        for a, b in zip(got, outs):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("config", ["tiny", "gqa-fp8"])
def test_decode_step_replays(config):
    w = W.make_workload(config, W.config_seed(config), device=G.DEV,
                        overrides=None if config == "tiny" else dict(S=8))
    run = G.GpuRun(w).setup()
    gen = torch.Generator(device=G.DEV).manual_seed(3)
    qs = [torch.randn(w.q.shape, generator=gen, device=G.DEV).to(w.q.dtype) for _ in range(3)]
    q = w.q.clone()

    def step():
        pa.pa_reshape_and_cache(w.new_k, w.new_v, run.new_slots, run.kc, run.vc, device_error=run.err,
                                **run.kw)
        pa.pa_decode(run.out, q, run.kc, run.vc, run.bt, run.sl, w.max_seq_len, w.scale,
                     partition_size=run.P, workspace=run.ws, device_error=run.err, **run.kw)
    _replay_matches_eager(w, step, [run.out], [(q, qs)])
    assert int(run.err.item()) == 0


def test_prefill_and_copy_replay():
    lens, q_lens = [300, 129, 64], [200, 129, 1]
    w = W.random_case(31, 3, 4, 2, 128, 16, "bf16", "bf16", lens, device=G.DEV)
    run = G.GpuRun(w).setup()
    run.step()
    gen = torch.Generator(device=G.DEV).manual_seed(4)
    T = sum(q_lens)
    qs = [torch.randn((T, 4, 128), generator=gen, device=G.DEV).bfloat16() for _ in range(3)]
    q = qs[0].clone()
    out = torch.empty_like(q)
    cu = torch.tensor([0, 200, 329, 330], dtype=torch.int32, device=G.DEV)
    used = {int(b) for s in range(w.S) for b in w.block_tables[s, :-(-int(w.seq_lens[s]) // w.bs)]}
    free = [b for b in range(w.num_blocks) if b not in used][:2]
    pairs = torch.tensor([[int(w.block_tables[0, 0]), free[0]], [int(w.block_tables[1, 0]), free[1]]],
                         dtype=torch.int64, device=G.DEV)

    def step():
        pa.pa_copy_blocks(run.kc, run.vc, pairs, device_error=run.err)
        pa.pa_prefill(out, q, cu, run.kc, run.vc, run.bt, run.sl, 200, w.scale, device_error=run.err)
    _replay_matches_eager(w, step, [out, run.kc], [(q, qs)])
    assert int(run.err.item()) == 0
