"""The library's calls recorded in a CUDA graph (with their programmatic
dependent launches) and replayed: the replay must match the same calls
issued one by one, and the oracle, also after the inputs change in place
between replays."""
import numpy as np
import pytest
import torch

import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg,kw,shared", [("cfg2", {"small": True}, False), ("cfg4", {"small": True}, False),
                                           ("cfg3", {"small": True, "prompt_len": 200}, True)])
def test_step_replayed_from_a_cuda_graph(cfg, kw, shared):
    wl = inputs.workload(cfg, **kw)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, decode=False)  # copies and the cache write done once, eagerly
    plan = None
    if shared:
        plan, info = pa.shared_prefix_plan(g["host_tables"], r["lens"], wl.block_size, wl.num_q_heads,
                                           wl.num_kv_heads)
        assert info["num_groups"] > 0
        plan = plan.cuda()
    ws = torch.empty(pa.pa_decode_workspace_bytes(g["k_cache"], wl.num_seqs, wl.num_q_heads, shared=shared),
                     dtype=torch.uint8, device="cuda")
    q = g["q"].clone()
    out = torch.empty_like(q)

    def decode():
        pa.pa_decode(q, g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out=out, workspace=ws,
                     shared_plan=plan)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        decode()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(out, eager)
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]
    # new queries written in place: the replay reads them
    q.copy_(torch.flip(g["q"], dims=[0]))
    host2 = dict(host)
    host2["q"] = np.ascontiguousarray(host["q"][::-1])
    graph.replay()
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_decode(wl, host2, r)) <= TOL["bf16"]


def test_calls_take_torchs_current_stream():
    assert (pa._stream().value or 0) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert pa._stream().value == side.cuda_stream
    assert (pa._stream().value or 0) == torch.cuda.current_stream().cuda_stream


def test_concurrent_decodes_on_two_streams_match_sequential_ones():
    """Two batches decoded at the same time on two streams, each with its
    own workspace: the library keeps no other per-call state on the device,
    so the outputs equal those of the same calls made one after another."""
    wls = [inputs.workload("cfg2", small=True), inputs.workload("cfg4", small=True)]
    steps = []
    for wl in wls:
        dev, host = host_values(wl, "cpu")
        g = gpu_step(wl, dev, decode=False)
        ws = torch.empty(pa.pa_decode_workspace_bytes(g["k_cache"], wl.num_seqs, wl.num_q_heads),
                         dtype=torch.uint8, device="cuda")
        steps.append((wl, g, ws))

    def decode(wl, g, ws, out):
        pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out=out, workspace=ws)

    ref = []
    for wl, g, ws in steps:
        out = torch.empty_like(g["q"])
        decode(wl, g, ws, out)
        ref.append(out)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(g["q"]) for _, g, _ in steps]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(20):
        for (wl, g, ws), s, out in zip(steps, streams, outs):
            with torch.cuda.stream(s):
                decode(wl, g, ws, out)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    for out, r in zip(outs, ref):
        assert torch.equal(out, r)
