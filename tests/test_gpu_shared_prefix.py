"""GPU parity of decode with a shared-prefix plan: blocks shared by several
sequences (parallel-sampling forks, prefix-cache hits, beams) are read once
for all sharers.  The output is the same attention, so it must match the fp64
oracle within the bf16 tolerance, for every head ratio, head size, block
size, layout and split count the tensor-core kernel covers; a plan that does
not match its call is reported and the affected sequences are computed
without sharing, still correctly."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step

pytestmark = pytest.mark.gpu

# (name, prompts, prompt_len, samples, max_append, H, Hk, D, B).  Rows per KV
# head = samples x query heads per KV head; the plan's rows per pass R is the
# smallest of 16, 32, 64 holding them (4, 2 or 1 KV heads per stage).  Passes
# of 64 rows in the row layout run on tcgen05 (accumulators in tensor
# memory), the others on mma.sync.
SAMPLING = [
    ("g4-s4", 6, 200, 4, 40, 32, 8, 128, 16),     # the parallel-sampling shape, reduced: 16 rows, R 16
    ("g8-s4", 4, 150, 4, 30, 64, 8, 128, 16),     # 8 query heads per KV head: 32 rows, R 32 (2 heads per stage)
    ("g1-s40", 2, 90, 40, 20, 32, 32, 128, 16),   # one query head per KV head, 40 sharers: R 64, one warp idle
    ("g2-b32", 3, 300, 5, 70, 16, 8, 128, 32),    # block size 32: 10 rows, R 16
    ("g4-d64", 3, 120, 6, 25, 32, 8, 64, 16),     # head_dim 64: 24 rows, R 32
    ("g4-s9-b32", 3, 64, 9, 10, 16, 4, 64, 32),   # 36 rows, R 64, head_dim 64, block 32
    ("g2-s4", 3, 80, 4, 12, 16, 8, 128, 16),      # 8 rows: R 16, the second MMA tile empty
    ("g8-s9", 2, 120, 9, 20, 64, 8, 128, 16),     # 72 rows: R 64, two passes, the second on one warp
    ("g4-s12-b32", 2, 200, 12, 30, 32, 8, 128, 32),  # 48 rows, R 64, block size 32: rounds of 2 blocks
    ("g2-s20-d64", 2, 150, 20, 20, 16, 8, 64, 16),  # 40 rows, R 64, head_dim 64
    ("g1-s64", 1, 700, 64, 9, 8, 8, 128, 16),     # 64 rows, R 64, 43 shared blocks: full rounds and a ragged one
]


def _sampling(name, prompts, prompt_len, samples, max_append, H, Hk, D, B, seed=4242):
    return inputs.sampling_workload(name, prompts, prompt_len, samples, max_append, H, Hk, D, B, "bf16", seed)


@pytest.mark.parametrize("spec", SAMPLING, ids=[s[0] for s in SAMPLING])
def test_shared_prefix_decode_matches_oracle(spec):
    wl = _sampling(*spec)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, shared=True)
    assert g["plan_info"]["num_groups"] == spec[1]  # every prompt's samples share its blocks
    assert max_abs_err(g["out"], ref) <= TOL["bf16"]
    plain = gpu_step(wl, {k: v.clone() for k, v in dev.items()})
    assert (g["out"].float() - plain["out"].float()).abs().max().item() <= TOL["bf16"]


@pytest.mark.parametrize("idx", [0, 10], ids=["R16", "R64"])
@pytest.mark.parametrize("splits", [2, 3, 7, 64, 0])
def test_shared_prefix_any_split_count(splits, idx):
    """Any split count: with 64-row passes (tcgen05 halves) odd counts leave
    a CTA whose halves are of different kinds, or a half with nothing to do."""
    wl = _sampling(*SAMPLING[idx])
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, dev, shared=True, num_splits=splits)
    assert max_abs_err(g["out"], ref) <= TOL["bf16"]


@pytest.mark.parametrize("idx", [0, 2], ids=["R16", "R64"])
def test_shared_prefix_split_layout(idx):
    wl = _sampling(*SAMPLING[idx])
    dev, host = host_values(wl, "cpu", layout="split")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, shared=True)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


def _growing_scores(wl, step):
    """Values whose cached keys grow with their position in the sequence
    (factor 1 + position / step), so that the scores of later shared blocks
    pass the running maximum of earlier ones many times over: the online
    softmax must rescale its accumulators in the middle of a prefix."""
    vals = inputs.make_values(wl, device="cpu")
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    kc = vals["k_cache"].float()
    seen = set()
    for table in r["tables"]:
        for b, blk in enumerate(table):
            if blk not in seen:
                seen.add(blk)
                f = 1.0 + (b * wl.block_size + torch.arange(wl.block_size, dtype=torch.float32)) / step
                kc[blk] *= f[:, None, None]
    vals["k_cache"] = kc.to(vals["k_cache"].dtype)
    dev = {n: v.to("cuda") for n, v in vals.items()}
    host = {n: inputs.to_numpy_elems(v).copy() for n, v in vals.items()}
    return dev, host


@pytest.mark.parametrize("idx", [0, 2, 10], ids=["R16", "R64", "R64-43-blocks"])
def test_shared_prefix_scores_growing_along_the_prefix(idx):
    spec = SAMPLING[idx]
    wl = _sampling(*spec)
    dev, host = _growing_scores(wl, 24.0)
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, shared=True)
    assert max_abs_err(g["out"], ref) <= TOL["bf16"]
    plain = gpu_step(wl, dev)
    assert max_abs_err(plain["out"], ref) <= TOL["bf16"]


@pytest.mark.parametrize("cfg,kw", [("cfg3", {"small": True}), ("cfg3", {"small": True, "prompt_len": 200}),
                                    ("prefix", {"small": True})])
def test_shared_prefix_small_workloads(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, shared=True)
    assert g["plan_info"]["num_groups"] > 0
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


@pytest.mark.parametrize("cfg,kw", [("cfg3", {"prompt_len": 2008}), ("cfg3", {}), ("prefix", {})])
def test_shared_prefix_full_size_every_output(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, shared=True)
    assert g["plan_info"]["num_groups"] in (64, 8)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]
    # every output against the decode without a plan
    plain = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale)
    assert (g["out"].float() - plain.float()).abs().max().item() <= TOL["bf16"]


def test_shared_prefix_beam_search_steps():
    wl = inputs.beam(False)
    vals = inputs.make_values(wl, "cuda")
    dev = {k: v.cuda() for k, v in vals.items()}
    host = {k: inputs.to_numpy_elems(v).copy() for k, v in vals.items()}
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    row = qrow = grouped = 0
    for st in wl.steps:
        r = oracle.run_script(0, wl.block_size, None, st["ops"], manager=m)
        slots, pairs = bm.apply_script(st["ops"])
        T = len(slots)
        oracle.copy_blocks(host["k_cache"], host["v_cache"], r["pairs"])
        oracle.reshape_and_cache(host["k"][row:row + T], host["v"][row:row + T], r["slots"], host["k_cache"],
                                 host["v_cache"])
        pa.pa_copy_blocks(dev["k_cache"], dev["v_cache"], torch.from_numpy(pairs).cuda())
        pa.pa_reshape_and_cache(dev["k"][row:row + T], dev["v"][row:row + T], torch.from_numpy(slots).cuda(),
                                dev["k_cache"], dev["v_cache"])
        seqs = st["decode"]
        mb = max(len(m.tables[s]) for s in seqs)
        tables, lens = bm.export(seqs, mb)
        plan, info = pa.shared_prefix_plan(tables, lens, wl.block_size, wl.num_q_heads, wl.num_kv_heads)
        grouped += info["num_groups"]
        q = dev["q"][qrow:qrow + len(seqs)]
        out = pa.pa_decode(q, dev["k_cache"], dev["v_cache"], torch.from_numpy(tables).cuda(),
                           torch.from_numpy(lens).cuda(), wl.scale, shared_plan=plan.cuda())
        ref = oracle.decode(host["q"][qrow:qrow + len(seqs)], host["k_cache"], host["v_cache"],
                            oracle.pad_tables([m.tables[s] for s in seqs], mb), [m.lens[s] for s in seqs],
                            wl.scale, num_threads=oracle.available_threads())
        assert np.abs(out.double().cpu().numpy() - ref).max() <= TOL["bf16"]
        oracle.run_script(0, wl.block_size, None, st["select"], manager=m)
        bm.apply_script(st["select"])
        row += T
        qrow += len(seqs)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert grouped > 0


def _plan_case():
    wl = _sampling("mismatch", 3, 100, 4, 20, 32, 8, 128, 16, seed=77)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, decode=False)
    tables, lens = g["host_tables"], r["lens"].astype(np.int32)
    plan, info = pa.shared_prefix_plan(tables, lens, wl.block_size, wl.num_q_heads, wl.num_kv_heads)
    assert info["num_groups"] == 3
    return wl, host, r, g, plan, lens


def test_member_without_own_positions_is_computed_without_sharing():
    wl, host, r, g, plan, lens = _plan_case()
    P = 100 // 16  # 6 shared blocks
    short = lens.copy()
    short[5] = P * wl.block_size  # on the device this member now ends with the shared prefix
    out = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], torch.from_numpy(short).cuda(), wl.scale,
                       shared_plan=plan.cuda())
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_PLAN
    ref = oracle.decode(host["q"], r["k_cache"], r["v_cache"], r["tables_padded"], short, wl.scale,
                        num_threads=oracle.available_threads())
    assert max_abs_err(out, ref) <= TOL["bf16"]


@pytest.mark.parametrize("corrupt", ["magic", "num_seqs", "member", "prefix", "back_pointer", "pass_count",
                                     "rows_per_pass"])
def test_plan_that_does_not_match_is_reported_and_ignored(corrupt):
    wl, host, r, g, plan, lens = _plan_case()
    w = plan.clone()
    N, ng, M = int(w[1]), int(w[4]), int(w[5])
    o_prefix = 8 + 2 * N
    o_vbase = o_prefix + ng
    o_members = o_vbase + 2 * (ng + 1)
    if corrupt == "magic":
        w[0] = 0
    elif corrupt == "num_seqs":
        w[1] = N + 1
    elif corrupt == "member":
        w[o_members + 1] = N + 5
    elif corrupt == "prefix":
        w[o_prefix] = 10 ** 6
    elif corrupt == "back_pointer":
        w[8 + N + 0] = 3  # seq_member of sequence 0
    elif corrupt == "pass_count":
        w[o_vbase + 1] += 1
    elif corrupt == "rows_per_pass":
        w[7] = 24
    out = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale,
                       shared_plan=w.cuda())
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_PLAN
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_back_to_back_calls_on_one_workspace_with_a_rejected_plan():
    """Calls queued on one stream and one workspace with no synchronisation
    between them, alternating a rejected plan (its merge grid has nothing to
    merge, and the call's attention launch takes every sequence) and a good
    one.  Each call's plan kernel re-zeroes the arrival counters the previous
    call's attention launch counts on, so every output matching the oracle
    shows that no call's work overlapped the one before it."""
    wl, host, r, g, plan, lens = _plan_case()
    bad = plan.clone()
    bad[0] = 0  # not a plan: rejected on the device
    plans = [bad.cuda(), plan.cuda()]
    ref = oracle_decode(wl, host, r)
    ws = torch.empty(pa.pa_decode_workspace_bytes(g["k_cache"], wl.num_seqs, wl.num_q_heads, shared=True),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    outs = [pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, workspace=ws,
                         shared_plan=plans[i % 2]) for i in range(12)]
    torch.cuda.synchronize()
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_PLAN
    for out in outs:
        assert max_abs_err(out, ref) <= TOL["bf16"]


def test_plan_with_one_cta_is_ignored_quietly():
    wl, host, r, g, plan, lens = _plan_case()
    out = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, num_splits=1,
                       shared_plan=plan.cuda())
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_plan_with_q_not_16_byte_aligned_is_ignored_quietly():
    wl, host, r, g, plan, lens = _plan_case()
    buf = torch.empty(g["q"].numel() + 8, dtype=g["q"].dtype, device="cuda")
    q = buf[2:2 + g["q"].numel()].view(g["q"].shape)  # 4-byte aligned, not 16
    q.copy_(g["q"])
    out = pa.pa_decode(q, g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, shared_plan=plan.cuda())
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_shared_prefix_plan_too_large_for_shared_memory():
    """4000 sequences in 1000 groups: the plan's words (about 112 KB) are read
    from global memory by the plan kernel instead of a shared-memory copy."""
    wl = _sampling("many-groups", 1000, 40, 4, 20, 32, 8, 128, 16, seed=91)
    assert 4 * (7 * wl.num_seqs + 16) > 96 * 1024
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, shared=True)
    assert g["plan_info"]["num_groups"] == 1000
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


@pytest.mark.parametrize("idx,layout", [(2, "row"), (8, "row"), (9, "row"), (2, "split")],
                         ids=["d128-b16", "d128-b32", "d64-b16", "split"])
def test_64_row_passes_choose_tcgen05_in_the_row_layout(idx, layout):
    """The host chooses the tcgen05 shared-prefix CTAs for plans of 64 rows
    per pass in the row layout (their tensor memory fits an SM), and the
    mma.sync ones in the split layout; both give the oracle's attention."""
    wl = _sampling(*SAMPLING[idx])
    dev, host = host_values(wl, "cpu", layout=layout)
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, decode=False)
    lens = g["lens"].cpu().numpy()
    plan, info = pa.shared_prefix_plan(g["host_tables"], lens, wl.block_size, wl.num_q_heads, wl.num_kv_heads)
    assert int(plan[7]) == 64
    plan_d = plan.cuda()
    assert pa.pa_decode_shared_tc(g["k_cache"], wl.num_seqs, wl.num_q_heads, plan_d) == (layout == "row")
    out = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, shared_plan=plan_d)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]
