"""One step of the hot path on both sides, from the same seeded inputs.

oracle side: the oracle's block-manager model -> block copy -> cache write ->
fp64 decode (all pairs, or a sample of (seq, head) pairs).
CUDA side:   the C++ block manager -> pa_copy_blocks -> pa_reshape_and_cache
-> pa_decode, through the C ABI.
"""
import numpy as np
import torch

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}


def host_values(wl, device, layout="row"):
    """Seeded values generated on ``device`` (caches in the row or the split
    layout); returns (device tensors, host numpy)."""
    vals = inputs.make_values(wl, device=device)
    if layout == "split":
        vals["k_cache"], vals["v_cache"] = inputs.to_split_layout(vals["k_cache"], vals["v_cache"])
    dev = {k: v.to("cuda") for k, v in vals.items()}
    host = {k: inputs.to_numpy_elems(v).copy() for k, v in vals.items()}
    return dev, host


def oracle_step(wl, host):
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    kc, vc = host["k_cache"].copy(), host["v_cache"].copy()
    oracle.copy_blocks(kc, vc, r["pairs"])
    bad = oracle.reshape_and_cache(host["k"], host["v"], r["slots"], kc, vc)
    assert bad == 0
    r["tables_padded"] = oracle.pad_tables(r["tables"], wl.max_blocks_per_seq)
    r["k_cache"], r["v_cache"] = kc, vc
    return r


def oracle_decode(wl, host, r, pairs=None):
    return oracle.decode(host["q"], r["k_cache"], r["v_cache"], r["tables_padded"], r["lens"], wl.scale,
                         pairs=pairs, num_threads=oracle.available_threads())


def gpu_step(wl, dev, kernel="auto", num_splits=0, decode=True, shared=False, host_lens=None):
    """``shared``: decode with a shared-prefix plan built from the host tables.
    ``host_lens``: the host-lengths hint of pa_decode, "exact" for the true
    lengths or any int32 array of num_seqs entries."""
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    slots, pairs = bm.apply_script(wl.script)
    tables, lens = bm.export(list(range(wl.num_seqs)), wl.max_blocks_per_seq)
    g = dict(dev)
    g["tables"] = torch.from_numpy(tables).cuda()
    g["lens"] = torch.from_numpy(lens).cuda()
    g["slots"] = torch.from_numpy(slots).cuda()
    g["pairs"] = torch.from_numpy(pairs).cuda()
    pa.pa_copy_blocks(g["k_cache"], g["v_cache"], g["pairs"])
    pa.pa_reshape_and_cache(g["k"], g["v"], g["slots"], g["k_cache"], g["v_cache"])
    plan = None
    if shared:
        plan, g["plan_info"] = pa.shared_prefix_plan(tables, lens, wl.block_size, wl.num_q_heads, wl.num_kv_heads)
        plan = plan.cuda()
    if decode:
        hint = lens if isinstance(host_lens, str) and host_lens == "exact" else host_lens
        g["out"] = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale,
                                kernel=kernel, num_splits=num_splits, shared_plan=plan, host_seq_lens=hint)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    g["host_tables"], g["host_slots"], g["host_pairs"] = tables, slots, pairs
    return g


def max_abs_err(out_dev, ref, pairs=None):
    out = out_dev.double().cpu().numpy()
    if pairs is None:
        return float(np.abs(out - ref).max())
    idx = np.asarray(pairs)
    return float(np.abs(out[idx[:, 0], idx[:, 1]] - ref[idx[:, 0], idx[:, 1]]).max())
