"""GPU parity for prefix caching: requests that share system prompts point at
the same physical blocks; only uncached positions are written (cached ones get
slot -1), and decode through the shared tables matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["row", "split"])
def test_prefix_cached_step_matches_oracle(layout):
    wl = inputs.workload("prefix", small=True)
    dev, host = host_values(wl, "cpu", layout=layout)
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    np.testing.assert_array_equal(g["host_slots"], r["slots"])
    assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"])
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_prefix_cached_full_size_every_output():
    wl = inputs.workload("prefix")
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    assert (g["host_slots"] == -1).sum() == 144000  # 9000 cached blocks of 16 positions
    np.testing.assert_array_equal(g["host_slots"], r["slots"])
    assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"])
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


@pytest.mark.parametrize("small", [True, False])
def test_retained_prompt_blocks_serve_a_later_wave(small):
    """With prefix retention on, a later wave decodes over system-prompt K/V
    that only the first wave wrote, while blocks evicted from under it are
    written again by their new owners.  Each phase's rows go through one
    cache write; caches are bit-exact and decode is within tolerance of the
    oracle replaying the same phases."""
    wl = inputs.retention(small)
    dev, host = host_values(wl, "cpu" if small else "cuda")
    kc, vc = host["k_cache"].copy(), host["v_cache"].copy()
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    op0 = row0 = 0
    for ops, rows in wl.extra["phases"]:
        script = wl.script[op0:op0 + ops]
        r = oracle.run_script(0, wl.block_size, None, script, manager=m)
        slots, pairs = bm.apply_script(script)
        np.testing.assert_array_equal(slots, r["slots"])
        assert len(slots) == rows and len(pairs) == 0
        rng = slice(row0, row0 + rows)
        assert oracle.reshape_and_cache(host["k"][rng], host["v"][rng], r["slots"], kc, vc) == 0
        pa.pa_reshape_and_cache(dev["k"][rng], dev["v"][rng], torch.from_numpy(slots).cuda(), dev["k_cache"],
                                dev["v_cache"])
        op0 += ops
        row0 += rows
    assert row0 == wl.num_new_tokens
    assert np.array_equal(inputs.to_numpy_elems(dev["k_cache"]), kc)
    assert np.array_equal(inputs.to_numpy_elems(dev["v_cache"]), vc)
    live = wl.extra["live"]
    tables, lens = bm.export(live, wl.max_blocks_per_seq)
    ref_tables = oracle.pad_tables([m.tables[s] for s in live], wl.max_blocks_per_seq)
    np.testing.assert_array_equal(tables, ref_tables)
    out = pa.pa_decode(dev["q"], dev["k_cache"], dev["v_cache"], torch.from_numpy(tables).cuda(),
                       torch.from_numpy(lens).cuda(), wl.scale)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    ref = oracle.decode(host["q"], kc, vc, ref_tables, lens, wl.scale, num_threads=oracle.available_threads())
    assert max_abs_err(out, ref) <= TOL["bf16"]
