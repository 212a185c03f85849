"""GPU parity for beam search: repeated fork / copy-on-write chains over many
steps.  At every step both sides apply the same block-manager ops, copy the
shared partly filled blocks, write each live beam's new token and decode all
live beams; outputs and caches are compared step by step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("small,gen_device", [(True, "cpu"), (False, "cuda")])
def test_beam_search_steps_match_oracle(small, gen_device):
    wl = inputs.beam(small)
    vals = inputs.make_values(wl, gen_device)
    dev = {k: v.cuda() for k, v in vals.items()}
    host = {k: inputs.to_numpy_elems(v).copy() for k, v in vals.items()}
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    row = qrow = copies = 0
    for st in wl.steps:
        r = oracle.run_script(0, wl.block_size, None, st["ops"], manager=m)
        slots, pairs = bm.apply_script(st["ops"])
        np.testing.assert_array_equal(slots, r["slots"])
        np.testing.assert_array_equal(pairs, r["pairs"])
        T = len(slots)
        copies += len(pairs)
        oracle.copy_blocks(host["k_cache"], host["v_cache"], r["pairs"])
        oracle.reshape_and_cache(host["k"][row:row + T], host["v"][row:row + T], r["slots"], host["k_cache"],
                                 host["v_cache"])
        pa.pa_copy_blocks(dev["k_cache"], dev["v_cache"], torch.from_numpy(pairs).cuda())
        pa.pa_reshape_and_cache(dev["k"][row:row + T], dev["v"][row:row + T], torch.from_numpy(slots).cuda(),
                                dev["k_cache"], dev["v_cache"])
        seqs = st["decode"]
        mb = max(len(m.tables[s]) for s in seqs)
        tables, lens = bm.export(seqs, mb)
        q = dev["q"][qrow:qrow + len(seqs)]
        out = pa.pa_decode(q, dev["k_cache"], dev["v_cache"], torch.from_numpy(tables).cuda(),
                           torch.from_numpy(lens).cuda(), wl.scale)
        ref = oracle.decode(host["q"][qrow:qrow + len(seqs)], host["k_cache"], host["v_cache"],
                            oracle.pad_tables([m.tables[s] for s in seqs], mb), [m.lens[s] for s in seqs],
                            wl.scale, num_threads=oracle.available_threads())
        assert np.abs(out.double().cpu().numpy() - ref).max() <= TOL["bf16"]
        oracle.run_script(0, wl.block_size, None, st["select"], manager=m)
        bm.apply_script(st["select"])
        row += T
        qrow += len(seqs)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert copies > 0
    assert np.array_equal(inputs.to_numpy_elems(dev["k_cache"]), host["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(dev["v_cache"]), host["v_cache"])
