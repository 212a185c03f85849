"""The N > 1 path on CPU with gloo, world size 2: sequences shard across ranks
with no data-path collective, every sequence lands on exactly one rank, the
per-rank results reassemble into the single-process result, and the timing
reduction takes the max over ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
from paged_kv_cache_150_gb300 import inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _reference(wl):
    vals = inputs.make_values(wl, "cpu")
    host = {k: inputs.to_numpy_elems(v).copy() for k, v in vals.items()}
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    oracle.copy_blocks(host["k_cache"], host["v_cache"], r["pairs"])
    oracle.reshape_and_cache(host["k"], host["v"], r["slots"], host["k_cache"], host["v_cache"])
    tables = oracle.pad_tables(r["tables"], wl.max_blocks_per_seq)
    return host, tables, r["lens"]


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = inputs.workload("cfg2", small=True)
        host, tables, lens = _reference(wl)
        per_seq = lens.astype(np.int64) * wl.num_kv_heads * wl.head_dim * 2 * wl.elem_bytes
        mine = inputs.shard_sequences(per_seq, world)[rank]
        pairs = [(int(s), h) for s in mine for h in range(wl.num_q_heads)]
        out = oracle.decode(host["q"], host["k_cache"], host["v_cache"], tables, lens, wl.scale, pairs=pairs)
        local = {int(s): out[s] for s in mine}
        gathered = [None] * world
        dist.all_gather_object(gathered, local)  # test-only gather of the results
        import bench

        t = bench.reduce_max(float(rank + 1) * 1.5, world)
        if rank == 0:
            out_q.put((gathered, t))
    finally:
        dist.destroy_process_group()


def test_shards_cover_every_sequence_once():
    rng = np.random.default_rng(0)
    for world in (1, 2, 3, 8):
        b = rng.integers(1, 10 ** 6, size=257)
        parts = inputs.shard_sequences(b, world)
        allidx = np.concatenate(parts)
        assert sorted(allidx.tolist()) == list(range(257))
        loads = [b[p].sum() for p in parts]
        assert max(loads) - min(loads) <= b.max()


def test_two_gloo_ranks_reassemble_the_single_process_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert tmax == 3.0
    wl = inputs.workload("cfg2", small=True)
    host, tables, lens = _reference(wl)
    full = oracle.decode(host["q"], host["k_cache"], host["v_cache"], tables, lens, wl.scale)
    seen = {}
    for part in gathered:
        for s, o in part.items():
            assert s not in seen
            seen[s] = o
    assert sorted(seen) == list(range(wl.num_seqs))
    for s, o in seen.items():
        np.testing.assert_array_equal(o, full[s])
