"""The product's C++ block manager against the oracle's model of the pages'
manager: identical tables, slots and copy-on-write pairs on every workload,
the pages' worked example, and the failure semantics."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


WORKLOADS = [("cfg0", {}), ("cfg1", {}), ("cfg1", {"small": True}), ("cfg2", {}),
             ("cfg2", {"small": True}), ("cfg3", {}), ("cfg3", {"prompt_len": 2008}),
             ("cfg3", {"small": True}), ("cfg3", {"small": True, "prompt_len": 200}),
             ("cfg4", {}), ("cfg4", {"block_size": 32}), ("cfg4", {"small": True}),
             ("prefix", {}), ("prefix", {"small": True})]


@pytest.mark.parametrize("cfg,kw", WORKLOADS)
def test_manager_matches_oracle_model(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    slots, pairs = bm.apply_script(wl.script)
    np.testing.assert_array_equal(slots, r["slots"])
    np.testing.assert_array_equal(pairs, r["pairs"])
    # the step writes every row in one call and copies every pair in another:
    # distinct written slots, distinct copy destinations, no destination read
    written = slots[slots >= 0]
    assert len(np.unique(written)) == len(written)
    if len(pairs):
        assert len(np.unique(pairs[:, 1])) == len(pairs) and not set(pairs[:, 1]) & set(pairs[:, 0])
    tables, lens = bm.export(list(range(wl.num_seqs)), wl.max_blocks_per_seq)
    np.testing.assert_array_equal(tables, oracle.pad_tables(r["tables"], wl.max_blocks_per_seq))
    np.testing.assert_array_equal(lens, r["lens"])
    np.testing.assert_array_equal(lens, wl.seq_lens)
    assert bm.stats() == r["manager"].stats()
    m = r["manager"]
    assert bm.cache_stats() == (len(m.cached), m.hits, m.lookups)
    for b, ref in list(r["manager"].ref.items())[:200]:
        assert bm.refcount(b) == ref


def test_go_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "go_worked_example.json")))
    bm = pa.BlockManager(g["num_blocks"], g["block_size"])
    seqs = {}
    for st in g["steps"]:
        if st["op"] == "new":
            seqs[st["name"]] = bm.new_seq(st["tokens"])
        else:
            bm.free_seq(seqs[st["name"]])
        free, used, _ = bm.stats()
        if "expect_free" in st:
            assert free == st["expect_free"]
        if "expect_used" in st:
            assert used == st["expect_used"]
    assert bm.block_table(seqs["e"]) == g["derived"]["table_e"]
    assert bm.physical_index(seqs["e"], 40) == g["derived"]["physical_index_e_40"]


def test_sharing_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sharing_examples.json")))["parallel_sampling"]
    B = g["block_size"]
    bm = pa.BlockManager(len(g["free_order"]), B, g["free_order"])
    parent = bm.new_seq(3 * B)
    seqs = [parent] + [bm.fork(parent) for _ in range(3)]
    assert all(bm.refcount(b) == 4 for b in g["prompt_blocks"])
    for s in seqs:
        assert bm.append_token(s)[1] is None
    assert [bm.block_table(s)[-1] for s in seqs] == g["extra_blocks"]
    assert bm.stats()[1] == g["physical_blocks"]


def test_copy_on_write_pair_and_in_place_last_writer():
    bm = pa.BlockManager(8, 4)
    s = bm.new_seq(6)  # blocks [0, 1] (Go order: top two ids in stack order)
    kids = [bm.fork(s) for _ in range(2)]
    shared_last = bm.block_table(s)[1]
    got = [bm.append_token(x) for x in [s] + kids]
    assert got[0][1] is not None and got[1][1] is not None and got[2][1] is None
    assert got[0][1][0] == shared_last and got[1][1][0] == shared_last
    assert bm.block_table(kids[1])[1] == shared_last and bm.refcount(shared_last) == 1
    for x in [s] + kids:
        slot = bm.physical_index(x, 6)
        assert bm.refcount(slot // 4) == 1


def _snapshot(bm, seqs):
    return (bm.stats(), [bm.block_table(s) for s in seqs], [bm.seq_len(s) for s in seqs])


def test_failures_change_nothing():
    bm = pa.BlockManager(3, 4)
    a = bm.new_seq(8)
    snap = _snapshot(bm, [a])
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.new_seq(9)
    assert e.value.status == -4 and _snapshot(bm, [a]) == snap
    with pytest.raises(pa.PagedAttentionError):
        bm.append_tokens(a, 5)  # needs 2 new blocks, 1 free: all or nothing
    assert _snapshot(bm, [a]) == snap
    bm2 = pa.BlockManager(2, 4)
    s = bm2.new_seq(6)
    t = bm2.fork(s)
    snap2 = _snapshot(bm2, [s, t])
    with pytest.raises(pa.PagedAttentionError):
        bm2.append_token(s)  # copy needed, pool empty
    assert _snapshot(bm2, [s, t]) == snap2
    bm2.free_seq(t)
    with pytest.raises(pa.PagedAttentionError):
        bm2.free_seq(t)  # double free
    slot, pair = bm2.append_token(s)  # now unshared: written in place
    assert pair is None and slot == bm2.block_table(s)[1] * 4 + 2


def test_bad_free_order_is_rejected():
    with pytest.raises(ValueError):
        pa.BlockManager(4, 4, [0, 1, 1, 2])
    with pytest.raises(ValueError):
        pa.BlockManager(4, 4, [0, 1, 2, 4])


def test_append_tokens_matches_repeated_append_token():
    rng = np.random.default_rng(3)
    order = rng.permutation(64).astype(np.int32)
    a = pa.BlockManager(64, 8, order)
    b = pa.BlockManager(64, 8, order)
    for m in (a, b):
        p = m.new_seq(13)
        m.fork(p)
        m.fork(p)
    for seq, count in [(0, 5), (1, 17), (2, 1), (0, 9)]:
        slots_a, pair_a = a.append_tokens(seq, count)
        singles = [b.append_token(seq) for _ in range(count)]
        assert slots_a.tolist() == [x[0] for x in singles]
        pairs_b = [x[1] for x in singles if x[1] is not None]
        assert (pair_a is None and not pairs_b) or [pair_a] == pairs_b
    assert a.stats() == b.stats()


def test_prefix_cache_matches_oracle_through_frees_and_reuse():
    rng = np.random.default_rng(5)
    order = rng.permutation(256).astype(np.int32)
    bm = pa.BlockManager(256, 8, order)
    m = oracle.OracleBlockManager(256, 8, order)
    prompts = [rng.integers(0, 50, size=int(rng.integers(20, 90))).tolist() for _ in range(4)]
    live = []
    for step in range(40):
        p = prompts[int(rng.integers(0, 4))]
        toks = p[:int(rng.integers(len(p) // 2, len(p) + 1))] + rng.integers(0, 50, size=int(rng.integers(0, 9))).tolist()
        got = bm.new_seq_cached(toks)
        want = m.new_sequence_cached(toks)
        assert got == want
        live.append(got[0])
        assert bm.block_table(got[0]) == m.tables[want[0]]
        if len(live) > 6:
            victim = live.pop(int(rng.integers(0, len(live))))
            bm.free_seq(victim)
            m.free_seq(victim)
        assert bm.stats() == m.stats()
        assert bm.cache_stats() == (len(m.cached), m.hits, m.lookups)


@pytest.mark.parametrize("small", [True, False])
def test_beam_search_manager_matches_oracle(small):
    wl = inputs.beam(small)
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    for st in wl.steps:
        r = oracle.run_script(0, wl.block_size, None, st["ops"], manager=m)
        slots, pairs = bm.apply_script(st["ops"])
        np.testing.assert_array_equal(slots, r["slots"])
        np.testing.assert_array_equal(pairs, r["pairs"])
        mb = max(len(m.tables[s]) for s in st["decode"])
        tables, lens = bm.export(st["decode"], mb)
        np.testing.assert_array_equal(tables, oracle.pad_tables([m.tables[s] for s in st["decode"]], mb))
        oracle.run_script(0, wl.block_size, None, st["select"], manager=m)
        bm.apply_script(st["select"])
        assert bm.stats() == m.stats()


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
def test_prefix_retention_matches_oracle_under_pool_pressure(seed):
    """Retention on, a pool small enough that allocations evict: the C++
    manager and the oracle model agree on every hit, table, free count,
    cache counter and evictable count, through forks, appends with
    copy-on-write, frees, failed allocations (no state change) and switching
    retention off."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(16).astype(np.int32)
    bm = pa.BlockManager(16, 8, order)
    m = oracle.OracleBlockManager(16, 8, order)
    bm.set_prefix_retention(True)
    m.set_retention(True)
    prompts = [rng.integers(0, 30, size=int(rng.integers(16, 70))).tolist() for _ in range(5)]
    live = []
    failures = most_evictable = evicted = forks = copies = 0
    for step in range(150):
        if step == 120:  # retention off: evictable blocks become free, oldest first
            bm.set_prefix_retention(False)
            m.set_retention(False)
        p = prompts[int(rng.integers(0, len(prompts)))]
        toks = p[:int(rng.integers(len(p) // 2, len(p) + 1))] + rng.integers(0, 30, size=int(rng.integers(0, 6))).tolist()
        registered = len(m.cached)
        want = m.new_sequence_cached(toks)
        if want is None:
            failures += 1
            with pytest.raises(pa.PagedAttentionError):
                bm.new_seq_cached(toks)
        else:
            got = bm.new_seq_cached(toks)
            assert got == want
            live.append(got[0])
            assert bm.block_table(got[0]) == m.tables[want[0]]
            # registered blocks only go away by eviction while retention is on
            evicted += step < 120 and len(m.cached) < registered
        if live and rng.random() < 0.25:  # a fork shares every block, cached ones included
            parent = live[int(rng.integers(0, len(live)))]
            child = m.fork(parent)
            assert bm.fork(parent) == child
            live.append(child)
            forks += 1
        if live and rng.random() < 0.6:  # growth of a live sequence, copying a shared partial block
            s = live[int(rng.integers(0, len(live)))]
            want = m.append_token(s)
            if want is None:
                with pytest.raises(pa.PagedAttentionError):
                    bm.append_tokens(s, 1)
            else:
                slots, pair = bm.append_tokens(s, 1)
                assert (int(slots[0]), pair) == want
                copies += pair is not None
        while len(live) > 4 or (live and rng.random() < 0.3):
            victim = live.pop(int(rng.integers(0, len(live))))
            bm.free_seq(victim)
            m.free_seq(victim)
        assert bm.stats() == m.stats()
        assert bm.cache_stats() == (len(m.cached), m.hits, m.lookups)
        assert bm.evictable() == len(m.evictable)
        most_evictable = max(most_evictable, len(m.evictable))
    assert failures > 0 and m.hits > 0 and most_evictable > 0 and evicted > 0 and forks > 0 and copies > 0


def test_retained_prompt_is_hit_again_after_its_sequence_is_freed():
    bm = pa.BlockManager(16, 4)
    bm.set_prefix_retention(True)
    toks = list(range(11))  # two full blocks and a partial one
    s, cached = bm.new_seq_cached(toks)
    assert cached == 0
    bm.free_seq(s)
    assert bm.evictable() == 2 and bm.stats()[0] == 16  # evictable blocks count as free
    s2, cached2 = bm.new_seq_cached(toks)
    assert cached2 == 8 and bm.evictable() == 0
    bm.free_seq(s2)
    bm.set_prefix_retention(False)
    assert bm.evictable() == 0 and bm.cache_stats()[0] == 0


def test_a_freed_prompt_loses_its_tail_before_its_head():
    bm = pa.BlockManager(4, 2)
    bm.set_prefix_retention(True)
    toks = [1, 2, 3, 4, 5, 6]
    s, _ = bm.new_seq_cached(toks)
    bm.free_seq(s)
    other = bm.new_seq(4)  # two blocks: the free one and the prompt's evicted last block
    assert bm.evictable() == 2
    bm.free_seq(other)
    _, cached = bm.new_seq_cached(toks)
    assert cached == 4 and bm.evictable() == 0


@pytest.mark.parametrize("small", [True, False])
def test_retention_waves_match_oracle(small):
    """The two-wave retention workload, phase by phase: identical slots and
    tables, the designed prefix hits, and the first prompt keeping exactly
    the blocks the fresh prompt did not evict (its tail went first)."""
    wl = inputs.retention(small)
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    op0 = 0
    for ops, rows in wl.extra["phases"]:
        script = wl.script[op0:op0 + ops]
        r = oracle.run_script(0, wl.block_size, None, script, manager=m)
        slots, pairs = bm.apply_script(script)
        np.testing.assert_array_equal(slots, r["slots"])
        assert len(slots) == rows and len(pairs) == 0 and len(r["pairs"]) == 0
        written = slots[slots >= 0]
        assert len(np.unique(written)) == len(written)  # one cache write per phase stays race-free
        assert bm.evictable() == len(m.evictable)
        assert bm.cache_stats() == (len(m.cached), m.hits, m.lookups)
        op0 += ops
    assert op0 == len(wl.script)
    live = wl.extra["live"]
    tables, lens = bm.export(live, wl.max_blocks_per_seq)
    np.testing.assert_array_equal(tables, oracle.pad_tables([m.tables[s] for s in live], wl.max_blocks_per_seq))
    np.testing.assert_array_equal(lens, wl.seq_lens)
    # the last phase: the fresh request freed, then the first prompt's request
    first_len = len(wl.script[op0 - 1 - len(live)][1])
    cached = int((slots[:first_len] < 0).sum())
    assert cached == wl.extra["cached_tokens_first_prompt"] and slots[cached] >= 0


def test_sampling_memory_matches_oracle():
    rng = np.random.default_rng(12)
    cases = [(48, [16] * 4, 16), (2000, [1, 256, 100, 37], 16), (2008, [5, 0, 9, 300], 16), (0, [3, 3], 4)]
    for _ in range(30):
        B = int(rng.choice([1, 8, 16, 32]))
        cases.append((int(rng.integers(0, 400)), [int(x) for x in rng.integers(0, 90, size=int(rng.integers(1, 6)))], B))
    for P, gens, B in cases:
        got = pa.sampling_memory(P, gens, B)
        assert (got["shared_blocks"], got["unshared_blocks"], got["copies"]) == oracle.sampling_memory(P, gens, B)
