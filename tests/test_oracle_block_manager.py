"""Pins for the oracle's block-manager model: the pages' worked examples,
sharing counts, copy-on-write invariants and failure semantics."""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_150_gb300 import inputs


def test_go_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "go_worked_example.json")))
    m = oracle.OracleBlockManager(g["num_blocks"], g["block_size"])
    seqs = {}
    for st in g["steps"]:
        if st["op"] == "new":
            s = m.new_sequence(st["tokens"])
            assert s is not None
            seqs[st["name"]] = s
            if "expect_blocks" in st:
                assert len(m.tables[s]) == st["expect_blocks"]
        else:
            m.free_seq(seqs[st["name"]])
        free, used, _ = m.stats()
        if "expect_free" in st:
            assert free == st["expect_free"]
        if "expect_used" in st:
            assert used == st["expect_used"]
    d = g["derived"]
    assert m.tables[seqs["e"]] == d["table_e"]
    assert m.tables[seqs["a"]] == d["table_a"] and m.tables[seqs["c"]] == d["table_c"]
    assert m.physical_index(seqs["e"], 40) == d["physical_index_e_40"]


def test_nano_vllm_free_list_pops_highest_first(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "slot_mapping_examples.json")))["free_list"]
    m = oracle.OracleBlockManager(g["num_blocks"], 256, list(range(g["num_blocks"])))
    s = m.new_sequence(1)
    assert m.tables[s] == [g["first_pop"]]
    m.free_seq(s)
    assert m.free[-1] == g["first_pop"]


def test_parallel_sampling_shares_prompt_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sharing_examples.json")))["parallel_sampling"]
    B = g["block_size"]
    m = oracle.OracleBlockManager(len(g["free_order"]), B, g["free_order"])
    parent = m.new_sequence(len(g["prompt_blocks"]) * B)
    seqs = [parent] + [m.fork(parent) for _ in range(g["samples"] - 1)]
    assert m.tables[parent] == g["prompt_blocks"]
    assert all(m.ref[b] == g["prompt_refcount"] for b in g["prompt_blocks"])
    pairs = []
    for s in seqs:
        slot, pair = m.append_token(s)
        pairs.append(pair)
    assert pairs == [None] * g["samples"]  # block-aligned prompt: no copy
    assert [m.tables[s][-1] for s in seqs] == g["extra_blocks"]
    free, used, shared = m.stats()
    assert used == g["physical_blocks"]
    unshared = sum(len(m.tables[s]) for s in seqs)
    assert unshared == g["unshared_blocks"]
    assert 1 - used / unshared == pytest.approx(g["saved_fraction"])
    assert shared == len(g["prompt_blocks"])


def test_three_requests_share_two_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sharing_examples.json")))["three_requests"]
    B = g["block_size"]
    tail = list(reversed(g["new_blocks"])) + g["shared_blocks"]
    top = max(tail) + 1
    order = [b for b in range(top) if b not in tail] + tail
    m = oracle.OracleBlockManager(top, B, order)
    first = m.new_sequence(len(g["shared_blocks"]) * B)
    seqs = [first] + [m.fork(first) for _ in range(g["requests"] - 1)]
    assert m.stats()[1] == len(g["shared_blocks"])
    assert all(m.ref[b] == g["shared_refcount"] for b in g["shared_blocks"])
    for s in seqs:
        m.append_token(s)
    assert [m.tables[s][-1] for s in seqs] == g["new_blocks"]
    assert all(m.tables[s][:2] == g["shared_blocks"] for s in seqs)
    assert m.stats()[1] == g["distinct_blocks"]


def _check_invariants(m):
    free, used, _ = m.stats()
    assert free + used == m.num_blocks
    assert sum(m.ref.values()) == sum(len(t) for t in m.tables.values())
    assert len(set(m.free)) == len(m.free) and not (set(m.free) & set(m.ref))


@pytest.mark.parametrize("prompt_len,expect_pairs", [(192, 0), (200, 3)])
def test_copy_on_write_in_parallel_sampling(prompt_len, expect_pairs):
    wl = inputs.workload("cfg3", small=True, prompt_len=prompt_len)
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    m = r["manager"]
    prompts = wl.extra["num_prompts"]
    assert len(r["pairs"]) == expect_pairs * prompts
    assert all(ref == 1 for ref in r["written_refcounts"])  # no shared block written in place
    dst = r["pairs"][:, 1].tolist()
    assert len(set(dst)) == len(dst) and not (set(dst) & set(r["pairs"][:, 0].tolist()))
    np.testing.assert_array_equal(r["lens"], wl.seq_lens)
    _check_invariants(m)
    if expect_pairs:
        # the last writer of each shared partial block writes it in place
        srcs = r["pairs"][:, 0]
        for s in set(srcs.tolist()):
            assert (srcs == s).sum() == wl.extra["samples"] - 1 and m.ref[s] == 1


def _state(m):
    return (list(m.free), dict(m.ref), {k: list(v) for k, v in m.tables.items()}, dict(m.lens))


def test_allocation_failure_changes_nothing():
    m = oracle.OracleBlockManager(3, 4)
    m.new_sequence(8)  # 2 blocks used, 1 free
    before = _state(m)
    assert m.new_sequence(9) is None  # needs 3 blocks
    assert _state(m) == before
    m2 = oracle.OracleBlockManager(2, 4)
    s = m2.new_sequence(6)  # partly filled last block, pool now empty
    m2.fork(s)
    before = _state(m2)
    assert m2.append_token(s) is None  # a copy is needed and no block is free
    assert _state(m2) == before
    m3 = oracle.OracleBlockManager(1, 4)
    s3 = m3.new_sequence(4)
    before = _state(m3)
    assert m3.append_token(s3) is None  # a new block is needed and none is free
    assert _state(m3) == before


def test_free_of_unknown_sequence_raises():
    m = oracle.OracleBlockManager(4, 4)
    s = m.new_sequence(4)
    m.free_seq(s)
    with pytest.raises(KeyError):
        m.free_seq(s)


def test_decode_workload_tables_cover_lengths():
    for cfg in ("cfg0", "cfg1", "cfg2"):
        wl = inputs.workload(cfg, small=True)
        r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
        np.testing.assert_array_equal(r["lens"], wl.seq_lens)
        for L, t in zip(wl.seq_lens, r["tables"]):
            assert len(t) == -(-int(L) // wl.block_size)
        assert len(r["slots"]) == wl.num_new_tokens
        _check_invariants(r["manager"])


# ------------------------------------------------------------ prefix caching
def test_fnv1a64_published_test_vectors():
    from oracle.block_manager import fnv1a64

    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_ten_requests_share_one_copy_of_the_system_prompt(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "prefix_sharing_example.json")))
    B, n = g["block_size"], g["requests"]
    rng = np.random.default_rng(0)
    system = rng.integers(0, 32000, size=g["system_prompt_tokens"]).tolist()
    m = oracle.OracleBlockManager(4096, B)
    seqs, cached, own = [], [], 0
    for i in range(n):
        suffix = rng.integers(0, 32000, size=int(rng.integers(1, 100))).tolist()
        s, c = m.new_sequence_cached(system + suffix)
        seqs.append(s)
        cached.append(c)
        own += m.blocks_needed(len(system) + len(suffix)) - g["system_prompt_blocks"]
    assert cached == [0] + [g["system_prompt_tokens"]] * (n - 1)
    assert all(m.tables[s][:125] == m.tables[seqs[0]][:125] for s in seqs)
    assert all(m.ref[b] == n for b in m.tables[seqs[0]][:g["system_prompt_blocks"]])
    assert m.stats()[1] == g["system_prompt_blocks"] + own  # one copy, not ten
    _check_invariants(m)


def test_prefix_match_is_chained_and_stops_at_the_first_miss():
    B = 4
    m = oracle.OracleBlockManager(64, B)
    a = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13]
    s0, c0 = m.new_sequence_cached(a)
    assert c0 == 0
    # same first and third block, different second block: only block 0 is reused
    b = [1, 2, 3, 4, 99, 6, 7, 8, 9, 10, 11, 12]
    s1, c1 = m.new_sequence_cached(b)
    assert c1 == 4 and m.tables[s1][0] == m.tables[s0][0] and m.tables[s1][2] != m.tables[s0][2]
    # block 1 of `a` after a different block 0: no hit (the key covers the prefix)
    s2, c2 = m.new_sequence_cached([0, 0, 0, 0, 5, 6, 7, 8])
    assert c2 == 0
    # the partial last block (token 13) was not registered
    s3, c3 = m.new_sequence_cached(a)
    assert c3 == 12 and m.tables[s3][3] != m.tables[s0][3]
    _check_invariants(m)


def test_cached_blocks_leave_the_map_when_their_last_user_frees_them():
    m = oracle.OracleBlockManager(32, 4)
    p = list(range(8))
    s0, _ = m.new_sequence_cached(p)
    s1, c1 = m.new_sequence_cached(p)
    assert c1 == 8
    m.free_seq(s0)
    assert len(m.cached) == 2  # still held by s1
    m.free_seq(s1)
    assert len(m.cached) == 0
    s2, c2 = m.new_sequence_cached(p)
    assert c2 == 0
    _check_invariants(m)


def test_prefix_cached_failure_changes_nothing():
    m = oracle.OracleBlockManager(3, 4)
    m.new_sequence_cached(list(range(8)))
    before = _state(m), dict(m.cached), m.hits, m.lookups
    assert m.new_sequence_cached(list(range(8)) + [5] * 8) is None  # needs 2 fresh, 1 free
    assert (_state(m), dict(m.cached), m.hits, m.lookups) == before


@pytest.mark.parametrize("small", [True, False])
def test_prefix_workload_never_writes_a_shared_block(small):
    wl = inputs.workload("prefix", small=small)
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    assert all(ref == 1 for ref in r["written_refcounts"])
    assert (r["slots"] == -1).sum() > 0  # some prompt positions were cached
    np.testing.assert_array_equal(r["lens"], wl.seq_lens)
    _check_invariants(r["manager"])


# -------------------------------------------------------------- beam search
@pytest.mark.parametrize("small", [True, False])
def test_beam_search_keeps_copy_on_write_invariants(small):
    wl = inputs.beam(small)
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    B = wl.block_size
    for st in wl.steps:
        setup = [op for op in st["ops"] if op[0] != "append"]  # the first step creates the beams
        appends = [op for op in st["ops"] if op[0] == "append"]
        oracle.run_script(0, B, None, setup, manager=m)
        # A shared partly filled block with refcount R written by n of its
        # holders is copied min(n, R - 1) times (the last holder writes in place).
        writers, refs = {}, {}
        for op in appends:
            if op[0] == "append" and op[1] in m.tables:
                pos = m.lens[op[1]]
                if pos % B:
                    b = m.tables[op[1]][pos // B]
                    if m.ref[b] > 1:
                        writers[b] = writers.get(b, 0) + 1
                        refs[b] = m.ref[b]
        r = oracle.run_script(0, B, None, appends, manager=m)
        assert len(r["pairs"]) == sum(min(n, refs[b] - 1) for b, n in writers.items())
        assert all(ref == 1 for ref in r["written_refcounts"])
        oracle.run_script(0, B, None, st["select"], manager=m)
        _check_invariants(m)


def test_retention_evicts_the_least_recently_released_block_first():
    """Retained blocks leave in the order they were released.  Prompts A and
    B each fill one block and are freed, A first; a request for three blocks
    then takes the two free ones and evicts A's block, so B's prompt still
    hits while A's prompt has left the map.  A request that neither free nor
    evictable blocks can cover fails and changes nothing."""
    m = oracle.OracleBlockManager(4, 2, free_order=[3, 2, 1, 0])  # block 0 is taken first
    m.set_retention(True)
    a, _ = m.new_sequence_cached([1, 2])
    b, _ = m.new_sequence_cached([3, 4])
    block_a, block_b = m.tables[a][0], m.tables[b][0]
    m.free_seq(a)
    m.free_seq(b)
    assert m.evictable == [block_a, block_b] and m.stats()[0] == 4
    c = m.new_sequence(5)  # three blocks: the two free ones and block_a
    assert c is not None and block_a in m.tables[c] and m.evictable == [block_b]
    assert list(m.cached.values()) == [block_b]  # A's prompt left the map
    _, hit = m.new_sequence_cached([3, 4])
    assert hit == 2 and m.evictable == [] and m.ref[block_b] == 1
    state = (list(m.free), dict(m.ref), dict(m.cached), m.hits, m.lookups)
    assert m.new_sequence_cached([1, 2, 9, 9]) is None  # two blocks wanted, none left
    assert (list(m.free), dict(m.ref), dict(m.cached), m.hits, m.lookups) == state


def test_retention_off_returns_retained_blocks_oldest_first():
    """Switching retention off unregisters every retained block and pushes
    them onto the free stack in release order, so the newest release is the
    next block handed out."""
    m = oracle.OracleBlockManager(3, 2, free_order=[2, 1, 0])
    m.set_retention(True)
    seqs = [m.new_sequence_cached([k, k])[0] for k in (1, 2, 3)]
    released = [m.tables[s][0] for s in seqs]
    for s in seqs:
        m.free_seq(s)
    m.set_retention(False)
    assert m.free == released and m.cached == {} and m.evictable == []
    assert m.allocate(1) == [released[-1]]


def test_a_freed_prompt_loses_its_tail_before_its_head():
    """Matching stops at a prompt's first miss, so evicting a prompt's first
    block would strand the rest.  A freed three-block prompt gives up its
    last block to the first eviction, and the same prompt still hits its
    first two blocks afterwards."""
    m = oracle.OracleBlockManager(4, 2)
    m.set_retention(True)
    s, _ = m.new_sequence_cached([1, 2, 3, 4, 5, 6])
    table = list(m.tables[s])
    m.free_seq(s)
    assert m.evictable == table[::-1]
    got = m.allocate(2)  # the one free block and the evicted tail
    assert table[2] in got and m.evictable == table[1::-1]
    m.free_blocks(got)
    _, hit = m.new_sequence_cached([1, 2, 3, 4, 5, 6])
    assert hit == 4


def test_sampling_memory_reproduces_the_page_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sharing_examples.json")))["parallel_sampling"]
    B = g["block_size"]
    shared, alone, copies = oracle.sampling_memory(len(g["prompt_blocks"]) * B, [B] * g["samples"], B)
    assert (shared, alone, copies) == (g["physical_blocks"], g["unshared_blocks"], 0)
    assert 1 - shared / alone == g["saved_fraction"]


def test_sampling_memory_closed_form():
    """Full prompt blocks are held once; each sample that writes ends up with
    its own blocks from the prompt's partly filled block on (the first n-1
    writers into that shared block copy it, the last writes in place).
    Unshared, every sample holds ceil((P + g) / B) blocks."""
    rng = np.random.default_rng(11)
    for _ in range(60):
        B = int(rng.choice([1, 4, 16, 32]))
        P = int(rng.integers(0, 300))
        gens = [int(x) for x in rng.integers(1, 80, size=int(rng.integers(1, 7)))]
        full = P // B
        expect_shared = full + sum(-(-(P + g) // B) - full for g in gens)
        expect_alone = sum(-(-(P + g) // B) for g in gens)
        expect_copies = (len(gens) - 1) if P % B else 0
        assert oracle.sampling_memory(P, gens, B) == (expect_shared, expect_alone, expect_copies)
    # samples that generate nothing keep sharing the whole prompt
    assert oracle.sampling_memory(2008, [0, 0, 0, 0], 16) == (126, 4 * 126, 0)


def test_sampling_saves_over_half_for_a_2000_token_prompt():
    """Exercise E's measurement: four samples of U[1, 256] tokens from a
    2000-token prompt; the table of section 7 quotes 55%+ saved."""
    rng = np.random.default_rng(1503)
    gens = [int(x) for x in rng.integers(1, 257, size=4)]
    for P in (2000, 2008):
        shared, alone, _ = oracle.sampling_memory(P, gens, 16)
        assert 1 - shared / alone >= 0.55
