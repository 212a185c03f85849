"""The shared-prefix plan builder (host): which sequences share leading
physical blocks, and the packed words the decode kernels read.

The words are decoded here with an independent reader of the documented
layout (include/pa.h, pa_common.cuh), and the grouping is checked against
what the tables themselves fix: every member of a group has the same first
P blocks, P is maximal (a member differs at block P, or P is the largest
prefix that leaves every member a position of its own), and sequences left
out of groups share no first block with a group."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def decode_plan(words):
    w = [int(x) for x in np.asarray(words)]
    magic, N, G, B, ng, M, V, R = w[:8]
    assert magic == 0x50415350
    pos = 8

    def take(n):
        nonlocal pos
        out = w[pos:pos + n]
        pos += n
        return out

    p = {"N": N, "G": G, "B": B, "groups": ng, "M": M, "V": V, "R": R}
    p["seq_group"], p["seq_member"] = take(N), take(N)
    p["prefix"], p["vbase"], p["begin"] = take(ng), take(ng + 1), take(ng + 1)
    p["members"], p["vgroup"], p["cu_s"] = take(M), take(V), take(V + 1)
    assert pos <= len(w)
    return p


def check_plan(p, tables, lens, B, G, min_blocks=1):
    N = len(lens)
    # query rows per pass: the smallest of 16, 32, 64 holding the largest group's rows
    sizes = [p["begin"][g + 1] - p["begin"][g] for g in range(p["groups"])]
    max_rows = max([n * G for n in sizes], default=0)
    assert p["R"] == (16 if max_rows <= 16 else 32 if max_rows <= 32 else 64)
    assert p["N"] == N and p["B"] == B and p["G"] == G
    sharing = G in (1, 2, 4, 8)
    if not sharing:
        assert p["groups"] == 0
    grouped = set()
    for g in range(p["groups"]):
        mem = p["members"][p["begin"][g]:p["begin"][g + 1]]
        P = p["prefix"][g]
        assert len(mem) >= 2 and P >= min_blocks
        rep = tables[mem[0]]
        for k, i in enumerate(mem):
            assert p["seq_group"][i] == g and p["seq_member"][i] == k
            assert list(tables[i][:P]) == list(rep[:P])
            assert P * B < lens[i]  # every member keeps a position of its own
            grouped.add(i)
        # maximal: one more block is either not common or not allowed
        cap = min((lens[i] - 1) // B for i in mem)
        assert P == cap or any(tables[i][P] != rep[P] for i in mem)
        passes = p["vbase"][g + 1] - p["vbase"][g]
        assert passes == -(-len(mem) * G // p["R"])
        for v in range(p["vbase"][g], p["vbase"][g + 1]):
            assert p["vgroup"][v] == g and p["cu_s"][v + 1] - p["cu_s"][v] == P
    assert p["cu_s"][0] == 0 and p["vbase"][p["groups"]] == p["V"] and p["begin"][p["groups"]] == p["M"]
    assert len(grouped) == p["M"]
    for i in range(N):
        if i not in grouped:
            assert p["seq_group"][i] == -1 and p["seq_member"][i] == -1
    # a sequence outside every group shares its first block with no group
    firsts = {int(tables[i][0]) for i in grouped}
    for i in range(N):
        if i not in grouped and (lens[i] - 1) // B >= 1 and sharing and min_blocks == 1:
            assert int(tables[i][0]) not in firsts or all(
                p["prefix"][p["seq_group"][j]] < 1 for j in grouped if tables[j][0] == tables[i][0])


def plan_for(wl, **kw):
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    tables = oracle.pad_tables(r["tables"], wl.max_blocks_per_seq)
    plan, info = pa.shared_prefix_plan(tables, r["lens"], wl.block_size, wl.num_q_heads, wl.num_kv_heads, **kw)
    return decode_plan(plan.numpy()), info, tables, r["lens"]


@pytest.mark.parametrize("prompt_len", [2000, 2008])
def test_parallel_sampling_groups_the_samples_of_each_prompt(prompt_len):
    wl = inputs.workload("cfg3", prompt_len=prompt_len)
    p, info, tables, lens = plan_for(wl)
    check_plan(p, tables, lens, wl.block_size, wl.num_q_heads // wl.num_kv_heads)
    # 64 prompts x 4 samples; the 125 full prompt blocks are shared (with a
    # 2008-token prompt the half-full 126th is copied on write for 3 samples)
    assert info["num_groups"] == 64 and info["num_members"] == 256
    assert set(p["prefix"]) == {125}
    assert p["R"] == 16 and p["V"] == 64  # 4 samples x 4 query heads = 16 rows: one pass of 16
    assert info["saved_blocks"] == 64 * 3 * 125


def test_prefix_cache_groups_requests_of_each_system_prompt():
    wl = inputs.workload("prefix")
    p, info, tables, lens = plan_for(wl)
    check_plan(p, tables, lens, wl.block_size, wl.num_q_heads // wl.num_kv_heads)
    assert info["num_groups"] == 8 and info["num_members"] == 80
    assert set(p["prefix"]) == {125}  # 2000-token system prompt
    assert p["R"] == 64 and p["V"] == 8  # 10 requests x 4 query heads = 40 rows: one pass of up to 64


@pytest.mark.parametrize("cfg,kw", [("cfg1", {}), ("cfg2", {}), ("cfg4", {})])
def test_batches_without_sharing_have_no_group(cfg, kw):
    p, info, tables, lens = plan_for(inputs.workload(cfg, **kw))
    assert info["num_groups"] == 0 and p["V"] == 0 and p["M"] == 0


@pytest.mark.parametrize("small", [True, False])
def test_beam_search_tables_at_every_step(small):
    wl = inputs.beam(small)
    m = oracle.OracleBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    G = wl.num_q_heads // wl.num_kv_heads
    for st in wl.steps:
        oracle.run_script(0, wl.block_size, None, st["ops"], manager=m)
        mb = max(len(m.tables[s]) for s in st["decode"])
        tables = oracle.pad_tables([m.tables[s] for s in st["decode"]], mb)
        lens = np.asarray([m.lens[s] for s in st["decode"]], dtype=np.int32)
        plan, _ = pa.shared_prefix_plan(tables, lens, wl.block_size, wl.num_q_heads, wl.num_kv_heads)
        check_plan(decode_plan(plan.numpy()), tables, lens, wl.block_size, G)
        oracle.run_script(0, wl.block_size, None, st["select"], manager=m)


def test_random_tables_and_thresholds():
    rng = np.random.default_rng(11)
    for trial in range(60):
        N, mb, B = int(rng.integers(1, 40)), int(rng.integers(1, 12)), int(rng.choice([4, 16]))
        base = rng.permutation(1000)[:mb * N].reshape(N, mb).astype(np.int32)
        # plant shared prefixes: copy the first k blocks of a few "parents"
        for i in range(N):
            if rng.random() < 0.6:
                j = int(rng.integers(0, N))
                k = int(rng.integers(0, mb + 1))
                base[i, :k] = base[j, :k]
        lens = rng.integers(0, mb * B + 1, size=N).astype(np.int32)
        G = int(rng.choice([1, 2, 3, 4, 8]))
        Hk = int(rng.choice([1, 2, 4]))
        mins = int(rng.integers(1, 4))
        plan, info = pa.shared_prefix_plan(base, lens, B, G * Hk, Hk, min_shared_blocks=mins)
        p = decode_plan(plan.numpy())
        check_plan(p, base, lens, B, G, mins)
        assert info["num_groups"] == p["groups"] and info["num_members"] == p["M"]


def test_bad_arguments():
    t = np.zeros((2, 3), dtype=np.int32)
    L = np.array([5, 6], dtype=np.int32)
    with pytest.raises(pa.PagedAttentionError):
        pa.shared_prefix_plan(t, np.array([5, 13], dtype=np.int32), 4, 8, 8)  # length past the table
    with pytest.raises(pa.PagedAttentionError):
        pa.shared_prefix_plan(t, L, 4, 8, 3)  # heads not a multiple of KV heads
    with pytest.raises(pa.PagedAttentionError):
        pa.shared_prefix_plan(t, L, 4, 8, 8, min_shared_blocks=0)
    with pytest.raises(ValueError):
        pa.shared_prefix_plan(t, L[:1], 4, 8, 8)
