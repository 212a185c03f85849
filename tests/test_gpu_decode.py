"""GPU parity of paged decode attention against the fp64 oracle.

Tolerances (max-abs against the fp64 result): 1e-5 for fp32 inputs, 2e-2 for
bf16 inputs with fp32 accumulation.  Every case compares every output, the
full-size ones in the benchmark's launch configuration (automatic kernel
choice, one wave of CTAs)."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step

pytestmark = pytest.mark.gpu

SMALL = [("cfg0", {}), ("cfg1", {"small": True}), ("cfg2", {"small": True}),
         ("cfg3", {"small": True}), ("cfg3", {"small": True, "prompt_len": 200}),
         ("cfg4", {"small": True}), ("cfg4", {"small": True, "block_size": 32}),
         ("cfg4", {"small": True, "placement": "contiguous"}), ("cfg2-f32", {"small": True}),
         ("d256", {"small": True})]


@pytest.mark.parametrize("cfg,kw", SMALL)
@pytest.mark.parametrize("kernel,splits", [("auto", 0), ("auto", 1), ("auto", 7), ("simt", 0), ("simt", 5)])
def test_decode_small(cfg, kw, kernel, splits):
    wl = inputs.workload(cfg, **kw)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, dev, kernel=kernel, num_splits=splits)
    err = max_abs_err(g["out"], ref)
    assert err <= TOL[wl.dtype], err


FULL = [("cfg1", {}), ("cfg2", {}), ("cfg3", {}), ("cfg3", {"prompt_len": 2008}),
        ("cfg4", {}), ("cfg4", {"block_size": 32}), ("cfg4", {"placement": "contiguous"}), ("cfg2-f32", {}),
        ("d256", {})]


@pytest.mark.parametrize("cfg,kw", FULL)
def test_decode_full_size_every_output(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    ref = oracle_decode(wl, host, r)
    err = max_abs_err(g["out"], ref)
    assert err <= TOL[wl.dtype], err
    assert torch.isfinite(g["out"].float()).all()


# ------------------------------------------------------------- shape sweep
SHAPES = [  # (dtype, H, Hk, D, B)
    ("bf16", 8, 8, 128, 16), ("bf16", 16, 8, 128, 16), ("bf16", 32, 8, 128, 32), ("bf16", 64, 8, 128, 32),
    ("bf16", 8, 1, 128, 16), ("bf16", 6, 2, 64, 16), ("bf16", 12, 4, 64, 32), ("bf16", 8, 8, 256, 16),
    ("bf16", 4, 4, 128, 8), ("f32", 8, 2, 128, 16), ("f32", 4, 4, 64, 4), ("f32", 3, 1, 64, 5),
    # block sizes without a tensor-core instance: the TMA-staged CUDA-core kernel (a ring of 2 to 8
    # stages), and fp32 blocks of 128 tokens, whose ring does not fit, on the per-token kernel
    ("bf16", 8, 8, 64, 1), ("f32", 32, 8, 64, 7), ("bf16", 16, 8, 256, 64), ("f32", 8, 2, 128, 64),
    ("f32", 16, 2, 128, 128),
    # eight query heads per KV head on the CUDA-core kernel (its largest accumulator sets)
    ("f32", 16, 2, 64, 16), ("f32", 16, 2, 128, 16), ("bf16", 16, 2, 256, 16), ("f32", 7, 1, 128, 32),
]


@pytest.mark.parametrize("dtype,H,Hk,D,B", SHAPES)
@pytest.mark.parametrize("splits", [0, 3])
def test_decode_shapes(dtype, H, Hk, D, B, splits):
    lens = [1, B - 1, B, B + 1, 5 * B + 3, 2, 0, 77]
    wl = inputs.decode_workload("shape", lens, H, Hk, D, B, dtype, seed=99, pool_factor=1.3)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    for kernel in ("auto", "simt"):
        g = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, kernel=kernel, num_splits=splits)
        err = max_abs_err(g["out"], ref)
        assert err <= TOL[dtype], (kernel, err)
        assert (g["out"][6] == 0).all()  # the empty sequence


def test_single_token_sequences_return_their_value_rows_exactly():
    wl = inputs.decode_workload("one", [1] * 10, 16, 2, 128, 16, "bf16", seed=5, pool_factor=2.0)
    dev, host = host_values(wl, "cpu")
    g = gpu_step(wl, dev)
    for i in range(10):
        slot = int(g["host_slots"][i])
        row = g["v_cache"].view(-1, 2, 128)[slot]
        for h in range(16):
            assert torch.equal(g["out"][i, h], row[h // 8])


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_stale_slots_full_of_nan_are_never_read(kernel):
    wl = inputs.decode_workload("nan", [3, 17, 40, 16, 100], 32, 8, 128, 16, "bf16", seed=6, pool_factor=1.5)
    dev, host = host_values(wl, "cpu")
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    live = np.zeros((wl.num_blocks, wl.block_size), bool)
    for t, L in zip(r["tables"], r["lens"]):
        for pos in range(int(L)):
            live[t[pos // wl.block_size], pos % wl.block_size] = True
    nan_bits = np.uint16(0x7FC0)
    for name in ("k_cache", "v_cache"):
        host[name][~live] = nan_bits
        dev[name].view(torch.int16)[torch.from_numpy(~live).cuda()] = int(np.int16(0x7FC0))
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    assert np.isfinite(ref).all()
    g = gpu_step(wl, dev, kernel=kernel, num_splits=4)
    assert torch.isfinite(g["out"].float()).all()
    assert max_abs_err(g["out"], ref) <= TOL["bf16"]


def test_split_count_does_not_change_the_result():
    wl = inputs.workload("cfg4", small=True)
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    outs = []
    for splits in (1, 2, 7, 33, 0):
        g = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, num_splits=splits)
        assert max_abs_err(g["out"], ref) <= TOL["bf16"]
        outs.append(g["out"].float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= TOL["bf16"]


def test_block_size_16_and_32_agree():
    lens = [4096 + 5, 35, 700]
    outs = []
    for B in (16, 32):
        wl = inputs.decode_workload("b%d" % B, lens, 64, 8, 128, B, "bf16", seed=7, pool_factor=1.05)
        # same logical rows for both layouts: write every token through the cache write
        q = torch.randn(3, 64, 128, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16).cuda()
        rows_k = torch.randn(sum(lens), 8, 128, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
        rows_v = torch.randn(sum(lens), 8, 128, generator=torch.Generator().manual_seed(10)).to(torch.bfloat16).cuda()
        bm = pa.BlockManager(wl.num_blocks, B, wl.free_order)
        slots = []
        for L in lens:
            s = bm.new_seq(0)
            slots.append(bm.append_tokens(s, L)[0])
        tables, lens_np = bm.export([0, 1, 2], max(-(-L // B) for L in lens))
        kc = torch.zeros(wl.num_blocks, B, 8, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        pa.pa_reshape_and_cache(rows_k, rows_v, torch.from_numpy(np.concatenate(slots)).cuda(), kc, vc)
        out = pa.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens_np).cuda(),
                           1 / math.sqrt(128))
        outs.append(out.float())
    assert (outs[0] - outs[1]).abs().max().item() <= TOL["bf16"]


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_bad_table_entry_and_length_are_reported_without_a_fault(kernel):
    wl = inputs.decode_workload("bad", [40, 33], 16, 8, 128, 16, "bf16", seed=11, pool_factor=1.0)
    dev, host = host_values(wl, "cpu")
    g = gpu_step(wl, dev, decode=False)
    tables = g["tables"].clone()
    tables[0, 1] = wl.num_blocks + 3
    pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], tables, g["lens"], wl.scale, kernel=kernel)
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_BOUNDS
    lens = g["lens"].clone()
    lens[1] = 10 ** 6
    out = pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], lens, wl.scale, kernel=kernel)
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_BOUNDS
    assert (out[1] == 0).all()  # an out-of-range length counts as 0
    pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, kernel=kernel)
    assert pa.pa_get_device_error(raise_on_error=False) == 0


def test_bounded_wait_times_out_and_the_context_stays_usable():
    import time

    t0 = time.perf_counter()
    pa.pa_selftest_wait_timeout(20_000_000)  # 20 ms; nothing ever arrives
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    wl = inputs.workload("cfg0")
    dev, host = host_values(wl, "cpu")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["f32"]


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("num_seqs", [3000, 4095, 4096])
def test_many_sequences_prefix_sums_in_global_memory(kernel, num_seqs):
    """3000 sequences: more than the plan kernel keeps in shared memory, so
    its prefix sums and start search run from global memory, while each
    tensor-core CTA still computes its own copy (chunks of 19 per thread).
    4095: the largest batch whose prefix sums (4096 entries, 16 KiB) a
    tensor-core CTA keeps; 4096: the smallest it leaves to the plan kernel.
    Empty sequences scattered through the batch."""
    rng = np.random.default_rng(31)
    lens = rng.integers(1, 45, size=num_seqs)
    lens[::97] = 0
    wl = inputs.decode_workload("many", lens, 16, 8, 128, 16, "bf16", seed=31, pool_factor=1.2)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, kernel=kernel)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]
    assert (g["out"][::97] == 0).all()


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_one_long_sequence_merged_from_every_cta(kernel):
    """A 131,077-token sequence beside short ones (one of them exactly 256
    blocks).  With the default split the tensor-core kernel cuts its blocks
    across about 147 CTAs per head group (the CUDA-core kernel across all of
    its CTAs), so the last arriver of each (sequence, KV head) merges that
    many pieces."""
    lens = [131072 + 5, 17, 1, 4096]
    wl = inputs.decode_workload("long", lens, 64, 8, 128, 16, "bf16", seed=41, pool_factor=1.05)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, kernel=kernel)
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]
    assert torch.isfinite(g["out"].float()).all()


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_batch_of_only_empty_sequences(kernel):
    """No blocks at all: every attention CTA leaves at once; the output is
    all zeros (written by the plan kernel) and no error is recorded."""
    wl = inputs.decode_workload("empty", [0, 0, 0, 0, 0], 16, 8, 128, 16, "bf16", seed=43, pool_factor=1.0)
    dev, host = host_values(wl, "cpu")
    out = torch.full_like(dev["q"], float("nan"))
    g = gpu_step(wl, dev, decode=False)
    pa.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out=out, kernel=kernel)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert (out == 0).all()


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_large_scores_underflow_cleanly_through_the_merge(kernel):
    """q scaled 50x: scores spread over about +-150, so most softmax weights
    underflow to exactly 0 and the pieces of a split sequence carry maxima
    far apart (their rescaling factors 2^(m_p - M) reach 0).  The result
    stays finite and matches the oracle."""
    lens = [20000, 3, 700, 17, 4096 + 5]
    wl = inputs.decode_workload("peaked", lens, 32, 8, 128, 16, "bf16", seed=47, pool_factor=1.1)
    dev, host = host_values(wl, "cpu")
    dev["q"] = (dev["q"].float() * 50.0).to(torch.bfloat16)
    host["q"] = inputs.to_numpy_elems(dev["q"]).copy()
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, dev, kernel=kernel)
    assert torch.isfinite(g["out"].float()).all()
    assert max_abs_err(g["out"], ref) <= TOL["bf16"]


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("hint", ["exact", "zeros", "all-long"])
def test_long_context_merge_kernel_whatever_the_host_hint(kernel, hint):
    """With the host copy of the lengths, sequences cut into 8 or more pieces
    are merged by long_merge_kernel instead of their last-arriving CTA.  The
    hint only chooses the merge path: exact lengths (the long sequence goes
    to the second kernel), zeros (no second kernel) and lengths that claim
    every sequence is as long as the table allows (the second kernel runs
    and the device still picks only the truly long sequence) all match the
    oracle.  The CUDA-core kernel ignores the hint."""
    lens = [131072 + 5, 17, 1, 4096 + 5, 300, 0]
    wl = inputs.decode_workload("longhint", lens, 64, 8, 128, 16, "bf16", seed=53, pool_factor=1.05)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    hints = {"exact": "exact", "zeros": np.zeros(len(lens), np.int32),
             "all-long": np.full(len(lens), wl.max_blocks_per_seq * wl.block_size, np.int32)}
    g = gpu_step(wl, dev, kernel=kernel, host_lens=hints[hint])
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]
    assert (g["out"][5] == 0).all()
    assert torch.isfinite(g["out"].float()).all()


def test_long_context_merge_full_size_with_host_lengths():
    """The long-context workload (every sequence cut into ~10 pieces) in the
    benchmark's launch configuration, with the host lengths given."""
    wl = inputs.workload("cfg4")
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, host_lens="exact")
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]


def test_host_hint_leaves_short_sequences_bit_identical():
    """In a batch where the hint does bring in the second merge kernel, the
    sequences below the piece threshold are still merged in the attention
    launch: with and without the hint their outputs are the same bits."""
    lens = [131072 + 5, 17, 1, 4096 + 5, 300, 0, 2000]
    wl = inputs.decode_workload("longhint2", lens, 64, 8, 128, 16, "bf16", seed=59, pool_factor=1.05)
    dev, host = host_values(wl, "cuda")
    a = gpu_step(wl, {k: v.clone() for k, v in dev.items()})
    b = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, host_lens="exact")
    assert torch.equal(a["out"][1:], b["out"][1:])
    assert (a["out"][0].float() - b["out"][0].float()).abs().max().item() <= TOL["bf16"]


def test_launch_count_follows_the_options():
    """pa_decode_launch_count: plan + attention, plus the long-context merge
    when the host lengths show a sequence cut into 8+ pieces, plus the
    shared-prefix merge with a plan."""
    wl = inputs.workload("cfg4")
    kc = torch.empty(4, wl.block_size, wl.num_kv_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lens = np.asarray(wl.seq_lens, np.int32)
    args = (kc, wl.num_seqs, wl.num_q_heads, wl.max_blocks_per_seq)
    assert pa.pa_decode_launch_count(*args) == 2
    assert pa.pa_decode_launch_count(*args, host_seq_lens=lens) == 3
    assert pa.pa_decode_launch_count(*args, host_seq_lens=np.zeros_like(lens)) == 2
    assert pa.pa_decode_launch_count(*args, kernel="simt", host_seq_lens=lens) == 2
    assert pa.pa_decode_launch_count(*args, shared=True, host_seq_lens=lens) == 3  # shared merge, no long merge
    w2 = inputs.workload("cfg2")
    k2 = torch.empty(4, w2.block_size, w2.num_kv_heads, w2.head_dim, dtype=torch.bfloat16, device="cuda")
    assert pa.pa_decode_launch_count(k2, w2.num_seqs, w2.num_q_heads, w2.max_blocks_per_seq,
                                     host_seq_lens=np.asarray(w2.seq_lens, np.int32)) == 2
    assert pa.pa_decode_launch_count(k2, 0, w2.num_q_heads, w2.max_blocks_per_seq) == 0


def test_long_merge_among_many_short_sequences():
    """Two long contexts among 298 short sequences: enough (head group,
    sequence) pairs that long_merge_kernel lists the long ones 256 pairs at a
    time before dealing out their merges."""
    rng = np.random.default_rng(61)
    lens = rng.integers(1, 500, size=300)
    lens[17], lens[250] = 65536 + 3, 40000
    lens[::41] = 0
    wl = inputs.decode_workload("manylong", lens, 32, 8, 128, 16, "bf16", seed=61, pool_factor=1.1)
    dev, host = host_values(wl, "cuda")
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, host_lens="exact")
    assert max_abs_err(g["out"], oracle_decode(wl, host, r)) <= TOL["bf16"]
    assert (g["out"][::41] == 0).all()


@pytest.mark.parametrize("cfg,kw,kernel,layout", [
    ("cfg0", {}, "auto", "row"), ("cfg1", {"small": True}, "auto", "row"), ("cfg2", {"small": True}, "auto", "row"),
    ("cfg2", {"small": True}, "simt", "row"), ("cfg4", {"small": True, "block_size": 32}, "auto", "row"),
    ("cfg2", {"small": True}, "auto", "split"), ("cfg2", {}, "auto", "row"), ("cfg4", {}, "auto", "row")])
def test_relabelled_physical_blocks_give_the_same_bits(cfg, kw, kernel, layout):
    """A block table may point at any physical blocks ("10 PagedAttention"
    (PidokuInfra), section 4 PhysicalIndex; "PagedAttention" (tokentrails),
    step 3: the same attention as over contiguous memory).  Moving every
    block's contents to a new physical id and rewriting the tables to match
    must not change a single bit of the output: the work split and the
    order of the arithmetic depend only on the lengths, never on where the
    blocks sit in the pool."""
    wl = inputs.workload(cfg, **kw)
    dev, _ = host_values(wl, "cuda", layout=layout)
    g = gpu_step(wl, dev, kernel=kernel)
    perm = torch.from_numpy(np.random.default_rng(71).permutation(wl.num_blocks)).cuda()  # new id of block b
    k2, v2 = torch.empty_like(g["k_cache"]), torch.empty_like(g["v_cache"])
    k2[perm] = g["k_cache"]
    v2[perm] = g["v_cache"]
    t = g["tables"]
    t2 = torch.where(t >= 0, perm[t.clamp(min=0).long()].to(torch.int32), t)
    assert not torch.equal(t2, t)
    out2 = pa.pa_decode(g["q"], k2, v2, t2, g["lens"], wl.scale, kernel=kernel)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(out2, g["out"])
