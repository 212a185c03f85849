"""Seeded synthetic workloads for the paged-KV decode path.

This module is shared by the tests, the benchmark and the smoke check, and by
both sides of every parity check (the CUDA library and the CPU oracle).  It
holds no arithmetic of the method itself: it draws sequence lengths, the order
of the free list, a script of block-manager operations and random K/V/q
values.  Block tables, slots and copy-on-write pairs are NOT computed here;
each side derives them from the script with its own block manager.

Workload shapes follow the pages' examples and the five benchmark workloads:
  cfg0  fp32 tiny decode: lengths {5,16,23,40}, 4 q heads = 4 KV heads,
        head_dim 64, block_size 4, pool of 32 blocks.
  cfg1  bf16 MHA decode: 32 sequences, lengths uniform in [128, 2048],
        32 = 32 heads, head_dim 128, block_size 16, pool 1.25x the need.
  cfg2  bf16 GQA mixed lengths: 256 sequences, lognormal lengths (median 512,
        sigma 1.0, clipped to [16, 8192]), 32 q / 8 KV heads, head_dim 128,
        block_size 16, pool 1.1x the need.
  cfg3  bf16 parallel sampling: 64 prompts of 2000 tokens (2008 in the
        copy-on-write variant), each forked into 4 samples, each sample
        appends 1..256 tokens; 32 q / 8 KV heads, head_dim 128, block_size 16.
        The reduced twin uses 4 prompts of 192 tokens (200 for copy-on-write)
        and appends of 1..40 tokens.
  cfg4  bf16 long context: 16 sequences of 32768 tokens, 64 q / 8 KV heads,
        head_dim 128, block_size 16 or 32, pool 1.05x the need.
  prefix  bf16 prefix caching: 8 system prompts of 2000 tokens, 10 requests
        each with a U[16, 512]-token suffix (32 q / 8 KV heads, head_dim 128,
        block_size 16); the reduced twin has 2 prompts of 200 tokens x 3.

Conventions (readings of the workload text):
  * Workload k is seeded with 1500 + k (numpy PCG64 for structure, a torch
    generator on the target device for values).  Reduced-size variants used by
    parity tests are seeded with 2500 + k.
  * For decode workloads a sequence's stated length L counts the token written
    in this step: the script creates it with L - 1 tokens, then appends one.
  * Every pool element is N(0, 1), cast to the workload's element type
    (round-to-nearest-even for bf16).  Blocks are placed by popping a
    seed-shuffled free list (pop from the end).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

NEW = "new"        # ("new", prompt_len): create a sequence holding prompt_len tokens
FORK = "fork"      # ("fork", parent): create a sequence sharing the parent's blocks
APPEND = "append"  # ("append", seq, count): append count new tokens to seq


@dataclass
class Workload:
    name: str
    dtype: str                    # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seed: int
    free_order: np.ndarray        # int32 [num_blocks]; the top of the stack is the last entry
    script: List[Tuple]           # block-manager operations, in order
    seq_lens: np.ndarray          # int32 [num_seqs]: final length of every sequence (decode order)
    num_new_tokens: int           # rows of k/v written by this step (in script order)
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-int(self.seq_lens.max(initial=0)) // self.block_size))

    def kv_bytes_read(self) -> int:
        """Bytes of K and V that one decode pass reads: sum_i L_i * Hk * D * 2 * elem."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 2 * self.elem_bytes

    def pool_bytes(self) -> int:
        return 2 * self.num_blocks * self.block_size * self.num_kv_heads * self.head_dim * self.elem_bytes


def _shuffled_free_order(rng: np.random.Generator, num_blocks: int) -> np.ndarray:
    return rng.permutation(num_blocks).astype(np.int32)


def decode_workload(name: str, lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    block_size: int, dtype: str, seed: int, pool_factor: float = 1.0,
                    num_blocks: Optional[int] = None, rng: Optional[np.random.Generator] = None,
                    note: str = "", placement: str = "random") -> Workload:
    """One decode step over independent sequences of the given final lengths.

    Each sequence is created with L-1 tokens and then receives one new token
    (the token this step writes); a length of 0 creates an empty sequence and
    writes nothing.  ``placement``: "random" (a seed-shuffled free list) or
    "contiguous" (an ascending free list: the manager hands every sequence
    consecutive physical blocks in order, as one contiguous KV region would)."""
    if placement not in ("random", "contiguous"):
        raise ValueError("placement must be 'random' or 'contiguous'")
    lens = np.asarray(lens, dtype=np.int32)
    if rng is None:
        rng = np.random.default_rng(seed)
    need = int(sum(-(-int(L) // block_size) for L in lens))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * need)))
    if placement == "contiguous":
        free_order = np.arange(num_blocks, dtype=np.int32)
    else:
        free_order = _shuffled_free_order(rng, num_blocks)
    script: List[Tuple] = []
    for L in lens:
        script.append((NEW, max(int(L) - 1, 0)))
    ntok = 0
    for i, L in enumerate(lens):
        if L > 0:
            script.append((APPEND, i, 1))
            ntok += 1
    return Workload(name, dtype, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                    seed, free_order, script, lens, ntok, note=note)


def sampling_workload(name: str, num_prompts: int, prompt_len: int, samples: int,
                      max_append: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      block_size: int, dtype: str, seed: int, spare_blocks: int = 64) -> Workload:
    """Parallel sampling: each prompt is forked into ``samples`` sequences that
    share its blocks, then every sample appends U[1, max_append] tokens, in
    sample order.  Decode runs over every sample."""
    rng = np.random.default_rng(seed)
    appends = rng.integers(1, max_append + 1, size=num_prompts * samples).astype(np.int32)
    script: List[Tuple] = []
    lens = []
    seq = 0
    sample_ids = []
    for p in range(num_prompts):
        parent = seq
        script.append((NEW, prompt_len))
        seq += 1
        ids = [parent]
        for _ in range(samples - 1):
            script.append((FORK, parent))
            ids.append(seq)
            seq += 1
        sample_ids.extend(ids)
    for j, s in enumerate(sample_ids):
        script.append((APPEND, s, int(appends[j])))
        lens.append(prompt_len + int(appends[j]))
    # Pool sizing: the prompt's blocks once, every sample's own growth, one
    # private copy of a partly filled shared last block per sample, plus spare.
    bs = block_size
    prompt_blocks = -(-prompt_len // bs)
    growth = sum(-(-(prompt_len + int(a)) // bs) - prompt_blocks for a in appends)
    partial_copies = num_prompts * samples if prompt_len % bs else 0
    num_blocks = num_prompts * prompt_blocks + growth + partial_copies + spare_blocks
    free_order = _shuffled_free_order(rng, num_blocks)
    return Workload(name, dtype, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                    seed, free_order, script, np.asarray(lens, dtype=np.int32),
                    int(appends.sum()),
                    note="%d prompts x %d samples, prompt %d, append U[1,%d]"
                         % (num_prompts, samples, prompt_len, max_append),
                    extra={"prompt_len": prompt_len, "samples": samples,
                           "num_prompts": num_prompts})


NEW_CACHED = "new_cached"  # ("new_cached", token_ids): a prompt that may reuse cached prefix blocks
FREE = "free"              # ("free", seq): release a sequence's blocks
RETAIN = "retain"          # ("retain", on): keep freed prompt blocks registered until evicted


@dataclass
class BeamWorkload:
    """Beam search over one prompt: a list of steps, each a block-manager
    script (one appended token per live beam) followed by a decode over the
    live beams; after the decode the step's selection ops (free the beams not
    chosen, fork the ones chosen more than once) run.  Values: one K/V row per
    appended token, in script order over all steps."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seed: int
    free_order: np.ndarray
    prompt_len: int
    beams: int
    steps: list              # [{"ops": [...], "decode": [seq ids], "select": [...]}]
    num_new_tokens: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


def beam_workload(name: str, prompt_len: int, beams: int, num_steps: int, num_q_heads: int, num_kv_heads: int,
                  head_dim: int, block_size: int, dtype: str, seed: int) -> BeamWorkload:
    """Each step every live beam appends a token; then `beams` parents are
    drawn (uniformly, with replacement) among the live beams: a parent drawn
    c >= 1 times stays and is forked c - 1 times, a parent never drawn is
    freed.  Sequence ids are assigned in creation order (the prompt is 0)."""
    rng = np.random.default_rng(seed)
    live = [0]
    next_id = 1
    steps = []
    init = [(NEW, prompt_len)]
    for _ in range(beams - 1):
        init.append((FORK, 0))
        live.append(next_id)
        next_id += 1
    ntok = 0
    for s in range(num_steps):
        ops = list(init) if s == 0 else []
        for b in live:
            ops.append((APPEND, b, 1))
            ntok += 1
        decode = list(live)
        picks = rng.integers(0, len(live), size=beams)
        counts = np.bincount(picks, minlength=len(live))
        select, new_live = [], []
        for i, b in enumerate(live):
            if counts[i] == 0:
                select.append((FREE, b))
            else:
                new_live.append(b)
                for _ in range(int(counts[i]) - 1):
                    select.append((FORK, b))
                    new_live.append(next_id)
                    next_id += 1
        steps.append({"ops": ops, "decode": decode, "select": select})
        live = new_live
    prompt_blocks = -(-prompt_len // block_size)
    num_blocks = prompt_blocks + beams * (num_steps // block_size + 2) * 2 + 16
    free_order = _shuffled_free_order(rng, num_blocks)
    return BeamWorkload(name, dtype, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, seed, free_order,
                        prompt_len, beams, steps, ntok)


def beam(small: bool = False) -> BeamWorkload:
    """4 beams over a 2008-token prompt (last block partly filled), 40 steps
    (the reduced twin: 4 beams, 40-token prompt, 24 steps); 32 q / 8 KV heads,
    head_dim 128, block_size 16, bf16."""
    if small:
        return beam_workload("beam-small", 40, 4, 24, 32, 8, 128, 16, "bf16", 2605)
    return beam_workload("beam", 2008, 4, 40, 32, 8, 128, 16, "bf16", 1605)


def prefix_workload(name: str, num_prompts: int, requests_per_prompt: int, system_len: int,
                    suffix_range, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                    dtype: str, seed: int, spare_blocks: int = 64) -> Workload:
    """Requests that share system prompts: each of num_prompts system prompts
    (system_len random token ids) is followed by a per-request random suffix of
    U[suffix_range] tokens; every request then decodes one token.  With prefix
    caching the full blocks of a shared system prompt are stored once
    ("10 PagedAttention" section 2: ten requests with the same 2000-token system
    prompt would otherwise store ten copies).  K/V rows exist for every prompt
    position (in script order) and for each decode token; rows of positions
    that turn out cached are simply not written."""
    rng = np.random.default_rng(seed)
    systems = [rng.integers(0, 32000, size=system_len).astype(np.int32) for _ in range(num_prompts)]
    script: List[Tuple] = []
    lens = []
    ntok = 0
    for r in range(requests_per_prompt):
        for p in range(num_prompts):
            suf = rng.integers(0, 32000, size=int(rng.integers(suffix_range[0], suffix_range[1] + 1)))
            toks = np.concatenate([systems[p], suf.astype(np.int32)])
            script.append((NEW_CACHED, toks))
            lens.append(len(toks) + 1)
            ntok += len(toks)
    for i in range(len(lens)):
        script.append((APPEND, i, 1))
        ntok += 1
    bs = block_size
    # pool: every request's own blocks plus one copy of each system prompt
    per_req = sum(-(-(L) // bs) for L in lens)
    num_blocks = per_req + spare_blocks
    free_order = _shuffled_free_order(rng, num_blocks)
    return Workload(name, dtype, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, seed,
                    free_order, script, np.asarray(lens, dtype=np.int32), ntok,
                    note="%d system prompts x %d requests, system %d tokens, suffix U[%d,%d]"
                         % (num_prompts, requests_per_prompt, system_len, suffix_range[0], suffix_range[1]),
                    extra={"system_len": system_len, "num_prompts": num_prompts,
                           "requests_per_prompt": requests_per_prompt})



def retention_workload(name: str, num_prompts: int, requests_per_prompt: int, system_blocks: int,
                       spare_blocks: int, evict_blocks: int, num_q_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, dtype: str, seed: int) -> Workload:
    """Two waves of requests over a pool with prefix retention switched on
    (the eviction of the hands-on exercise, "10 PagedAttention" section 10 A).

    Wave 1 switches retention on, requests each of num_prompts system prompts
    (system_blocks whole blocks of random token ids) requests_per_prompt times,
    each followed by its own suffix of U[1, B-1] tokens (so every request ends
    in a partly filled block of its own), and frees every request: the system
    prompts' blocks stay registered, the first prompt's released first.

    Wave 2 requests every prompt but the first once (prefix hits), then a
    fresh prompt of whole blocks, as many as the free stack then holds plus
    evict_blocks, so it evicts that many of the first prompt's blocks; the
    fresh request is freed again, the first prompt is requested (it hits the
    blocks it kept) and every live request appends one decode token.

    ``script`` is wave 1 followed by wave 2.  Its K/V rows must be written in
    three phases, ``extra["phases"]`` (ops, rows) each: wave 1; wave 2 up to
    the fresh prompt; the rest.  Within a phase every slot is distinct, but
    blocks the fresh prompt wrote are evicted and written again later in
    wave 2.  ``extra`` also holds the live sequence ids (decode order) and the
    counts the design fixes."""
    assert 0 < evict_blocks <= system_blocks and block_size >= 2
    rng = np.random.default_rng(seed)
    B = block_size
    systems = [rng.integers(0, 32000, size=system_blocks * B).astype(np.int32) for _ in range(num_prompts)]

    def request(p):
        suf = rng.integers(0, 32000, size=int(rng.integers(1, B))).astype(np.int32)
        return np.concatenate([systems[p], suf])

    wave1: List[Tuple] = [(RETAIN, True)]
    rows1 = 0
    for r in range(requests_per_prompt):
        for p in range(num_prompts):
            toks = request(p)
            wave1.append((NEW_CACHED, toks))
            rows1 += len(toks)
    n1 = num_prompts * requests_per_prompt
    wave1 += [(FREE, i) for i in range(n1)]
    # free stack after wave 1: the spare blocks and every request's partly
    # filled block; each later request for a kept prompt takes one of them
    free_after_hits = spare_blocks + n1 - (num_prompts - 1)
    fresh_blocks = free_after_hits + evict_blocks
    wave2: List[Tuple] = []
    prompts2, rows2, lens = [], 0, []
    for p in range(num_prompts - 1, 0, -1):
        toks = request(p)
        wave2.append((NEW_CACHED, toks))
        prompts2.append(toks)
    fresh = rng.integers(0, 32000, size=fresh_blocks * B).astype(np.int32)
    wave2.append((NEW_CACHED, fresh))
    ops2a, rows2a = len(wave2), sum(len(t) for t in prompts2) + len(fresh)
    fresh_id = n1 + num_prompts - 1
    wave2.append((FREE, fresh_id))
    toks0 = request(0)
    wave2.append((NEW_CACHED, toks0))
    prompts2.append(toks0)
    live = list(range(n1, fresh_id)) + [fresh_id + 1]
    for seq in live:
        wave2.append((APPEND, seq, 1))
    rows2 = sum(len(t) for t in prompts2) + len(fresh) + len(live)
    lens = [len(t) + 1 for t in prompts2]
    num_blocks = num_prompts * system_blocks + n1 + spare_blocks
    free_order = _shuffled_free_order(rng, num_blocks)
    return Workload(name, dtype, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, seed, free_order,
                    wave1 + wave2, np.asarray(lens, dtype=np.int32), rows1 + rows2,
                    note="%d prompts of %d blocks x %d requests, then a wave that evicts %d blocks"
                         % (num_prompts, system_blocks, requests_per_prompt, evict_blocks),
                    extra={"phases": [(len(wave1), rows1), (ops2a, rows2a),
                                      (len(wave2) - ops2a, rows2 - rows2a)], "live": live,
                           "evicted_first_prompt": evict_blocks, "fresh_blocks": fresh_blocks,
                           "cached_tokens_first_prompt": (system_blocks - evict_blocks) * B})


def retention(small: bool = False) -> Workload:
    """Prefix retention over two waves: 3 prompts of 8 blocks requested twice,
    4 blocks evicted (the reduced case), or 4 prompts of 2000 tokens requested
    three times, 60 blocks evicted; 32 q / 8 KV heads, head_dim 128,
    block_size 16, bf16."""
    if small:
        return retention_workload("retention-small", 3, 2, 8, 9, 4, 32, 8, 128, 16, "bf16", 2700)
    return retention_workload("retention", 4, 3, 125, 20, 60, 32, 8, 128, 16, "bf16", 1700)

def workload(cfg: str, small: bool = False, block_size: Optional[int] = None,
             prompt_len: Optional[int] = None, placement: str = "random") -> Workload:
    """The named benchmark workload ("cfg0".."cfg4"), or its reduced-size twin.

    ``block_size`` selects 16 or 32 for cfg4; ``prompt_len`` overrides cfg3's
    prompt (2000 as written, 2008 for the copy-on-write variant)."""
    if cfg == "prefix":
        if small:
            return prefix_workload("prefix-small", 2, 3, 200, (1, 40), 32, 8, 128, 16, "bf16", 2600, spare_blocks=8)
        return prefix_workload("prefix", 8, 10, 2000, (16, 512), 32, 8, 128, 16, "bf16", 1600)
    if cfg in ("cfg2-f32", "d256"):
        # The mixed-length batch where only the CUDA-core kernel applies: in
        # fp32 (cfg2's shape), and in bf16 with head_dim 256 (16 query / 8 KV
        # heads, lengths lognormal around 1024).
        f32 = cfg == "cfg2-f32"
        seed = (2700 if small else 1700) + (0 if f32 else 1)
        rng = np.random.default_rng(seed)
        n, median = (20, 160.0) if small else ((256, 512.0) if f32 else (128, 1024.0))
        lens = np.clip(np.rint(np.exp(rng.normal(math.log(median), 1.0, size=n))), 16, 8192).astype(np.int32)
        if small:
            lens = np.concatenate([[1, 15, 16, 17, 33], lens]).astype(np.int32)
        H, D = (32, 128) if f32 else (16, 256)
        return decode_workload(cfg + ("-small" if small else ""), lens, H, 8, D, 16, "f32" if f32 else "bf16", seed,
                               pool_factor=1.1, rng=rng,
                               note="mixed lengths, lognormal(median %d, sigma 1), %s" %
                                    (int(median), "fp32" if f32 else "head_dim 256"))
    k = int(cfg[-1])
    seed = (2500 if small else 1500) + k
    rng = np.random.default_rng(seed)
    if k == 0:
        return decode_workload("cfg0", [5, 16, 23, 40], 4, 4, 64, 4, "f32", seed,
                               num_blocks=32, rng=rng, note="tiny fp32 decode")
    if k == 1:
        if small:
            lens = rng.integers(128, 700, size=6)
        else:
            lens = rng.integers(128, 2049, size=32)
        return decode_workload("cfg1" + ("-small" if small else ""), lens, 32, 32, 128, 16,
                               "bf16", seed, pool_factor=1.25, rng=rng,
                               note="MHA decode, lengths U[128,2048]")
    if k == 2:
        if small:
            body = np.clip(np.rint(np.exp(rng.normal(math.log(160.0), 1.0, size=20))), 16, 1500)
            lens = np.concatenate([[1, 15, 16, 17, 33], body]).astype(np.int32)
        else:
            lens = np.clip(np.rint(np.exp(rng.normal(math.log(512.0), 1.0, size=256))), 16, 8192)
        return decode_workload("cfg2" + ("-small" if small else ""), lens.astype(np.int32), 32, 8,
                               128, 16, "bf16", seed, pool_factor=1.1, rng=rng,
                               note="GQA mixed lengths, lognormal(median 512, sigma 1)")
    if k == 3:
        if prompt_len is None:
            prompt_len = 192 if small else 2000
        if small:
            return sampling_workload("cfg3-small-p%d" % prompt_len, 4, prompt_len, 4, 40, 32, 8,
                                     128, 16, "bf16", seed, spare_blocks=8)
        return sampling_workload("cfg3-p%d" % prompt_len, 64, prompt_len, 4, 256, 32, 8, 128, 16,
                                 "bf16", seed)
    if k == 4:
        bs = block_size or 16
        if small:
            lens = [4096 + 5, 2 * bs + 3]
        else:
            lens = [32768] * 16
        contiguous = placement == "contiguous"
        return decode_workload("cfg4-b%d" % bs + ("-small" if small else "") + ("-contiguous" if contiguous else ""),
                               lens, 64, 8, 128, bs, "bf16", seed, pool_factor=1.05, rng=rng,
                               note="long-context decode, block_size %d%s"
                                    % (bs, ", blocks of each sequence physically contiguous" if contiguous else ""),
                               placement=placement)
    raise ValueError("unknown workload %r" % cfg)


# ---------------------------------------------------------------- values
def torch_dtype(dtype: str):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _randn(shape, dtype: str, gen, device, chunk_elems: int = 1 << 27):
    """N(0,1) fp32 draws cast to the element type, produced in chunks."""
    import torch
    out = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    flat = out.view(-1)
    total = flat.numel()
    start = 0
    while start < total:
        n = min(chunk_elems, total - start)
        flat[start:start + n].copy_(torch.randn(n, generator=gen, device=device, dtype=torch.float32))
        start += n
    return out


def make_values(wl, device="cpu"):
    """Random tensors for one step: q [N,H,D], k/v new rows [T,Hk,D] and the
    pool caches [NB,B,Hk,D], all N(0,1) in the workload's element type.  For a
    beam-search workload q holds one row per (step, decoded beam) in order."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    cache_shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    k_cache = _randn(cache_shape, wl.dtype, gen, device)
    v_cache = _randn(cache_shape, wl.dtype, gen, device)
    nq = sum(len(s["decode"]) for s in wl.steps) if isinstance(wl, BeamWorkload) else wl.num_seqs
    q = _randn((nq, wl.num_q_heads, wl.head_dim), wl.dtype, gen, device)
    k_new = _randn((wl.num_new_tokens, wl.num_kv_heads, wl.head_dim), wl.dtype, gen, device)
    v_new = _randn((wl.num_new_tokens, wl.num_kv_heads, wl.head_dim), wl.dtype, gen, device)
    return {"q": q, "k": k_new, "v": v_new, "k_cache": k_cache, "v_cache": v_cache}


def to_numpy_elems(t):
    """Host numpy view of a tensor's elements: float32, or uint16 bits for bf16."""
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def shard_sequences(seq_bytes, world_size: int):
    """Greedy longest-first split of sequences over ranks by their KV bytes.

    Returns a list (one per rank) of sequence index arrays.  Ranks share no
    sequence, and every sequence goes to exactly one rank."""
    seq_bytes = np.asarray(seq_bytes, dtype=np.int64)
    order = np.argsort(-seq_bytes, kind="stable")
    loads = np.zeros(world_size, dtype=np.int64)
    parts: List[list] = [[] for _ in range(world_size)]
    for i in order:
        r = int(np.argmin(loads))
        parts[r].append(int(i))
        loads[r] += seq_bytes[i]
    return [np.asarray(sorted(p), dtype=np.int64) for p in parts]


def to_split_layout(k_cache, v_cache):
    """The same cache contents in the split layout: K [NB, Hk, D/x, B, x] and
    V [NB, Hk, D, B], x = 16 / element bytes (a reshape/permute of the random
    values, for workloads run in that layout)."""
    nb, bs, hk, d = k_cache.shape
    x = 16 // k_cache.element_size()
    k = k_cache.view(nb, bs, hk, d // x, x).permute(0, 2, 3, 1, 4).contiguous()
    v = v_cache.permute(0, 2, 3, 1).contiguous()
    return k, v


def request_stream(seed: int, num_requests: int, rate: float, prompt_median: float = 256.0,
                   output_median: float = 128.0, sigma: float = 1.0, max_prompt: int = 2048,
                   max_new_tokens: int = 2048):
    """A synthetic serving stream: Poisson arrivals (``rate`` requests per
    decode step), lognormal prompt and output lengths (given medians, shape
    sigma), clipped to [1, max_prompt] and [1, max_new_tokens].  Returns
    int32 arrays (arrival_step non-decreasing, prompt_len, output_len)."""
    rng = np.random.default_rng(seed)
    gaps = rng.exponential(1.0 / rate, size=num_requests)
    arrival = np.floor(np.cumsum(gaps)).astype(np.int32)
    prompt = np.clip(np.rint(np.exp(rng.normal(math.log(prompt_median), sigma, size=num_requests))), 1, max_prompt)
    output = np.clip(np.rint(np.exp(rng.normal(math.log(output_median), sigma, size=num_requests))), 1,
                     max_new_tokens)
    return arrival, prompt.astype(np.int32), output.astype(np.int32)
