"""Paged-KV decode attention for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libpa.so`` (hand-written CUDA, see
include/pa.h).  This package only marshals arguments to it: tensors must
already live on the GPU, and every call runs on torch's current stream.  The
library is loaded on first use; a missing library raises, there is no
fallback.

Calls (same names as the C ABI):
  pa_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache)
  pa_copy_blocks(k_cache, v_cache, src_dst_pairs)
  pa_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, ...)
  pa_get_device_error()
  BlockManager: the host block manager (free list, refcounts, fork,
  copy-on-write, slot mapping).
"""
import ctypes

import numpy as np

from . import _lib
from ._lib import (PA_BF16, PA_F32, PA_KERNEL_AUTO, PA_KERNEL_MMA, PA_KERNEL_SIMT, PA_OK,
                   PagedAttentionError)

_KERNELS = {"auto": PA_KERNEL_AUTO, "simt": PA_KERNEL_SIMT, "mma": PA_KERNEL_MMA}


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError("element type must be float32 or bfloat16, got %s" % t.dtype)


def _cache_desc(k_cache, v_cache):
    """Descriptor read off the cache shapes: K and V [NB, B, Hk, D] (row
    layout) or K [NB, Hk, D/x, B, x] with V [NB, Hk, D, B] (split layout,
    x = 16 / element bytes)."""
    if k_cache.dtype != v_cache.dtype:
        raise TypeError("k_cache and v_cache element types differ")
    if k_cache.dim() == 4 and v_cache.shape == k_cache.shape:
        nb, bs, hk, d = k_cache.shape
        return _lib.CacheDesc(nb, bs, hk, d, _dtype_code(k_cache), _lib.PA_LAYOUT_ROW)
    if k_cache.dim() == 5 and v_cache.dim() == 4:
        nb, hk, dx, bs, x = k_cache.shape
        if x * k_cache.element_size() == 16 and tuple(v_cache.shape) == (nb, hk, dx * x, bs):
            return _lib.CacheDesc(nb, bs, hk, dx * x, _dtype_code(k_cache), _lib.PA_LAYOUT_SPLIT)
    raise ValueError("caches must be K, V [num_blocks, block_size, num_kv_heads, head_dim], or "
                     "K [num_blocks, num_kv_heads, head_dim/x, block_size, x] with "
                     "V [num_blocks, num_kv_heads, head_dim, block_size], x = 16 / element bytes")


def _current_device():
    """Index of torch's current CUDA device: the library enqueues on that
    device's current stream and looks up its per-device state there."""
    return _torch().cuda.current_device()


def _dev(t, name, dtype=None, device=None):
    """Device pointer of contiguous CUDA tensor ``t``.  ``device``: the index
    the tensor must be on (the current device; the library works there, so a
    tensor on another GPU would be read through a foreign pointer)."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device.index != device:
        raise ValueError("%s is on cuda:%s but the current device is cuda:%d: make its device current "
                         "(torch.cuda.device) before the call" % (name, t.device.index, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    """torch's current stream on the current device, as a cudaStream_t.  The
    raw getter returns the same handle as current_stream().cuda_stream
    without building a Stream object (about 3 us of host time per call)."""
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return ctypes.c_void_p(raw(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def pa_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache):
    """Write new tokens' K/V rows into the paged caches at their slots."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache)
    T = k.shape[0]
    if k.shape != v.shape or tuple(k.shape[1:]) != (desc.num_kv_heads, desc.head_dim):
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim] matching the cache")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    for name, t in (("k", k), ("v", v)):
        if t.dtype != k_cache.dtype:
            raise TypeError("%s element type differs from the cache" % name)
    d = _current_device()
    st = _lib.load().pa_reshape_and_cache(
        _dev(k, "k", device=d), _dev(v, "v", device=d), _dev(slot_mapping, "slot_mapping", torch.int32, d), T,
        _dev(k_cache, "k_cache", device=d), _dev(v_cache, "v_cache", device=d), ctypes.byref(desc), _stream())
    _lib.check("pa_reshape_and_cache", st)


def pa_copy_blocks(k_cache, v_cache, src_dst_pairs):
    """Copy whole blocks: for each (src, dst) row of the int32 [P, 2] tensor."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache)
    pairs = src_dst_pairs.reshape(-1, 2) if src_dst_pairs.numel() else src_dst_pairs
    P = pairs.shape[0] if pairs.numel() else 0
    if P == 0:
        return
    d = _current_device()
    st = _lib.load().pa_copy_blocks(_dev(k_cache, "k_cache", device=d), _dev(v_cache, "v_cache", device=d),
                                    ctypes.byref(desc), _dev(pairs, "src_dst_pairs", torch.int32, d), P,
                                    _stream())
    _lib.check("pa_copy_blocks", st)


def _opts(num_splits, kernel, events, shared_plan=None, device=None):
    o = _lib.DecodeOpts(int(num_splits), _KERNELS[kernel], None, None, None)
    if shared_plan is not None:
        o.shared_plan = _dev(shared_plan, "shared_plan", _torch().int32, device).value
    if events is not None:
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event on its first record
                e.record()
        o.ev_partial_begin = ctypes.c_void_p(events[0].cuda_event)
        o.ev_partial_end = ctypes.c_void_p(events[1].cuda_event)
    return o


def _set_host_lens(o, host_seq_lens, num_seqs):
    """Put the host-lengths hint into options ``o``; returns the int32 array,
    which the caller keeps alive until the call returns (or None)."""
    if host_seq_lens is None:
        return None
    host_lens = np.ascontiguousarray(np.asarray(host_seq_lens, dtype=np.int32))
    if host_lens.shape != (int(num_seqs),):
        raise ValueError("host_seq_lens must be [num_seqs]")
    o.host_seq_lens = host_lens.ctypes.data
    return host_lens


def _cache_desc_from_k(k_cache):
    """Descriptor from the K cache alone (its shape fixes the layout)."""
    if k_cache.dim() == 5:
        nb, hk, dx, bs, x = k_cache.shape
        return _cache_desc(k_cache, k_cache.new_empty((nb, hk, dx * x, bs)))
    return _cache_desc(k_cache, k_cache)


def pa_decode_workspace_bytes(k_cache, num_seqs, num_heads, num_splits=0, kernel="auto", shared=False):
    """Workspace bytes of pa_decode; ``shared`` sizes it for a call with a
    shared-prefix plan."""
    desc = _cache_desc_from_k(k_cache)
    o = _opts(num_splits, kernel, None)
    if shared:
        o.shared_plan = ctypes.c_void_p(1)  # only tested for NULL when sizing
    n = _lib.load().pa_decode_workspace_bytes(ctypes.byref(desc), int(num_seqs), int(num_heads),
                                              ctypes.byref(o))
    if n == 0:
        raise PagedAttentionError("pa_decode_workspace_bytes", _lib.PA_ERR_UNSUPPORTED)
    return int(n)


def pa_decode_launch_count(k_cache, num_seqs, num_heads, max_blocks_per_seq, num_splits=0, kernel="auto",
                           shared=False, host_seq_lens=None):
    """Kernels one pa_decode call with these arguments launches (plan kernel,
    attention kernel and the merge kernels its options bring in)."""
    desc = _cache_desc_from_k(k_cache)
    o = _opts(num_splits, kernel, None)
    if shared:
        o.shared_plan = ctypes.c_void_p(1)  # only tested for NULL here
    host_lens = _set_host_lens(o, host_seq_lens, num_seqs)  # noqa: F841 (alive for the call)
    n = _lib.load().pa_decode_launch_count(ctypes.byref(desc), int(num_seqs), int(num_heads),
                                           int(max_blocks_per_seq), ctypes.byref(o))
    if n < 0:
        raise PagedAttentionError("pa_decode_launch_count", n)
    return int(n)


def pa_decode_default_splits(k_cache, num_heads, kernel="auto"):
    desc = _cache_desc_from_k(k_cache)
    o = _opts(0, kernel, None)
    n = _lib.load().pa_decode_default_splits(ctypes.byref(desc), int(num_heads), ctypes.byref(o))
    if n < 0:
        raise PagedAttentionError("pa_decode_default_splits", n)
    return int(n)


def pa_decode_shared_tc(k_cache, num_seqs, num_heads, shared_plan, num_splits=0):
    """True when pa_decode with this device plan would run its 64-row shared
    passes on tcgen05 (host-side choice; plans of 16 or 32 rows per pass run
    on mma.sync whatever this says)."""
    desc = _cache_desc_from_k(k_cache)
    o = _opts(num_splits, "auto", None, shared_plan, _current_device())
    n = _lib.load().pa_decode_shared_tc(ctypes.byref(desc), int(num_seqs), int(num_heads), ctypes.byref(o))
    if n < 0:
        raise PagedAttentionError("pa_decode_shared_tc", n)
    return n == 1


def pa_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, out=None, workspace=None,
              num_splits=0, kernel="auto", events=None, shared_plan=None, host_seq_lens=None):
    """Decode attention through block tables; returns ``out`` [N, H, D].

    ``events``: optional (begin, end) torch.cuda.Event pair recorded around the
    attention kernel on the current stream.  ``shared_plan``: optional device
    int32 tensor from shared_prefix_plan (built from the same tables and
    lengths), so that blocks shared by several sequences are read once.
    ``host_seq_lens``: optional host copy of seq_lens (numpy or CPU tensor), a
    hint that lets long contexts be merged across the GPU; the results do
    not depend on it."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache)
    N, H, D = q.shape
    if D != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [num_seqs, num_heads, head_dim] in the cache's element type")
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.shape != (N,):
        raise ValueError("block_tables must be [num_seqs, max_blocks] and seq_lens [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    d = _current_device()
    o = _opts(num_splits, kernel, events, shared_plan, d)
    host_lens = _set_host_lens(o, host_seq_lens, N)  # noqa: F841 (alive for the call)
    lib = _lib.load()
    if workspace is None:  # a caller's workspace is checked by the library (PA_ERR_WORKSPACE)
        need = lib.pa_decode_workspace_bytes(ctypes.byref(desc), N, H, ctypes.byref(o))
        if need == 0:
            raise PagedAttentionError("pa_decode_workspace_bytes", _lib.PA_ERR_UNSUPPORTED)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.pa_decode(_dev(out, "out", device=d), _dev(q, "q", device=d), _dev(k_cache, "k_cache", device=d),
                       _dev(v_cache, "v_cache", device=d), ctypes.byref(desc),
                       _dev(block_tables, "block_tables", torch.int32, d), block_tables.shape[1],
                       _dev(seq_lens, "seq_lens", torch.int32, d), N, H, float(scale),
                       _dev(workspace, "workspace", device=d), workspace.numel(), ctypes.byref(o), _stream())
    _lib.check("pa_decode", st)
    return out


def shared_prefix_plan(block_tables, seq_lens, block_size, num_heads, num_kv_heads, min_shared_blocks=1):
    """Shared-prefix plan of one batch from HOST tables [N, max_blocks] and
    lengths [N] (numpy or CPU tensors): sequences whose tables start with the
    same physical blocks, and their common prefix.  Returns (plan, info):
    plan is a CPU int32 tensor to copy to the device and pass to pa_decode
    as ``shared_plan``; info is a dict (num_groups, num_members,
    shared_blocks, saved_blocks)."""
    torch = _torch()
    t = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    L = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if t.ndim != 2 or L.shape != (t.shape[0],):
        raise ValueError("block_tables must be [num_seqs, max_blocks] and seq_lens [num_seqs]")
    lib = _lib.load()
    n = int(lib.pa_shared_plan_ints(t.shape[0]))
    plan = np.zeros(n, dtype=np.int32)
    info = _lib.SharedPlanInfo()
    st = lib.pa_shared_plan_build(_i32p(t), t.shape[1], _i32p(L), t.shape[0], int(block_size), int(num_heads),
                                  int(num_kv_heads), int(min_shared_blocks), _i32p(plan), n, ctypes.byref(info))
    _lib.check("pa_shared_plan_build", st)
    return torch.from_numpy(plan), {"num_groups": info.num_groups, "num_members": info.num_members,
                                    "shared_blocks": info.shared_blocks, "saved_blocks": info.saved_blocks}


def pa_decode_no_alloc(q, k_cache, v_cache, block_tables, seq_lens, scale, out, num_splits=0, kernel="auto",
                       host_seq_lens=None):
    """pa_decode without a workspace argument, for callers that cannot allocate
    device memory (a pool that took all free memory at startup, a framework
    that owns the allocator, a loop that cannot afford cudaMalloc's implicit
    synchronisation).  Its scratch is a fixed array of
    PA_NO_ALLOC_SCRATCH_BYTES inside the library, shared by every call on a
    device; calls that can overlap on the GPU race on it.  ``out`` is
    required: this path allocates nothing.  ``host_seq_lens`` as in
    pa_decode."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache)
    N, H, D = q.shape
    if D != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [num_seqs, num_heads, head_dim] in the cache's element type")
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.shape != (N,):
        raise ValueError("block_tables must be [num_seqs, max_blocks] and seq_lens [num_seqs]")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    d = _current_device()
    o = _opts(num_splits, kernel, None)
    host_lens = _set_host_lens(o, host_seq_lens, N)  # noqa: F841 (alive for the call)
    st = _lib.load().pa_decode_no_alloc(
        _dev(out, "out", device=d), _dev(q, "q", device=d), _dev(k_cache, "k_cache", device=d),
        _dev(v_cache, "v_cache", device=d), ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32, d),
        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32, d), N, H, float(scale), ctypes.byref(o),
        _stream())
    _lib.check("pa_decode_no_alloc", st)
    return out


def pa_get_device_error(raise_on_error=True):
    """Synchronise the current stream and read/clear the device error word."""
    st = _lib.load().pa_get_device_error(_stream())
    if raise_on_error:
        _lib.check("kernel", st)
    return st


def pa_selftest_wait_timeout(limit_ns):
    """Launch the bounded-wait self-test kernel (its wait runs out by design)."""
    _lib.check("pa_selftest_wait_timeout", _lib.load().pa_selftest_wait_timeout(int(limit_ns), _stream()))


def pa_split_range(total_blocks, num_splits, c):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    _lib.load().pa_split_range(int(total_blocks), int(num_splits), int(c), ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def pa_split_owner(total_blocks, num_splits, x):
    return int(_lib.load().pa_split_owner(int(total_blocks), int(num_splits), int(x)))


def _i32p(arr):
    return arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class BlockManager:
    """Host block manager (C++ in libpa.so)."""

    def __init__(self, num_blocks, block_size, free_order=None):
        lib = _lib.load()
        self._lib = lib
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if free_order is None:
            h = lib.pa_bm_create(self.num_blocks, self.block_size, None)
        else:
            fo = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
            if fo.shape != (self.num_blocks,):
                raise ValueError("free_order must hold num_blocks ids")
            h = lib.pa_bm_create(self.num_blocks, self.block_size, _i32p(fo))
        if not h:
            raise ValueError("pa_bm_create rejected its arguments")
        self._h = ctypes.c_void_p(h)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pa_bm_destroy(h)
            self._h = None

    def _call(self, name, *args):
        st = getattr(self._lib, name)(self._h, *args)
        _lib.check(name, st)

    def new_seq(self, num_tokens):
        s = ctypes.c_int32()
        self._call("pa_bm_new_seq", int(num_tokens), ctypes.byref(s))
        return s.value

    def new_seq_cached(self, token_ids):
        """Prompt with prefix caching: (seq, cached_tokens); positions below
        cached_tokens already have K/V in shared blocks."""
        toks = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        s, c = ctypes.c_int32(), ctypes.c_int32()
        self._call("pa_bm_new_seq_cached", _i32p(toks), toks.shape[0], ctypes.byref(s), ctypes.byref(c))
        return s.value, c.value

    def slots(self, seq, first_pos, count):
        out = np.empty(max(int(count), 1), dtype=np.int32)
        self._call("pa_bm_slots", int(seq), int(first_pos), int(count), _i32p(out))
        return out[:int(count)]

    def set_prefix_retention(self, on=True):
        """Keep prefix-cached blocks registered when their refcount reaches 0
        (evictable, least recently released evicted first) instead of freeing
        them; off turns the evictable blocks into free ones."""
        self._call("pa_bm_set_prefix_retention", 1 if on else 0)

    def evictable(self):
        """Number of retained blocks at refcount 0."""
        n = ctypes.c_int32()
        self._call("pa_bm_evictable", ctypes.byref(n))
        return n.value

    def cache_stats(self):
        """(registered blocks, block hits, block lookups) of the prefix cache."""
        n, h, l = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
        self._call("pa_bm_cache_stats", ctypes.byref(n), ctypes.byref(h), ctypes.byref(l))
        return n.value, h.value, l.value

    def fork(self, parent):
        s = ctypes.c_int32()
        self._call("pa_bm_fork", int(parent), ctypes.byref(s))
        return s.value

    def free_seq(self, seq):
        self._call("pa_bm_free_seq", int(seq))

    def append_token(self, seq):
        slot, src, dst = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._call("pa_bm_append_token", int(seq), ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_tokens(self, seq, count):
        slots = np.empty(max(int(count), 1), dtype=np.int32)
        pair = np.full(2, -1, dtype=np.int32)
        npairs = ctypes.c_int32()
        self._call("pa_bm_append_tokens", int(seq), int(count), _i32p(slots), _i32p(pair), ctypes.byref(npairs))
        return slots[:int(count)], (tuple(int(x) for x in pair) if npairs.value else None)

    def seq_len(self, seq):
        n, nb = ctypes.c_int32(), ctypes.c_int32()
        self._call("pa_bm_seq_len", int(seq), ctypes.byref(n), ctypes.byref(nb))
        return n.value

    def block_table(self, seq):
        n, nb = ctypes.c_int32(), ctypes.c_int32()
        self._call("pa_bm_seq_len", int(seq), ctypes.byref(n), ctypes.byref(nb))
        out = np.empty(max(nb.value, 1), dtype=np.int32)
        ln = ctypes.c_int32()
        self._call("pa_bm_block_table", int(seq), _i32p(out), out.shape[0], ctypes.byref(ln))
        return out[:ln.value].tolist()

    def physical_index(self, seq, pos):
        s = ctypes.c_int32()
        self._call("pa_bm_physical_index", int(seq), int(pos), ctypes.byref(s))
        return s.value

    def refcount(self, block):
        r = ctypes.c_int32()
        self._call("pa_bm_refcount", int(block), ctypes.byref(r))
        return r.value

    def stats(self):
        """(free, used, shared) block counts."""
        f, u, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._call("pa_bm_stats", ctypes.byref(f), ctypes.byref(u), ctypes.byref(s))
        return f.value, u.value, s.value

    def export(self, seqs, max_blocks):
        """(tables int32 [n, max_blocks] padded with -1, lens int32 [n])."""
        seqs = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = seqs.shape[0]
        tables = np.empty((max(n, 1), max(int(max_blocks), 1)), dtype=np.int32)
        lens = np.empty(max(n, 1), dtype=np.int32)
        self._call("pa_bm_export", _i32p(seqs), n, int(max_blocks), _i32p(tables), _i32p(lens))
        return tables[:n], lens[:n]

    def apply_script(self, script):
        """Run a workload script ("new", tokens) / ("new_cached", token_ids) /
        ("fork", parent) / ("free", seq) / ("append", seq, count) /
        ("retain", on).  Returns (slots int32 [T], pairs int32 [P, 2]), slots
        in script order and pairs in the order they were made."""
        slots, pairs = [], []
        for op in script:
            if op[0] == "new":
                self.new_seq(op[1])
            elif op[0] == "new_cached":
                # every prompt position has a K/V row; cached positions get
                # slot -1 (padding: the cache write skips them)
                seq, cached = self.new_seq_cached(op[1])
                n = len(op[1])
                s = np.full(n, -1, dtype=np.int32)
                s[cached:] = self.slots(seq, cached, n - cached)
                slots.append(s)
            elif op[0] == "fork":
                self.fork(op[1])
            elif op[0] == "free":
                self.free_seq(op[1])
            elif op[0] == "retain":
                self.set_prefix_retention(op[1])
            elif op[0] == "append":
                s, pair = self.append_tokens(op[1], op[2])
                slots.append(s)
                if pair is not None:
                    pairs.append(pair)
            else:
                raise ValueError("unknown op %r" % (op,))
        slots = np.concatenate(slots).astype(np.int32) if slots else np.zeros(0, np.int32)
        return slots, np.asarray(pairs, dtype=np.int32).reshape(-1, 2)



def sampling_memory(prompt_len, gen_lens, block_size=16):
    """Parallel sampling of len(gen_lens) completions from one prompt, with and
    without block sharing (hands-on exercise E of "10 PagedAttention"
    (PidokuInfra); the sharing of its section 5 "Copy-on-write sharing").

    Shared: one sequence holds the prompt, the other samples fork it, and
    each sample in turn appends its generated tokens (a write into a shared,
    partly filled block copies it first).  Unshared: every sample holds its
    own copy of the prompt.  Returns the blocks each way holds at the end,
    the fraction sharing saves and the copy-on-write copies it made."""
    gen_lens = [int(g) for g in gen_lens]
    B = int(block_size)
    n = len(gen_lens)
    if n == 0 or prompt_len < 0 or min(gen_lens) < 0:
        raise ValueError("need at least one sample and non-negative lengths")
    pool = sum(-(-(prompt_len + g) // B) for g in gen_lens) + 1
    shared = BlockManager(pool, B)
    root = shared.new_seq(prompt_len)
    seqs = [root] + [shared.fork(root) for _ in range(n - 1)]
    copies = 0
    for seq, g in zip(seqs, gen_lens):
        if g:
            copies += shared.append_tokens(seq, g)[1] is not None
    alone = BlockManager(pool, B)
    for g in gen_lens:
        seq = alone.new_seq(prompt_len)
        if g:
            alone.append_tokens(seq, g)
    used_shared, used_alone = shared.stats()[1], alone.stats()[1]
    return {"shared_blocks": used_shared, "unshared_blocks": used_alone,
            "saved_fraction": 1.0 - used_shared / used_alone if used_alone else 0.0, "copies": copies}

def simulate(policy, arrival_step, prompt_len, output_len, total_slots, block_size=16, max_new_tokens=2048,
             max_steps=10 ** 7):
    """Run the host allocation simulator (pa_sim_run): policy "contiguous"
    (max-length reservation) or "paged".  Returns a dict of its totals."""
    a = np.ascontiguousarray(np.asarray(arrival_step, dtype=np.int32))
    p = np.ascontiguousarray(np.asarray(prompt_len, dtype=np.int32))
    o = np.ascontiguousarray(np.asarray(output_len, dtype=np.int32))
    cfg = _lib.SimConfig(1 if policy == "paged" else 0, int(block_size), int(max_new_tokens), int(max_steps),
                         int(total_slots))
    res = _lib.SimResult()
    _lib.check("pa_sim_run", _lib.load().pa_sim_run(ctypes.byref(cfg), _i32p(a), _i32p(p), _i32p(o), a.shape[0],
                                                    ctypes.byref(res)))
    return {name: getattr(res, name) for name, _ in _lib.SimResult._fields_}


def version():
    return _lib.load().pa_version().decode()


__all__ = [
    "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_decode_workspace_bytes", "pa_decode_no_alloc",
    "pa_decode_default_splits", "pa_decode_shared_tc", "pa_decode_launch_count", "pa_get_device_error", "pa_selftest_wait_timeout",
    "pa_split_range", "pa_split_owner",
    "BlockManager", "PagedAttentionError", "sampling_memory", "simulate", "version",
]
