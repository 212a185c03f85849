"""The C-ABI library loads, exports every symbol include/pa.h declares, and
validates host-visible arguments without touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, "binding lacks a signature for %s" % n


def test_status_strings_and_version(lib):
    assert lib.pa_status_string(0) == b"ok"
    assert b"workspace" in lib.pa_status_string(-7)
    names = [lib.pa_status_string(c) for c in range(0, -10, -1)]
    assert len(set(names)) == 10 and b"unknown status" not in names  # every code, PA_ERR_HOST_MEMORY included
    assert lib.pa_status_string(-10) == b"unknown status"
    assert b"sm_103a" in lib.pa_version()


def _desc(nb=8, bs=16, hk=8, d=128, dt=_lib.PA_BF16):
    return _lib.CacheDesc(nb, bs, hk, d, dt)


def _gpu_present():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001 (no torch or no driver: no GPU)
        return False


def test_host_validation_rejects_bad_arguments_without_a_gpu(lib):
    """Host checks that come before any CUDA call.  Device pointers are None
    except where the check under test needs a non-null one; those few cases
    pass a non-null address that is never dereferenced and therefore run only
    where no GPU is present (a regressed check then fails to find a device
    instead of launching)."""
    d = _desc()
    # null pointers / negative sizes / bad descriptors are caught before any CUDA call
    assert lib.pa_reshape_and_cache(None, None, None, 4, None, None, ctypes.byref(d), None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(None, None, None, -1, None, None, ctypes.byref(d), None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(None, None, None, 0, None, None, ctypes.byref(d), None) == _lib.PA_OK
    assert lib.pa_copy_blocks(None, None, ctypes.byref(d), None, 0, None) == _lib.PA_OK
    assert lib.pa_copy_blocks(None, None, ctypes.byref(d), None, 3, None) == _lib.PA_ERR_INVALID_ARG
    bad = _desc(dt=7)
    assert lib.pa_copy_blocks(None, None, ctypes.byref(bad), None, 1, None) == _lib.PA_ERR_INVALID_ARG
    big = _desc(nb=1 << 28, bs=16)
    assert lib.pa_copy_blocks(None, None, ctypes.byref(big), None, 1, None) == _lib.PA_ERR_INVALID_ARG
    o = _lib.DecodeOpts(4, _lib.PA_KERNEL_AUTO, None, None)
    # H not a multiple of Hk, group above 8, unsupported head_dim: the plan is made first
    args = (None, None, None, None)
    assert lib.pa_decode(*args, ctypes.byref(d), None, 4, None, 2, 12, 1.0, None, 1 << 20, ctypes.byref(o),
                         None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_decode(*args, ctypes.byref(d), None, 4, None, 2, 128, 1.0, None, 1 << 20, ctypes.byref(o),
                         None) == _lib.PA_ERR_UNSUPPORTED
    d96 = _desc(d=96)
    assert lib.pa_decode(*args, ctypes.byref(d96), None, 4, None, 2, 32, 1.0, None, 1 << 20, ctypes.byref(o),
                         None) == _lib.PA_ERR_UNSUPPORTED
    # the tensor-core kernel needs bf16 and a block size multiple of 16
    d32 = _desc(dt=_lib.PA_F32, d=64)
    om = _lib.DecodeOpts(4, _lib.PA_KERNEL_MMA, None, None)
    assert lib.pa_decode(*args, ctypes.byref(d32), None, 4, None, 2, 32, 1.0, None, 1 << 20, ctypes.byref(om),
                         None) == _lib.PA_ERR_UNSUPPORTED
    # null workspace; zero sequences is a no-op
    assert lib.pa_decode(*args, ctypes.byref(d), None, 4, None, 2, 32, 1.0, None, 1 << 20, ctypes.byref(o),
                         None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_decode(*args, ctypes.byref(d), None, 4, None, 0, 32, 1.0, None, 1 << 20, ctypes.byref(o),
                         None) == _lib.PA_OK
    if _gpu_present():
        return  # the checks below need non-null device pointers
    p = ctypes.c_void_p(0x1000)
    # workspace too small, misaligned workspace
    assert lib.pa_decode(p, p, p, p, ctypes.byref(d), p, 4, p, 2, 32, 1.0, p, 16, ctypes.byref(o),
                         None) == _lib.PA_ERR_WORKSPACE
    assert lib.pa_decode(p, p, p, p, ctypes.byref(d), p, 4, p, 2, 32, 1.0, ctypes.c_void_p(0x1010),
                         1 << 20, ctypes.byref(o), None) == _lib.PA_ERR_INVALID_ARG


def test_workspace_size_follows_the_split_count(lib):
    d = _desc()
    sizes = []
    for c in (1, 152, 304):
        o = _lib.DecodeOpts(c, _lib.PA_KERNEL_MMA, None, None)
        sizes.append(lib.pa_decode_workspace_bytes(ctypes.byref(d), 256, 32, ctypes.byref(o)))
    assert sizes[0] < sizes[1] < sizes[2]
    # Documented layout: pieces for (C + NG*N) slots of HPG heads x (D + 2)
    # floats, plus lengths, prefix sums and counters.  Tensor-core kernel:
    # NH = 4 KV heads per CTA for Hk = 8, so NG = 2 groups of HPG = 16 heads.
    o = _lib.DecodeOpts(152, _lib.PA_KERNEL_MMA, None, None)
    n = lib.pa_decode_workspace_bytes(ctypes.byref(d), 256, 32, ctypes.byref(o))
    pieces = (152 + 2 * 256) * 16 * 130 * 4
    assert pieces <= n < pieces + 4 * (256 + 257 + 256 * 8) + 4 * 256


def test_split_covers_every_block_once(lib):
    rng = np.random.default_rng(0)
    for W, C in [(1, 1), (10, 3), (7, 20), (13264, 152), (32768, 152), (1 << 20, 1000)]:
        begins = [pa.pa_split_range(W, C, c) for c in range(C)]
        assert begins[0][0] == 0 and begins[-1][1] == W
        for c in range(1, C):
            assert begins[c][0] == begins[c - 1][1]
        for x in rng.integers(0, W, size=50).tolist() + [0, W - 1]:
            c = pa.pa_split_owner(W, C, x)
            b, e = begins[c]
            assert b <= x < e


def test_partial_slots_are_unique():
    # slot = c + (flattened sequence); check with random ragged sequences
    import paged_kv_cache_150_gb300 as pa

    rng = np.random.default_rng(1)
    for _ in range(20):
        nb = rng.integers(0, 9, size=int(rng.integers(1, 30)))
        cu = np.concatenate([[0], np.cumsum(nb)])
        W = int(cu[-1])
        if W == 0:
            continue
        C = int(rng.integers(1, 40))
        seen = set()
        for c in range(C):
            b, e = pa.pa_split_range(W, C, c)
            for x in range(b, e):
                seq = int(np.searchsorted(cu, x, side="right") - 1)
                seen.add((c, seq))
        slots = [c + s for c, s in seen]
        assert len(slots) == len(set(slots))
        assert max(slots) < C + len(nb)


def test_reduce_visits_exactly_the_ctas_holding_a_piece():
    # The reduce walks CTAs split_owner(first block) .. split_owner(last block)
    # and skips empty ranges; that set must equal the owners of the blocks,
    # also when there are more CTAs than blocks.
    rng = np.random.default_rng(2)
    for _ in range(200):
        nb = rng.integers(0, 6, size=int(rng.integers(1, 12)))
        W = int(nb.sum())
        if W == 0:
            continue
        C = int(rng.integers(1, 60))
        cu = np.concatenate([[0], np.cumsum(nb)])
        for i in range(len(nb)):
            if nb[i] == 0:
                continue
            c0 = pa.pa_split_owner(W, C, int(cu[i]))
            c1 = pa.pa_split_owner(W, C, int(cu[i + 1] - 1))
            visited = {c for c in range(c0, c1 + 1) if pa.pa_split_range(W, C, c)[0] < pa.pa_split_range(W, C, c)[1]}
            owners = {pa.pa_split_owner(W, C, x) for x in range(int(cu[i]), int(cu[i + 1]))}
            assert visited == owners


def test_launch_count_with_host_lengths_follows_the_split(lib):
    """Host-only (the split count is given, so no occupancy query): with a
    host copy of the lengths, pa_decode_launch_count is 3 exactly when some
    (head group, sequence) overlaps 8 or more of the split's CTA ranges
    (counted here over the ranges pa_split_range returns), else 2; the
    CUDA-core kernel and a shared-prefix plan never bring in that merge."""
    d = _desc()
    rng = np.random.default_rng(5)
    NH, NG, B, max_blocks = 4, 2, 16, 4096
    for trial in range(60):
        N = int(rng.integers(1, 40))
        C = int(rng.choice([7, 64, 152, 304]))
        lens = rng.integers(0, 3000, size=N)
        if trial % 3 == 0:
            lens[rng.integers(0, N)] = int(rng.integers(10000, max_blocks * B))
        if trial % 7 == 0:
            lens[rng.integers(0, N)] = max_blocks * B + 5  # out of range: counts as 0
        lens = np.ascontiguousarray(lens, np.int32)
        nb = [0 if (L < 0 or L > max_blocks * B) else -(-int(L) // B) for L in lens]
        cu = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
        Wg = int(cu[-1])
        W = NG * Wg
        expect = 2
        if W > 0:
            Ce = min(C, W)
            ranges = [pa.pa_split_range(W, Ce, c) for c in range(Ce)]
            for g in range(NG):
                for i in range(N):
                    if nb[i] == 0:
                        continue
                    a, b = g * Wg + int(cu[i]), g * Wg + int(cu[i + 1])
                    if sum(1 for lo, hi in ranges if lo < b and a < hi) >= 8:
                        expect = 3
        o = _lib.DecodeOpts(C, _lib.PA_KERNEL_MMA, None, None, None, lens.ctypes.data)
        assert lib.pa_decode_launch_count(ctypes.byref(d), N, 32, max_blocks, ctypes.byref(o)) == expect
        o_simt = _lib.DecodeOpts(C, _lib.PA_KERNEL_SIMT, None, None, None, lens.ctypes.data)
        assert lib.pa_decode_launch_count(ctypes.byref(d), N, 32, max_blocks, ctypes.byref(o_simt)) == 2
        if C >= 2:
            o_plan = _lib.DecodeOpts(C, _lib.PA_KERNEL_MMA, None, None, ctypes.c_void_p(1), lens.ctypes.data)
            assert lib.pa_decode_launch_count(ctypes.byref(d), N, 32, max_blocks, ctypes.byref(o_plan)) == 3


def test_a_run_of_blocks_spans_at_most_its_share_plus_two_ctas():
    """The host's long-context decision skips the exact count for sequences
    with nb * Ce < 6 * W: nb consecutive blocks of a W-block list cut into Ce
    even ranges touch at most nb * Ce / W + 2 of them."""
    rng = np.random.default_rng(9)
    for _ in range(3000):
        W = int(rng.integers(1, 1 << 22))
        Ce = int(min(rng.integers(1, 5000), W))
        nb = int(rng.integers(1, W + 1))
        x0 = int(rng.integers(0, W - nb + 1))
        pieces = pa.pa_split_owner(W, Ce, x0 + nb - 1) - pa.pa_split_owner(W, Ce, x0) + 1
        assert pieces <= nb * Ce / W + 2
        if nb * Ce < 6 * W:
            assert pieces < 8


class _FakeCudaTensor:
    """Just enough of a CUDA tensor for the binding's checks (no GPU needed):
    it reports a device index and never gets as far as a C call."""

    def __init__(self, shape, dtype, index):
        import torch
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device("cuda", index)
        self.is_cuda = True

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for x in self.shape:
            n *= x
        return n

    def reshape(self, *shape):
        return self

    def element_size(self):
        return 2

    def is_contiguous(self):
        return True

    def data_ptr(self):
        raise AssertionError("a tensor on another device reached the C call")


def test_tensors_on_another_device_are_refused_before_the_call(monkeypatch):
    """The library works on the current device (its stream, its error word,
    its scratch); a tensor on another GPU is refused with ValueError."""
    import torch
    monkeypatch.setattr(pa, "_current_device", lambda: 0)
    bf = torch.bfloat16
    kc = _FakeCudaTensor((8, 16, 8, 128), bf, 1)
    vc = _FakeCudaTensor((8, 16, 8, 128), bf, 1)
    pairs = _FakeCudaTensor((2, 2), torch.int32, 1)
    with pytest.raises(ValueError, match="current device"):
        pa.pa_copy_blocks(kc, vc, pairs)
    k = _FakeCudaTensor((4, 8, 128), bf, 1)
    slots = _FakeCudaTensor((4,), torch.int32, 1)
    with pytest.raises(ValueError, match="current device"):
        pa.pa_reshape_and_cache(k, k, slots, kc, vc)
    q = _FakeCudaTensor((2, 32, 128), bf, 1)
    tables = _FakeCudaTensor((2, 4), torch.int32, 1)
    lens = _FakeCudaTensor((2,), torch.int32, 1)
    ws = _FakeCudaTensor((1 << 20,), torch.uint8, 1)
    with pytest.raises(ValueError, match="current device"):
        pa.pa_decode(q, kc, vc, tables, lens, 0.088, out=q, workspace=ws)
    with pytest.raises(ValueError, match="current device"):
        pa.pa_decode_no_alloc(q, kc, vc, tables, lens, 0.088, q)
