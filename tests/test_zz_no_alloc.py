"""pa_decode_no_alloc: decode for callers that cannot allocate device memory.

Such callers (a server whose KV pool took nearly all device memory at
startup, a plugin whose host framework owns the allocator, a loop that cannot
pay for cudaMalloc's implicit synchronisation) cannot pass pa_decode a
workspace.  The no-allocation entry point uses a fixed scratch array inside the
library instead.  This file checks, through the C ABI, that calls in a row
give the same bits as pa_decode with a caller-provided workspace and the same
split (also right after a larger call with more splits has left its counters
and partials in the shared array), and that a shape too large for the fixed
array is refused before anything is launched.  It is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import _lib, inputs
from _pipeline import TOL, gpu_step, host_values

pytestmark = pytest.mark.gpu


def _no_alloc(g, wl, num_splits=0):
    out = torch.full_like(g["out"], float("nan"))
    pa.pa_decode_no_alloc(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out,
                          num_splits=num_splits)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    return out


@pytest.mark.parametrize("cfg,kw", [("cfg2", {"small": True}), ("cfg4", {"small": True}), ("cfg0", {})])
def test_no_alloc_gives_the_bits_of_pa_decode_on_two_calls_in_a_row(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    dev, _ = host_values(wl, "cpu")
    g = gpu_step(wl, dev)  # pa_decode with a workspace from the caller, default split
    for _ in range(2):
        assert torch.equal(_no_alloc(g, wl), g["out"])


def test_no_alloc_after_a_larger_call_with_more_splits():
    """A 256-sequence batch on 608 CTAs leaves more arrival counters and
    partials in the shared array than the smaller call after it uses; each
    call must still match pa_decode bit for bit."""
    big_wl = inputs.workload("cfg2")
    big_dev, _ = host_values(big_wl, "cuda")
    big = gpu_step(big_wl, big_dev, num_splits=608)
    small_wl = inputs.workload("cfg4", small=True)
    small_dev, _ = host_values(small_wl, "cpu")
    small = gpu_step(small_wl, small_dev)
    for _ in range(2):
        assert torch.equal(_no_alloc(big, big_wl, num_splits=608), big["out"])
        assert torch.equal(_no_alloc(small, small_wl), small["out"])


def test_no_alloc_refuses_a_shape_beyond_its_scratch():
    desc = _lib.CacheDesc(1 << 16, 16, 8, 128, _lib.PA_BF16)
    opts = _lib.DecodeOpts(0, _lib.PA_KERNEL_AUTO, None, None)
    need = _lib.load().pa_decode_workspace_bytes(ctypes.byref(desc), 8192, 64, ctypes.byref(opts))
    assert need > _lib.PA_NO_ALLOC_SCRATCH_BYTES
    # Null device pointers: the size check comes first, and if it ever did
    # not, pa_decode's null-pointer check would refuse the call before any
    # launch.
    st = _lib.load().pa_decode_no_alloc(None, None, None, None, ctypes.byref(desc), None, 4, None, 8192, 64, 0.088,
                                        ctypes.byref(opts), None)
    assert st == _lib.PA_ERR_WORKSPACE


def test_no_alloc_with_the_host_lengths_matches_pa_decode():
    """The long-context merge path (a host copy of the lengths) through the
    no-allocation entry point: the same bits as pa_decode with the same
    hint, and the oracle within tolerance."""
    import numpy as np

    from _pipeline import max_abs_err, oracle_decode, oracle_step

    lens = [131072 + 5, 17, 1, 4096 + 5, 300, 0]
    wl = inputs.decode_workload("noalloc-long", lens, 64, 8, 128, 16, "bf16", seed=53, pool_factor=1.05)
    dev, host = host_values(wl, "cuda")
    g = gpu_step(wl, dev, host_lens="exact")
    host_lens = np.asarray(wl.seq_lens, np.int32)
    out = torch.full_like(g["out"], float("nan"))
    pa.pa_decode_no_alloc(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out,
                          host_seq_lens=host_lens)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(out, g["out"])
    r = oracle_step(wl, host)
    assert max_abs_err(out, oracle_decode(wl, host, r)) <= TOL["bf16"]
