"""pa_decode_no_alloc: decode for callers that cannot allocate device memory.

Such callers (a server whose KV pool took nearly all device memory at
startup, a plugin whose host framework owns the allocator, a loop that cannot
pay for cudaMalloc's implicit synchronisation) cannot pass pa_decode a
workspace.  The no-allocation entry point uses a fixed scratch array inside the
library instead.  This file checks, through the C ABI, that two calls in a row
give the same output as pa_decode with a caller-provided workspace (within the
suite's bf16 tolerance), and that a shape too large for the fixed array is
refused before anything is launched.  It is named so that pytest collects it
last.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import _lib, inputs
from _pipeline import TOL, gpu_step, host_values

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg,kw", [("cfg2", {"small": True}), ("cfg4", {"small": True}), ("cfg0", {})])
def test_no_alloc_matches_pa_decode_on_two_calls_in_a_row(cfg, kw):
    wl = inputs.workload(cfg, **kw)
    dev, _ = host_values(wl, "cpu")
    g = gpu_step(wl, dev)  # pa_decode with a workspace from the caller
    ref = g["out"].float()
    for _ in range(2):
        out = torch.full_like(g["out"], float("nan"))
        pa.pa_decode_no_alloc(g["q"], g["k_cache"], g["v_cache"], g["tables"], g["lens"], wl.scale, out)
        assert pa.pa_get_device_error(raise_on_error=False) == 0
        assert torch.isfinite(out.float()).all()
        assert (out.float() - ref).abs().max().item() <= TOL[wl.dtype]


def test_no_alloc_refuses_a_shape_beyond_its_scratch():
    desc = _lib.CacheDesc(1 << 16, 16, 8, 128, _lib.PA_BF16)
    opts = _lib.DecodeOpts(0, _lib.PA_KERNEL_AUTO, None, None)
    need = _lib.load().pa_decode_workspace_bytes(ctypes.byref(desc), 8192, 64, ctypes.byref(opts))
    assert need > _lib.PA_NO_ALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    st = _lib.load().pa_decode_no_alloc(p, p, p, p, ctypes.byref(desc), p, 4, p, 8192, 64, 0.088,
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
    pairs = [(0, h) for h in range(0, 64, 9)] + [(3, 5), (4, 60)]
    assert max_abs_err(out, oracle_decode(wl, host, r, pairs=pairs), pairs) <= TOL["bf16"]
