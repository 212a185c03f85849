"""GPU parity of the paged KV write and the copy-on-write block copy: the
caches after the step must equal the oracle's byte for byte."""
import numpy as np
import pytest
import torch

import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs
from _pipeline import gpu_step, host_values, oracle_step

pytestmark = pytest.mark.gpu

SMALL = [("cfg0", {}), ("cfg1", {"small": True}), ("cfg2", {"small": True}),
         ("cfg3", {"small": True, "prompt_len": 200}), ("cfg3", {"small": True}),
         ("cfg4", {"small": True}), ("cfg4", {"small": True, "block_size": 32})]
FULL = [("cfg1", {}), ("cfg2", {}), ("cfg3", {"prompt_len": 2008}), ("cfg4", {})]


def _check(wl, gen_device):
    dev, host = host_values(wl, gen_device)
    r = oracle_step(wl, host)
    g = gpu_step(wl, dev, decode=False)
    np.testing.assert_array_equal(g["host_slots"], r["slots"])
    np.testing.assert_array_equal(g["host_pairs"], r["pairs"])
    np.testing.assert_array_equal(g["host_tables"], r["tables_padded"])
    assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"])
    assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"])
    return r


@pytest.mark.parametrize("cfg,kw", SMALL)
def test_write_and_copy_bit_exact(cfg, kw):
    r = _check(inputs.workload(cfg, **kw), "cpu")
    if kw.get("prompt_len") == 200:
        assert len(r["pairs"]) == 3 * 4


@pytest.mark.parametrize("cfg,kw", FULL)
def test_write_and_copy_bit_exact_full_size(cfg, kw):
    r = _check(inputs.workload(cfg, **kw), "cuda")
    if kw.get("prompt_len") == 2008:
        assert len(r["pairs"]) == 192


def _cache(nb, bs, hk, d, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(nb, bs, hk, d, generator=g, device="cuda").to(dtype),
            torch.randn(nb, bs, hk, d, generator=g, device="cuda").to(dtype))


@pytest.mark.parametrize("hk,d,dtype", [(2, 3, torch.bfloat16), (1, 6, torch.float32), (8, 128, torch.bfloat16),
                                        (1, 3, torch.bfloat16), (3, 4, torch.bfloat16), (8, 256, torch.bfloat16),
                                        (8, 128, torch.float32), (5, 104, torch.bfloat16)])
def test_write_any_row_width_and_padding_slots(hk, d, dtype):
    nb, bs = 5, 4
    kc, vc = _cache(nb, bs, hk, d, dtype, 1)
    T = 7
    g = torch.Generator(device="cuda").manual_seed(2)
    k = torch.randn(T, hk, d, generator=g, device="cuda").to(dtype)
    v = torch.randn(T, hk, d, generator=g, device="cuda").to(dtype)
    slots = torch.tensor([0, 19, -1, 5, 7, -3, 12], dtype=torch.int32, device="cuda")
    ref_k, ref_v = kc.clone().view(nb * bs, hk, d), vc.clone().view(nb * bs, hk, d)
    keep = slots >= 0
    ref_k[slots[keep].long()] = k[keep]
    ref_v[slots[keep].long()] = v[keep]
    pa.pa_reshape_and_cache(k, v, slots, kc, vc)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(kc.view(nb * bs, hk, d), ref_k) and torch.equal(vc.view(nb * bs, hk, d), ref_v)


def test_out_of_range_slot_and_pair_are_skipped_and_reported():
    nb, bs, hk, d = 4, 16, 8, 128
    kc, vc = _cache(nb, bs, hk, d, torch.bfloat16, 3)
    before_k = kc.clone()
    k = torch.ones(2, hk, d, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([nb * bs, 3], dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(k, k, slots, kc, vc)
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_BOUNDS
    before_k.view(nb * bs, hk, d)[3] = 1
    assert torch.equal(kc, before_k)
    assert pa.pa_get_device_error(raise_on_error=False) == 0  # the word was cleared
    pairs = torch.tensor([[0, 1], [2, nb]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, pairs)
    assert pa.pa_get_device_error(raise_on_error=False) == pa._lib.PA_ERR_DEVICE_BOUNDS
    assert torch.equal(kc[1], kc[0]) and torch.equal(vc[1], vc[0])


def test_copy_of_many_pairs():
    nb, bs, hk, d = 64, 32, 8, 128
    kc, vc = _cache(nb, bs, hk, d, torch.bfloat16, 4)
    src = torch.arange(0, 20, dtype=torch.int32)
    dst = torch.arange(30, 50, dtype=torch.int32)
    ref_k, ref_v = kc.clone(), vc.clone()
    ref_k[dst.long()] = kc[src.long()]
    ref_v[dst.long()] = vc[src.long()]
    pa.pa_copy_blocks(kc, vc, torch.stack([src, dst], 1).cuda())
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(kc, ref_k) and torch.equal(vc, ref_v)


def test_write_many_tokens_several_grid_passes():
    """More tokens than one pass of the write's grid covers (32 tokens per warp
    per pass), a third of them padding, each row one 16-byte vector."""
    T, nslots, hk, d = 400_000, 500_000, 1, 8
    bs = 16
    kc, vc = _cache(nslots // bs, bs, hk, d, torch.bfloat16, 5)
    g = torch.Generator(device="cuda").manual_seed(6)
    k = torch.randn(T, hk, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(T, hk, d, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(7)
    slots = rng.permutation(nslots)[:T].astype(np.int32)
    slots[rng.random(T) < 1 / 3] = -1
    slots_d = torch.from_numpy(slots).cuda()
    ref_k, ref_v = kc.clone().view(-1, hk, d), vc.clone().view(-1, hk, d)
    keep = slots_d >= 0
    ref_k[slots_d[keep].long()] = k[keep]
    ref_v[slots_d[keep].long()] = v[keep]
    pa.pa_reshape_and_cache(k, v, slots_d, kc, vc)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(kc.view(-1, hk, d), ref_k) and torch.equal(vc.view(-1, hk, d), ref_v)


@pytest.mark.parametrize("cfg,kw", [("cfg3", {"small": True, "prompt_len": 200}), ("cfg3", {"small": True}),
                                    ("cfg3", {"prompt_len": 2008})])
def test_shared_blocks_are_never_written_in_place(cfg, kw):
    """Copy-on-write invariant on the device: in the parallel-sampling step
    (the prompt's rows predate it; the step writes only the samples' new
    tokens) every block still shared (refcount > 1) after the manager's
    operations keeps its bytes through the block copies and the cache write.
    (With prefix caching the first holder writes a prompt block in the same
    step that later requests come to share it, so the test does not apply.)"""
    wl = inputs.workload(cfg, **kw)
    dev, _ = host_values(wl, "cuda" if not kw.get("small") else "cpu")
    bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    slots, pairs = bm.apply_script(wl.script)
    shared = [b for b in range(wl.num_blocks) if bm.refcount(b) > 1]
    assert shared
    idx = torch.tensor(shared, dtype=torch.long, device="cuda")
    before_k, before_v = dev["k_cache"][idx].clone(), dev["v_cache"][idx].clone()
    pa.pa_copy_blocks(dev["k_cache"], dev["v_cache"], torch.from_numpy(pairs).cuda())
    pa.pa_reshape_and_cache(dev["k"], dev["v"], torch.from_numpy(slots).cuda(), dev["k_cache"], dev["v_cache"])
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    assert torch.equal(dev["k_cache"][idx], before_k) and torch.equal(dev["v_cache"][idx], before_v)
    # and the written slots all lie in blocks held by one sequence
    written = np.unique(slots[slots >= 0] // wl.block_size)
    assert not set(written.tolist()) & set(shared)
