"""Seeded random sweeps against the oracle.

Independent sequences: element type, KV heads, query heads per KV head
(including 3), head dim, block size, cache layout, batch size, lengths
(with 0, 1 and values at block edges) and split counts, on both kernels;
the cache write is compared byte for byte, decode within the tolerance of
its element type.  Parallel sampling with a shared-prefix plan: random
prompt counts and lengths, samples, appended tokens, head ratios, head
dims, block sizes, layouts and split counts.  Block copy then cache write:
random shapes, layouts, pairs and padded slot lists, byte for byte."""
import numpy as np
import pytest

from paged_kv_cache_150_gb300 import inputs
from _pipeline import TOL, gpu_step, host_values, max_abs_err, oracle_decode, oracle_step

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(10_000 + seed)
    dtype = "f32" if rng.random() < 0.25 else "bf16"
    Hk = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8]))
    if dtype == "f32":
        D, B = int(rng.choice([64, 128])), int(rng.choice([4, 8, 16, 32]))
    else:
        D, B = int(rng.choice([64, 128, 128, 256])), int(rng.choice([8, 16, 16, 32]))
    layout = "split" if rng.random() < 0.25 else "row"
    N = int(rng.integers(1, 24))
    edges = [0, 1, B - 1, B, B + 1, 2 * B, 3 * B + 1]
    lens = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 40 * B)) for _ in range(N)]
    splits = int(rng.choice([0, 0, 1, 2, 5, 13]))
    return dtype, Hk * G, Hk, D, B, layout, lens, splits


@pytest.mark.parametrize("seed", range(160))
def test_random_shapes_match_the_oracle(seed):
    dtype, H, Hk, D, B, layout, lens, splits = _case(seed)
    wl = inputs.decode_workload("fuzz%d" % seed, lens, H, Hk, D, B, dtype, seed=20_000 + seed, pool_factor=1.3)
    dev, host = host_values(wl, "cpu", layout=layout)
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    shape = (dtype, H, Hk, D, B, layout, splits)
    for kernel in ("auto", "simt"):
        g = gpu_step(wl, {k: v.clone() for k, v in dev.items()}, kernel=kernel, num_splits=splits)
        assert np.array_equal(inputs.to_numpy_elems(g["k_cache"]), r["k_cache"]), shape
        assert np.array_equal(inputs.to_numpy_elems(g["v_cache"]), r["v_cache"]), shape
        err = max_abs_err(g["out"], ref)
        assert err <= TOL[dtype], (kernel, err, shape)


def _sampling_case(seed):
    rng = np.random.default_rng(30_000 + seed)
    Hk, G = int(rng.choice([4, 8])), int(rng.choice([1, 2, 4, 8]))
    D, B = int(rng.choice([64, 128])), int(rng.choice([16, 32]))
    prompts, samples = int(rng.integers(1, 6)), int(rng.integers(2, 12))
    prompt_len = int(rng.integers(B + 1, 40 * B))  # at least one whole block to share
    max_append = int(rng.integers(1, 3 * B))
    layout = "split" if rng.random() < 0.25 else "row"
    splits = int(rng.choice([0, 0, 2, 5, 13]))
    return prompts, prompt_len, samples, max_append, Hk * G, Hk, D, B, layout, splits


@pytest.mark.parametrize("seed", range(40))
def test_random_parallel_sampling_with_a_shared_prefix_plan(seed):
    """Forked prompts decoded with a shared-prefix plan, over random prompt
    counts and lengths, samples per prompt, appended tokens, head ratios,
    head dims, block sizes, layouts and split counts."""
    prompts, plen, samples, max_append, H, Hk, D, B, layout, splits = _sampling_case(seed)
    wl = inputs.sampling_workload("sfuzz%d" % seed, prompts, plen, samples, max_append, H, Hk, D, B, "bf16",
                                  40_000 + seed)
    dev, host = host_values(wl, "cpu", layout=layout)
    r = oracle_step(wl, host)
    ref = oracle_decode(wl, host, r)
    g = gpu_step(wl, dev, shared=True, num_splits=splits)
    assert g["plan_info"]["num_groups"] == prompts
    err = max_abs_err(g["out"], ref)
    assert err <= TOL["bf16"], (err, prompts, plen, samples, max_append, H, Hk, D, B, layout, splits)


@pytest.mark.parametrize("seed", range(60))
def test_random_block_copy_then_cache_write_bit_exact(seed):
    """Copy-on-write pairs, then a cache write, over random element types,
    KV heads, row widths (down to 3 elements), block sizes (down to 1), both
    layouts, pair counts and slot lists with padding: the caches equal the
    oracle's byte for byte."""
    import torch

    import oracle
    import paged_kv_cache_150_gb300 as pa

    rng = np.random.default_rng(50_000 + seed)
    dtype = "f32" if rng.random() < 0.3 else "bf16"
    tdt, eb = (torch.float32, 4) if dtype == "f32" else (torch.bfloat16, 2)
    hk, d = int(rng.integers(1, 9)), int(rng.choice([3, 6, 8, 64, 104, 128, 256]))
    B, nb = int(rng.choice([1, 4, 5, 8, 16, 32])), int(rng.integers(4, 120))
    split = (d * eb) % 16 == 0 and rng.random() < 0.35
    gen = torch.Generator(device="cuda").manual_seed(60_000 + seed)
    kc = torch.randn(nb, B, hk, d, generator=gen, device="cuda").to(tdt)
    vc = torch.randn(nb, B, hk, d, generator=gen, device="cuda").to(tdt)
    if split:
        kc, vc = inputs.to_split_layout(kc, vc)
    P = int(rng.integers(0, nb // 3 + 1))
    perm = rng.permutation(nb)
    pairs = np.stack([rng.choice(perm[P:], size=P), perm[:P]], 1).astype(np.int32)  # distinct dsts, none a src
    T = int(rng.integers(0, nb * B // 2 + 1))
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.int32)
    slots[rng.random(T) < 0.2] = -1  # padding
    k = torch.randn(T, hk, d, generator=gen, device="cuda").to(tdt)
    v = torch.randn(T, hk, d, generator=gen, device="cuda").to(tdt)
    ref_k, ref_v = inputs.to_numpy_elems(kc).copy(), inputs.to_numpy_elems(vc).copy()
    oracle.copy_blocks(ref_k, ref_v, pairs)
    oracle.reshape_and_cache(inputs.to_numpy_elems(k), inputs.to_numpy_elems(v), slots, ref_k, ref_v)
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    pa.pa_reshape_and_cache(k, v, torch.from_numpy(slots).cuda(), kc, vc)
    assert pa.pa_get_device_error(raise_on_error=False) == 0
    shape = (dtype, hk, d, B, nb, split, P, T)
    assert np.array_equal(inputs.to_numpy_elems(kc), ref_k), shape
    assert np.array_equal(inputs.to_numpy_elems(vc), ref_v), shape
