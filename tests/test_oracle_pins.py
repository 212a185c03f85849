"""Pins for the CPU oracle: values the pages print, closed forms, invariants and
brute force on tiny inputs.  None of these re-types the oracle's own loops:
the references are the pages' worked numbers, textbook identities, or an
independent formulation (torch.cat of the table's blocks, then dense fp64
softmax attention, as the tokentrails "PagedAttention" Code sketch gathers K).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_150_gb300 import inputs

def _rand_case(dtype, n_seqs, lens, H, Hk, D, B, num_blocks, seed, pad_extra=1):
    """Random pool/q and tables drawn from a shuffled pool (test-local helper)."""
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.randn(num_blocks, B, Hk, D, generator=g).to(tdt)
    vc = torch.randn(num_blocks, B, Hk, D, generator=g).to(tdt)
    q = torch.randn(n_seqs, H, D, generator=g).to(tdt)
    perm = torch.randperm(num_blocks, generator=g).tolist()
    max_blocks = max(1, max(-(-L // B) for L in lens)) + pad_extra
    tables = np.full((n_seqs, max_blocks), -1, dtype=np.int32)
    used = 0
    for i, L in enumerate(lens):
        nb = -(-L // B)
        tables[i, :nb] = perm[used:used + nb]
        used += nb
    assert used <= num_blocks
    return q, kc, vc, tables, np.asarray(lens, dtype=np.int32)


def _np(t):
    return inputs.to_numpy_elems(t)


def _torch_dense_reference(q, kc, vc, tables, lens, scale):
    """Gather each sequence's K/V by concatenating its blocks in table order,
    then softmax(scale * q K^T) V in fp64 with torch; GQA by repeat_interleave."""
    n, H, D = q.shape
    Hk = kc.shape[2]
    G = H // Hk
    out = torch.zeros(n, H, D, dtype=torch.float64)
    for i in range(n):
        L = int(lens[i])
        if L == 0:
            continue
        B = kc.shape[1]
        nb = -(-L // B)
        K = torch.cat([kc[int(b)] for b in tables[i, :nb]])[:L].double()  # [L, Hk, D]
        V = torch.cat([vc[int(b)] for b in tables[i, :nb]])[:L].double()
        K = K.repeat_interleave(G, dim=1)  # [L, H, D]
        V = V.repeat_interleave(G, dim=1)
        s = torch.einsum("hd,lhd->hl", q[i].double(), K) * scale
        w = torch.softmax(s, dim=-1)
        out[i] = torch.einsum("hl,lhd->hd", w, V)
    return out.numpy()


def _oracle(q, kc, vc, tables, lens, scale, **kw):
    return oracle.decode(_np(q), _np(kc), _np(vc), tables, lens, scale, **kw)


# ----------------------------------------------------------------- attention
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token_returns_its_value_row(dtype):
    q, kc, vc, tables, lens = _rand_case(dtype, 3, [1, 1, 1], 4, 2, 64, 4, 8, 1)
    out = _oracle(q, kc, vc, tables, lens, 0.125)
    for i in range(3):
        b = int(tables[i, 0])
        for h in range(4):
            np.testing.assert_array_equal(out[i, h], vc[b, 0, h // 2].double().numpy())


def test_equal_keys_give_mean_of_values():
    q, kc, vc, tables, lens = _rand_case("f32", 2, [7, 13], 2, 2, 32, 4, 12, 2)
    kc[:] = kc[0, 0]  # every key row identical -> every score identical
    out = _oracle(q, kc, vc, tables, lens, 0.3)
    for i, L in enumerate(lens):
        nb = -(-int(L) // 4)
        V = torch.cat([vc[int(b)] for b in tables[i, :nb]])[:L].double()
        np.testing.assert_allclose(out[i], V.mean(0).numpy(), rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_values():
    q, kc, vc, tables, lens = _rand_case("bf16", 2, [9, 30], 4, 4, 64, 8, 10, 3)
    q.zero_()
    out = _oracle(q, kc, vc, tables, lens, 1.0)
    for i, L in enumerate(lens):
        nb = -(-int(L) // 8)
        V = torch.cat([vc[int(b)] for b in tables[i, :nb]])[:L].double()
        np.testing.assert_allclose(out[i], V.mean(0).numpy(), rtol=0, atol=1e-14)


def test_two_tokens_follow_the_logistic_closed_form():
    # q = e_0 and K_j = (a_j, 0, ...): scores are scale * a_j exactly.
    D, B, scale = 8, 2, 0.5
    a0, a1 = 1.5, -2.25
    kc = torch.zeros(3, B, 1, D)
    vc = torch.randn(3, B, 1, D, generator=torch.Generator().manual_seed(5))
    kc[2, 0, 0, 0] = a0
    kc[2, 1, 0, 0] = a1
    q = torch.zeros(1, 1, D)
    q[0, 0, 0] = 1.0
    tables = np.array([[2]], dtype=np.int32)
    out = _oracle(q, kc, vc, tables, [2], scale)
    w0 = 1.0 / (1.0 + math.exp(scale * (a1 - a0)))
    expect = w0 * vc[2, 0, 0].double().numpy() + (1.0 - w0) * vc[2, 1, 0].double().numpy()
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-15)


def test_large_score_gaps_stay_finite():
    # Scores (0, -1000, 1000): the true softmax is (e^-1000, e^-2000, 1), so the
    # output equals the last value row to double precision; an exponent taken
    # without the maximum over every score would overflow.
    D, B = 4, 4
    kc = torch.zeros(1, B, 1, D)
    vc = torch.randn(1, B, 1, D, generator=torch.Generator().manual_seed(6))
    kc[0, 1, 0, 0] = -1.0
    kc[0, 2, 0, 0] = 1.0
    q = torch.zeros(1, 1, D)
    q[0, 0, 0] = 1000.0
    out = _oracle(q, kc, vc, np.array([[0]], np.int32), [3], 1.0)
    np.testing.assert_allclose(out[0, 0], vc[0, 2, 0].double().numpy(), rtol=0, atol=1e-300)


@pytest.mark.parametrize("dtype,H,Hk,D,B", [("f32", 4, 4, 64, 4), ("bf16", 8, 2, 32, 16),
                                           ("bf16", 8, 1, 16, 1), ("f32", 6, 3, 8, 5)])
def test_matches_dense_attention_on_gathered_blocks(dtype, H, Hk, D, B):
    lens = [1, B - 1 if B > 1 else 2, B, B + 1, 3 * B + 2, 0]
    nblocks = sum(-(-L // B) for L in lens) + 5
    q, kc, vc, tables, lens = _rand_case(dtype, len(lens), lens, H, Hk, D, B, nblocks, 7)
    scale = 1.0 / math.sqrt(D)
    out = _oracle(q, kc, vc, tables, lens, scale)
    ref = _torch_dense_reference(q, kc, vc, tables, lens, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_grouped_heads_read_kv_head_h_div_group():
    # KV head 0 holds values +1, KV head 1 holds -1: with H=4, Hk=2 (group 2),
    # heads 0,1 must average +1 and heads 2,3 must average -1.
    q, kc, vc, tables, lens = _rand_case("f32", 1, [11], 4, 2, 16, 4, 5, 8)
    vc[:, :, 0, :] = 1.0
    vc[:, :, 1, :] = -1.0
    out = _oracle(q, kc, vc, tables, lens, 0.25)
    np.testing.assert_allclose(out[0, :2], 1.0, atol=1e-14)
    np.testing.assert_allclose(out[0, 2:], -1.0, atol=1e-14)


def test_invariant_under_permutation_of_physical_blocks():
    q, kc, vc, tables, lens = _rand_case("bf16", 4, [5, 40, 17, 64], 4, 2, 32, 8, 24, 9)
    out = _oracle(q, kc, vc, tables, lens, 0.2)
    perm = torch.randperm(24, generator=torch.Generator().manual_seed(10))
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = np.where(tables >= 0, perm.numpy()[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = _oracle(q, kc2, vc2, t2, lens, 0.2)
    np.testing.assert_array_equal(out, out2)


def test_invariant_under_block_size():
    # The same logical K/V rows stored with block size 4 and with block size 16.
    g = torch.Generator().manual_seed(11)
    lens = [3, 21, 50]
    Hk, D, H = 2, 16, 4
    q = torch.randn(3, H, D, generator=g)
    rows_k = [torch.randn(L, Hk, D, generator=g) for L in lens]
    rows_v = [torch.randn(L, Hk, D, generator=g) for L in lens]
    outs = []
    for B in (4, 16):
        nbs = [-(-L // B) for L in lens]
        kc = torch.full((sum(nbs) + 2, B, Hk, D), float("nan"))
        vc = torch.full_like(kc, float("nan"))
        order = torch.randperm(kc.shape[0], generator=g).tolist()
        tables = np.full((3, max(nbs)), -1, dtype=np.int32)
        used = 0
        for i, L in enumerate(lens):
            for j in range(nbs[i]):
                b = order[used]
                used += 1
                tables[i, j] = b
                lo, hi = j * B, min(L, (j + 1) * B)
                kc[b, :hi - lo] = rows_k[i][lo:hi]
                vc[b, :hi - lo] = rows_v[i][lo:hi]
        outs.append(_oracle(q, kc, vc, tables, lens, 0.25))
    np.testing.assert_array_equal(outs[0], outs[1])
    assert np.isfinite(outs[0]).all()


def test_stale_slots_and_padding_are_never_read():
    q, kc, vc, tables, lens = _rand_case("bf16", 3, [6, 17, 31], 4, 4, 32, 8, 12, 12, pad_extra=3)
    clean = _oracle(q, kc, vc, tables, lens, 0.3)
    kc2, vc2 = kc.clone(), vc.clone()
    live = set()
    for i, L in enumerate(lens):
        for pos in range(int(L)):
            live.add((int(tables[i, pos // 8]), pos % 8))
    for b in range(kc.shape[0]):
        for o in range(8):
            if (b, o) not in live:
                kc2[b, o] = float("nan")
                vc2[b, o] = float("nan")
    out = _oracle(q, kc2, vc2, tables, lens, 0.3)
    np.testing.assert_array_equal(out, clean)


def test_zero_length_sequence_gives_zeros():
    q, kc, vc, tables, lens = _rand_case("f32", 2, [0, 5], 2, 2, 16, 4, 4, 13)
    out = _oracle(q, kc, vc, tables, lens, 0.25)
    assert (out[0] == 0).all()
    assert np.isfinite(out[1]).all()


def test_bf16_widening_is_exact():
    # 1.0, -2.5, 0.15625 and the smallest subnormal 2^-133, as raw bf16 bits.
    bits = np.array([0x3F80, 0xC020, 0x3E20, 0x0001], dtype=np.uint16)
    vc = np.zeros((1, 1, 1, 4), dtype=np.uint16)
    vc[0, 0, 0] = bits
    kc = np.zeros_like(vc)
    q = np.zeros((1, 1, 4), dtype=np.uint16)
    out = oracle.decode(q, kc, vc, np.array([[0]], np.int32), [1], 1.0)
    np.testing.assert_array_equal(out[0, 0], [1.0, -2.5, 0.15625, 2.0 ** -133])


def test_out_of_range_table_entry_is_rejected():
    q, kc, vc, tables, lens = _rand_case("f32", 1, [5], 2, 2, 16, 4, 4, 14)
    tables[0, 1] = 4  # pool has blocks 0..3
    with pytest.raises(ValueError):
        _oracle(q, kc, vc, tables, lens, 0.25)


def test_thread_count_does_not_change_results():
    q, kc, vc, tables, lens = _rand_case("bf16", 5, [3, 30, 77, 1, 64], 8, 2, 32, 16, 20, 15)
    a = _oracle(q, kc, vc, tables, lens, 0.2, num_threads=1)
    b = _oracle(q, kc, vc, tables, lens, 0.2, num_threads=4)
    np.testing.assert_array_equal(a, b)


def test_pair_subset_matches_full_run():
    q, kc, vc, tables, lens = _rand_case("bf16", 3, [12, 40, 7], 4, 2, 32, 8, 12, 16)
    full = _oracle(q, kc, vc, tables, lens, 0.2)
    pairs = [(2, 3), (0, 1), (1, 0)]
    part = _oracle(q, kc, vc, tables, lens, 0.2, pairs=pairs)
    for s, h in pairs:
        np.testing.assert_array_equal(part[s, h], full[s, h])
    assert np.isnan(part[0, 0]).all()


def test_repeated_pairs_give_the_same_values_on_many_threads():
    """A pair listed several times is computed once: with 8 threads the
    repeats would otherwise race on the same output row."""
    q, kc, vc, tables, lens = _rand_case("bf16", 3, [6000, 40, 7], 4, 2, 32, 16, 400, 17)
    full = _oracle(q, kc, vc, tables, lens, 0.2)
    pairs = [(0, 1)] * 16 + [(0, 2)] * 16 + [(1, 2), (2, 3)] * 3
    part = _oracle(q, kc, vc, tables, lens, 0.2, pairs=pairs, num_threads=8)
    for s, h in set(pairs):
        np.testing.assert_array_equal(part[s, h], full[s, h])


# ----------------------------------------------------------- write and copy
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cache_write_matches_indexed_assignment(dtype):
    g = torch.Generator().manual_seed(20)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    NB, B, Hk, D, T = 6, 4, 3, 8, 9
    kc = torch.randn(NB, B, Hk, D, generator=g).to(tdt)
    vc = torch.randn(NB, B, Hk, D, generator=g).to(tdt)
    k = torch.randn(T, Hk, D, generator=g).to(tdt)
    v = torch.randn(T, Hk, D, generator=g).to(tdt)
    slots = torch.randperm(NB * B, generator=g)[:T].clone()
    slots[2] = -1  # padding token
    ok = slots >= 0
    ref_k = kc.clone().view(NB * B, Hk, D)
    ref_v = vc.clone().view(NB * B, Hk, D)
    ref_k[slots[ok]] = k[ok]
    ref_v[slots[ok]] = v[ok]
    kn, vn = _np(kc), _np(vc)
    bad = oracle.reshape_and_cache(_np(k), _np(v), slots.numpy(), kn, vn)
    assert bad == 0
    np.testing.assert_array_equal(kn, _np(ref_k.view(NB, B, Hk, D)))
    np.testing.assert_array_equal(vn, _np(ref_v.view(NB, B, Hk, D)))


def test_cache_write_skips_and_counts_slots_beyond_the_pool():
    kc = np.zeros((2, 4, 1, 4), np.float32)
    vc = np.zeros_like(kc)
    k = np.ones((2, 1, 4), np.float32)
    bad = oracle.reshape_and_cache(k, k, np.array([8, 3]), kc, vc)
    assert bad == 1
    assert (kc[0, 3] == 1).all() and kc.sum() == 4


def test_copy_blocks_matches_indexing():
    g = torch.Generator().manual_seed(21)
    kc = torch.randn(8, 4, 2, 8, generator=g).to(torch.bfloat16)
    vc = torch.randn(8, 4, 2, 8, generator=g).to(torch.bfloat16)
    pairs = np.array([[1, 5], [1, 6], [3, 0]], np.int32)
    ref_k, ref_v = kc.clone(), vc.clone()
    ref_k[torch.tensor([5, 6, 0])] = kc[torch.tensor([1, 1, 3])]
    ref_v[torch.tensor([5, 6, 0])] = vc[torch.tensor([1, 1, 3])]
    kn, vn = _np(kc), _np(vc)
    oracle.copy_blocks(kn, vn, pairs)
    np.testing.assert_array_equal(kn, _np(ref_k))
    np.testing.assert_array_equal(vn, _np(ref_v))


# ------------------------------------------------------ slots (pages' values)
def test_slot_mapping_worked_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "slot_mapping_examples.json")))
    B = g["block_size"]
    table = np.array(g["table"], np.int32)
    for case in g["cases"]:
        assert oracle.physical_index(table, B, case["token"]) == case["slot"]
        slot = oracle.slot_mapping(table[None, :], [0], [case["token"]], B)[0]
        assert slot == case["slot"]
        assert slot // B == case["physical_block"] and slot % B == case["offset"]
    m = oracle.OracleBlockManager(1, B)
    for c in g["blocks_needed"]:
        assert m.blocks_needed(c["tokens"]) == c["blocks"]


# ------------------------------------------------ split (vLLM) cache layout
def _to_split(kc, vc):
    """Row layout [NB, B, Hk, D] -> K [NB, Hk, D/x, B, x], V [NB, Hk, D, B] with
    x = 16 / element bytes, by torch reshapes and permutes ("10 PagedAttention",
    section 5, "The layout, more precisely")."""
    nb, bs, hk, d = kc.shape
    x = 16 // kc.element_size()
    k = kc.view(nb, bs, hk, d // x, x).permute(0, 2, 3, 1, 4).contiguous()
    v = vc.permute(0, 2, 3, 1).contiguous()
    return k, v


@pytest.mark.parametrize("dtype,x", [("bf16", 8), ("f32", 4)])
def test_split_layout_vector_width(dtype, x):
    q, kc, vc, tables, lens = _rand_case(dtype, 1, [5], 2, 2, 32, 4, 4, 30)
    ks, vs = _to_split(kc, vc)
    layout, nb, bs, hk, d = oracle.cache_geometry(_np(ks), _np(vs))
    assert layout == oracle.SPLIT and ks.shape[-1] == x and (nb, bs, hk, d) == (4, 4, 2, 32)


@pytest.mark.parametrize("dtype,H,Hk,D,B", [("bf16", 8, 2, 32, 16), ("f32", 4, 4, 16, 4), ("bf16", 6, 3, 64, 8)])
def test_split_layout_decode_equals_row_layout_decode(dtype, H, Hk, D, B):
    lens = [1, B - 1, B + 1, 3 * B + 2, 0]
    nblocks = sum(-(-L // B) for L in lens) + 3
    q, kc, vc, tables, lens = _rand_case(dtype, len(lens), lens, H, Hk, D, B, nblocks, 31)
    ks, vs = _to_split(kc, vc)
    row = _oracle(q, kc, vc, tables, lens, 0.2)
    split = _oracle(q, ks, vs, tables, lens, 0.2)
    np.testing.assert_array_equal(row, split)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_layout_write_equals_permuted_row_write(dtype):
    g = torch.Generator().manual_seed(32)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    NB, B, Hk, D, T = 5, 8, 2, 16, 11
    kc = torch.randn(NB, B, Hk, D, generator=g).to(tdt)
    vc = torch.randn(NB, B, Hk, D, generator=g).to(tdt)
    k = torch.randn(T, Hk, D, generator=g).to(tdt)
    v = torch.randn(T, Hk, D, generator=g).to(tdt)
    slots = torch.randperm(NB * B, generator=g)[:T].numpy()
    slots[3] = -1
    ks, vs = (_np(t).copy() for t in _to_split(kc, vc))
    kr, vr = _np(kc).copy(), _np(vc).copy()
    assert oracle.reshape_and_cache(_np(k), _np(v), slots, kr, vr) == 0
    assert oracle.reshape_and_cache(_np(k), _np(v), slots, ks, vs) == 0
    tk = torch.from_numpy(kr.view(np.int16) if dtype == "bf16" else kr)
    tv = torch.from_numpy(vr.view(np.int16) if dtype == "bf16" else vr)
    ek, ev = _to_split(tk, tv)
    np.testing.assert_array_equal(ks.view(ek.numpy().dtype), ek.numpy())
    np.testing.assert_array_equal(vs.view(ev.numpy().dtype), ev.numpy())
