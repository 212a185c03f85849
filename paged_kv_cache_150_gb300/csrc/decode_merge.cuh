// Split-K merge of decode pieces (used by every decode translation unit).
//
// A piece is the partial result (running max, sum, accumulator) of one
// (sequence, KV head) over one CTA's part of its blocks; the merge folds all
// pieces of a pair with the max/sum rescaling.  Done by the pair's last
// arriver inside the attention kernels for sequences without a shared prefix
// (in the block loop for the CUDA-core kernel, merge_pieces; after the block
// loop for the tensor-core kernel, merge_online), and by shared_merge_kernel
// for sequences with one.
#pragma once

#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------ output stores
__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// A lane's slice of E merged outputs, a[j] * inv: 16-byte (or, for slices
// of 4, 8-byte) stores where the slice allows (bf16, aligned), else element
// by element.
template <typename T, int E>
__device__ __forceinline__ void store_slice(T *o, const float (&a)[E], float inv) {
    if constexpr (sizeof(T) == 2 && E == 4) {
        if (((uintptr_t)o & 7) == 0) {
            uint2 u;
            u.x = pack_bf16x2(a[0] * inv, a[1] * inv);
            u.y = pack_bf16x2(a[2] * inv, a[3] * inv);
            *reinterpret_cast<uint2 *>(o) = u;
            return;
        }
    }
    if constexpr (sizeof(T) == 2 && E % 8 == 0) {
        if (((uintptr_t)o & 15) == 0) {
#pragma unroll
            for (int j8 = 0; j8 < E / 8; ++j8) {
                uint4 u;
                u.x = pack_bf16x2(a[8 * j8 + 0] * inv, a[8 * j8 + 1] * inv);
                u.y = pack_bf16x2(a[8 * j8 + 2] * inv, a[8 * j8 + 3] * inv);
                u.z = pack_bf16x2(a[8 * j8 + 4] * inv, a[8 * j8 + 5] * inv);
                u.w = pack_bf16x2(a[8 * j8 + 6] * inv, a[8 * j8 + 7] * inv);
                *reinterpret_cast<uint4 *>(o + 8 * j8) = u;
            }
            return;
        }
    }
#pragma unroll
    for (int j = 0; j < E; ++j) store_out(o + j, a[j] * inv);
}

// ------------------------------------------------------------ piece merge
// Partial results of one (sequence, KV head) are "pieces": (m, l) in ml[] and
// the unnormalised accumulator in acc[] (D floats), for each of the G query
// heads.  A PieceRange names the pieces held by CTAs c0..c1 of one split:
// head h of the piece of CTA c is element (c + base) * stride + col + h.  The
// own-block pieces of a sequence form one range; with a shared-prefix plan,
// the pieces of its shared prefix form a second one.
struct PieceRange {
    const float2 *ml;
    const float *acc;
    int64_t base;
    int32_t stride, col, c0, c1;  // empty when c0 > c1
};

// Merge of both ranges for the G query heads of one (sequence, KV head), one
// piece per L2 round trip (few registers: it runs inside the CUDA-core
// kernel's block loop).  Lanes split the G heads x D outputs: LPH lanes per
// head, each a contiguous slice of E = D / LPH elements, so every load of a
// piece is issued back to back; two passes, the maximum over all pieces
// first, then the weighted sums.
template <typename T, int D, int LPH>
__device__ __forceinline__ void merge_pieces_lph(T *__restrict__ out_base, const PieceRange (&rg)[2], int32_t G,
                                                 int lane) {
    constexpr int E = D / LPH;
    static_assert(E % 4 == 0, "slices are whole float4s");
    const int h = lane / LPH;
    const int part = lane % LPH;
    if (h >= G) return;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const PieceRange &p = rg[k];
#pragma unroll 8
        for (int32_t c = p.c0; c <= p.c1; ++c)
            M = fmaxf(M, __ldcg(&p.ml[(c + p.base) * p.stride + p.col + h]).x);
    }
    float a[E];
#pragma unroll
    for (int j = 0; j < E; ++j) a[j] = 0.f;
    float Ls = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const PieceRange &p = rg[k];
#pragma unroll 1
        for (int32_t c = p.c0; c <= p.c1; ++c) {
            const int64_t idx = (c + p.base) * p.stride + p.col + h;
            const float4 *ap = reinterpret_cast<const float4 *>(p.acc + idx * D + part * E);
            float4 x[E / 4];
#pragma unroll
            for (int j4 = 0; j4 < E / 4; ++j4) x[j4] = __ldcg(ap + j4);
            const float2 v = __ldcg(&p.ml[idx]);
            const float wgt = ex2_approx(v.x - M);
            Ls = fmaf(wgt, v.y, Ls);
#pragma unroll
            for (int j4 = 0; j4 < E / 4; ++j4) {
                a[4 * j4 + 0] = fmaf(wgt, x[j4].x, a[4 * j4 + 0]);
                a[4 * j4 + 1] = fmaf(wgt, x[j4].y, a[4 * j4 + 1]);
                a[4 * j4 + 2] = fmaf(wgt, x[j4].z, a[4 * j4 + 2]);
                a[4 * j4 + 3] = fmaf(wgt, x[j4].w, a[4 * j4 + 3]);
            }
        }
    }
    const float inv = 1.f / Ls;
    T *o = out_base + (int64_t)h * D + part * E;
    store_slice<T, E>(o, a, inv);
}

// Lanes per head: 32 / (G rounded up to a power of two), with slices of at
// least 4 elements.
template <typename T, int D>
__device__ __forceinline__ void merge_pieces(T *__restrict__ out_base, const PieceRange (&rg)[2], int32_t G,
                                             int lane) {
    constexpr int kMaxLph = D / 4 < 32 ? D / 4 : 32;
    constexpr int kL8 = 8 < kMaxLph ? 8 : kMaxLph, kL16 = 16 < kMaxLph ? 16 : kMaxLph;
    if (G > 4)
        merge_pieces_lph<T, D, 4>(out_base, rg, G, lane);
    else if (G > 2)
        merge_pieces_lph<T, D, kL8>(out_base, rg, G, lane);
    else if (G > 1)
        merge_pieces_lph<T, D, kL16>(out_base, rg, G, lane);
    else
        merge_pieces_lph<T, D, kMaxLph>(out_base, rg, G, lane);
}

// Pieces of the sequence's own blocks: its range of the flattened (head
// group g, sequence, own block) list of W blocks cut over Ce CTAs; warp w of
// the group holds KV head g * NH + w.
__device__ __forceinline__ PieceRange own_range(const float2 *ml, const float *acc, const int32_t *__restrict__ cu,
                                                int32_t N, int32_t seq, int32_t g, int32_t w, int32_t G,
                                                int32_t HPG, int64_t W, int32_t Ce) {
    const int64_t x0 = (int64_t)g * cu[N] + cu[seq];
    const int32_t nb = cu[seq + 1] - cu[seq];
    return PieceRange{ml, acc, (int64_t)g * N + seq, HPG, w * G, split_owner(x0, W, Ce),
                      split_owner(x0 + nb - 1, W, Ce)};
}

__device__ __forceinline__ PieceRange no_range() { return PieceRange{nullptr, nullptr, 0, 0, 0, 0, -1}; }

// The shared-prefix part of a launch, as the merge needs it: the shared
// split is the flattened (stage head group hg of plan_stage_heads(R) KV
// heads, virtual sequence, block) list of Ws entries cut over Ce_s CTAs.
struct SharedView {
    PlanView pv;
    const int32_t *skip;
    const float2 *ml_s;
    const float *acc_s;
    int64_t Ws;
    int32_t Ce_s;
};

__device__ __forceinline__ SharedView shared_view(const int32_t *plan, const int32_t *skip, const float2 *ml_s,
                                                  const float *acc_s, int32_t Hk, int32_t Cs) {
    SharedView sv;
    sv.pv = PlanView::at(plan);
    sv.skip = skip;
    sv.ml_s = ml_s;
    sv.acc_s = acc_s;
    sv.Ws = (int64_t)(Hk / plan_stage_heads(sv.pv.R)) * sv.pv.cu_s[sv.pv.V];
    sv.Ce_s = (int32_t)(sv.Ws < (int64_t)Cs ? sv.Ws : (int64_t)Cs);
    return sv;
}

// Pieces of the shared prefix of sequence seq for KV head kvh (none when the
// sequence is computed without sharing): the virtual sequence v that holds
// its G query rows, in slots c + hg * V + v (hg = kvh / heads per stage),
// rows (kvh % heads per stage) * R + row % R.
__device__ __forceinline__ PieceRange shared_range(const SharedView &sv, int32_t seq, int32_t kvh, int32_t G) {
    if (sv.skip[seq] <= 0) return no_range();
    const PlanView &pv = sv.pv;
    const int32_t R = pv.R, nhb = plan_stage_heads(R);
    const int32_t hg = kvh / nhb;
    const int32_t grp = pv.seq_group[seq];
    const int32_t row0 = pv.seq_member[seq] * G;
    const int32_t v = pv.group_vbase[grp] + row0 / R;
    const int64_t xs = (int64_t)hg * pv.cu_s[pv.V] + pv.cu_s[v];
    const int32_t P = pv.cu_s[v + 1] - pv.cu_s[v];
    return PieceRange{sv.ml_s, sv.acc_s, (int64_t)hg * pv.V + v, kPlanSlotRows, (kvh - hg * nhb) * R + row0 % R,
                      split_owner(xs, sv.Ws, sv.Ce_s), split_owner(xs + P - 1, sv.Ws, sv.Ce_s)};
}

// After a warp published a piece of (sequence seq, KV head kvh): count the
// arrival.  True for the warp whose piece arrived last; that warp merges.
__device__ __forceinline__ bool arrive_piece(unsigned int *__restrict__ counters, const PieceRange (&rg)[2],
                                             int64_t counter, int lane) {
    const unsigned int total = (unsigned int)(rg[0].c1 - rg[0].c0 + 1) +
                               (unsigned int)(rg[1].c1 >= rg[1].c0 ? rg[1].c1 - rg[1].c0 + 1 : 0);
    __threadfence();  // this lane's partial stores, before the arrival below
    __syncwarp();
    unsigned int last = 0;
    if (lane == 0) last = atomicAdd(&counters[counter], 1u) + 1u == total;
    return __shfl_sync(0xffffffffu, last, 0) != 0;
}

// Arrival counter of (sequence seq, KV head kvh): [head group][seq][head in group].
__device__ __forceinline__ int64_t counter_index(int32_t seq, int32_t kvh, int32_t N, int32_t NH) {
    const int32_t g = kvh / NH;
    return ((int64_t)g * N + seq) * NH + (kvh - g * NH);
}

// Count a published piece; the last arriver merges every piece of the pair.
template <typename T, int D>
__device__ __forceinline__ void finish_piece(T *__restrict__ out, const PieceRange (&rg)[2],
                                             unsigned int *__restrict__ counters, int32_t N, int32_t NH, int32_t H,
                                             int32_t G, int32_t seq, int32_t kvh, int lane) {
    if (!arrive_piece(counters, rg, counter_index(seq, kvh, N, NH), lane)) return;
    __threadfence();  // every other piece is published: read them
    merge_pieces<T, D>(out + ((int64_t)seq * H + (int64_t)kvh * G) * D, rg, G, lane);
}

// Workspace of the shared-prefix part of a launch (all nullptr without a plan).
struct SharedArgs {
    const int32_t *plan;   // the plan's words (device)
    const int32_t *skip;   // [N] shared blocks of each sequence, 0 = none (plan kernel)
    const int32_t *ctl;    // ctl[0]: CTAs given to shared prefixes (plan kernel)
    const int32_t *start_s;
    const int32_t *rowseq; // [V][R] sequence of each query row of each virtual sequence, -1 past
                           // the group's rows (plan kernel)
    float2 *ml_s;          // shared-prefix pieces: [slot][kPlanSlotRows] (m, l)
    float *acc_s;          //                       [slot][kPlanSlotRows][D]
    int32_t tc;            // 1: plans of 64 rows per pass run on tcgen05 (decode_tc.cuh)
};

// Single-pass merge (after the tensor-core kernel's block loop and in
// shared_merge_kernel, where registers are free): pieces are loaded kBatch at
// a time and folded in with a running maximum, so a merge costs one dependent
// load per batch.  Lanes as in merge_pieces_lph.
template <typename T, int D, int LPH, int kWideBatch>
__device__ __forceinline__ void merge_online_lph(T *__restrict__ out_base, const PieceRange (&rg)[2], int32_t G,
                                                 int lane) {
    // kBatch * E floats of pieces in flight; slices of 32 take kWideBatch
    constexpr int E = D / LPH, kBatch = E >= 32 ? kWideBatch : 4;
    static_assert(E % 4 == 0, "slices are whole float4s");
    const int h = lane / LPH, part = lane % LPH;
    if (h >= G) return;
    float a[E];
#pragma unroll
    for (int j = 0; j < E; ++j) a[j] = 0.f;
    float M = -INFINITY, Ls = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const PieceRange &p = rg[k];
#pragma unroll 1
        for (int32_t cb = p.c0; cb <= p.c1; cb += kBatch) {
            float4 x[kBatch][E / 4];
            float2 v[kBatch];
            float mb = -INFINITY;
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (cb + b <= p.c1) {
                    const int64_t idx = (cb + b + p.base) * p.stride + p.col + h;
                    const float4 *ap = reinterpret_cast<const float4 *>(p.acc + idx * D + part * E);
#pragma unroll
                    for (int j4 = 0; j4 < E / 4; ++j4) x[b][j4] = __ldcg(ap + j4);
                    v[b] = __ldcg(&p.ml[idx]);
                    mb = fmaxf(mb, v[b].x);
                }
            }
            const float Mn = fmaxf(M, mb);
            const float sc = M == -INFINITY ? 0.f : ex2_approx(M - Mn);  // every piece has a finite max
            Ls *= sc;
#pragma unroll
            for (int j = 0; j < E; ++j) a[j] *= sc;
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (cb + b <= p.c1) {
                    const float wgt = ex2_approx(v[b].x - Mn);
                    Ls = fmaf(wgt, v[b].y, Ls);
#pragma unroll
                    for (int j4 = 0; j4 < E / 4; ++j4) {
                        a[4 * j4 + 0] = fmaf(wgt, x[b][j4].x, a[4 * j4 + 0]);
                        a[4 * j4 + 1] = fmaf(wgt, x[b][j4].y, a[4 * j4 + 1]);
                        a[4 * j4 + 2] = fmaf(wgt, x[b][j4].z, a[4 * j4 + 2]);
                        a[4 * j4 + 3] = fmaf(wgt, x[b][j4].w, a[4 * j4 + 3]);
                    }
                }
            }
            M = Mn;
        }
    }
    const float inv = 1.f / Ls;
    T *o = out_base + (int64_t)h * D + part * E;
    store_slice<T, E>(o, a, inv);
}

// merge_online_lph with lanes per head chosen from G (as merge_pieces).
template <typename T, int D, int kWideBatch>
__device__ __forceinline__ void merge_online(T *__restrict__ out_base, const PieceRange (&rg)[2], int32_t G,
                                             int lane) {
    constexpr int kMaxLph = D / 4 < 32 ? D / 4 : 32;
    constexpr int kL8 = 8 < kMaxLph ? 8 : kMaxLph, kL16 = 16 < kMaxLph ? 16 : kMaxLph;
    if (G > 4)
        merge_online_lph<T, D, 4, kWideBatch>(out_base, rg, G, lane);
    else if (G > 2)
        merge_online_lph<T, D, kL8, kWideBatch>(out_base, rg, G, lane);
    else if (G > 1)
        merge_online_lph<T, D, kL16, kWideBatch>(out_base, rg, G, lane);
    else
        merge_online_lph<T, D, kMaxLph, kWideBatch>(out_base, rg, G, lane);
}

// One (sequence, KV head) merge of long_merge_kernel: thread i owns float4
// i of the G x D output (threads with i >= G * D / 4 have none) and folds the
// pieces kBatch at a time with a running maximum, in the same order on every
// call.
template <int D>
__device__ __forceinline__ void long_merge_one(__nv_bfloat16 *__restrict__ out, const PieceRange &p, int32_t H,
                                               int32_t G, int32_t NH, int32_t seq, int32_t g, int32_t w) {
    constexpr int kQ = D / 4, kBatch = 8;
    const int h = (int)threadIdx.x / kQ, q4 = (int)threadIdx.x - h * kQ;
    if (h >= G) return;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, Ls = 0.f;
#pragma unroll 1
    for (int32_t cb = p.c0; cb <= p.c1; cb += kBatch) {
        float4 x[kBatch];
        float2 v[kBatch];
        float mb = -INFINITY;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (cb + b <= p.c1) {
                const int64_t idx = (cb + b + p.base) * p.stride + p.col + h;
                x[b] = __ldcg(reinterpret_cast<const float4 *>(p.acc + idx * D) + q4);
                v[b] = __ldcg(&p.ml[idx]);
                mb = fmaxf(mb, v[b].x);
            }
        }
        const float Mn = fmaxf(M, mb);
        const float sc = M == -INFINITY ? 0.f : ex2_approx(M - Mn);  // every piece has a finite max
        Ls *= sc;
        a.x *= sc, a.y *= sc, a.z *= sc, a.w *= sc;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (cb + b <= p.c1) {
                const float wgt = ex2_approx(v[b].x - Mn);
                Ls = fmaf(wgt, v[b].y, Ls);
                a.x = fmaf(wgt, x[b].x, a.x), a.y = fmaf(wgt, x[b].y, a.y);
                a.z = fmaf(wgt, x[b].z, a.z), a.w = fmaf(wgt, x[b].w, a.w);
            }
        }
        M = Mn;
    }
    const float inv = 1.f / Ls;
    __nv_bfloat16 *o = out + ((int64_t)seq * H + (int64_t)(g * NH + w) * G + h) * D + q4 * 4;
    const uint32_t lo = pack_bf16x2(a.x * inv, a.y * inv), hi = pack_bf16x2(a.z * inv, a.w * inv);
    if (((uintptr_t)o & 7u) == 0) {  // out itself is only 4-byte aligned
        *reinterpret_cast<uint2 *>(o) = make_uint2(lo, hi);
    } else {
        reinterpret_cast<uint32_t *>(o)[0] = lo;
        reinterpret_cast<uint32_t *>(o)[1] = hi;
    }
}

// Whether the split cuts (head group g, sequence seq) into min_pieces or more.
__device__ __forceinline__ bool pair_is_long(const int32_t *cu, int32_t Wg, int64_t W, int32_t Ce, int32_t min_pieces,
                                             int32_t g, int32_t seq) {
    const int32_t nb = cu[seq + 1] - cu[seq];
    if (nb == 0) return false;
    const int64_t x0 = (int64_t)g * Wg + cu[seq];
    return split_owner(x0 + nb - 1, W, Ce) - split_owner(x0, W, Ce) + 1 >= min_pieces;
}

// Merge of the long sequences (after the attention launch, which leaves to
// this kernel every (sequence, KV head) cut into at least min_pieces pieces;
// whether a (head group, sequence) pair is long is decided from cu[] here
// exactly as there, so both agree whatever the caller's host hint was).
// With few pairs each CTA tests the pair of its own (pair, KV head) tasks.
// With many, the pairs are tested 256 at a time, one per thread, the long
// ones of each chunk listed in order in shared memory (every CTA builds the
// same list), and their merges dealt out over the grid.
template <int D>
__global__ void __launch_bounds__(256) long_merge_kernel(
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G,
    int32_t NH, int32_t C, const float2 *__restrict__ ml_ws, const float *__restrict__ acc_ws, int32_t min_pieces) {
    constexpr int kSmemCu = 4096, kChunk = 256;
    __shared__ int32_t cu_s[kSmemCu];
    __shared__ int32_t longs[kChunk];
    __shared__ int32_t warp_count[kChunk / 32];
    grid_dependency_wait();  // the attention launch's pieces (after the plan kernel's cu[])
    const bool in_smem = N + 1 <= kSmemCu;
    if (in_smem) {
        for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) cu_s[i] = cu[i];
        __syncthreads();
    }
    const int32_t *c = in_smem ? cu_s : cu;
    const int32_t NG = Hk / NH, Wg = c[N];
    const int64_t W = (int64_t)NG * Wg;
    const int32_t Ce = (int32_t)(W < (int64_t)C ? W : (int64_t)C);
    const int64_t pairs = (int64_t)NG * N;
    const bool direct = pairs * NH <= 2 * (int64_t)gridDim.x;
    const int i = threadIdx.x, lane = i & 31, wid = i >> 5;
    for (int64_t k0 = 0; k0 < pairs; k0 += direct ? pairs : kChunk) {
        int64_t total = pairs;  // direct: every pair is a candidate, tested by its CTA
        if (!direct) {
            const int64_t k = k0 + i;
            const bool is_long =
                k < pairs && pair_is_long(c, Wg, W, Ce, min_pieces, (int32_t)(k / N), (int32_t)(k - (k / N) * N));
            const unsigned int bal = __ballot_sync(0xffffffffu, is_long);
            if (lane == 0) warp_count[wid] = __popc(bal);
            __syncthreads();
            int32_t before = 0, cnt = 0;
            for (int w = 0; w < kChunk / 32; ++w) {
                before += w < wid ? warp_count[w] : 0;
                cnt += warp_count[w];
            }
            if (is_long) longs[before + __popc(bal & ((1u << lane) - 1u))] = (int32_t)(k - k0);
            __syncthreads();
            total = cnt;
        }
        for (int64_t t = blockIdx.x; t < total * NH; t += gridDim.x) {
            const int64_t kk = direct ? t / NH : k0 + longs[t / NH];
            const int32_t g = (int32_t)(kk / N), seq = (int32_t)(kk - (int64_t)g * N), w = (int32_t)(t % NH);
            if (direct && c[seq + 1] == c[seq]) continue;  // empty
            const PieceRange p = own_range(ml_ws, acc_ws, c, N, seq, g, w, G, NH * G, W, Ce);
            if (direct && p.c1 - p.c0 + 1 < min_pieces) continue;  // merged in the attention launch
            long_merge_one<D>(out, p, H, G, NH, seq, g, w);
        }
        if (!direct) __syncthreads();  // the list is rebuilt for the next chunk
    }
}

// Merge of the sequences with a shared prefix (after the attention launch,
// which left their pieces in the workspace): one warp per (member of a
// group, KV head).  The piece ranges depend only on the plan kernel's output,
// so they are worked out before waiting for the attention launch (which lets
// this grid start as its CTAs finish); only the pieces are read after it.
// Every thread waits, also those with nothing to merge (a rejected plan, a
// sequence computed without sharing): this grid must not end before the
// attention launch, since work after it on the stream may rely on both.
template <int D>
__global__ void __launch_bounds__(256, 2) shared_merge_kernel(
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G,
    int32_t NH, int32_t C, const float2 *__restrict__ ml_ws, const float *__restrict__ acc_ws, const SharedArgs sh) {
    const int32_t Cs = sh.ctl[0];
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    int32_t seq = -1, kvh = 0;
    PieceRange own = no_range(), shr = no_range();
    // Cs <= 0: plan rejected, every sequence was merged in the attention launch
    if (Cs > 0) {
        const SharedView sv = shared_view(sh.plan, sh.skip, sh.ml_s, sh.acc_s, Hk, Cs);
        if (wid < (int64_t)sv.pv.M * Hk) {
            seq = sv.pv.members[wid / Hk];
            kvh = (int32_t)(wid % Hk);
            if (sh.skip[seq] > 0) {
                const int64_t W = (int64_t)(Hk / NH) * cu[N];
                const int32_t Ce = (int32_t)(W < (int64_t)(C - Cs) ? W : (int64_t)(C - Cs));
                own = own_range(ml_ws, acc_ws, cu, N, seq, kvh / NH, kvh % NH, G, NH * G, W, Ce);
                shr = shared_range(sv, seq, kvh, G);
            } else {
                seq = -1;  // computed without sharing: merged in the attention launch
            }
        }
    }
    grid_dependency_wait();  // the attention launch's pieces
    if (seq >= 0) {
        // the ranges' arrays are these parameters: only their indexes were kept across the wait
        const PieceRange rg[2] = {PieceRange{ml_ws, acc_ws, own.base, own.stride, own.col, own.c0, own.c1},
                                  PieceRange{sh.ml_s, sh.acc_s, shr.base, shr.stride, shr.col, shr.c0, shr.c1}};
        merge_online<__nv_bfloat16, D, 2>(out + ((int64_t)seq * H + (int64_t)kvh * G) * D, rg, G, lane);
    }
}

}  // namespace pa
