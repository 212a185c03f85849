// Paged decode attention (pa_decode).
//
// What is computed: for every sequence i and query head h,
//   out[i, h] = softmax_j(scale * q[i, h] . K_j) V_j   over j < seq_lens[i],
// with K_j, V_j the cache rows of slot table[i][j / B] * B + j % B
// ("10 PagedAttention" (PidokuInfra), section 4 PhysicalIndex and section 5
// "The kernel side"; "PagedAttention" (tokentrails), step 3: the same
// attention as over contiguous memory).  Query head h reads KV head
// h / (H / Hk).
//
// How (GB300 design; the pages give only a one-CTA-per-(seq, head) sketch):
// 1. decode_plan_kernel: one CTA turns seq_lens into block counts and their
//    exclusive prefix sums cu[], clamps bad lengths (recording them), zeroes
//    the merge counters and writes the zero output of empty sequences.
// 2. A persistent grid of C CTAs splits the flattened list of
//    (KV-head group, sequence, block) into Ce = min(C, W) equal contiguous
//    ranges (split_begin).  A CTA walks its range; each of its consumer warps
//    owns one KV head and all G query heads that share it, so each KV byte is
//    read from HBM once.  A range piece covering a whole sequence writes `out`
//    directly.  A piece of a longer sequence writes an unnormalised partial
//    (running max m in log2 units, sum l, accumulator) to the workspace and
//    bumps an arrival counter for its (sequence, KV head); the warp that
//    arrives last merges every piece (the split-K reduce, fused):
//      out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
//    Nothing ever waits for another CTA: the merge is done by whoever is last.
//
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

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

// ---------------------------------------------------------------- plan kernel
// Checks a shared-prefix plan's words against the call (sizes, heads per KV
// head, block size, and every index it holds), so that a bad plan can only
// switch sharing off, never send a kernel out of bounds.  Block-wide; every
// thread returns the verdict.
__device__ bool plan_valid(const int32_t *__restrict__ w, int32_t N, int32_t G, int32_t B, int32_t max_blocks,
                           int *s_flag, int *s_count) {
    if (threadIdx.x == 0) {
        const int32_t groups = w[4], M = w[5], V = w[6];
        const int32_t R = w[7];
        bool ok = w[0] == kPlanMagic && w[1] == N && w[2] == G && w[3] == B && groups >= 0 && groups <= N &&
                  M >= 0 && M <= N && V >= 0 && V <= N && R == kPlanRows && G <= 8 && 8 % G == 0 &&
                  PlanView::words(N, groups, M, V) <= 7 * (int64_t)N + 16;
        if (ok) {
            const PlanView pv = PlanView::at(w);
            ok = pv.group_begin[0] == 0 && pv.group_begin[groups] == M && pv.group_vbase[0] == 0 &&
                 pv.group_vbase[groups] == V && pv.cu_s[0] == 0;
        }
        *s_flag = ok ? 1 : 0;
        *s_count = 0;
    }
    __syncthreads();
    if (!*s_flag) return false;
    const PlanView pv = PlanView::at(w);
    bool ok = true;
    for (int32_t g = threadIdx.x; g < pv.groups; g += blockDim.x) {
        const int32_t S = pv.group_begin[g + 1] - pv.group_begin[g];
        const int32_t passes = pv.group_vbase[g + 1] - pv.group_vbase[g];
        ok = ok && S >= 1 && passes == (S * G + kPlanRows - 1) / kPlanRows && pv.group_prefix[g] >= 1 &&
             pv.group_prefix[g] <= max_blocks;
    }
    // From here group_begin and group_vbase are increasing from 0 to M and V,
    // so indexes built from them stay inside members[] and the virtual list.
    if (!__syncthreads_and(ok)) return false;
    for (int32_t k = threadIdx.x; k < pv.M; k += blockDim.x) ok = ok && pv.members[k] >= 0 && pv.members[k] < N;
    for (int32_t v = threadIdx.x; v < pv.V; v += blockDim.x) {
        const int32_t g = pv.vgroup[v];
        ok = ok && g >= 0 && g < pv.groups && pv.group_vbase[g] <= v && v < pv.group_vbase[g + 1] &&
             pv.cu_s[v + 1] - pv.cu_s[v] == pv.group_prefix[g];
    }
    int32_t grouped = 0;
    for (int32_t i = threadIdx.x; i < N; i += blockDim.x) {
        const int32_t g = pv.seq_group[i];
        if (g == -1) continue;
        ++grouped;
        if (g < 0 || g >= pv.groups) {
            ok = false;
            continue;
        }
        const int32_t m = pv.seq_member[i];
        ok = ok && m >= 0 && m < pv.group_begin[g + 1] - pv.group_begin[g] && pv.members[pv.group_begin[g] + m] == i;
    }
    if (grouped) atomicAdd(s_count, grouped);
    // Every grouped sequence points at a distinct member slot holding it, and
    // there are as many grouped sequences as slots: the two agree exactly.
    ok = __syncthreads_and(ok) != 0;
    return ok && *s_count == pv.M;
}

template <typename T>
__global__ void __launch_bounds__(1024) decode_plan_kernel(const int32_t *__restrict__ seq_lens, int32_t N,
                                                           int32_t B, int32_t max_len, int32_t HD,
                                                           int32_t *__restrict__ lens_ws,
                                                           int32_t *__restrict__ cu,
                                                           unsigned int *__restrict__ counters,
                                                           int32_t num_counters, T *__restrict__ out,
                                                           int32_t NG, int32_t C,
                                                           int32_t *__restrict__ start_seq,
                                                           unsigned int *__restrict__ err,
                                                           const int32_t *__restrict__ plan, int32_t G,
                                                           int32_t Hk, int32_t NH, int32_t *__restrict__ skip,
                                                           int32_t *__restrict__ ctl,
                                                           int32_t *__restrict__ start_s, int32_t plan_in_smem) {
    grid_dependency_wait();     // inputs written by earlier work on the stream
    grid_launch_dependents();   // the attention kernel may become resident now
    constexpr int32_t kSmemCu = 2048;  // prefix sums kept in shared memory for the start search
    __shared__ int32_t warp_incl[32];
    __shared__ int32_t carry;
    __shared__ int32_t n_empty;
    __shared__ int32_t empty_ids[1024];
    __shared__ int32_t cu_s[kSmemCu];
    __shared__ int s_flag, s_count, s_cs;
    const bool cu_in_smem = N + 1 <= kSmemCu;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    for (int32_t i = threadIdx.x; i < num_counters; i += blockDim.x) counters[i] = 0u;
    // The plan's words (the caller's buffer holds 7 N + 16 of them), copied to
    // shared memory in one coalesced pass when they fit, so that its checks
    // and lookups below are not chains of global loads.
    extern __shared__ int32_t plan_sm[];
    if (plan && plan_in_smem) {
        const int32_t words = 7 * N + 16;
        for (int32_t i = threadIdx.x; i < words; i += blockDim.x) plan_sm[i] = plan[i];
        __syncthreads();
        plan = plan_sm;
    }
    // A shared-prefix plan that does not match the call switches sharing off.
    const bool plan_ok = plan && plan_valid(plan, N, G, B, max_len / B, &s_flag, &s_count);
    if (plan && !plan_ok && threadIdx.x == 0) atomicOr(err, kErrPlan);
    const PlanView pv = plan_ok ? PlanView::at(plan) : PlanView{};
    for (int32_t base = 0; base < N; base += blockDim.x) {
        if (threadIdx.x == 0) n_empty = 0;
        __syncthreads();
        const int32_t i = base + threadIdx.x;
        int32_t nb = 0;
        if (i < N) {
            int32_t L = seq_lens[i];
            if (L < 0 || L > max_len) {
                atomicOr(err, kErrLength);
                L = 0;
            }
            lens_ws[i] = L;
            nb = (L + B - 1) / B;
            if (L == 0) empty_ids[atomicAdd(&n_empty, 1)] = i;
            // Shared prefix blocks are read by the shared-prefix CTAs; this
            // sequence keeps the rest (at least one position, else no sharing).
            int32_t sk = 0;
            if (plan_ok && pv.seq_group[i] >= 0) {
                const int32_t P = pv.group_prefix[pv.seq_group[i]];
                if ((int64_t)P * B < L)
                    sk = P;
                else
                    atomicOr(err, kErrPlan);
            }
            if (skip) skip[i] = sk;
            nb -= sk;
        }
        int32_t x = nb;  // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_incl[w] = x;
        __syncthreads();
        if (w == 0) {
            int32_t s = lane < nwarps ? warp_incl[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_incl[lane] = s;
        }
        __syncthreads();
        const int32_t incl = x + (w > 0 ? warp_incl[w - 1] : 0) + carry;
        if (i < N) {
            cu[i] = incl - nb;
            if (cu_in_smem) cu_s[i] = incl - nb;
        }
        // empty sequences of this pass: their output is zero
        for (int32_t k = 0; k < n_empty; ++k) {
            T *o = out + (int64_t)empty_ids[k] * HD;
            for (int32_t e = threadIdx.x; e < HD; e += blockDim.x) store_out(o + e, 0.f);
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        cu[N] = carry;
        if (cu_in_smem) cu_s[N] = carry;
        // CTAs for the shared prefixes, in proportion to the bytes they read
        // (a shared unit is one KV head of a block, an own unit NH heads).
        int32_t cs = 0;
        if (plan_ok) {
            const int64_t Ws = (int64_t)Hk * pv.cu_s[pv.V], Wo = (int64_t)NG * carry * NH;
            if (Ws > 0) {
                const double share = (double)Ws / (double)(Ws + Wo);
                cs = (int32_t)((double)C * share + 0.5);
                cs = cs < 1 ? 1 : (cs > C - 1 ? C - 1 : cs);
            }
        }
        s_cs = cs;
        if (ctl) ctl[0] = cs;
    }
    __syncthreads();
    // Sequence holding the first block of each own-block CTA's range, so the
    // CTA starts without searching cu[].
    const int32_t *cus = cu_in_smem ? cu_s : cu;
    const int32_t Wg = cus[N];
    const int64_t W = (int64_t)NG * Wg;
    const int32_t Co = C - s_cs;
    const int32_t Ce = (int32_t)(W < (int64_t)Co ? W : (int64_t)Co);
    for (int32_t c = threadIdx.x; c < Ce; c += blockDim.x) {
        const int32_t r = (int32_t)(split_begin(c, W, Ce) % Wg);
        int32_t lo = 0, hi = N - 1;  // largest seq with cu[seq] <= r
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (cus[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        start_seq[c] = lo;
    }
    // The same for the shared-prefix CTAs over the virtual sequences.
    if (s_cs > 0) {
        const int32_t Wv = pv.cu_s[pv.V];
        const int64_t Ws = (int64_t)(Hk / kPlanHeads) * Wv;
        const int32_t Ce_s = (int32_t)(Ws < (int64_t)s_cs ? Ws : (int64_t)s_cs);
        for (int32_t c = threadIdx.x; c < Ce_s; c += blockDim.x) {
            const int32_t r = (int32_t)(split_begin(c, Ws, Ce_s) % Wv);
            int32_t lo = 0, hi = pv.V - 1;
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (pv.cu_s[mid] <= r)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            start_s[c] = lo;
        }
    }
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

// Run by the warp that finished the last piece of one (sequence, KV head):
// merges both ranges for its G query heads.  Lanes split the G heads x D
// outputs: LPH lanes per head, each a contiguous slice of E = D / LPH
// elements.  With LPH a compile-time constant every load of a piece is issued
// back to back (the merge runs at the end of the kernel, so its L2 latency is
// on the kernel's critical path); two passes, the maximum over all pieces
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
// split is the flattened (head group hg of kPlanHeads heads, virtual
// sequence, block) list of Ws entries cut over Ce_s CTAs.
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
    sv.Ws = (int64_t)(Hk / kPlanHeads) * sv.pv.cu_s[sv.pv.V];
    sv.Ce_s = (int32_t)(sv.Ws < (int64_t)Cs ? sv.Ws : (int64_t)Cs);
    return sv;
}

// Pieces of the shared prefix of sequence seq for KV head kvh (none when the
// sequence is computed without sharing): the virtual sequence v that holds
// its G query rows, in slots c + hg * V + v, rows (kvh % 4) * 16 + row % 16.
__device__ __forceinline__ PieceRange shared_range(const SharedView &sv, int32_t seq, int32_t kvh, int32_t G) {
    if (sv.skip[seq] <= 0) return no_range();
    const PlanView &pv = sv.pv;
    const int32_t hg = kvh / kPlanHeads;
    const int32_t grp = pv.seq_group[seq];
    const int32_t row0 = pv.seq_member[seq] * G;
    const int32_t v = pv.group_vbase[grp] + row0 / kPlanRows;
    const int64_t xs = (int64_t)hg * pv.cu_s[pv.V] + pv.cu_s[v];
    const int32_t P = pv.cu_s[v + 1] - pv.cu_s[v];
    return PieceRange{sv.ml_s, sv.acc_s, (int64_t)hg * pv.V + v, kPlanSlotRows,
                      (kvh - hg * kPlanHeads) * kPlanRows + row0 % kPlanRows, split_owner(xs, sv.Ws, sv.Ce_s),
                      split_owner(xs + P - 1, sv.Ws, sv.Ce_s)};
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

// ------------------------------------------------------- CUDA-core kernel
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T, int VPL>
__device__ __forceinline__ void load_row_slice(const T *__restrict__ p, float (&x)[VPL]) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) x[j] = to_f32<T>(p[j]);
}

// Block tile: NH warps, warp w handles KV head g*NH + w and its G (<= GMAX)
// query heads, one token at a time (lane holds D/32 consecutive elements).
template <typename T, int D, int GMAX, int LAYOUT>
__global__ void __launch_bounds__(256) decode_simt_kernel(
    const T *__restrict__ q, T *__restrict__ out, const T *__restrict__ k_cache,
    const T *__restrict__ v_cache, const int32_t *__restrict__ tables, int32_t max_blocks,
    const int32_t *__restrict__ lens, const int32_t *__restrict__ cu, int32_t N, int32_t H,
    int32_t Hk, int32_t G, int32_t B, int32_t NB, int32_t NH, float scale_log2, int32_t C,
    float2 *__restrict__ ml_ws, float *__restrict__ acc_ws, unsigned int *__restrict__ counters,
    const int32_t *__restrict__ start_seq, unsigned int *__restrict__ err) {
    constexpr int VPL = D / 32;
    grid_dependency_wait();  // the plan kernel's cu[] / lens (programmatic launch)
    const int32_t NG = Hk / NH;
    const int32_t HPG = NH * G;
    const int64_t W = (int64_t)NG * cu[N];
    const int32_t Ce = (int32_t)(W < (int64_t)C ? W : (int64_t)C);  // no CTA with an empty range
    const int32_t c = blockIdx.x;
    if (c >= Ce) return;
    const int64_t lo = split_begin(c, W, Ce), hi = split_begin(c + 1, W, Ce);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    BlockCursor cur;
    cur.init_at(lo, start_seq[c], cu, N);
    float qv[GMAX][VPL], acc[GMAX][VPL], m[GMAX], l[GMAX];
    bool seg_start = true, seg_from_first = false;
    int32_t L = 0;
    for (int64_t x = lo; x < hi; ++x) {
        const int32_t kvh = cur.g * NH + warp;
        if (seg_start) {
            L = lens[cur.seq];
            const T *qp = q + ((int64_t)cur.seq * H + (int64_t)kvh * G) * D + lane * VPL;
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                if (h < G) {
                    load_row_slice<T, VPL>(qp + (int64_t)h * D, qv[h]);
                } else {
#pragma unroll
                    for (int j = 0; j < VPL; ++j) qv[h][j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < VPL; ++j) acc[h][j] = 0.f;
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
            seg_from_first = (cur.blk == 0);
            seg_start = false;
        }
        int32_t phys = tables[(int64_t)cur.seq * max_blocks + cur.blk];
        const bool valid = phys >= 0 && phys < NB;
        if (!valid && lane == 0) atomicOr(err, kErrBounds);
        const int32_t tok0 = cur.blk * B;
        const int32_t ntok = min(B, L - tok0);
        for (int32_t t = 0; t < ntok; ++t) {
            float kx[VPL], vx[VPL];
            if (valid && LAYOUT == PA_LAYOUT_ROW) {
                const int64_t row = (((int64_t)phys * B + t) * Hk + kvh) * D + lane * VPL;
                load_row_slice<T, VPL>(k_cache + row, kx);
                load_row_slice<T, VPL>(v_cache + row, vx);
            } else if (valid) {
                // split layout: K [NB, Hk, D/X, B, X], V [NB, Hk, D, B]
                constexpr int X = 16 / (int)sizeof(T);
                const int64_t head = (int64_t)phys * Hk + kvh;
#pragma unroll
                for (int j = 0; j < VPL; ++j) {
                    const int d = lane * VPL + j;
                    kx[j] = to_f32<T>(k_cache[((head * (D / X) + d / X) * B + t) * X + d % X]);
                    vx[j] = to_f32<T>(v_cache[(head * D + d) * B + t]);
                }
            } else {  // an invalid block id reads zeros (as the TMA kernel does)
#pragma unroll
                for (int j = 0; j < VPL; ++j) kx[j] = vx[j] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                if (h >= G) break;
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < VPL; ++j) s = fmaf(qv[h][j], kx[j], s);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                const float xs = s * scale_log2;
                const float mn = fmaxf(m[h], xs);
                const float alpha = ex2_approx(m[h] - mn);
                const float p = ex2_approx(xs - mn);
                l[h] = l[h] * alpha + p;
#pragma unroll
                for (int j = 0; j < VPL; ++j) acc[h][j] = fmaf(acc[h][j], alpha, p * vx[j]);
                m[h] = mn;
            }
        }
        const bool last_blk = (cur.blk == cur.nb - 1);
        if (last_blk || x + 1 == hi) {
            const int32_t sp = cur.g * N + cur.seq;
            if (seg_from_first && last_blk) {
                T *op = out + ((int64_t)cur.seq * H + (int64_t)kvh * G) * D + lane * VPL;
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h >= G) break;
                    const float inv = 1.f / l[h];
#pragma unroll
                    for (int j = 0; j < VPL; ++j) store_out(op + (int64_t)h * D + j, acc[h][j] * inv);
                }
            } else {
                const int64_t slot = partial_slot(c, sp);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h >= G) break;
                    const int64_t hh = slot * HPG + warp * G + h;
                    float *ap = acc_ws + hh * D + lane * VPL;
#pragma unroll
                    for (int j = 0; j < VPL; ++j) ap[j] = acc[h][j];
                    if (lane == 0) ml_ws[hh] = make_float2(m[h], l[h]);
                }
                const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, cur.seq, cur.g, warp, G, HPG, W, Ce),
                                          no_range()};
                finish_piece<T, D>(out, rg, counters, N, NH, H, G, cur.seq, kvh, lane);
            }
            seg_start = true;
        }
        cur.advance(cu, N);
    }
}

// ------------------------------------------------- TMA + tensor-core kernel
// Shared-memory tile of one stage and one tensor (K or V): the TMA box
// {64 elements, B tokens, D/64 halves, NH heads}, i.e. [head][half][token][64]
// with 128-byte lines swizzled (16-byte chunk index XOR line % 8).
template <int D, int B>
struct MmaTile {
    static constexpr int kHalves = D / 64;
    static constexpr int kSlabBytes = kHalves * B * 128;  // one head
    static constexpr int kStages = kMmaStages;
};

__device__ __forceinline__ uint32_t swz_addr(uint32_t slab, int line, int chunk) {
    return slab + (uint32_t)line * 128u + ((uint32_t)(chunk ^ (line & 7)) << 4);
}

// One staged block for one consumer warp: S^T (16 tokens x 8 query rows) =
// K Q^T per 16-token slice, online softmax in log2 units, O^T (D x 8) +=
// V^T P^T.  Token rows at or past L are masked (their V rows must be finite).
template <int D, int B, int LAYOUT>
__device__ __forceinline__ void mma_block(uint32_t kslab, uint32_t vslab, int32_t tok0, int32_t L,
                                          float scale_log2, const uint32_t (&qf)[D / 16][2],
                                          float (&o)[D / 16][4], float &m0, float &m1, float &l0, float &l1,
                                          int lane) {
    constexpr int KT = D / 16;
    const int r = lane >> 2;                  // mma groupID
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix id / row id
#pragma unroll
    for (int mt = 0; mt < B / 16; ++mt) {
        if (tok0 + mt * 16 >= L) break;
        // S^T (16 tokens x 8 heads) = K (16 x D) Q^T (D x 8)
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            const int t = mt * 16 + rr + (mi & 1) * 8;
            const int d = kk * 16 + (mi >> 1) * 8;
            uint32_t a0, a1, a2, a3;
            if (LAYOUT == PA_LAYOUT_ROW)
                ldmatrix_x4(swz_addr(kslab, (d >> 6) * B + t, (d & 63) >> 3), a0, a1, a2, a3);
            else  // split K tile [d / 8][token][8]: 8 tokens of a chunk are 128 contiguous bytes
                ldmatrix_x4(kslab + (uint32_t)(((d >> 3) * B + t) * 16), a0, a1, a2, a3);
            mma_bf16_16816(sacc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
        // online softmax in log2 units; rows = tokens, columns = heads
        const int ta = tok0 + mt * 16 + r, tb = ta + 8;
        const float x0 = ta < L ? sacc[0] * scale_log2 : -INFINITY;
        const float x1 = ta < L ? sacc[1] * scale_log2 : -INFINITY;
        const float x2 = tb < L ? sacc[2] * scale_log2 : -INFINITY;
        const float x3 = tb < L ? sacc[3] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = ex2_approx(m0 - mn0), al1 = ex2_approx(m1 - mn1);
        const float p0 = ex2_approx(x0 - mn0), p1 = ex2_approx(x1 - mn1);
        const float p2 = ex2_approx(x2 - mn0), p3 = ex2_approx(x3 - mn1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int dm = 0; dm < KT; ++dm) {
            o[dm][0] *= al0;
            o[dm][1] *= al1;
            o[dm][2] *= al0;
            o[dm][3] *= al1;
        }
        // P^T as the B operand: transpose the two 8x8 bf16 quadrants.
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
        // O^T (D x 8 heads) += V^T (D x 16 tokens) P^T (16 tokens x 8 heads)
#pragma unroll
        for (int dm = 0; dm < KT; ++dm) {
            uint32_t a0, a1, a2, a3;
            if (LAYOUT == PA_LAYOUT_ROW) {  // rows are tokens: transpose on load
                const int t = mt * 16 + rr + (mi >> 1) * 8;
                const int d = dm * 16 + (mi & 1) * 8;
                ldmatrix_x4_trans(swz_addr(vslab, (d >> 6) * B + t, (d & 63) >> 3), a0, a1, a2, a3);
            } else {  // split V tile [d][token]: rows are already V^T
                const int d = dm * 16 + rr + (mi & 1) * 8;
                const int t = mt * 16 + (mi >> 1) * 8;
                ldmatrix_x4(vslab + (uint32_t)((d * B + t) * 2), a0, a1, a2, a3);
            }
            mma_bf16_16816(o[dm], a0, a1, a2, a3, pb0, pb1);
        }
    }
}

// Shared-memory rows of the query block of one shared-prefix warp: 16 rows
// of D bf16, padded by 16 bytes so that the 8 rows an ldmatrix reads fall in
// distinct banks.
template <int D>
struct QRows {
    static constexpr int kRowBytes = D * 2 + 16;
    static constexpr int kBytes = kPlanRows * kRowBytes;
};

// The same as mma_block for NT 8-column tiles of query rows (NT * 8 rows) that
// share the staged block: every K and V fragment is loaded from shared memory
// once and used for all NT tiles.  The query rows are in shared memory at qsm
// (QRows layout) and are read per k-step, so they hold no registers across
// blocks.  All B tokens are valid (shared-prefix blocks are full).
template <int D, int B, int LAYOUT, int NT>
__device__ __forceinline__ void mma_block_tiles(uint32_t kslab, uint32_t vslab, uint32_t qsm, float scale_log2,
                                                float (&o)[NT][D / 16][4], float (&m)[NT][2], float (&l)[NT][2],
                                                int lane) {
    static_assert(NT == 2, "one ldmatrix.x4 gives the B fragments of two tiles");
    constexpr int KT = D / 16;
    const int mi = lane >> 3, rr = lane & 7;
    // ldmatrix.x4 of the query rows: matrix mi = (tile mi >> 1, d half mi & 1)
    const uint32_t qrow = qsm + (uint32_t)(((mi >> 1) * 8 + rr) * QRows<D>::kRowBytes + (mi & 1) * 16);
#pragma unroll
    for (int mt = 0; mt < B / 16; ++mt) {
        float sacc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) sacc[t][0] = sacc[t][1] = sacc[t][2] = sacc[t][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            const int tk = mt * 16 + rr + (mi & 1) * 8;
            const int d = kk * 16 + (mi >> 1) * 8;
            uint32_t a0, a1, a2, a3, b00, b01, b10, b11;
            if (LAYOUT == PA_LAYOUT_ROW)
                ldmatrix_x4(swz_addr(kslab, (d >> 6) * B + tk, (d & 63) >> 3), a0, a1, a2, a3);
            else
                ldmatrix_x4(kslab + (uint32_t)(((d >> 3) * B + tk) * 16), a0, a1, a2, a3);
            ldmatrix_x4(qrow + (uint32_t)(kk * 32), b00, b01, b10, b11);
            mma_bf16_16816(sacc[0], a0, a1, a2, a3, b00, b01);
            mma_bf16_16816(sacc[1], a0, a1, a2, a3, b10, b11);
        }
        uint32_t pb0[NT], pb1[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float x0 = sacc[t][0] * scale_log2, x1 = sacc[t][1] * scale_log2;
            const float x2 = sacc[t][2] * scale_log2, x3 = sacc[t][3] * scale_log2;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
            const float al0 = ex2_approx(m[t][0] - mn0), al1 = ex2_approx(m[t][1] - mn1);
            const float p0 = ex2_approx(x0 - mn0), p1 = ex2_approx(x1 - mn1);
            const float p2 = ex2_approx(x2 - mn0), p3 = ex2_approx(x3 - mn1);
            l[t][0] = l[t][0] * al0 + (p0 + p2);
            l[t][1] = l[t][1] * al1 + (p1 + p3);
            m[t][0] = mn0;
            m[t][1] = mn1;
#pragma unroll
            for (int dm = 0; dm < KT; ++dm) {
                o[t][dm][0] *= al0;
                o[t][dm][1] *= al1;
                o[t][dm][2] *= al0;
                o[t][dm][3] *= al1;
            }
            pb0[t] = movmatrix_trans(pack_bf16x2(p0, p1));
            pb1[t] = movmatrix_trans(pack_bf16x2(p2, p3));
        }
#pragma unroll
        for (int dm = 0; dm < KT; ++dm) {
            uint32_t a0, a1, a2, a3;
            if (LAYOUT == PA_LAYOUT_ROW) {
                const int tk = mt * 16 + rr + (mi >> 1) * 8;
                const int d = dm * 16 + (mi & 1) * 8;
                ldmatrix_x4_trans(swz_addr(vslab, (d >> 6) * B + tk, (d & 63) >> 3), a0, a1, a2, a3);
            } else {
                const int d = dm * 16 + rr + (mi & 1) * 8;
                const int tk = mt * 16 + (mi >> 1) * 8;
                ldmatrix_x4(vslab + (uint32_t)((d * B + tk) * 2), a0, a1, a2, a3);
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) mma_bf16_16816(o[t][dm], a0, a1, a2, a3, pb0[t], pb1[t]);
        }
    }
}

// Workspace of the shared-prefix part of a launch (all nullptr without a plan).
struct SharedArgs {
    const int32_t *plan;   // the plan's words (device)
    const int32_t *skip;   // [N] shared blocks of each sequence, 0 = none (plan kernel)
    const int32_t *ctl;    // ctl[0]: CTAs given to shared prefixes (plan kernel)
    const int32_t *start_s;
    float2 *ml_s;          // shared-prefix pieces: [slot][kPlanSlotRows] (m, l)
    float *acc_s;          //                       [slot][kPlanSlotRows][D]
};

// A CTA of the shared-prefix part.  Its range of the flattened (head group
// hg, virtual sequence v, block) list: W_s = (Hk / 4) * cu_s[V] entries cut
// over Ce_s CTAs.  The ring, its stages and the TMA box of 4 KV heads are the
// own-block CTAs'.  Each block of a group's prefix is read once (the table of
// the group's first member) and warp w applies head hg * 4 + w to the pass's
// 16 query rows (member m = row / G, query head h = kvh * G + row % G), as
// two 8-column MMA tiles.  A piece's partial goes to slot c + hg * V + v, and
// each member sequence whose rows it holds gets an arrival on its
// (sequence, KV head) counter; the last arriver merges.
template <int D, int B, int LAYOUT>
__device__ __forceinline__ void shared_prefix_cta(
    uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const __nv_bfloat16 *__restrict__ q,
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ tables, int32_t max_blocks, int32_t H,
    int32_t G, int32_t NB, float scale_log2, unsigned int *__restrict__ counters,
    const int32_t *__restrict__ cu, int32_t N, int32_t NH, int32_t Hk, int32_t C, int32_t Cs, float2 *ml_ws,
    float *acc_ws, const SharedArgs &sh, unsigned int *__restrict__ err) {
    using Tile = MmaTile<D, B>;
    constexpr int S = Tile::kStages;
    constexpr int KT = D / 16;
    constexpr int NT = kPlanRows / 8;  // MMA tiles per warp
    constexpr uint32_t tile_bytes = kPlanHeads * Tile::kSlabBytes, stage_bytes = 2 * tile_bytes;
    uint64_t *full = (uint64_t *)(smem + S * stage_bytes);
    uint64_t *empty = full + S;
    uint8_t *qbuf = smem + S * stage_bytes + 256;  // QRows of each consumer warp
    const SharedView sv = shared_view(sh.plan, sh.skip, sh.ml_s, sh.acc_s, Hk, Cs);
    const PlanView &pv = sv.pv;
    const int32_t c = blockIdx.x;
    if (c >= sv.Ce_s) return;
    const int64_t lo = split_begin(c, sv.Ws, sv.Ce_s), hi = split_begin(c + 1, sv.Ws, sv.Ce_s);
    const int64_t n = hi - lo;
    const int32_t V = pv.V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), (uint32_t)kPlanHeads);
        }
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == kPlanHeads) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(tmk);
            prefetch_tmap(tmv);
            const uint64_t kv_policy = l2_policy_evict_first();  // each shared block is read once
            BlockCursor cur, ahead;
            cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
            ahead.init_at(lo, sh.start_s[c], pv.cu_s, V);
            // table row of a virtual sequence: its group's first member
            auto rep_row = [&](int32_t v) {
                return (int64_t)pv.members[pv.group_begin[pv.vgroup[v]]] * max_blocks;
            };
            int32_t ahead_v = ahead.seq;
            int64_t ahead_row = rep_row(ahead_v);
            constexpr int PD = kTablePrefetch;
            int32_t ring[PD];
#pragma unroll
            for (int j = 0; j < PD; ++j) {
                if (j < n) {
                    if (ahead.seq != ahead_v) {
                        ahead_v = ahead.seq;
                        ahead_row = rep_row(ahead_v);
                    }
                    ring[j] = tables[ahead_row + ahead.blk];
                    ahead.advance(pv.cu_s, V);
                } else {
                    ring[j] = 0;
                }
            }
            int64_t issued = 0;
            for (; issued < n; ++issued) {
                const int s = (int)(issued % S);
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                int32_t phys = ring[0];
#pragma unroll
                for (int j = 0; j + 1 < PD; ++j) ring[j] = ring[j + 1];
                if (issued + PD < n) {
                    if (ahead.seq != ahead_v) {
                        ahead_v = ahead.seq;
                        ahead_row = rep_row(ahead_v);
                    }
                    ring[PD - 1] = tables[ahead_row + ahead.blk];
                    ahead.advance(pv.cu_s, V);
                }
                if (issued >= S && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u)) {
                    atomicOr(err, kErrTimeout);
                    break;
                }
                if (phys < 0 || phys >= NB) {  // read zeros: the box lies past the pool
                    atomicOr(err, kErrBounds);
                    phys = NB;
                }
                const uint32_t fb = smem_u32(&full[s]);
                const uint32_t dst = smem_u32(smem + (size_t)s * stage_bytes);
                mbar_arrive_expect_tx(fb, stage_bytes);
                if (LAYOUT == PA_LAYOUT_ROW) {
                    tma_load_4d_hint(dst, tmk, fb, 0, phys * B, 0, cur.g * kPlanHeads, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, tmv, fb, 0, phys * B, 0, cur.g * kPlanHeads, kv_policy);
                } else {
                    tma_load_4d_hint(dst, tmk, fb, 0, 0, cur.g * kPlanHeads, phys, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, tmv, fb, 0, 0, cur.g * kPlanHeads, phys, kv_policy);
                }
                cur.advance(pv.cu_s, V);
            }
            // Let every copy still in flight land before the CTA may exit.
            for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1));
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int r = lane >> 2, cq = lane & 3;
    uint8_t *qw = qbuf + warp * QRows<D>::kBytes;
    float o[NT][KT][4];
    float mm[NT][2], ll[NT][2];
    BlockCursor cur;
    cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
    bool seg_start = true;
    int32_t grp = 0, rows = 0, row_base = 0;
    for (int64_t it = 0; it < n; ++it) {
        const int s = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        const int32_t kvh = cur.g * kPlanHeads + warp, v = cur.seq;
        if (seg_start) {
            grp = pv.vgroup[v];
            rows = (pv.group_begin[grp + 1] - pv.group_begin[grp]) * G;
            row_base = (v - pv.group_vbase[grp]) * kPlanRows;
            // The pass's 16 query rows of this warp's head into shared memory
            // (zeros past the group's rows): row i = member i / G, head i % G.
            __syncwarp();  // the previous segment's reads of qw are done
            constexpr int kChunks = D / 8;  // 16-byte pieces of a row
            for (int e = lane; e < kPlanRows * kChunks; e += 32) {
                const int i = e / kChunks, ch = e - i * kChunks;
                const int32_t gr = row_base + i;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (gr < rows) {
                    const int32_t m = gr / G;
                    const int32_t seq = pv.members[pv.group_begin[grp] + m];
                    const __nv_bfloat16 *qp = q + ((int64_t)seq * H + (int64_t)kvh * G + (gr - m * G)) * D;
                    val = *reinterpret_cast<const uint4 *>(qp + ch * 8);  // q is 16-byte aligned with a plan
                }
                *reinterpret_cast<uint4 *>(qw + i * QRows<D>::kRowBytes + ch * 16) = val;
            }
            __syncwarp();
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[t][kk][e] = 0.f;
                mm[t][0] = mm[t][1] = -INFINITY;
                ll[t][0] = ll[t][1] = 0.f;
            }
            seg_start = false;
        }
        const bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(err, kErrTimeout);
            return;
        }
        const uint32_t kslab = smem_u32(smem + (size_t)s * stage_bytes) + (uint32_t)warp * Tile::kSlabBytes;
        mma_block_tiles<D, B, LAYOUT, NT>(kslab, kslab + tile_bytes, smem_u32(qw), scale_log2, o, mm, ll, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        if (cur.blk == cur.nb - 1 || it + 1 == n) {
            const int64_t slot = partial_slot(c, cur.g * V + v);
            const int64_t wrow = slot * kPlanSlotRows + warp * kPlanRows;  // this warp's 16 rows
            const int h0 = 2 * cq, h1 = 2 * cq + 1;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float lt0 = ll[t][0], lt1 = ll[t][1];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
                    lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
                }
                const bool v0 = row_base + t * 8 + h0 < rows, v1 = row_base + t * 8 + h1 < rows;
                float *ab = sh.acc_s + (wrow + t * 8) * D;
#pragma unroll
                for (int dm = 0; dm < KT; ++dm) {
                    const int d = dm * 16 + r;
                    if (v0) {
                        ab[h0 * D + d] = o[t][dm][0];
                        ab[h0 * D + d + 8] = o[t][dm][2];
                    }
                    if (v1) {
                        ab[h1 * D + d] = o[t][dm][1];
                        ab[h1 * D + d + 8] = o[t][dm][3];
                    }
                }
                if (r == 0) {
                    if (v0) sh.ml_s[wrow + t * 8 + h0] = make_float2(mm[t][0], lt0);
                    if (v1) sh.ml_s[wrow + t * 8 + h1] = make_float2(mm[t][1], lt1);
                }
            }
            seg_start = true;
        }
        cur.advance(pv.cu_s, V);
    }
}

// A CTA of the own-block part (the whole grid without a plan): CTA c of Co
// takes its range of the flattened (head group, sequence, own block) list.
// Consumer warp w owns KV head g * NH + w and its G query heads.  kShared:
// sequences may start after a shared prefix (skip[seq] blocks).
template <int D, int B, int LAYOUT, bool kShared>
__device__ __forceinline__ void own_block_cta(
    uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const __nv_bfloat16 *__restrict__ q,
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ tables, int32_t max_blocks,
    const int32_t *__restrict__ lens, const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t G, int32_t NB,
    int32_t NH, float scale_log2, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, int32_t Hk, int32_t C,
    int32_t Cs, const SharedArgs &sh, unsigned int *__restrict__ err) {
    using Tile = MmaTile<D, B>;
    constexpr int S = Tile::kStages;
    constexpr int KT = D / 16;  // k-steps of q.k and m-tiles of O^T
    const uint32_t tile_bytes = (uint32_t)NH * Tile::kSlabBytes;
    const uint32_t stage_bytes = 2u * tile_bytes;
    uint64_t *full = (uint64_t *)(smem + S * stage_bytes);
    uint64_t *empty = full + S;
    const int32_t *skip = kShared && Cs > 0 ? sh.skip : nullptr;  // nullptr without shared prefixes
    const int64_t W = (int64_t)(Hk / NH) * cu[N];
    const int32_t Ce = (int32_t)(W < (int64_t)(C - Cs) ? W : (int64_t)(C - Cs));  // no CTA with an empty range
    const int32_t c = (int32_t)blockIdx.x - Cs;
    if (c >= Ce) return;
    const int64_t lo = split_begin(c, W, Ce), hi = split_begin(c + 1, W, Ce);
    const int64_t n = hi - lo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), (uint32_t)NH);
        }
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == NH) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(tmk);
            prefetch_tmap(tmv);
            // KV tiles stream through once: evict them first, so that L2 keeps
            // the partials, q and tables that are read again.
            const uint64_t kv_policy = l2_policy_evict_first();
            BlockCursor cur, ahead;
            cur.init_at(lo, start_seq[c], cu, N, skip);
            ahead.init_at(lo, start_seq[c], cu, N, skip);
            // Block-table entries are loaded kTablePrefetch blocks ahead of their
            // TMA issue (a register shift ring), so the L2 latency of the table
            // read is off the issue path.
            constexpr int PD = kTablePrefetch;
            int32_t ring[PD];
#pragma unroll
            for (int j = 0; j < PD; ++j) {
                ring[j] = (j < n) ? tables[(int64_t)ahead.seq * max_blocks + ahead.b0 + ahead.blk] : 0;
                if (j < n) ahead.advance(cu, N, skip);
            }
            int64_t issued = 0;
            for (; issued < n; ++issued) {
                const int s = (int)(issued % S);
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                int32_t phys = ring[0];
#pragma unroll
                for (int j = 0; j + 1 < PD; ++j) ring[j] = ring[j + 1];
                if (issued + PD < n) {
                    ring[PD - 1] = tables[(int64_t)ahead.seq * max_blocks + ahead.b0 + ahead.blk];
                    ahead.advance(cu, N, skip);
                }
                if (issued >= S && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u)) {
                    atomicOr(err, kErrTimeout);
                    break;
                }
                if (phys < 0 || phys >= NB) {  // read zeros: the box lies past the pool
                    atomicOr(err, kErrBounds);
                    phys = NB;
                }
                const uint32_t fb = smem_u32(&full[s]);
                const uint32_t dst = smem_u32(smem + (size_t)s * stage_bytes);
                mbar_arrive_expect_tx(fb, stage_bytes);
                if (LAYOUT == PA_LAYOUT_ROW) {
                    tma_load_4d_hint(dst, tmk, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, tmv, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                } else {
                    tma_load_4d_hint(dst, tmk, fb, 0, 0, cur.g * NH, phys, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, tmv, fb, 0, 0, cur.g * NH, phys, kv_policy);
                }
                cur.advance(cu, N, skip);
            }
            // Let every copy still in flight land before the CTA may exit.
            for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1));
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int r = lane >> 2, cq = lane & 3;  // mma groupID / thread-in-group
    uint32_t qf[KT][2], qn[KT][2];
    float o[KT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    BlockCursor cur;
    cur.init_at(lo, start_seq[c], cu, N, skip);
    bool seg_start = true, seg_from_first = false, have_next_q = false;
    // B operand of S^T = K Q^T: column n = query head r of this KV head.
    auto load_q = [&](uint32_t (&dst)[KT][2], int32_t seq, int32_t grp) {
        const bool hv = r < G;
        const __nv_bfloat16 *qp =
            q + ((int64_t)seq * H + (int64_t)(grp * NH + warp) * G + (hv ? r : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            dst[kk][0] = hv ? *reinterpret_cast<const uint32_t *>(qp + kk * 16 + 2 * cq) : 0u;
            dst[kk][1] = hv ? *reinterpret_cast<const uint32_t *>(qp + kk * 16 + 8 + 2 * cq) : 0u;
        }
    };

    int32_t L = 0;
    for (int64_t it = 0; it < n; ++it) {
        const int s = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        const int32_t kvh = cur.g * NH + warp;
        if (seg_start) {
            L = lens[cur.seq];
            if (have_next_q) {
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    qf[kk][0] = qn[kk][0];
                    qf[kk][1] = qn[kk][1];
                }
            } else {
                load_q(qf, cur.seq, cur.g);
            }
            have_next_q = false;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[kk][e] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            // a piece from the sequence's first block, with no shared prefix
            seg_from_first = (cur.blk == 0 && cur.b0 == 0);
            seg_start = false;
        }
        // Last block of this sequence with more range after it: fetch the next
        // segment's q now, so the switch does not wait on a global load.
        if (cur.blk == cur.nb - 1 && it + 1 < n) {
            BlockCursor nx = cur;
            nx.advance(cu, N, skip);
            load_q(qn, nx.seq, nx.g);
            have_next_q = true;
        }

        const bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(err, kErrTimeout);
            return;
        }
        const uint32_t kslab = smem_u32(smem + (size_t)s * stage_bytes) + (uint32_t)warp * Tile::kSlabBytes;
        const uint32_t vslab = kslab + tile_bytes;
        const int32_t tok0 = (cur.b0 + cur.blk) * B;
        const int32_t ntok = min(B, L - tok0);
        if (ntok < B) {
            // Token rows past the sequence end hold stale data (maybe NaN):
            // zero them in V so that p = 0 rows contribute exactly 0.
            const int rows = B - ntok;
            if (LAYOUT == PA_LAYOUT_ROW) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int e = lane; e < Tile::kHalves * rows * 8; e += 32) {
                    const int chunk = e & 7;
                    const int ri = e >> 3;
                    const int half = ri / rows;
                    const int t = ntok + (ri - half * rows);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     vslab + (uint32_t)((half * B + t) * 128 + chunk * 16)),
                                 "r"(z.x), "r"(z.y), "r"(z.z), "r"(z.w)
                                 : "memory");
                }
            } else {  // split V tile: [d][token], tokens contiguous
                for (int e = lane; e < D * rows; e += 32) {
                    const int d = e / rows;
                    const int t = ntok + (e - d * rows);
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(vslab + (uint32_t)((d * B + t) * 2)),
                                 "h"((unsigned short)0)
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        mma_block<D, B, LAYOUT>(kslab, vslab, tok0, L, scale_log2, qf, o, m0, m1, l0, l1, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        const bool last_blk = (cur.blk == cur.nb - 1);
        if (last_blk || it + 1 == n) {
            float lt0 = l0, lt1 = l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
            }
            const int h0 = 2 * cq, h1 = 2 * cq + 1;
            if (seg_from_first && last_blk) {
                const float i0 = 1.f / lt0, i1 = 1.f / lt1;
                __nv_bfloat16 *ob = out + ((int64_t)cur.seq * H + (int64_t)kvh * G) * D;
#pragma unroll
                for (int dm = 0; dm < KT; ++dm) {
                    const int d = dm * 16 + r;
                    if (h0 < G) {
                        ob[h0 * D + d] = __float2bfloat16_rn(o[dm][0] * i0);
                        ob[h0 * D + d + 8] = __float2bfloat16_rn(o[dm][2] * i0);
                    }
                    if (h1 < G) {
                        ob[h1 * D + d] = __float2bfloat16_rn(o[dm][1] * i1);
                        ob[h1 * D + d + 8] = __float2bfloat16_rn(o[dm][3] * i1);
                    }
                }
            } else {
                const int32_t HPG = NH * G;
                const int64_t slot = partial_slot(c, cur.g * N + cur.seq);
                float *ab = acc_ws + (slot * HPG + (int64_t)warp * G) * D;
#pragma unroll
                for (int dm = 0; dm < KT; ++dm) {
                    const int d = dm * 16 + r;
                    if (h0 < G) {
                        ab[h0 * D + d] = o[dm][0];
                        ab[h0 * D + d + 8] = o[dm][2];
                    }
                    if (h1 < G) {
                        ab[h1 * D + d] = o[dm][1];
                        ab[h1 * D + d + 8] = o[dm][3];
                    }
                }
                if (r == 0) {
                    if (h0 < G) ml_ws[slot * HPG + warp * G + h0] = make_float2(m0, lt0);
                    if (h1 < G) ml_ws[slot * HPG + warp * G + h1] = make_float2(m1, lt1);
                }
                // A sequence with a shared prefix is merged by shared_merge_kernel
                // after this launch; every other one by its last arriver here.
                if (!(kShared && cur.b0 > 0)) {
                    const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, cur.seq, cur.g, warp, G, HPG, W, Ce),
                                              no_range()};
                    finish_piece<__nv_bfloat16, D>(out, rg, counters, N, NH, H, G, cur.seq, kvh, lane);
                }
            }
            seg_start = true;
        }
        cur.advance(cu, N, skip);
    }
}

// The attention launch.  Without a plan (kShared = false) every CTA is an
// own-block CTA.  With one, the plan kernel gives CTAs [0, Cs) to the shared
// prefixes and the rest to the sequences' own blocks; both kinds run at once
// and meet only at the arrival counters.
template <int D, int B, int LAYOUT, bool kShared>
__global__ void __launch_bounds__(32 * (kMmaMaxHeads + 1), 2) decode_mma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ out,
    const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G, int32_t NB,
    int32_t NH, float scale_log2, int32_t C, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, unsigned int *__restrict__ err,
    const SharedArgs sh) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

    grid_dependency_wait();  // the plan kernel's cu[] / lens / split (programmatic launch)
    // With a plan, the merge kernel may become resident as CTAs finish and
    // work out its piece ranges from the plan while the last ones run.
    if (kShared) grid_launch_dependents();
    const int32_t Cs = kShared ? sh.ctl[0] : 0;
    if (kShared && (int32_t)blockIdx.x < Cs)
        shared_prefix_cta<D, B, LAYOUT>(smem, &tmk, &tmv, q, out, tables, max_blocks, H, G, NB, scale_log2,
                                        counters, cu, N, NH, Hk, C, Cs, ml_ws, acc_ws, sh, err);
    else
        own_block_cta<D, B, LAYOUT, kShared>(smem, &tmk, &tmv, q, out, tables, max_blocks, lens, cu, N, H, G, NB,
                                             NH, scale_log2, ml_ws, acc_ws, counters, start_seq, Hk, C, Cs, sh,
                                             err);
}

// Single-pass merge for the merge kernel: pieces are loaded kBatch at a
// time and folded in with a running maximum, so a merge costs one dependent
// load per batch.  Lanes as in merge_pieces_lph.
template <typename T, int D, int LPH>
__device__ __forceinline__ void merge_online_lph(T *__restrict__ out_base, const PieceRange (&rg)[2], int32_t G,
                                                 int lane) {
    constexpr int E = D / LPH, kBatch = E >= 32 ? 2 : 4;  // kBatch * E floats of pieces in flight
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

// Merge of the sequences with a shared prefix (after the attention launch,
// which left their pieces in the workspace): one warp per (member of a
// group, KV head).  The piece ranges depend only on the plan kernel's output,
// so they are worked out before waiting for the attention launch (which lets
// this grid start as its CTAs finish); only the pieces are read after it.
template <int D>
__global__ void __launch_bounds__(256) shared_merge_kernel(
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G,
    int32_t NH, int32_t C, const float2 *__restrict__ ml_ws, const float *__restrict__ acc_ws, const SharedArgs sh) {
    const int32_t Cs = sh.ctl[0];
    if (Cs <= 0) return;  // plan rejected: every sequence was merged in the attention launch
    const SharedView sv = shared_view(sh.plan, sh.skip, sh.ml_s, sh.acc_s, Hk, Cs);
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)sv.pv.M * Hk) return;
    const int32_t seq = sv.pv.members[wid / Hk];
    const int32_t kvh = (int32_t)(wid % Hk);
    if (sh.skip[seq] <= 0) return;  // computed without sharing: merged in the attention launch
    const int64_t W = (int64_t)(Hk / NH) * cu[N];
    const int32_t Ce = (int32_t)(W < (int64_t)(C - Cs) ? W : (int64_t)(C - Cs));
    const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, seq, kvh / NH, kvh % NH, G, NH * G, W, Ce),
                              shared_range(sv, seq, kvh, G)};
    grid_dependency_wait();  // the attention launch's pieces
    __nv_bfloat16 *ob = out + ((int64_t)seq * H + (int64_t)kvh * G) * D;
    constexpr int kMaxLph = D / 4 < 32 ? D / 4 : 32;
    constexpr int kL8 = 8 < kMaxLph ? 8 : kMaxLph, kL16 = 16 < kMaxLph ? 16 : kMaxLph;
    if (G > 4)
        merge_online_lph<__nv_bfloat16, D, 4>(ob, rg, G, lane);
    else if (G > 2)
        merge_online_lph<__nv_bfloat16, D, kL8>(ob, rg, G, lane);
    else if (G > 1)
        merge_online_lph<__nv_bfloat16, D, kL16>(ob, rg, G, lane);
    else
        merge_online_lph<__nv_bfloat16, D, kMaxLph>(ob, rg, G, lane);
}

// ====================================================================== host
namespace {

struct DecodePlan {
    int kernel;    // PA_KERNEL_SIMT or PA_KERNEL_MMA
    int NH;        // KV heads per CTA (consumer warps)
    int NG;        // head groups = Hk / NH
    int HPG;       // query heads per group = NH * G
    int C;         // persistent CTAs
    bool shared;   // a shared-prefix plan is used
    size_t smem;   // dynamic shared memory of the attention kernel
    // workspace layout (byte offsets)
    size_t off_lens, off_cu, off_cnt, off_start, off_ml, off_acc;
    size_t off_skip, off_ctl, off_start_s, off_ml_s, off_acc_s;  // shared-prefix part
    size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int largest_divisor_at_most(int n, int cap) {
    for (int d = std::min(n, cap); d >= 1; --d)
        if (n % d == 0) return d;
    return 1;
}

bool mma_supported(const pa_cache_desc_t *c, int G) {
    return c->dtype == PA_BF16 && (c->head_dim == 64 || c->head_dim == 128) &&
           (c->block_size == 16 || c->block_size == 32) && G >= 1 && G <= 8;
}

bool simt_supported(const pa_cache_desc_t *c, int G) {
    const bool d_ok = c->dtype == PA_F32 ? (c->head_dim == 64 || c->head_dim == 128)
                                         : (c->head_dim == 64 || c->head_dim == 128 || c->head_dim == 256);
    return d_ok && G >= 1 && G <= 8;
}

int simt_gmax(int G) { return G <= 1 ? 1 : (G <= 4 ? 4 : 8); }

// kMmaStages stages of NH head slabs of K and of V (the shared-prefix CTAs
// use the same ring with NH = kPlanHeads), mbarriers after the tiles, with
// shared prefixes the query rows of the shared-prefix warps (QRows, 256
// bytes after the tiles); 1024 bytes to align the base.
size_t mma_smem_bytes(int D, int B, int NH, bool shared) {
    const size_t slab = (size_t)(D / 64) * B * 128;
    size_t bytes = (size_t)kMmaStages * 2 * NH * slab + 2 * (size_t)kMmaStages * sizeof(uint64_t) + 1024;
    if (shared) bytes += 256 + (size_t)kPlanHeads * kPlanRows * (D * 2 + 16);  // QRows of the shared-prefix warps
    return bytes;
}

template <typename T, int D, int GMAX>
const void *simt_fn(int layout) {
    return layout == PA_LAYOUT_SPLIT ? (const void *)decode_simt_kernel<T, D, GMAX, PA_LAYOUT_SPLIT>
                                     : (const void *)decode_simt_kernel<T, D, GMAX, PA_LAYOUT_ROW>;
}

const void *simt_kernel_ptr(int dtype, int D, int G, int layout) {
    const int gm = simt_gmax(G);
#define PA_SIMT_CASE(TT, DD)                                        \
    if (D == DD) {                                                  \
        if (gm == 1) return simt_fn<TT, DD, 1>(layout);             \
        if (gm == 4) return simt_fn<TT, DD, 4>(layout);             \
        return simt_fn<TT, DD, 8>(layout);                          \
    }
    if (dtype == PA_F32) {
        PA_SIMT_CASE(float, 64)
        PA_SIMT_CASE(float, 128)
    } else {
        PA_SIMT_CASE(__nv_bfloat16, 64)
        PA_SIMT_CASE(__nv_bfloat16, 128)
        PA_SIMT_CASE(__nv_bfloat16, 256)
    }
#undef PA_SIMT_CASE
    return nullptr;
}

template <int LAYOUT, bool kShared>
const void *mma_fn(int D, int B) {
    if (D == 128 && B == 16) return (const void *)decode_mma_kernel<128, 16, LAYOUT, kShared>;
    if (D == 128 && B == 32) return (const void *)decode_mma_kernel<128, 32, LAYOUT, kShared>;
    if (D == 64 && B == 16) return (const void *)decode_mma_kernel<64, 16, LAYOUT, kShared>;
    if (D == 64 && B == 32) return (const void *)decode_mma_kernel<64, 32, LAYOUT, kShared>;
    return nullptr;
}

const void *mma_kernel_ptr(int D, int B, int layout, bool shared) {
    if (shared)
        return layout == PA_LAYOUT_SPLIT ? mma_fn<PA_LAYOUT_SPLIT, true>(D, B) : mma_fn<PA_LAYOUT_ROW, true>(D, B);
    return layout == PA_LAYOUT_SPLIT ? mma_fn<PA_LAYOUT_SPLIT, false>(D, B) : mma_fn<PA_LAYOUT_ROW, false>(D, B);
}

// Occupancy-based default split count: one full wave of resident CTAs.
int default_ctas(const void *fn, int threads, size_t smem) {
    const int sms = num_sms();
    if (sms <= 0) return -1;
    int per_sm = 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return -1;
    return sms * std::max(per_sm, 1);
}

pa_status_t make_plan(const pa_cache_desc_t *c, int32_t N, int32_t H, const pa_decode_opts_t *opts,
                      bool need_default_splits, DecodePlan *p) {
    pa_status_t st = validate_cache_desc(c);
    if (st != PA_OK) return st;
    if (N < 0 || H <= 0 || H % c->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int G = H / c->num_kv_heads;
    const int want = opts ? opts->kernel : PA_KERNEL_AUTO;
    if (want != PA_KERNEL_AUTO && want != PA_KERNEL_SIMT && want != PA_KERNEL_MMA) return PA_ERR_INVALID_ARG;
    if (opts && opts->num_splits < 0) return PA_ERR_INVALID_ARG;
    int kernel;
    if (want == PA_KERNEL_MMA || (want == PA_KERNEL_AUTO && mma_supported(c, G))) {
        if (!mma_supported(c, G)) return PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_MMA;
    } else {
        if (!simt_supported(c, G)) return PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_SIMT;
    }
    p->kernel = kernel;
    p->shared = false;
    if (kernel == PA_KERNEL_MMA) {
        p->NH = largest_divisor_at_most(c->num_kv_heads, kMmaMaxHeads);
        // Shared-prefix CTAs use 4 consumer warps: the launch shape must match.
        p->shared = opts && opts->shared_plan && p->NH == kPlanHeads;
        p->smem = mma_smem_bytes(c->head_dim, c->block_size, p->NH, p->shared);
    } else {
        p->NH = largest_divisor_at_most(c->num_kv_heads, 8);
        p->smem = 0;
    }
    p->NG = c->num_kv_heads / p->NH;
    p->HPG = p->NH * G;
    int C = opts ? opts->num_splits : 0;
    if (C == 0) {
        if (!need_default_splits) return PA_ERR_INVALID_ARG;
        const void *fn = kernel == PA_KERNEL_MMA ? mma_kernel_ptr(c->head_dim, c->block_size, c->layout, p->shared)
                                                 : simt_kernel_ptr(c->dtype, c->head_dim, G, c->layout);
        const int threads = kernel == PA_KERNEL_MMA ? (p->NH + 1) * 32 : p->NH * 32;
        C = default_ctas(fn, threads, p->smem);
        if (C <= 0) return PA_ERR_CUDA;
    }
    p->C = C;
    if (p->shared && C < 2) {  // shared prefixes need a CTA of each kind
        p->shared = false;
        p->smem = mma_smem_bytes(c->head_dim, c->block_size, p->NH, false);
    }
    const size_t slots = (size_t)C + (size_t)p->NG * N;
    size_t off = 0;
    p->off_lens = off;
    off = align256(off + sizeof(int32_t) * (size_t)std::max(N, 1));
    p->off_cu = off;
    off = align256(off + sizeof(int32_t) * ((size_t)N + 1));
    p->off_cnt = off;
    off = align256(off + sizeof(uint32_t) * (size_t)std::max(N, 1) * c->num_kv_heads);
    p->off_start = off;
    off = align256(off + sizeof(int32_t) * (size_t)C);
    p->off_ml = off;
    off = align256(off + sizeof(float2) * slots * p->HPG);
    p->off_acc = off;
    off = align256(off + sizeof(float) * slots * p->HPG * c->head_dim);
    p->off_skip = p->off_ctl = p->off_start_s = p->off_ml_s = p->off_acc_s = 0;
    if (p->shared) {
        // virtual sequences V <= N (checked on the device), so at most
        // C + Hk * N shared-prefix slots of kPlanSlotRows query rows
        const size_t slots_s = (size_t)C + (size_t)c->num_kv_heads * N;
        p->off_skip = off;
        off = align256(off + sizeof(int32_t) * (size_t)std::max(N, 1));
        p->off_ctl = off;
        off = align256(off + sizeof(int32_t) * 8);
        p->off_start_s = off;
        off = align256(off + sizeof(int32_t) * (size_t)C);
        p->off_ml_s = off;
        off = align256(off + sizeof(float2) * slots_s * kPlanSlotRows);
        p->off_acc_s = off;
        off = align256(off + sizeof(float) * slots_s * kPlanSlotRows * c->head_dim);
    }
    p->total = off;
    return PA_OK;
}

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel on the stream finishes; the kernel itself calls
// griddepcontrol.wait before touching anything that kernel produced.
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    });
    return fn;
}

// 4-D maps over one bf16 cache (both use 128-byte rows of 64 elements).
// Row layout: {64, NB*B, D/64, Hk} with byte strides {Hk*D*2, 128, D*2}, box
// {64, B, D/64, NH}, 128-byte swizzle -> shared [head][half][token][64].
// Split layout (K [NB, Hk, D/8, B, 8] or V [NB, Hk, D, B]): each (block, head)
// slab is D*B contiguous elements, viewed as {64, D*B/64, Hk, NB} with strides
// {128, D*B*2, Hk*D*B*2}, box {64, D*B/64, NH, 1}, no swizzle -> the slab's
// own byte order in shared memory.
bool encode_cache_map(CUtensorMap *map, const void *base, const pa_cache_desc_t *c, int NH) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int D = c->head_dim;
    const int B = c->block_size;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r;
    if (c->layout == PA_LAYOUT_SPLIT) {
        cuuint64_t dims[4] = {64, (cuuint64_t)D * B / 64, (cuuint64_t)c->num_kv_heads, (cuuint64_t)c->num_blocks};
        cuuint64_t strides[3] = {128, (cuuint64_t)D * B * 2, (cuuint64_t)c->num_kv_heads * D * B * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)(D * B / 64), (cuuint32_t)NH, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {64, (cuuint64_t)c->num_blocks * B, (cuuint64_t)(D / 64), (cuuint64_t)c->num_kv_heads};
        cuuint64_t strides[3] = {(cuuint64_t)c->num_kv_heads * D * 2, 128, (cuuint64_t)D * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)B, (cuuint32_t)(D / 64), (cuuint32_t)NH};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_bytes(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                                            const pa_decode_opts_t *opts) {
    DecodePlan p;
    if (make_plan(cache, num_seqs, num_heads, opts, true, &p) != PA_OK) return 0;
    return p.total;
}

extern "C" int32_t pa_decode_default_splits(const pa_cache_desc_t *cache, int32_t num_heads,
                                            const pa_decode_opts_t *opts) {
    pa_decode_opts_t o = opts ? *opts : pa_decode_opts_t{0, PA_KERNEL_AUTO, nullptr, nullptr, nullptr};
    o.num_splits = 0;
    DecodePlan p;
    const pa_status_t st = make_plan(cache, 1, num_heads, &o, true, &p);
    return st == PA_OK ? p.C : (int32_t)st;
}

extern "C" void pa_split_range(int64_t total_blocks, int32_t num_splits, int32_t c, int64_t *begin,
                               int64_t *end) {
    if (begin) *begin = split_begin(c, total_blocks, num_splits);
    if (end) *end = split_begin((int64_t)c + 1, total_blocks, num_splits);
}

extern "C" int32_t pa_split_owner(int64_t total_blocks, int32_t num_splits, int64_t x) {
    return split_owner(x, total_blocks, num_splits);
}

extern "C" pa_status_t pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const pa_cache_desc_t *cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                 int32_t num_heads, float scale, void *workspace, size_t workspace_bytes,
                                 const pa_decode_opts_t *opts, pa_stream_t stream) {
    DecodePlan p;
    pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || (int64_t)num_seqs * max_blocks_per_seq >= ((int64_t)1 << 31) ||
        (int64_t)max_blocks_per_seq * cache->block_size >= ((int64_t)1 << 31))
        return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255) != 0) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < p.total) return PA_ERR_WORKSPACE;
    const int eb = dtype_bytes(cache->dtype);
    if (((uintptr_t)q | (uintptr_t)out) % (size_t)(eb * 2) != 0) return PA_ERR_INVALID_ARG;
    if (p.shared && (uintptr_t)q % 16 != 0) {  // shared-prefix warps read q rows in 16-byte pieces
        p.shared = false;
        p.smem = mma_smem_bytes(cache->head_dim, cache->block_size, p.NH, false);
    }
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;

    uint8_t *ws = (uint8_t *)workspace;
    int32_t *lens_ws = (int32_t *)(ws + p.off_lens);
    int32_t *cu = (int32_t *)(ws + p.off_cu);
    unsigned int *cnt = (unsigned int *)(ws + p.off_cnt);
    int32_t *start_seq = (int32_t *)(ws + p.off_start);
    float2 *ml = (float2 *)(ws + p.off_ml);
    float *acc = (float *)(ws + p.off_acc);
    const int G = num_heads / cache->num_kv_heads;
    const float scale_log2 = scale * 1.4426950408889634f;
    const int32_t max_len = max_blocks_per_seq * cache->block_size;
    cudaStream_t s = (cudaStream_t)stream;
    cudaGetLastError();  // clear a stale launch error so the checks below are ours

    const int32_t HD = num_heads * cache->head_dim;
    const int32_t ncnt = num_seqs * cache->num_kv_heads;
    SharedArgs sh{};
    if (p.shared) {
        sh.plan = opts->shared_plan;
        sh.skip = (const int32_t *)(ws + p.off_skip);
        sh.ctl = (const int32_t *)(ws + p.off_ctl);
        sh.start_s = (const int32_t *)(ws + p.off_start_s);
        sh.ml_s = (float2 *)(ws + p.off_ml_s);
        sh.acc_s = (float *)(ws + p.off_acc_s);
    }
    {
        int32_t Nv = num_seqs, Bv = cache->block_size, ml_v = max_len, HDv = HD, nc = ncnt, NGv = p.NG, Cv = p.C;
        int32_t Gv = G, Hkv = cache->num_kv_heads, NHv = p.NH;
        void *outp = out;
        const int32_t *planp = sh.plan;
        int32_t *skipp = (int32_t *)sh.skip, *ctlp = (int32_t *)sh.ctl, *start_sp = (int32_t *)sh.start_s;
        // the plan's words in shared memory when they fit (at most 96 KiB)
        const size_t plan_bytes = sizeof(int32_t) * (7 * (size_t)num_seqs + 16);
        int32_t in_smem = p.shared && plan_bytes <= 96 * 1024 ? 1 : 0;
        const void *pfn = cache->dtype == PA_BF16 ? (const void *)decode_plan_kernel<__nv_bfloat16>
                                                  : (const void *)decode_plan_kernel<float>;
        const size_t psmem = in_smem ? plan_bytes : 0;
        if (psmem > 48 * 1024 &&
            cudaFuncSetAttribute(pfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem) != cudaSuccess)
            return PA_ERR_CUDA;
        void *pargs[] = {&seq_lens, &Nv, &Bv, &ml_v, &HDv, &lens_ws, &cu, &cnt, &nc, &outp, &NGv, &Cv, &start_seq,
                         &err, &planp, &Gv, &Hkv, &NHv, &skipp, &ctlp, &start_sp, &in_smem};
        if (launch_pdl(pfn, dim3(1), dim3(1024), pargs, psmem, s) != cudaSuccess) return PA_ERR_CUDA;
    }

    if (opts && opts->ev_partial_begin && cudaEventRecord((cudaEvent_t)opts->ev_partial_begin, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (p.kernel == PA_KERNEL_MMA) {
        if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0) return PA_ERR_INVALID_ARG;
        CUtensorMap tmk, tmv;
        if (!encode_cache_map(&tmk, k_cache, cache, p.NH) || !encode_cache_map(&tmv, v_cache, cache, p.NH))
            return PA_ERR_CUDA;
        const void *fn = mma_kernel_ptr(cache->head_dim, cache->block_size, cache->layout, p.shared);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
            return PA_ERR_CUDA;
        const dim3 grid(p.C), block((p.NH + 1) * 32);
        const __nv_bfloat16 *qb = (const __nv_bfloat16 *)q;
        __nv_bfloat16 *ob = (__nv_bfloat16 *)out;
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq;
        float sl = scale_log2;
        void *args[] = {&tmk, &tmv, &qb, &ob, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk,
                        &Gv, &NB, &NHv, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err, &sh};
        if (launch_pdl(fn, grid, block, args, p.smem, s) != cudaSuccess) return PA_ERR_CUDA;
        if (p.shared) {
            // one warp per (sequence, KV head) bound: members <= N
            const int64_t warps = (int64_t)num_seqs * Hk;
            const dim3 mgrid((unsigned)((warps + 7) / 8)), mblock(256);
            void *margs[] = {&ob, &cu, &Nv, &Hv, &Hk, &Gv, &NHv, &Cv, &ml, &acc, &sh};
            const void *mfn = cache->head_dim == 128 ? (const void *)shared_merge_kernel<128>
                                                     : (const void *)shared_merge_kernel<64>;
            if (launch_pdl(mfn, mgrid, mblock, margs, 0, s) != cudaSuccess) return PA_ERR_CUDA;
        }
    } else {
        const void *fn = simt_kernel_ptr(cache->dtype, cache->head_dim, G, cache->layout);
        if (!fn) return PA_ERR_UNSUPPORTED;
        const dim3 grid(p.C), block(p.NH * 32);
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq, Bv = cache->block_size;
        float sl = scale_log2;
        void *args[] = {&q, &out, &k_cache, &v_cache, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk,
                        &Gv, &Bv, &NB, &NHv, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err};
        if (launch_pdl(fn, grid, block, args, 0, s) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (opts && opts->ev_partial_end && cudaEventRecord((cudaEvent_t)opts->ev_partial_end, s) != cudaSuccess)
        return PA_ERR_CUDA;

    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ------------------------------------------------------------ no-alloc entry
// Scratch of pa_decode_no_alloc: a fixed array in the library's device image
// (one per GPU that loads the library, alive until exit).  Host code must not
// pass `g_decode_scratch` itself to a kernel: on the host that name is only a
// stand-in, so its device address is looked up per device below.
static __device__ __align__(256) unsigned char g_decode_scratch[PA_NO_ALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_addr[64];

// Device address of g_decode_scratch on the current device, looked up on the
// first call per device (with that device current) and cached; nullptr on
// failure.
void *no_alloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}
}  // namespace

extern "C" pa_status_t pa_decode_no_alloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                          const pa_cache_desc_t *cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                          int32_t num_heads, float scale, const pa_decode_opts_t *opts,
                                          pa_stream_t stream) {
    DecodePlan p;
    const pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return st;
    if (p.total > (size_t)PA_NO_ALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void *scratch = no_alloc_scratch();
    if (!scratch) return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     num_heads, scale, scratch, (size_t)PA_NO_ALLOC_SCRATCH_BYTES, opts, stream);
}
