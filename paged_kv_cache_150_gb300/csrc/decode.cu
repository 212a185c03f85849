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

// ---------------------------------------------------------------- plan kernel
template <typename T>
__global__ void __launch_bounds__(1024) decode_plan_kernel(const int32_t *__restrict__ seq_lens, int32_t N,
                                                           int32_t B, int32_t max_len, int32_t HD,
                                                           int32_t *__restrict__ lens_ws,
                                                           int32_t *__restrict__ cu,
                                                           unsigned int *__restrict__ counters,
                                                           int32_t num_counters, T *__restrict__ out,
                                                           int32_t NG, int32_t C,
                                                           int32_t *__restrict__ start_seq,
                                                           unsigned int *__restrict__ err) {
    grid_dependency_wait();     // inputs written by earlier work on the stream
    grid_launch_dependents();   // the attention kernel may become resident now
    constexpr int32_t kSmemCu = 2048;  // prefix sums kept in shared memory for the start search
    __shared__ int32_t warp_incl[32];
    __shared__ int32_t carry;
    __shared__ int32_t n_empty;
    __shared__ int32_t empty_ids[1024];
    __shared__ int32_t cu_s[kSmemCu];
    const bool cu_in_smem = N + 1 <= kSmemCu;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    for (int32_t i = threadIdx.x; i < num_counters; i += blockDim.x) counters[i] = 0u;
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
    }
    __syncthreads();
    // Sequence holding the first block of each attention CTA's range, so the
    // CTA starts without searching cu[].
    const int32_t *cus = cu_in_smem ? cu_s : cu;
    const int32_t Wg = cus[N];
    const int64_t W = (int64_t)NG * Wg;
    const int32_t Ce = (int32_t)(W < (int64_t)C ? W : (int64_t)C);
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
}

// ------------------------------------------------------------ piece merge
// Run by the warp that finished the last piece of one (sequence, KV head):
// merges the pieces held by CTAs c0..c1 for its G query heads.  Lanes split
// the G heads x D outputs: LPH lanes per head, each a contiguous slice of
// E = D / LPH elements.  With LPH a compile-time constant every load of a
// piece is issued back to back (the merge runs at the end of the kernel, so
// its L2 latency is on the kernel's critical path); two passes, the maximum
// over all pieces first, then the weighted sums.
template <typename T, int D, int LPH>
__device__ __forceinline__ void merge_pieces_lph(T *__restrict__ out_base, const float2 *__restrict__ ml_ws,
                                                 const float *__restrict__ acc_ws, int32_t c0, int32_t c1,
                                                 int32_t sp, int32_t HPG, int32_t hoff, int32_t G, int lane) {
    constexpr int E = D / LPH;
    static_assert(E % 4 == 0, "slices are whole float4s");
    const int h = lane / LPH;
    const int part = lane % LPH;
    if (h >= G) return;
    const int64_t base = partial_slot(0, sp) * HPG + hoff + h;  // piece c is at base + c * HPG
    float M = -INFINITY;
#pragma unroll 8
    for (int32_t c = c0; c <= c1; ++c) M = fmaxf(M, __ldcg(&ml_ws[base + (int64_t)c * HPG]).x);
    float a[E];
#pragma unroll
    for (int j = 0; j < E; ++j) a[j] = 0.f;
    float Ls = 0.f;
#pragma unroll 1
    for (int32_t c = c0; c <= c1; ++c) {
        const int64_t idx = base + (int64_t)c * HPG;
        const float4 *ap = reinterpret_cast<const float4 *>(acc_ws + idx * D + part * E);
        float4 x[E / 4];
#pragma unroll
        for (int j4 = 0; j4 < E / 4; ++j4) x[j4] = __ldcg(ap + j4);
        const float2 v = __ldcg(&ml_ws[idx]);
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
    const float inv = 1.f / Ls;
    T *o = out_base + (int64_t)h * D + part * E;
#pragma unroll
    for (int j = 0; j < E; ++j) store_out(o + j, a[j] * inv);
}

// Lanes per head: 32 / (G rounded up to a power of two), with slices of at
// least 4 elements.
template <typename T, int D>
__device__ __forceinline__ void merge_pieces(T *__restrict__ out_base, const float2 *__restrict__ ml_ws,
                                             const float *__restrict__ acc_ws, int32_t c0, int32_t c1,
                                             int32_t sp, int32_t HPG, int32_t hoff, int32_t G, int lane) {
    constexpr int kMaxLph = D / 4 < 32 ? D / 4 : 32;
    if (G > 4)
        merge_pieces_lph<T, D, 4>(out_base, ml_ws, acc_ws, c0, c1, sp, HPG, hoff, G, lane);
    else if (G > 2)
        merge_pieces_lph<T, D, (8 < kMaxLph ? 8 : kMaxLph)>(out_base, ml_ws, acc_ws, c0, c1, sp, HPG, hoff, G, lane);
    else if (G > 1)
        merge_pieces_lph<T, D, (16 < kMaxLph ? 16 : kMaxLph)>(out_base, ml_ws, acc_ws, c0, c1, sp, HPG, hoff, G, lane);
    else
        merge_pieces_lph<T, D, kMaxLph>(out_base, ml_ws, acc_ws, c0, c1, sp, HPG, hoff, G, lane);
}

// After a warp wrote its partial for (sequence seq of group g, KV head kvh):
// publish it, count the arrival, and merge if this warp is the last one.
template <typename T, int D>
__device__ __forceinline__ void finish_piece(T *__restrict__ out, const float2 *__restrict__ ml_ws,
                                             const float *__restrict__ acc_ws, unsigned int *__restrict__ counters,
                                             const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t G,
                                             int32_t NH, int32_t warp, int32_t g, int32_t seq, int32_t nb,
                                             int64_t W, int32_t Ce, int lane) {
    const int32_t sp = g * N + seq;
    const int64_t x0 = (int64_t)g * cu[N] + cu[seq];
    const int32_t c0 = split_owner(x0, W, Ce);
    const int32_t c1 = split_owner(x0 + nb - 1, W, Ce);
    __threadfence();  // this lane's partial stores, before the arrival below
    __syncwarp();
    unsigned int last = 0;
    if (lane == 0) last = atomicAdd(&counters[(int64_t)sp * NH + warp], 1u) == (unsigned int)(c1 - c0);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();  // every other piece is published: read them
    const int32_t kvh = g * NH + warp;
    merge_pieces<T, D>(out + ((int64_t)seq * H + (int64_t)kvh * G) * D, ml_ws, acc_ws, c0, c1, sp, NH * G,
                       warp * G, G, lane);
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
                finish_piece<T, D>(out, ml_ws, acc_ws, counters, cu, N, H, G, NH, warp, cur.g, cur.seq, cur.nb, W,
                                   Ce, lane);
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

template <int D, int B, int LAYOUT>
__global__ void __launch_bounds__(32 * (kMmaMaxHeads + 1), 2) decode_mma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ out,
    const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G, int32_t NB,
    int32_t NH, float scale_log2, int32_t C, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, unsigned int *__restrict__ err) {
    using Tile = MmaTile<D, B>;
    constexpr int S = Tile::kStages;
    constexpr int KT = D / 16;  // k-steps of q.k and m-tiles of O^T
    const uint32_t tile_bytes = (uint32_t)NH * Tile::kSlabBytes;
    const uint32_t stage_bytes = 2u * tile_bytes;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + S * stage_bytes);
    uint64_t *empty = full + S;

    grid_dependency_wait();  // the plan kernel's cu[] / lens (programmatic launch)
    const int32_t NG = Hk / NH;
    const int64_t W = (int64_t)NG * cu[N];
    const int32_t Ce = (int32_t)(W < (int64_t)C ? W : (int64_t)C);  // no CTA with an empty range
    const int32_t c = blockIdx.x;
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
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
            // KV tiles stream through once: evict them first, so that L2 keeps
            // the partials, q and tables that are read again.
            const uint64_t kv_policy = l2_policy_evict_first();
            BlockCursor cur, ahead;
            cur.init_at(lo, start_seq[c], cu, N);
            ahead.init_at(lo, start_seq[c], cu, N);
            // Block-table entries are loaded kTablePrefetch blocks ahead of their
            // TMA issue (a register shift ring), so the L2 latency of the table
            // read is off the issue path.
            constexpr int PD = kTablePrefetch;
            int32_t ring[PD];
#pragma unroll
            for (int j = 0; j < PD; ++j) {
                ring[j] = (j < n) ? tables[(int64_t)ahead.seq * max_blocks + ahead.blk] : 0;
                if (j < n) ahead.advance(cu, N);
            }
            int64_t issued = 0;
            for (; issued < n; ++issued) {
                const int s = (int)(issued % S);
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                int32_t phys = ring[0];
#pragma unroll
                for (int j = 0; j + 1 < PD; ++j) ring[j] = ring[j + 1];
                if (issued + PD < n) {
                    ring[PD - 1] = tables[(int64_t)ahead.seq * max_blocks + ahead.blk];
                    ahead.advance(cu, N);
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
                    tma_load_4d_hint(dst, &tmk, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, &tmv, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                } else {
                    tma_load_4d_hint(dst, &tmk, fb, 0, 0, cur.g * NH, phys, kv_policy);
                    tma_load_4d_hint(dst + tile_bytes, &tmv, fb, 0, 0, cur.g * NH, phys, kv_policy);
                }
                cur.advance(cu, N);
            }
            // Let every copy still in flight land before the CTA may exit.
            for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1));
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int r = lane >> 2, cq = lane & 3;  // mma groupID / thread-in-group
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix id / row id
    uint32_t qf[KT][2], qn[KT][2];
    float o[KT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    BlockCursor cur;
    cur.init_at(lo, start_seq[c], cu, N);
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
            seg_from_first = (cur.blk == 0);
            seg_start = false;
        }
        // Last block of this sequence with more range after it: fetch the next
        // segment's q now, so the switch does not wait on a global load.
        if (cur.blk == cur.nb - 1 && it + 1 < n) {
            BlockCursor nx = cur;
            nx.advance(cu, N);
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
        const int32_t tok0 = cur.blk * B;
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
                finish_piece<__nv_bfloat16, D>(out, ml_ws, acc_ws, counters, cu, N, H, G, NH, warp, cur.g,
                                               cur.seq, cur.nb, W, Ce, lane);
            }
            seg_start = true;
        }
        cur.advance(cu, N);
    }
}

// ====================================================================== host
namespace {

struct DecodePlan {
    int kernel;    // PA_KERNEL_SIMT or PA_KERNEL_MMA
    int NH;        // KV heads per CTA (consumer warps)
    int NG;        // head groups = Hk / NH
    int HPG;       // query heads per group = NH * G
    int C;         // persistent CTAs
    size_t smem;   // dynamic shared memory of the attention kernel
    // workspace layout (byte offsets)
    size_t off_lens, off_cu, off_cnt, off_start, off_ml, off_acc, total;
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

size_t mma_smem_bytes(int D, int B, int NH) {
    const size_t tile = (size_t)NH * (D / 64) * B * 128;
    return (size_t)kMmaStages * 2 * tile + 2 * kMmaStages * sizeof(uint64_t) + 1024;
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

template <int LAYOUT>
const void *mma_fn(int D, int B) {
    if (D == 128 && B == 16) return (const void *)decode_mma_kernel<128, 16, LAYOUT>;
    if (D == 128 && B == 32) return (const void *)decode_mma_kernel<128, 32, LAYOUT>;
    if (D == 64 && B == 16) return (const void *)decode_mma_kernel<64, 16, LAYOUT>;
    if (D == 64 && B == 32) return (const void *)decode_mma_kernel<64, 32, LAYOUT>;
    return nullptr;
}

const void *mma_kernel_ptr(int D, int B, int layout) {
    return layout == PA_LAYOUT_SPLIT ? mma_fn<PA_LAYOUT_SPLIT>(D, B) : mma_fn<PA_LAYOUT_ROW>(D, B);
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
    if (kernel == PA_KERNEL_MMA) {
        p->NH = largest_divisor_at_most(c->num_kv_heads, kMmaMaxHeads);
        p->smem = mma_smem_bytes(c->head_dim, c->block_size, p->NH);
    } else {
        p->NH = largest_divisor_at_most(c->num_kv_heads, 8);
        p->smem = 0;
    }
    p->NG = c->num_kv_heads / p->NH;
    p->HPG = p->NH * G;
    int C = opts ? opts->num_splits : 0;
    if (C == 0) {
        if (!need_default_splits) return PA_ERR_INVALID_ARG;
        const void *fn = kernel == PA_KERNEL_MMA ? mma_kernel_ptr(c->head_dim, c->block_size, c->layout)
                                                 : simt_kernel_ptr(c->dtype, c->head_dim, G, c->layout);
        const int threads = kernel == PA_KERNEL_MMA ? (p->NH + 1) * 32 : p->NH * 32;
        C = default_ctas(fn, threads, p->smem);
        if (C <= 0) return PA_ERR_CUDA;
    }
    p->C = C;
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
    pa_decode_opts_t o = opts ? *opts : pa_decode_opts_t{0, PA_KERNEL_AUTO, nullptr, nullptr};
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
    {
        int32_t Nv = num_seqs, Bv = cache->block_size, ml_v = max_len, HDv = HD, nc = ncnt, NGv = p.NG, Cv = p.C;
        void *outp = out;
        void *pargs[] = {&seq_lens, &Nv, &Bv, &ml_v, &HDv, &lens_ws, &cu, &cnt, &nc, &outp, &NGv, &Cv, &start_seq, &err};
        const void *pfn = cache->dtype == PA_BF16 ? (const void *)decode_plan_kernel<__nv_bfloat16>
                                                  : (const void *)decode_plan_kernel<float>;
        if (launch_pdl(pfn, dim3(1), dim3(1024), pargs, 0, s) != cudaSuccess) return PA_ERR_CUDA;
    }

    if (opts && opts->ev_partial_begin && cudaEventRecord((cudaEvent_t)opts->ev_partial_begin, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (p.kernel == PA_KERNEL_MMA) {
        if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0) return PA_ERR_INVALID_ARG;
        CUtensorMap tmk, tmv;
        if (!encode_cache_map(&tmk, k_cache, cache, p.NH) || !encode_cache_map(&tmv, v_cache, cache, p.NH))
            return PA_ERR_CUDA;
        const void *fn = mma_kernel_ptr(cache->head_dim, cache->block_size, cache->layout);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
            return PA_ERR_CUDA;
        const dim3 grid(p.C), block((p.NH + 1) * 32);
        const __nv_bfloat16 *qb = (const __nv_bfloat16 *)q;
        __nv_bfloat16 *ob = (__nv_bfloat16 *)out;
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq;
        float sl = scale_log2;
        void *args[] = {&tmk, &tmv, &qb, &ob, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk, &Gv,
                        &NB, &NHv, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err};
        if (launch_pdl(fn, grid, block, args, p.smem, s) != cudaSuccess) return PA_ERR_CUDA;
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
