// CUDA-core decode kernel with TMA-staged blocks (instantiated in decode_simt.cu).
//
// For what the tensor-core kernel does not cover in the row layout: fp32
// (whose 1e-5 tolerance rules out bf16 and tf32 tensor cores), head_dim 256,
// block sizes other than 16 and 32.  Same work split, plan kernel, pieces and
// merges as the tensor-core kernel; the blocks arrive the same way (a producer
// warp issues TMA loads of (block, NH KV heads) tiles into an mbarrier ring,
// 128-byte swizzled), and each consumer warp owns one KV head and its G query
// heads.  A staged block is worked in two phases:
//   1. scores: lane (token t, slice p) takes a dot product over its D / LPT
//      elements of K row t for every query head (q in shared memory, in fp32),
//      the LPT slices of a token are summed with shuffles, and the block's
//      maximum and probabilities come from one shuffle reduction per head;
//      the probabilities go to shared memory;
//   2. P V: lane l owns D / 32 consecutive elements of the output and adds
//      p[h][t] * V[t] for every token of the block (probabilities read as
//      shared-memory broadcasts).
// The online softmax is in log2 units, as in the tensor-core kernel; the
// accumulators are rescaled only when a head's running maximum moved.
#pragma once

#include <cuda.h>  // CUtensorMap

#include "pa_internal.h"
#include "decode_merge.cuh"  // pieces and merges
#include "decode_simt.cuh"   // to_f32

namespace pa {

template <typename T>
struct FmaElt;
template <>
struct FmaElt<float> {
    static constexpr int kLine = 32;   // elements per 128-byte line (TMA box inner dimension)
    static constexpr int kChunk = 4;   // elements per 16-byte chunk
};
template <>
struct FmaElt<__nv_bfloat16> {
    static constexpr int kLine = 64;
    static constexpr int kChunk = 8;
};

// Elements of a 16-byte chunk as fp32.
__device__ __forceinline__ void chunk_f32(const uint4 &u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void chunk_f32(const uint4 &u, float (&x)[8]) {
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16);
    x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16);
    x[7] = __uint_as_float(u.w & 0xffff0000u);
}

// Byte offset of (line, 16-byte chunk) in a 128-byte-swizzled box whose base
// is 1024-byte aligned: the chunk index is XORed with the line index mod 8.
__device__ __forceinline__ uint32_t swz_off(int line, int chunk) {
    return (uint32_t)line * 128u + ((uint32_t)(chunk ^ (line & 7)) << 4);
}

// EPL consecutive elements of a line (EPL * sizeof(T) = 4, 8 or 16 bytes,
// never crossing a 16-byte chunk) as fp32.
template <typename T, int EPL>
__device__ __forceinline__ void load_elems(const uint8_t *p, float (&x)[EPL]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (EPL == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(p);
            x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
        } else {
            static_assert(EPL == 2, "fp32 slices are 2 or 4 elements");
            const float2 v = *reinterpret_cast<const float2 *>(p);
            x[0] = v.x, x[1] = v.y;
        }
    } else {
        if constexpr (EPL == 8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(p);
            chunk_f32(u, x);
        } else if constexpr (EPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(p);
            x[0] = __uint_as_float(u.x << 16), x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16), x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            static_assert(EPL == 2, "bf16 slices are 2, 4 or 8 elements");
            const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
            x[0] = __uint_as_float(u << 16), x[1] = __uint_as_float(u & 0xffff0000u);
        }
    }
}

// Shared memory of one CTA (host and device agree through these helpers).
struct FmaSmem {
    // one tensor's box of NH heads: (D / kLine) * B lines of 128 bytes per head
    __host__ __device__ static uint32_t box_bytes(int NH, int D, int B, int line_elems) {
        return (uint32_t)(((size_t)NH * (D / line_elems) * B * 128 + 1023) & ~(size_t)1023);
    }
    // per consumer warp: q of its G (<= GMAX) heads in fp32, [head][slice][D / LPT + 4]
    __host__ __device__ static uint32_t q_floats(int GMAX, int D, int LPT) { return (uint32_t)GMAX * (D + 4 * LPT); }
    // per consumer warp: probabilities of one pass of tokens, [token][GMAX]
    __host__ __device__ static uint32_t p_floats(int GMAX, int LPT) { return (uint32_t)(32 / LPT) * GMAX; }
    __host__ __device__ static size_t bytes(int S, int NH, int D, int B, int line_elems, int GMAX, int LPT) {
        return (size_t)S * 2 * box_bytes(NH, D, B, line_elems) + 256 +
               (size_t)NH * (q_floats(GMAX, D, LPT) + p_floats(GMAX, LPT)) * sizeof(float) + 1024;
    }
};

// Lanes per token in the score phase (each takes half of D), so tokens are
// taken 16 at a time: one pass for blocks of up to 16 tokens.  A fixed count
// keeps every loop of the consumers' inner code at a compile-time length.
constexpr int kFmaLanesPerToken = 2;
__host__ __device__ __forceinline__ int fma_lanes_per_token(int) { return kFmaLanesPerToken; }

// Up to 4 consumer warps and a producer; three CTAs per SM (the ring and q
// rows of a CTA take at most ~70 KB of shared memory for the common shapes),
// two for the instances whose accumulators need more registers.
template <int D, int GMAX>
constexpr int fma_min_ctas() { return (GMAX == 8 || GMAX * D >= 1024) ? 2 : 3; }

template <typename T, int D, int GMAX>
__global__ void __launch_bounds__(160, fma_min_ctas<D, GMAX>()) decode_fma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const T *__restrict__ q,
    T *__restrict__ out, const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G, int32_t B, int32_t NB, int32_t NH,
    int32_t S, float scale_log2, int32_t C, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, unsigned int *__restrict__ err) {
    constexpr int E = FmaElt<T>::kLine, EC = FmaElt<T>::kChunk;
    constexpr int DL = D / E;     // 128-byte lines per token row
    constexpr int EPL = D / 32;   // output elements per lane in the P V phase
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    grid_dependency_wait();  // the plan kernel's cu[] / lens / start table (programmatic launch)

    constexpr int LPT = kFmaLanesPerToken, TPP = 32 / LPT;
    const uint32_t box = FmaSmem::box_bytes(NH, D, B, E), stage_bytes = 2 * box;
    uint64_t *full = (uint64_t *)(smem + (size_t)S * stage_bytes);
    uint64_t *empty = full + S;
    float *qsm_all = (float *)(smem + (size_t)S * stage_bytes + 256);
    const uint32_t qf = FmaSmem::q_floats(GMAX, D, LPT), pf = FmaSmem::p_floats(GMAX, LPT);

    const int32_t NG = Hk / NH, HPG = NH * G;
    const int64_t W = (int64_t)NG * cu[N];
    const int32_t Ce = (int32_t)(W < (int64_t)C ? W : (int64_t)C);  // no CTA with an empty range
    const int32_t c = blockIdx.x;
    if (c >= Ce) return;
    const int64_t lo = split_begin(c, W, Ce), hi = split_begin(c + 1, W, Ce);
    const int64_t n = hi - lo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
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
            const uint64_t kv_policy = l2_policy_evict_first();  // KV streams through once
            BlockCursor cur, ahead;
            cur.init_at(lo, start_seq[c], cu, N);
            ahead = cur;
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
                mbar_arrive_expect_tx(fb, 2u * (uint32_t)NH * DL * B * 128u);
                tma_load_4d_hint(dst, &tmk, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                tma_load_4d_hint(dst + box, &tmv, fb, 0, phys * B, 0, cur.g * NH, kv_policy);
                cur.advance(cu, N);
            }
            // Let every copy still in flight land before the CTA may exit.
            for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1));
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    constexpr int kPer = D / LPT;           // score-phase elements per lane
    constexpr int kQStride = kPer + 4;      // padded slice: the two slices fall in distinct banks
    constexpr int kChunks = kPer / EC;      // 16-byte K chunks per lane and token
    constexpr int kChains = GMAX <= 4 ? 2 : 1;  // independent partial sums per head (shorter FMA chains)
    float *qs = qsm_all + (size_t)warp * (qf + pf);  // [GMAX][LPT][kQStride]
    float *ps = qs + qf;                             // [TPP][GMAX]
    const int tl = lane / LPT, part = lane - tl * LPT;
    // Sequences whose merge falls to this warp, done after the block loop
    // where its registers are free (only a range's first and last segments
    // are pieces: at most two).
    int32_t pend0 = -1, pend1 = -1;
    float acc[GMAX][EPL], m[GMAX], l[GMAX];
    BlockCursor cur;
    cur.init_at(lo, start_seq[c], cu, N);
    bool seg_start = true, seg_from_first = false;
    int32_t L = 0;
    for (int64_t it = 0; it < n; ++it) {
        const int s = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        const int32_t kvh = cur.g * NH + warp;
        if (seg_start) {
            L = lens[cur.seq];
            // this warp's q rows, as fp32, into its padded slices
            __syncwarp();  // the previous segment's reads of qs are done
            const T *qp = q + ((int64_t)cur.seq * H + (int64_t)kvh * G) * D;
#pragma unroll 4
            for (int e = lane; e < GMAX * D; e += 32) {
                const int h = e / D, d = e - h * D;
                const float v = h < G ? to_f32<T>(qp[(int64_t)h * D + d]) : 0.f;
                const int pp = d / kPer;
                qs[h * (LPT * kQStride) + pp * kQStride + (d - pp * kPer)] = v;
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
#pragma unroll
                for (int j = 0; j < EPL; ++j) acc[h][j] = 0.f;
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
            seg_from_first = (cur.blk == 0);
            seg_start = false;
        }
        const bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(err, kErrTimeout);
            return;
        }
        const uint8_t *kbox = smem + (size_t)s * stage_bytes;
        const uint8_t *vbox = kbox + box;
        const int32_t ntok = min(B, L - cur.blk * B);
        for (int t0 = 0; t0 < ntok; t0 += TPP) {
            // ---- scores of tokens t0 .. t0 + TPP - 1 (lane: token t0 + tl, slice part)
            const int t = t0 + tl;
            float sc[GMAX];
            {
                float sp[kChains][GMAX];
#pragma unroll
                for (int k = 0; k < kChains; ++k)
#pragma unroll
                    for (int h = 0; h < GMAX; ++h) sp[k][h] = 0.f;
                if (t < B) {
                    const float *qv = qs + part * kQStride;
#pragma unroll 4
                    for (int i = 0; i < kChunks; ++i) {
                        const int e0 = part * kPer + i * EC;
                        const int line = (warp * DL + e0 / E) * B + t;
                        const uint4 raw = *reinterpret_cast<const uint4 *>(kbox + swz_off(line, (e0 % E) / EC));
                        float kx[EC];
                        chunk_f32(raw, kx);
#pragma unroll
                        for (int h = 0; h < GMAX; ++h) {
                            if (h < G) {
#pragma unroll
                                for (int j = 0; j < EC; j += 4) {
                                    const float4 qq =
                                        *reinterpret_cast<const float4 *>(qv + h * LPT * kQStride + i * EC + j);
                                    float &a = sp[i % kChains][h];
                                    a = fmaf(qq.x, kx[j], a);
                                    a = fmaf(qq.y, kx[j + 1], a);
                                    a = fmaf(qq.z, kx[j + 2], a);
                                    a = fmaf(qq.w, kx[j + 3], a);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    sc[h] = sp[0][h];
#pragma unroll
                    for (int k = 1; k < kChains; ++k) sc[h] += sp[k][h];
                }
            }
            // the two slices of a token are adjacent lanes
#pragma unroll
            for (int o = 1; o < LPT; o <<= 1)
#pragma unroll
                for (int h = 0; h < GMAX; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
            const bool valid = t < ntok;
            float alpha[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                const float x = valid ? sc[h] * scale_log2 : -INFINITY;  // stale rows (maybe NaN) never count
                float mx = x;
#pragma unroll
                for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = fmaxf(m[h], mx);  // every pass has a valid token: finite
                alpha[h] = ex2_approx(m[h] - mn);
                const float p = ex2_approx(x - mn);
                if (part == 0) ps[tl * GMAX + h] = p;
                m[h] = mn;
            }
            __syncwarp();
            // ---- P V over this pass's valid tokens (lane: elements lane * EPL ..)
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                if (alpha[h] != 1.f) {  // the same for every lane: no divergence
                    l[h] *= alpha[h];
#pragma unroll
                    for (int j = 0; j < EPL; ++j) acc[h][j] *= alpha[h];
                }
            }
            const int d0 = lane * EPL;
            const int nt = min(TPP, ntok - t0);
            const uint8_t *vrow = vbox + swz_off(0, 0);  // lines below: (warp * DL + d0 / E) * B + t0 + k
            const int vline0 = (warp * DL + d0 / E) * B + t0;
            const uint32_t vbyte = (uint32_t)((d0 % EC) * sizeof(T));
#pragma unroll 4
            for (int k = 0; k < nt; ++k) {
                const int line = vline0 + k;
                float vx[EPL];
                load_elems<T, EPL>(vrow + swz_off(line, (d0 % E) / EC) + vbyte, vx);
                float pk[GMAX];
                if constexpr (GMAX % 4 == 0) {
#pragma unroll
                    for (int h = 0; h < GMAX; h += 4) {
                        const float4 p4 = *reinterpret_cast<const float4 *>(ps + k * GMAX + h);
                        pk[h] = p4.x, pk[h + 1] = p4.y, pk[h + 2] = p4.z, pk[h + 3] = p4.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < GMAX; ++h) pk[h] = ps[k * GMAX + h];
                }
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    l[h] += pk[h];
#pragma unroll
                    for (int j = 0; j < EPL; ++j) acc[h][j] = fmaf(pk[h], vx[j], acc[h][j]);
                }
            }
            __syncwarp();  // the pass's probabilities are read before the next pass writes them
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        const bool last_blk = (cur.blk == cur.nb - 1);
        if (last_blk || it + 1 == n) {
            if (seg_from_first && last_blk) {
                T *op = out + ((int64_t)cur.seq * H + (int64_t)kvh * G) * D + lane * EPL;
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h < G) {
                        const float inv = 1.f / l[h];
#pragma unroll
                        for (int j = 0; j < EPL; ++j) store_out(op + (int64_t)h * D + j, acc[h][j] * inv);
                    }
                }
            } else {
                const int64_t slot = partial_slot(c, cur.g * N + cur.seq);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h < G) {
                        const int64_t hh = slot * HPG + warp * G + h;
                        float *ap = acc_ws + hh * D + lane * EPL;
#pragma unroll
                        for (int j = 0; j < EPL; ++j) ap[j] = acc[h][j];
                        if (lane == 0) ml_ws[hh] = make_float2(m[h], l[h]);
                    }
                }
                const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, cur.seq, cur.g, warp, G, HPG, W, Ce),
                                          no_range()};
                if (arrive_piece(counters, rg, counter_index(cur.seq, kvh, N, NH), lane)) {
                    if (pend0 < 0)
                        pend0 = cur.g * N + cur.seq;
                    else
                        pend1 = cur.g * N + cur.seq;
                }
            }
            seg_start = true;
        }
        cur.advance(cu, N);
    }
    // Merges whose last piece this warp published (the split-K reduce).
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
        const int32_t sp = k == 0 ? pend0 : pend1;
        if (sp < 0) continue;
        const int32_t g = sp / N, seq = sp - g * N;
        const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, seq, g, warp, G, HPG, W, Ce), no_range()};
        __threadfence();  // every other piece is published: read them
        merge_pieces<T, D>(out + ((int64_t)seq * H + (int64_t)(g * NH + warp) * G) * D, rg, G, lane);
    }
}

}  // namespace pa
