// CUDA-core decode kernel (instantiated in decode_simt.cu).
//
// fp32 (and bf16 shapes the tensor-core kernel does not cover): one warp per
// KV head, warp-shuffle q.k and online softmax over one token at a time.
#pragma once

#include "pa_internal.h"

namespace pa {

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

}  // namespace pa
