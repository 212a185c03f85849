// TMA + tensor-core decode kernel (instantiated in decode_mma_plain.cu and
// decode_mma_shared.cu).
//
// TMA tiles of (block, up to 4 KV heads) through an mbarrier ring, mma.sync for
// S^T = K Q^T and O^T += V^T P^T; own-block CTAs and, with a plan,
// shared-prefix CTAs in one launch.
#pragma once

#include <cuda.h>  // CUtensorMap

#include "pa_internal.h"

namespace pa {

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

// Barrier of one CTA, or of one half of a two-half CTA (named barrier
// 1 + half over its 32 * (kMmaMaxHeads + 1) threads; 0: the whole CTA).
__device__ __forceinline__ void cta_sync(uint32_t bar) {
    if (bar == 0)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * (kMmaMaxHeads + 1)) : "memory");
}

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
        // Lazy maximum: the column maxima (shuffles over the 8 lanes of a
        // column) and the rescale only when some score passes the running
        // maximum by more than kLazyMaxSlack (always on a segment's first
        // tokens, where the maximum is -inf).
        if (__any_sync(0xffffffffu, mx0 > m0 + kLazyMaxSlack || mx1 > m1 + kLazyMaxSlack)) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = ex2_approx(m0 - mn0), al1 = ex2_approx(m1 - mn1);
            l0 *= al0;
            l1 *= al1;
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int dm = 0; dm < KT; ++dm) {
                o[dm][0] *= al0;
                o[dm][1] *= al1;
                o[dm][2] *= al0;
                o[dm][3] *= al1;
            }
        }
        const float p0 = ex2_approx(x0 - m0), p1 = ex2_approx(x1 - m1);
        const float p2 = ex2_approx(x2 - m0), p3 = ex2_approx(x3 - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
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
    static constexpr int kBytes = kPlanWarpRows * kRowBytes;
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
        // Two accumulators per tile (even and odd k-steps), summed at the end:
        // the dependent MMA chain is half as long.
        float sacc[NT][2][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) sacc[t][h][0] = sacc[t][h][1] = sacc[t][h][2] = sacc[t][h][3] = 0.f;
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
            mma_bf16_16816(sacc[0][kk & 1], a0, a1, a2, a3, b00, b01);
            mma_bf16_16816(sacc[1][kk & 1], a0, a1, a2, a3, b10, b11);
        }
        uint32_t pb0[NT], pb1[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float x0 = (sacc[t][0][0] + sacc[t][1][0]) * scale_log2;
            const float x1 = (sacc[t][0][1] + sacc[t][1][1]) * scale_log2;
            const float x2 = (sacc[t][0][2] + sacc[t][1][2]) * scale_log2;
            const float x3 = (sacc[t][0][3] + sacc[t][1][3]) * scale_log2;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
            // Lazy maximum, as in mma_block: shuffles and rescale only when a
            // score passes the running maximum by more than kLazyMaxSlack.
            if (__any_sync(0xffffffffu, mx0 > m[t][0] + kLazyMaxSlack || mx1 > m[t][1] + kLazyMaxSlack)) {
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
                const float al0 = ex2_approx(m[t][0] - mn0), al1 = ex2_approx(m[t][1] - mn1);
                l[t][0] *= al0;
                l[t][1] *= al1;
                m[t][0] = mn0;
                m[t][1] = mn1;
#pragma unroll
                for (int dm = 0; dm < KT; ++dm) {
                    o[t][dm][0] *= al0;
                    o[t][dm][1] *= al1;
                    o[t][dm][2] *= al0;
                    o[t][dm][3] *= al1;
                }
            }
            const float p0 = ex2_approx(x0 - m[t][0]), p1 = ex2_approx(x1 - m[t][1]);
            const float p2 = ex2_approx(x2 - m[t][0]), p3 = ex2_approx(x3 - m[t][1]);
            l[t][0] += p0 + p2;
            l[t][1] += p1 + p3;
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

// The TMA producer of a shared-prefix CTA (one thread): its range [lo, lo + n)
// of the flattened (stage head group, virtual sequence, block) list through a
// ring of S stages of stage_bytes, nhb one-head boxes of K then of V per
// stage (tile_bytes each).  Each block is read through the table row of the
// sequence of the pass's first query row (a member of the group).
template <int D, int B, int LAYOUT>
__device__ __forceinline__ void shared_prefix_producer(uint8_t *smem, uint64_t *full, uint64_t *empty, int S,
                                                       uint32_t stage_bytes, uint32_t tile_bytes, int32_t nhb,
                                                       const CUtensorMap *tmk1, const CUtensorMap *tmv1,
                                                       const int32_t *__restrict__ tables, int32_t max_blocks,
                                                       int32_t NB, const PlanView &pv, const SharedArgs &sh,
                                                       int32_t c, int64_t lo, int64_t n,
                                                       unsigned int *__restrict__ err) {
    using Tile = MmaTile<D, B>;
    const int32_t V = pv.V;
    prefetch_tmap(tmk1);
    prefetch_tmap(tmv1);
    const uint64_t kv_policy = l2_policy_evict_first();  // a pass streams each shared block once
    BlockCursor cur, ahead;
    cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
    ahead.init_at(lo, sh.start_s[c], pv.cu_s, V);
    // table row of a virtual sequence: the sequence of its first query row
    // (the plan kernel's row table), a member of the group that shares the
    // prefix: one load rather than the chain through the plan's arrays
    auto rep_row = [&](int32_t v) { return (int64_t)sh.rowseq[(int64_t)v * pv.R] * max_blocks; };
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
        const int st = (int)(issued % S);
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
        if (issued >= S && !mbar_wait_bounded(smem_u32(&empty[st]), ph ^ 1u)) {
            atomicOr(err, kErrTimeout);
            break;
        }
        if (phys < 0 || phys >= NB) {  // read zeros: the box lies past the pool
            atomicOr(err, kErrBounds);
            phys = NB;
        }
        const uint32_t fb = smem_u32(&full[st]);
        const uint32_t dst = smem_u32(smem + (size_t)st * stage_bytes);
        mbar_arrive_expect_tx(fb, stage_bytes);
        for (int32_t h = 0; h < nhb; ++h) {  // nhb one-head boxes land as one nhb-head box would
            const int32_t head = cur.g * nhb + h;
            const uint32_t off = (uint32_t)h * Tile::kSlabBytes;
            if (LAYOUT == PA_LAYOUT_ROW) {
                tma_load_4d_hint(dst + off, tmk1, fb, 0, phys * B, 0, head, kv_policy);
                tma_load_4d_hint(dst + tile_bytes + off, tmv1, fb, 0, phys * B, 0, head, kv_policy);
            } else {
                tma_load_4d_hint(dst + off, tmk1, fb, 0, 0, head, phys, kv_policy);
                tma_load_4d_hint(dst + tile_bytes + off, tmv1, fb, 0, 0, head, phys, kv_policy);
            }
        }
        cur.advance(pv.cu_s, V);
    }
    // Let every copy still in flight land before the CTA may exit.
    for (int64_t j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1));
}

// A CTA of the shared-prefix part.  Its range of the flattened (stage head
// group hg, virtual sequence v, block) list: W_s = (Hk / nhb) * cu_s[V]
// entries cut over Ce_s CTAs, nhb = plan_stage_heads(R) KV heads per stage.
// The ring has the own-block CTAs' bytes, cut into 2, 4 or 8 stages of nhb
// one-head TMA boxes of K and of V (tmk1 / tmv1).  Each block of a group's
// prefix is read once per pass (the table of one of its members), and
// warp w applies head hg * nhb + w / (R / 16) of the stage to its 16 query
// rows of the pass (member m = row / G, query head h = kvh * G + row % G), as
// two 8-column MMA tiles; a warp whose rows are all past the group's rows
// only keeps the ring's phases.  A piece's partial goes to slot
// c + hg * V + v, rows w * 16 .. + 15; shared_merge_kernel merges the
// members' pieces after the launch.
template <int D, int B, int LAYOUT>
__device__ __forceinline__ void shared_prefix_cta(uint8_t *smem, const CUtensorMap *tmk1, const CUtensorMap *tmv1,
                                                  const __nv_bfloat16 *__restrict__ q,
                                                  const int32_t *__restrict__ tables, int32_t max_blocks, int32_t H,
                                                  int32_t G, int32_t NB, float scale_log2, int32_t Hk, int32_t Cs,
                                                  const SharedArgs &sh, unsigned int *__restrict__ err, int32_t cta,
                                                  int tid, uint32_t bar) {
    using Tile = MmaTile<D, B>;
    constexpr int KT = D / 16;
    constexpr int NT = kPlanWarpRows / 8;  // MMA tiles per warp
    constexpr uint32_t ring_bytes = (uint32_t)Tile::kStages * 2 * kPlanWarps * Tile::kSlabBytes;
    const SharedView sv = shared_view(sh.plan, sh.skip, sh.ml_s, sh.acc_s, Hk, Cs);
    const PlanView &pv = sv.pv;
    const int32_t R = pv.R, nhb = plan_stage_heads(R), wph = R / kPlanWarpRows;
    const uint32_t tile_bytes = (uint32_t)nhb * Tile::kSlabBytes, stage_bytes = 2 * tile_bytes;
    const int S = (int)(ring_bytes / stage_bytes);  // 2, 4 or 8 stages
    uint64_t *full = (uint64_t *)(smem + ring_bytes);
    uint64_t *empty = full + S;                     // 2 * S <= 16 barriers in the 256 bytes after the ring
    uint8_t *qbuf = smem + ring_bytes + 256;        // QRows of each consumer warp
    const int32_t c = cta;
    if (c >= sv.Ce_s) return;
    const int64_t lo = split_begin(c, sv.Ws, sv.Ce_s), hi = split_begin(c + 1, sv.Ws, sv.Ce_s);
    const int64_t n = hi - lo;
    const int32_t V = pv.V;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), (uint32_t)kPlanWarps);
        }
        fence_mbarrier_init();
    }
    cta_sync(bar);

    if (warp == kPlanWarps) {
        // ------------------------------------------------------- producer
        if (lane == 0)
            shared_prefix_producer<D, B, LAYOUT>(smem, full, empty, S, stage_bytes, tile_bytes, nhb, tmk1, tmv1, tables,
                                                 max_blocks, NB, pv, sh, c, lo, n, err);
        return;
    }

    // ----------------------------------------------------------- consumers
    const int r = lane >> 2, cq = lane & 3;
    const int hb = warp / wph, sub = warp - hb * wph;  // this warp's head in the stage, rows of the pass
    uint8_t *qw = qbuf + warp * QRows<D>::kBytes;
    float o[NT][KT][4];
    float mm[NT][2], ll[NT][2];
    BlockCursor cur;
    cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
    bool seg_start = true, active = false;
    uint32_t row_valid = 0;  // bit i: this warp's row i of the pass belongs to a member
    for (int64_t it = 0; it < n; ++it) {
        const int st = (int)(it % S);
        const uint32_t ph = (uint32_t)((it / S) & 1);
        const int32_t kvh = cur.g * nhb + hb, v = cur.seq;
        if (seg_start) {
            // This warp's rows of the pass: sub * 16 .. + 15 (member row / G,
            // query head row % G); lane i < 16 loads row i's sequence from the
            // plan kernel's table, then every load of the rows is issued at
            // once: two round trips per segment.
            int32_t row_seq = -1;
            if (lane < kPlanWarpRows) row_seq = sh.rowseq[(int64_t)v * R + sub * kPlanWarpRows + lane];
            row_valid = __ballot_sync(0xffffffffu, row_seq >= 0) & ((1u << kPlanWarpRows) - 1u);
            active = row_valid != 0;
            if (active) {
                // The warp's 16 query rows of its head into shared memory
                // (zeros for rows past the group's).
                __syncwarp();  // the previous segment's reads of qw are done
                constexpr int kChunks = D / 8;  // 16-byte pieces of a row
                uint4 val[kPlanWarpRows * kChunks / 32];
#pragma unroll
                for (int k = 0; k < kPlanWarpRows * kChunks / 32; ++k) {
                    const int e = lane + 32 * k, i = e / kChunks, ch = e - i * kChunks;
                    const int32_t seq = __shfl_sync(0xffffffffu, row_seq, i);
                    val[k] = make_uint4(0u, 0u, 0u, 0u);
                    if (seq >= 0) {  // q is 16-byte aligned with a plan; passes start on a member
                        const int hq = (sub * kPlanWarpRows + i) % G;
                        const __nv_bfloat16 *qp = q + ((int64_t)seq * H + (int64_t)kvh * G + hq) * D;
                        val[k] = *reinterpret_cast<const uint4 *>(qp + ch * 8);
                    }
                }
#pragma unroll
                for (int k = 0; k < kPlanWarpRows * kChunks / 32; ++k) {
                    const int e = lane + 32 * k, i = e / kChunks, ch = e - i * kChunks;
                    *reinterpret_cast<uint4 *>(qw + i * QRows<D>::kRowBytes + ch * 16) = val[k];
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
            }
            seg_start = false;
        }
        const bool ok = mbar_wait_bounded(smem_u32(&full[st]), ph);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(err, kErrTimeout);
            return;
        }
        if (active) {
            const uint32_t kslab = smem_u32(smem + (size_t)st * stage_bytes) + (uint32_t)hb * Tile::kSlabBytes;
            mma_block_tiles<D, B, LAYOUT, NT>(kslab, kslab + tile_bytes, smem_u32(qw), scale_log2, o, mm, ll, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));

        if (cur.blk == cur.nb - 1 || it + 1 == n) {
            if (active) {
                const int64_t slot = partial_slot(c, cur.g * V + v);
                const int64_t wrow = slot * kPlanSlotRows + warp * kPlanWarpRows;  // this warp's 16 rows
                const int h0 = 2 * cq, h1 = 2 * cq + 1;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float lt0 = ll[t][0], lt1 = ll[t][1];
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
                        lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
                    }
                    const bool v0 = (row_valid >> (t * 8 + h0)) & 1u, v1 = (row_valid >> (t * 8 + h1)) & 1u;
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
            }
            seg_start = true;
        }
        cur.advance(pv.cu_s, V);
    }
}

// A CTA of the own-block part (the whole grid without a plan): CTA c of Co
// takes its range of the flattened (head group, sequence, own block) list.
// Consumer warp w owns KV head g * NH + w and its G query heads.  kShared:
// sequences may start after a shared prefix (skip[seq] blocks).  cu[] is the
// plan kernel's (global memory) or the CTA's own copy (shared memory); lens[]
// is clamped here as the plan kernel clamps it; without a start table
// (start_seq == nullptr) the CTA finds its first sequence by search.
template <int D, int B, int LAYOUT, bool kShared>
__device__ __forceinline__ void own_block_cta(
    uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const __nv_bfloat16 *__restrict__ q,
    __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ tables, int32_t max_blocks,
    const int32_t *__restrict__ lens, const int32_t *cu, int32_t N, int32_t H, int32_t G, int32_t NB,
    int32_t NH, float scale_log2, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, int32_t Hk, int32_t C,
    int32_t Cs, const SharedArgs &sh, unsigned int *__restrict__ err, int32_t min_pieces, int32_t cta, int tid,
    uint32_t bar) {
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
    const int32_t c = cta - Cs;
    if (c >= Ce) return;
    const int64_t lo = split_begin(c, W, Ce), hi = split_begin(c + 1, W, Ce);
    const int64_t n = hi - lo;
    const int warp = tid >> 5, lane = tid & 31;
    // Sequences whose merge falls to a consumer warp, done after its block
    // loop where the loop's registers are free for the pieces' loads.  Only
    // the first and the last segment of a range are pieces: at most two.
    // One table per half of a two-half CTA.
    __shared__ int32_t pending_tab[kShared ? 2 : 1][kMmaMaxHeads][2];
    int32_t(&pending)[kMmaMaxHeads][2] = pending_tab[kShared && bar == 2 ? 1 : 0];
    if (tid < 2 * kMmaMaxHeads) pending[tid >> 1][tid & 1] = -1;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), (uint32_t)NH);
        }
        fence_mbarrier_init();
    }
    cta_sync(bar);

    if (warp == NH) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(tmk);
            prefetch_tmap(tmv);
            // KV tiles stream through once: evict them first, so that L2 keeps
            // the partials, q and tables that are read again.
            const uint64_t kv_policy = l2_policy_evict_first();
            BlockCursor cur, ahead;
            if (start_seq) {
                cur.init_at(lo, start_seq[c], cu, N, skip);
            } else {
                cur.init(lo, cu, N, skip);
            }
            ahead = cur;
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
    if (start_seq) {
        cur.init_at(lo, start_seq[c], cu, N, skip);
    } else {
        cur.init(lo, cu, N, skip);
    }
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
            L = (L < 0 || L > max_blocks * B) ? 0 : L;  // as the plan kernel clamps it
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
                // after this launch, one cut into min_pieces or more pieces by
                // long_merge_kernel, every other one by its last arriver after
                // its block loop (pending).
                const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, cur.seq, cur.g, warp, G, HPG, W, Ce),
                                          no_range()};
                const bool long_seq = min_pieces > 0 && rg[0].c1 - rg[0].c0 + 1 >= min_pieces;
                if (!(kShared && cur.b0 > 0) && !long_seq) {
                    // The plan kernel zeroes the arrival counters: it has
                    // finished before the first arrival (at once if it has).
                    grid_dependency_wait();
                    if (arrive_piece(counters, rg, counter_index(cur.seq, kvh, N, NH), lane) && lane == 0)
                        pending[warp][pending[warp][0] >= 0 ? 1 : 0] = cur.g * N + cur.seq;
                }
            }
            seg_start = true;
        }
        cur.advance(cu, N, skip);
    }
    __syncwarp();
    const int32_t sp0 = pending[warp][0], sp1 = pending[warp][1];
    if (sp0 >= 0) {
        const int32_t g = sp0 / N, seq = sp0 - g * N;
        const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, seq, g, warp, G, NH * G, W, Ce), no_range()};
        __threadfence();  // every other piece is published: read them
        merge_online<__nv_bfloat16, D, 3>(out + ((int64_t)seq * H + (int64_t)(g * NH + warp) * G) * D, rg, G, lane);
    }
    if (sp1 >= 0) {
        const int32_t g = sp1 / N, seq = sp1 - g * N;
        const PieceRange rg[2] = {own_range(ml_ws, acc_ws, cu, N, seq, g, warp, G, NH * G, W, Ce), no_range()};
        __threadfence();
        merge_online<__nv_bfloat16, D, 3>(out + ((int64_t)seq * H + (int64_t)(g * NH + warp) * G) * D, rg, G, lane);
    }
}

// Block counts of the N sequences and their exclusive prefix sums, written to
// cu_l[0..N] in shared memory by the whole CTA: the plan kernel's cu[] (the
// same clamping of bad lengths to 0), without waiting for that kernel.  Each
// thread scans a contiguous chunk; one block-wide scan joins the chunks.
__device__ __forceinline__ void local_prefix_sums(const int32_t *__restrict__ seq_lens, int32_t N, int32_t B,
                                                  int32_t max_len, int32_t *cu_l) {
    __shared__ int32_t warp_sum[32];
    const int32_t t = threadIdx.x, nt = blockDim.x;
    const int lane = t & 31, w = t >> 5, nw = (nt + 31) >> 5;
    for (int32_t i = t; i < N; i += nt) {
        int32_t L = seq_lens[i];
        L = (L < 0 || L > max_len) ? 0 : L;
        cu_l[i] = (L + B - 1) / B;
    }
    __syncthreads();
    const int32_t per = (N + nt - 1) / nt;
    const int32_t i0 = min(t * per, N), i1 = min(i0 + per, N);
    int32_t mine = 0;
    for (int32_t i = i0; i < i1; ++i) mine += cu_l[i];
    int32_t x = mine;  // inclusive scan of the chunk sums within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[w] = x;
    __syncthreads();
    if (w == 0) {
        int32_t v = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_sum[lane] = v;
    }
    __syncthreads();
    int32_t run = x - mine + (w > 0 ? warp_sum[w - 1] : 0);  // exclusive prefix of this chunk
    for (int32_t i = i0; i < i1; ++i) {
        const int32_t nb = cu_l[i];
        cu_l[i] = run;
        run += nb;
    }
    if (t == nt - 1) cu_l[N] = run;  // the last chunk ends at N: run is the total
    __syncthreads();
}

}  // namespace pa

#include "decode_tc.cuh"  // the tcgen05 shared-prefix CTA

namespace pa {

// The attention launch.  Without a plan (kShared = false) every CTA is an
// own-block CTA (two resident per SM at block size 16).  With one, each CTA
// is shared_halves(D, B) halves of 32 * (kMmaMaxHeads + 1) threads and
// shared_half_bytes of shared memory, one logical CTA each (halves * blockIdx
// + half): a kernel that holds tcgen05 instructions is resident once per SM,
// so two halves keep two logical CTAs per SM where they fit.  The plan kernel gives logical CTAs [0, Cs) to the shared prefixes
// and the rest to the sequences' own blocks; both kinds run at once and meet
// only at the arrival counters.  tmk / tmv hold NH-head boxes (the own-block
// CTAs'), tmk1 / tmv1 one-head boxes (the mma.sync shared-prefix CTAs'),
// tmkp / tmvp one-head, one-panel boxes (the tcgen05 ones').
template <int D, int B, int LAYOUT, bool kShared>
__global__ void __launch_bounds__(32 * (kMmaMaxHeads + 1) * (kShared ? shared_halves(D, B) : 1), kShared ? 1 : 2)
    decode_mma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __grid_constant__ CUtensorMap tmk1, const __grid_constant__ CUtensorMap tmv1,
    const __grid_constant__ CUtensorMap tmkp, const __grid_constant__ CUtensorMap tmvp,
    const __nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ out,
    const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ cu, int32_t N, int32_t H, int32_t Hk, int32_t G, int32_t NB,
    int32_t NH, float scale_log2, int32_t C, float2 *__restrict__ ml_ws, float *__restrict__ acc_ws,
    unsigned int *__restrict__ counters, const int32_t *__restrict__ start_seq, unsigned int *__restrict__ err,
    const SharedArgs sh, const int32_t *__restrict__ seq_lens, int32_t local_cu, int32_t min_pieces) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

    // local_cu (no plan, N + 1 <= kLocalCuMax; the host adds the room): the
    // CTA computes cu[] from seq_lens itself and starts on its blocks while
    // the plan kernel still runs; it waits for that kernel only before its
    // first arrival (the counters) and before it ends.  Otherwise it waits
    // here for the plan kernel's cu[], lens and start table.
    const bool local = !kShared && local_cu != 0;
    const int32_t *cu_p = cu, *lens_p = lens, *start_p = start_seq;  // generic: global or shared memory
    if (local) {
        using Tile = MmaTile<D, B>;
        int32_t *cu_l = (int32_t *)(smem + (size_t)Tile::kStages * 2 * NH * Tile::kSlabBytes +
                                    2 * Tile::kStages * sizeof(uint64_t));
        local_prefix_sums(seq_lens, N, B, max_blocks * B, cu_l);
        cu_p = cu_l;
        lens_p = seq_lens;
        start_p = nullptr;
    } else {
        grid_dependency_wait();  // the plan kernel's cu[] / lens / split (programmatic launch)
    }
    // With a plan or with long sequences, the merge kernel that follows may
    // become resident now and wait for this launch there.
    if (kShared || min_pieces > 0) grid_launch_dependents();
    if constexpr (kShared) {
        const int32_t Cs = sh.ctl[0];
        constexpr int kHalf = 32 * (kMmaMaxHeads + 1);
        const int half = (int)threadIdx.x / kHalf, tid = (int)threadIdx.x - half * kHalf;
        const int32_t cta = shared_halves(D, B) * (int32_t)blockIdx.x + half;
        uint8_t *hs = smem + (size_t)half * shared_half_bytes(D, B);
        const uint32_t bar = 1u + (uint32_t)half;
        if (cta < Cs) {
            bool tc = false;
            if constexpr (LAYOUT == PA_LAYOUT_ROW) tc = sh.tc != 0 && sh.plan[7] == kPlanSlotRows;
            if (tc)
                shared_prefix_cta_tc<D, B>(hs, &tmkp, &tmvp, q, tables, max_blocks, H, G, NB, scale_log2, Hk, Cs, sh,
                                           err, cta, tid, bar, half);
            else
                shared_prefix_cta<D, B, LAYOUT>(hs, &tmk1, &tmv1, q, tables, max_blocks, H, G, NB, scale_log2, Hk,
                                                Cs, sh, err, cta, tid, bar);
        } else {
            own_block_cta<D, B, LAYOUT, true>(hs, &tmk, &tmv, q, out, tables, max_blocks, lens_p, cu_p, N, H, G, NB,
                                              NH, scale_log2, ml_ws, acc_ws, counters, start_p, Hk, C, Cs, sh, err, 0,
                                              cta, tid, bar);
        }
    } else {
        own_block_cta<D, B, LAYOUT, false>(smem, &tmk, &tmv, q, out, tables, max_blocks, lens_p, cu_p, N, H, G, NB,
                                           NH, scale_log2, ml_ws, acc_ws, counters, start_p, Hk, C, 0, sh, err,
                                           min_pieces, (int32_t)blockIdx.x, (int)threadIdx.x, 0u);
    }
    // The grid ends after the plan kernel (which also writes the zero output
    // of empty sequences), as a grid that waited at its start does.
    if (local) grid_dependency_wait();
}

}  // namespace pa
