// Shared-prefix CTAs on the fifth-generation tensor cores (part of
// decode_mma.cuh, included after the shared-prefix producer).
//
// A pass of up to 64 query rows over one KV head's shared blocks is a
// product with M = rows: S = Q K^T and O += P V are tcgen05 MMAs whose
// operands are the TMA tiles as they land (128-byte swizzle), the query rows
// and the probabilities staged in shared memory, and whose accumulators S and
// O live in tensor memory.  One thread per query row reads its scores back
// with tcgen05.ld, so the softmax needs no shuffles and the running maximum
// is per thread ("10 PagedAttention" (PidokuInfra), section 5 "The kernel
// side": each block's scores, softmax and weighted V, here for all sharers'
// rows at once; "The relationship to prefix caching").
#pragma once

namespace pa {

// ------------------------------------------------------------ tcgen05 PTX
// Tensor memory: 128 lanes x 512 columns of 32 bits per SM.  Warp w of a CTA
// reaches lanes 32 (w % 4) .. + 31; an address is (lane << 16) | column.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) = A B (+ D when accumulate != 0); A and B from shared
// memory descriptors, bf16 inputs and fp32 accumulators (idesc).  Issued by
// one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One arrival on the barrier once every MMA this thread issued before has
// completed (and its shared-memory operands may be overwritten).
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive columns of this thread's lane, waited for in the same
// statement (the registers are not valid before the wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// The same for 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand (the layout
// TMA's 128-byte swizzle writes: 128-byte lines, 16-byte chunk index XOR
// line % 8, 1024-byte atoms of 8 lines).  K-major operands step 8-line
// groups by sbo along M / N (lbo unused); MN-major ones step 64-element
// atoms by lbo along M / N and 8-line groups by sbo along K.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of a dense bf16 x bf16 -> fp32 MMA of M x N.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------- shared-memory map (tc)
// One half of a two-half CTA: [P: 64 rows x 64 tokens bf16][Q: 64 rows x D
// bf16 in D/64 panels][two round slots][barriers].  A round slot holds up to
// 64 tokens (64 / B blocks) of one KV head as panels of 64 columns: K panel
// p at p * kPanel, V panel p at (D/64 + p) * kPanel, token t of the round at
// line t of each (128-byte lines, 128-byte swizzle, as TMA writes a box of
// B lines).  So the round's tokens are one operand of N = 64 (S = Q K^T) and
// of K = 64 (O += P V).  The MMAs are M = 128: in the first half rows
// 64..127 of P read Q's bytes and those of Q's last panel read slot 0; the
// second half's descriptors start 8 KiB before P and Q, so its rows 0..63
// read the bytes before them.  Those rows' results land in tensor-memory
// lanes that are never read.
template <int D, int B>
struct TcSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kRB = 64 / B;  // blocks per round
    static constexpr uint32_t kPanel = 64 * 128;
    static constexpr uint32_t kP = 64 * 64 * 2;
    static constexpr uint32_t kQ = 64 * D * 2;
    static constexpr uint32_t kSlot = 2 * kPanels * kPanel;
    static constexpr uint32_t kBars = 256;
    static constexpr uint32_t kBytes = kP + kQ + 2 * kSlot + kBars;
    static constexpr uint32_t kCols = D == 128 ? 256 : 128;  // S: 64 columns, O: D columns
    static_assert(kBytes <= shared_half_bytes(D, B), "the tcgen05 map fits one half");
    static_assert(kSlot >= 8192, "the last Q panel's unused rows read 8 KiB past Q");
};

// Rounds of a tcgen05 shared-prefix CTA: up to 64 / B blocks of one segment
// (virtual sequence and KV head), cut at the segment's and the range's end.
__device__ __forceinline__ int tc_round_blocks(const BlockCursor &cur, int64_t it, int64_t n, int rb) {
    int nblk = cur.nb - cur.blk;
    if (nblk > rb) nblk = rb;
    if ((int64_t)nblk > n - it) nblk = (int)(n - it);
    return nblk;
}

// The TMA producer of a tcgen05 shared-prefix CTA (one thread): round r into
// slot r % 2, each block as 2 * D/64 one-panel boxes (tmkp / tmvp), through
// the table row of the sequence of the pass's first query row.
template <int D, int B>
__device__ __forceinline__ void shared_prefix_producer_tc(uint8_t *slots, uint64_t *full, uint64_t *empty,
                                                          const CUtensorMap *tmkp, const CUtensorMap *tmvp,
                                                          const int32_t *__restrict__ tables, int32_t max_blocks,
                                                          int32_t NB, const PlanView &pv, const SharedArgs &sh,
                                                          int32_t c, int64_t lo, int64_t n,
                                                          unsigned int *__restrict__ err) {
    using L = TcSmem<D, B>;
    const int32_t V = pv.V;
    prefetch_tmap(tmkp);
    prefetch_tmap(tmvp);
    const uint64_t kv_policy = l2_policy_evict_first();  // a pass streams each shared block once
    BlockCursor cur, ahead;
    cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
    ahead = cur;
    // table row of a virtual sequence: the sequence of its first query row
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
    int64_t it = 0, r = 0;
    for (; it < n; ++r) {
        const int nblk = tc_round_blocks(cur, it, n, L::kRB);
        const int slot = (int)(r & 1);
        if (r >= 2 && !mbar_wait_bounded(smem_u32(&empty[slot]), (uint32_t)(((r >> 1) & 1) ^ 1))) {
            atomicOr(err, kErrTimeout);
            break;
        }
        const uint32_t fb = smem_u32(&full[slot]);
        const uint32_t base = smem_u32(slots + (size_t)slot * L::kSlot);
        mbar_arrive_expect_tx(fb, (uint32_t)nblk * 2u * (uint32_t)D * (uint32_t)B * 2u);
        for (int b = 0; b < nblk; ++b) {
            int32_t phys = ring[0];
#pragma unroll
            for (int j = 0; j + 1 < PD; ++j) ring[j] = ring[j + 1];
            if (it + b + PD < n) {
                if (ahead.seq != ahead_v) {
                    ahead_v = ahead.seq;
                    ahead_row = rep_row(ahead_v);
                }
                ring[PD - 1] = tables[ahead_row + ahead.blk];
                ahead.advance(pv.cu_s, V);
            }
            if (phys < 0 || phys >= NB) {  // read zeros: the box lies past the pool
                atomicOr(err, kErrBounds);
                phys = NB;
            }
            const uint32_t line = (uint32_t)(b * B * 128);
#pragma unroll
            for (int p = 0; p < L::kPanels; ++p) {
                tma_load_4d_hint(base + (uint32_t)p * L::kPanel + line, tmkp, fb, 0, phys * B, p, cur.g, kv_policy);
                tma_load_4d_hint(base + (uint32_t)(L::kPanels + p) * L::kPanel + line, tmvp, fb, 0, phys * B, p, cur.g,
                                 kv_policy);
            }
        }
        for (int b = 0; b < nblk; ++b) cur.advance(pv.cu_s, V);
        it += nblk;
    }
    // Let every copy still in flight land before the CTA may exit.
    for (int64_t j = r > 2 ? r - 2 : 0; j < r; ++j) mbar_wait_bounded(smem_u32(&full[j & 1]), (uint32_t)((j >> 1) & 1));
}

// A shared-prefix CTA on tcgen05 (plans of 64 rows per pass: one KV head
// per segment), one half of a two-half CTA.  Warp 4 of the half streams the
// CTA's range of (KV head, virtual sequence, block) in rounds of up to 64
// tokens of one segment.  A consumer thread of a warp without query rows
// issues the MMAs.  A consumer thread owns
// the tensor-memory lane its warp reaches (CTA warp w: lanes 32 (w % 4) ..,
// so the halves' consumer warps cover the four quadrants in different
// orders); lane rbase + t holds query row t < 64 of the pass (member t / G,
// query head kvh * G + t % G), rbase = 0 in the first half and 64 in the
// second (its Q and P descriptors start 8 KiB early, so its rows sit in
// quadrants 2 and 3 and the halves' softmax warps use different SM
// partitions).  Per round:
//   S[rows][64] = Q K^T   (D/16 MMAs of N = the round's tokens),
//   rows: lazy running maximum, P = 2^(x - m) to shared memory as bf16,
//   O[rows][D] += P V     (one MMA of N = D per 16 tokens).
// At a segment's end O, m and l of each valid row go to the partial slot
// c + kvh * V + v, row t, as in the mma.sync version.
template <int D, int B>
__device__ __forceinline__ void shared_prefix_cta_tc(uint8_t *smem, const CUtensorMap *tmkp,
                                                     const CUtensorMap *tmvp, const __nv_bfloat16 *__restrict__ q,
                                                     const int32_t *__restrict__ tables, int32_t max_blocks,
                                                     int32_t H, int32_t G, int32_t NB, float scale_log2, int32_t Hk,
                                                     int32_t Cs, const SharedArgs &sh, unsigned int *__restrict__ err,
                                                     int32_t cta, int tid, uint32_t bar, int half) {
    using L = TcSmem<D, B>;
    constexpr int KT = D / 16;  // k-steps of Q K^T
    constexpr uint32_t IDESC_S = tc_idesc_bf16(128, 8, false, false) & ~(0x3Fu << 17);  // N set per round
    constexpr uint32_t IDESC_O = tc_idesc_bf16(128, D, false, true);
    const SharedView sv = shared_view(sh.plan, sh.skip, sh.ml_s, sh.acc_s, Hk, Cs);
    const PlanView &pv = sv.pv;
    const int32_t c = cta;
    if (c >= sv.Ce_s) return;
    const int64_t lo = split_begin(c, sv.Ws, sv.Ce_s), hi = split_begin(c + 1, sv.Ws, sv.Ce_s);
    const int64_t n = hi - lo;
    const int32_t V = pv.V;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t cons_bar = 3u + (uint32_t)half;  // the half's 4 consumer warps
    uint8_t *Ps = smem, *Qs = smem + L::kP, *slots = smem + L::kP + L::kQ;
    uint64_t *full = (uint64_t *)(slots + 2 * L::kSlot);
    uint64_t *empty = full + 2;
    uint64_t *sbar = empty + 2;  // S of a round computed
    uint64_t *obar = sbar + 1;   // O of a segment complete
    uint32_t *tmem_slot = (uint32_t *)(obar + 1);

    if (tid == 0) {
        for (int st = 0; st < 2; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), 1);  // one commit per round
        }
        mbar_init(smem_u32(sbar), 1);
        mbar_init(smem_u32(obar), 1);
        fence_mbarrier_init();
    }
    // Each half holds its own columns (two halves: at most 512, one SM's
    // tensor memory); the permit is kept, as the other half may allocate later.
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), L::kCols);
    tc_fence_before();
    cta_sync(bar);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kPlanWarps) {
        // ------------------------------------------------------- producer
        if (lane == 0)
            shared_prefix_producer_tc<D, B>(slots, full, empty, tmkp, tmvp, tables, max_blocks, NB, pv, sh, c, lo, n,
                                            err);
        return;
    }

    // -------------------------------------------------------- consumers
    const int row = (int)((threadIdx.x >> 5) & 3) * 32 + lane;  // this thread's tensor-memory lane
    const uint32_t t_lane = (uint32_t)(row & ~31) << 16;
    // The second half keeps its query rows in lanes 64..127 (quadrants 2 and
    // 3), so that the two halves' softmax warps run on different SM
    // partitions: its Q and P descriptors start 8 KiB before the rows (rows
    // 0..63 of its products read the preceding bytes and are never used).
    const int rbase = half ? 64 : 0;
    const int qi = row - rbase;  // query row of the pass this lane holds (0..63), if any
    const uint32_t a_shift = half ? 8192u : 0u;
    // The MMAs are issued by lane 0 of a consumer warp that holds no query
    // rows (quadrant 2 in the first half, quadrant 1 in the second), so that
    // a softmax warp never waits on a full MMA queue.
    const int issuer = half ? 0 : 64;
    const uint32_t tS = tmem, tO = tmem + 64;
    const uint32_t q_base = smem_u32(Qs), p_base = smem_u32(Ps), slot_base = smem_u32(slots);
    float m_run = -INFINITY, l_run = 0.f;
    bool valid = false;      // this thread's lane holds a query row of a member
    bool warp_rows = false;  // some row of this warp does
    bool seg_start = true, first_round = true, abort = false;
    uint32_t sph = 0, oph = 0;
    BlockCursor cur;
    cur.init_at(lo, sh.start_s[c], pv.cu_s, V);
    for (int64_t it = 0, r = 0; it < n; ++r) {
        const int32_t kvh = cur.g, v = cur.seq;
        const int nblk = tc_round_blocks(cur, it, n, L::kRB);
        const int ntok = nblk * B;
        const bool seg_end = cur.blk + nblk == cur.nb || it + nblk == n;
        const int slot = (int)(r & 1);
        const uint32_t kbase = slot_base + (uint32_t)slot * L::kSlot, vbase = kbase + L::kPanels * L::kPanel;
        if (seg_start) {
            // The pass's rows into Q (zeros past the group's rows): two
            // threads per row, D/2 elements each.
            const int i = tid >> 1, hf = tid & 1;
            const int32_t sq = sh.rowseq[(int64_t)v * 64 + i];
            uint4 val[D / 16];
            const __nv_bfloat16 *qp =
                q + ((int64_t)(sq < 0 ? 0 : sq) * H + (int64_t)kvh * G + i % G) * D + hf * (D / 2);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                val[k] = sq >= 0 ? *reinterpret_cast<const uint4 *>(qp + 8 * k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const int ch = hf * (D / 16) + k;  // 16-byte chunk of the row
                *reinterpret_cast<uint4 *>(Qs + (ch >> 3) * L::kPanel + i * 128 + (((ch & 7) ^ (i & 7)) << 4)) = val[k];
            }
            fence_proxy_async_smem();
            valid = qi >= 0 && qi < 64 && sh.rowseq[(int64_t)v * 64 + qi] >= 0;
            warp_rows = __any_sync(0xffffffffu, valid);
            m_run = -INFINITY;
            l_run = 0.f;
            first_round = true;
            named_bar_sync(cons_bar, 4 * 32);  // Q complete before the first S MMA
            seg_start = false;
        }
        if (tid == issuer) {
            if (!abort && !mbar_wait_bounded(smem_u32(&full[slot]), (uint32_t)((r >> 1) & 1))) {
                atomicOr(err, kErrTimeout);
                abort = true;  // the MMAs still run (on stale tiles), so that every wait below ends
            }
            tc_fence_after();
            const uint32_t idesc = IDESC_S | ((uint32_t)(ntok >> 3) << 17);
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                const uint32_t koff = (uint32_t)(k >> 2) * L::kPanel + (uint32_t)(k & 3) * 32;
                const uint64_t a = smem_desc_sw128(q_base - a_shift + koff, 16, 1024);  // Q panels: the same stride
                tc_mma_bf16(tS, a, smem_desc_sw128(kbase + koff, 16, 1024), idesc, k > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(sbar));
        }
        if (!abort && !mbar_wait_bounded(smem_u32(sbar), sph)) {
            atomicOr(err, kErrTimeout);
            abort = true;  // later waits are skipped: the call's output is flagged as unreliable
        }
        sph ^= 1u;
        tc_fence_after();
        if (warp_rows) {
            float xa[32], xb[32];  // tokens 0..31 and 32..63 of the round
            tmem_ld32(tS + t_lane, xa);
            tmem_ld32(tS + t_lane + 32, xb);
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                xa[j] = j < ntok ? xa[j] * scale_log2 : -INFINITY;
                xb[j] = 32 + j < ntok ? xb[j] * scale_log2 : -INFINITY;
                mx = fmaxf(mx, fmaxf(xa[j], xb[j]));
            }
            // Lazy running maximum: move it (and rescale l and O) only when a
            // score passes it by more than kLazyMaxSlack.
            const bool grow = valid && mx > m_run + kLazyMaxSlack;
            if (__any_sync(0xffffffffu, grow)) {
                const float m_new = grow ? fmaxf(m_run, mx) : m_run;
                const float alpha = grow ? ex2_approx(m_run - m_new) : 1.f;
                m_run = m_new;
                l_run *= alpha;
                if (!first_round) {
#pragma unroll 1
                    for (int d0 = 0; d0 < D; d0 += 16) {
                        float o[16];
                        tmem_ld16(tO + t_lane + (uint32_t)d0, o);
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] *= alpha;
                        tmem_st16(tO + t_lane + (uint32_t)d0, o);
                    }
                }
            }
            const float mref = valid ? m_run : 0.f;  // rows outside the pass: finite zeros
            // P row qi as bf16, one 16-byte chunk of 8 tokens at a time, in the
            // 128-byte-swizzled K-major layout.
            float lsum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = ch * 8 + 2 * k;
                    const float x0 = j < 32 ? xa[j] : xb[j - 32], x1 = j + 1 < 32 ? xa[j + 1] : xb[j - 31];
                    const float p0 = ex2_approx(x0 - mref), p1 = ex2_approx(x1 - mref);
                    lsum += p0 + p1;
                    w[k] = pack_bf16x2(p0, p1);
                }
                if (qi >= 0 && qi < 64)
                    *reinterpret_cast<uint4 *>(Ps + qi * 128 + ((ch ^ (qi & 7)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
            }
            l_run += lsum;
            fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar_sync(cons_bar, 4 * 32);  // P written, S and O reads done
        if (tid == issuer) {
            tc_fence_after();
            for (int j = 0; j < ntok / 16; ++j) {
                const uint64_t a = smem_desc_sw128(p_base - a_shift + (uint32_t)j * 32, 16, 1024);
                const uint64_t bv = smem_desc_sw128(vbase + (uint32_t)j * 2048, L::kPanel, 1024);
                tc_mma_bf16(tO, a, bv, IDESC_O, first_round && j == 0 ? 0u : 1u);
            }
            tc_commit(smem_u32(&empty[slot]));
            if (seg_end) tc_commit(smem_u32(obar));
        }
        first_round = false;
        if (seg_end) {
            if (!abort && !mbar_wait_bounded(smem_u32(obar), oph)) {
                atomicOr(err, kErrTimeout);
                abort = true;
            }
            oph ^= 1u;
            tc_fence_after();
            if (warp_rows) {
                const int64_t slot_p = partial_slot(c, kvh * V + v);
                const int64_t prow = slot_p * kPlanSlotRows + qi;
                float *ab = sh.acc_s + prow * D;
#pragma unroll 1
                for (int d0 = 0; d0 < D; d0 += 32) {
                    float o[32];
                    tmem_ld32(tO + t_lane + (uint32_t)d0, o);
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(ab + d0 + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                    }
                }
                if (valid) sh.ml_s[prow] = make_float2(m_run, l_run);
            }
            seg_start = true;
        }
        for (int b = 0; b < nblk; ++b) cur.advance(pv.cu_s, V);
        it += nblk;
    }
    // Every MMA has completed (the last round ends a segment and its O was
    // waited for); free the tensor memory.
    tc_fence_before();
    named_bar_sync(cons_bar, 4 * 32);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kCols);
    }
}

}  // namespace pa
