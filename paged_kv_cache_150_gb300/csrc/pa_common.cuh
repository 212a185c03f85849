// Shared device helpers for the paged-KV kernels (sm_103a).
//
// - the device error word bits,
// - the even split of the flattened (KV-head group, sequence, block) list over
//   persistent CTAs (host and device use these same integer formulas),
// - thin inline-PTX wrappers: mbarrier, TMA tensor loads, ldmatrix,
//   movmatrix, mma.sync, ex2.approx, globaltimer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Bits of the per-device error word.
enum : unsigned int {
    kErrBounds = 1u,   // slot / table entry / block id outside the pool
    kErrLength = 2u,   // sequence length outside [0, max_blocks * B]
    kErrTimeout = 4u,  // a bounded mbarrier wait ran out
    kErrPlan = 8u,     // a shared-prefix plan that does not match its decode call
};

// Bound on any single mbarrier wait (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Block-table entries the TMA producer reads ahead of their use.
constexpr int kTablePrefetch = 4;

// Tensor-core decode pipeline: stages in the shared-memory ring, and the
// most KV heads one CTA covers (NH = the largest divisor of Hk not above it).
// A stage holds one (block, head-group) tile of K and of V: 32 KiB at
// block_size 16 and 64 KiB at 32 for head_dim 128, so about 128 KiB is in
// flight per SM (two CTAs per SM at block_size 16, one at 32).  Measured
// on GB300 against 3-4 stages and 8 heads per CTA: deeper rings (192 KiB per
// SM) were 2-3% slower on every workload.
constexpr int kMmaStages = 2;
// Online softmax with a lazy running maximum (log2 units): the column-wide
// maximum is recomputed (shuffles) and the accumulators rescaled only when a
// score exceeds the running maximum by more than this, so between updates the
// probabilities 2^(s - m) stay at most 2^8.  The result is the same softmax:
// numerator and denominator carry the same subtracted constant.
constexpr float kLazyMaxSlack = 8.f;
constexpr int kMmaMaxHeads = 4;
// Sequences (+ 1) whose block-count prefix sums a tensor-core CTA computes in
// its own shared memory (16 KiB) instead of waiting for the plan kernel's.
constexpr int kLocalCuMax = 4096;

// ---------------------------------------------------------------- work split
// CTA c of C owns flattened blocks [split_begin(c), split_begin(c + 1)).
__host__ __device__ __forceinline__ int64_t split_begin(int64_t c, int64_t W, int64_t C) {
    return c * W / C;
}
// Largest c with split_begin(c) <= x, i.e. the CTA that owns block x (0 <= x < W).
__host__ __device__ __forceinline__ int32_t split_owner(int64_t x, int64_t W, int64_t C) {
    return (int32_t)(((x + 1) * C + W - 1) / W - 1);
}

// Partial-result slot of (CTA c, flattened sequence sp = group * N + seq).
// Unique because CTA ranges and sequences are both ordered along the
// flattened block list; there are at most C + NG * N slots.
__host__ __device__ __forceinline__ int64_t partial_slot(int32_t c, int32_t sp) {
    return (int64_t)c + sp;
}

// ------------------------------------------------------- shared-prefix plan
// Packed int32 words written by pa_shared_plan_build, read by the decode
// plan and attention kernels:
//   header[kPlanHeader] = {magic, N, G, B, groups, members, V, R}
//   seq_group[N]  seq_member[N]  group_prefix[groups]  group_vbase[groups + 1]
//   group_begin[groups + 1]  members[members]  vgroup[V]  cu_s[V + 1]
// A group's sharers contribute G query rows each (member m: rows m*G ..
// m*G + G - 1); the rows are cut into passes of R (16, 32 or 64, one value
// per plan), and each pass is one "virtual sequence" v over the group's P
// shared blocks (cu_s = prefix sums of P over virtual sequences).  A
// shared-prefix CTA has kPlanWarps consumer warps of kPlanWarpRows rows each:
// a stage holds kPlanSlotRows / R KV heads (1-head TMA boxes side by side),
// and warp w applies head w / (R / 16) of the stage to rows
// (w % (R / 16)) * 16 .. + 15 of the pass (two 8-column MMA tiles).  So one
// streamed tile serves up to 64 query rows of its KV head.  G divides 8, so a
// member's rows never straddle an MMA tile or a pass.
constexpr int32_t kPlanMagic = 0x50415350;
constexpr int kPlanHeader = 8;
constexpr int kPlanWarps = 4;                               // consumer warps of a shared-prefix CTA
constexpr int kPlanWarpRows = 16;                           // query rows of one consumer warp
constexpr int kPlanSlotRows = kPlanWarps * kPlanWarpRows;   // rows of one shared-prefix partial slot

// Relative cost of a one-head shared-prefix stage on tcgen05 against an
// own-block stage of the same launch (the CTA split of the plan kernel).
constexpr float kTcStageWeight = 0.6f;

// Shared memory of one half of a two-half CTA of the shared-plan attention
// launch (1024-byte multiple): the largest of the own-block map (the ring of
// kMmaStages stages of kPlanWarps heads, barriers), the mma.sync
// shared-prefix map (the same ring, 256 bytes of barriers, 16 query rows of
// D + 8 elements per consumer warp) and the tcgen05 one (64 x 64 bf16
// probabilities, 64 query rows of D, two rounds of 64 tokens of K and V,
// barriers).
__host__ __device__ constexpr uint32_t shared_half_bytes(int D, int B) {
    const uint32_t slab = (uint32_t)(D / 64) * (uint32_t)B * 128u;
    const uint32_t ring = (uint32_t)kMmaStages * 2u * (uint32_t)kPlanWarps * slab;
    const uint32_t own = ring + 2u * (uint32_t)kMmaStages * 8u;
    const uint32_t mma = ring + 256u + (uint32_t)kPlanWarps * (uint32_t)kPlanWarpRows * (uint32_t)(D * 2 + 16);
    const uint32_t tc = 64u * 64u * 2u + 64u * (uint32_t)D * 2u + 2u * (2u * 64u * (uint32_t)D * 2u) + 256u;
    const uint32_t m = own > mma ? (own > tc ? own : tc) : (mma > tc ? mma : tc);
    return (m + 1023u) & ~1023u;
}
// Halves per CTA of the shared-plan launch: two when both fit the 227 KiB a
// CTA may hold (block size 16, and head_dim 64 at 32), else one.
__host__ __device__ constexpr int shared_halves(int D, int B) {
    return 2u * shared_half_bytes(D, B) + 1024u <= 227u * 1024u ? 2 : 1;
}

// Rows per pass R that a plan may carry, and the KV heads of a stage for it.
__host__ __device__ __forceinline__ bool plan_rows_ok(int32_t R) { return R == 16 || R == 32 || R == 64; }
__host__ __device__ __forceinline__ int32_t plan_stage_heads(int32_t R) { return kPlanSlotRows / R; }

struct PlanView {
    const int32_t *seq_group, *seq_member, *group_prefix, *group_vbase, *group_begin, *members, *vgroup, *cu_s;
    int32_t N, G, B, groups, M, V, R;

    __host__ __device__ __forceinline__ static int64_t words(int32_t N, int32_t groups, int32_t M, int32_t V) {
        return (int64_t)kPlanHeader + 2 * (int64_t)N + 3 * (int64_t)groups + 2 + M + 2 * (int64_t)V + 1;
    }
    // Pointers into the words; the header's counts must be validated first.
    __host__ __device__ __forceinline__ static PlanView at(const int32_t *w) {
        PlanView p;
        p.N = w[1];
        p.G = w[2];
        p.B = w[3];
        p.groups = w[4];
        p.M = w[5];
        p.V = w[6];
        p.R = w[7];
        const int32_t *x = w + kPlanHeader;
        p.seq_group = x;
        x += p.N;
        p.seq_member = x;
        x += p.N;
        p.group_prefix = x;
        x += p.groups;
        p.group_vbase = x;
        x += p.groups + 1;
        p.group_begin = x;
        x += p.groups + 1;
        p.members = x;
        x += p.M;
        p.vgroup = x;
        x += p.V;
        p.cu_s = x;
        return p;
    }
};

// ------------------------------------------------------------- small helpers
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------- programmatic dependent launch
// Wait until the preceding grid on the stream has completed and its memory
// is visible (a no-op when this grid was not launched programmatically).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid on the stream (if launched programmatically) to start.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after
// limit_ns nanoseconds of %globaltimer.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Same load with an L2 cache policy (e.g. evict-first for streamed data).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const void *tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
        : "memory");
}

// L2 policy that evicts these lines first: KV tiles are read once per step.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ----------------------------------------------------------- warp-level MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------- block cursor
// Walks the flattened (group, sequence, block) list.  cu[] holds the
// exclusive prefix sums of per-sequence block counts (cu[N] = Wg).
struct BlockCursor {
    int32_t g, seq, blk;
    int32_t nb;  // blocks of the current sequence
    int32_t b0;  // blocks of the current sequence before the list's first (skip[seq]; 0 without skip)

    __device__ __forceinline__ void init(int64_t x, const int32_t *__restrict__ cu, int32_t N,
                                         const int32_t *__restrict__ skip = nullptr) {
        const int32_t Wg = cu[N];
        g = (int32_t)(x / Wg);
        const int32_t r = (int32_t)(x - (int64_t)g * Wg);
        // largest seq with cu[seq] <= r (skips empty sequences: cu[seq+1] > r)
        int32_t lo = 0, hi = N - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        seq = lo;
        blk = r - cu[seq];
        nb = cu[seq + 1] - cu[seq];
        b0 = skip ? skip[seq] : 0;
    }

    // Position at flattened block x when the sequence holding it is known
    // (from the plan kernel's per-CTA start table): no search.
    __device__ __forceinline__ void init_at(int64_t x, int32_t s, const int32_t *__restrict__ cu, int32_t N,
                                            const int32_t *__restrict__ skip = nullptr) {
        const int32_t Wg = cu[N];
        g = (int32_t)(x / Wg);
        seq = s;
        blk = (int32_t)(x - (int64_t)g * Wg) - cu[s];
        nb = cu[s + 1] - cu[s];
        b0 = skip ? skip[s] : 0;
    }

    __device__ __forceinline__ void advance(const int32_t *__restrict__ cu, int32_t N,
                                            const int32_t *__restrict__ skip = nullptr) {
        if (++blk < nb) return;
        blk = 0;
        do {
            if (++seq == N) {
                seq = 0;
                ++g;
            }
            nb = cu[seq + 1] - cu[seq];
        } while (nb == 0);
        b0 = skip ? skip[seq] : 0;
    }
};

}  // namespace pa
