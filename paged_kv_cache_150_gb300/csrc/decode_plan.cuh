// Decode plan kernel and shared-prefix plan checks (part of decode.cu).
//
// One CTA per call: lengths to block counts and prefix sums, arrival
// counters, empty outputs, per-CTA start sequences, and the check of an
// optional shared-prefix plan with the split of CTAs between the two kinds.
#pragma once

#include "pa_internal.h"

namespace pa {

// ---------------------------------------------------------------- plan kernel
// Checks a shared-prefix plan's words against the call (sizes, heads per KV
// head, block size, rows per pass, and every index it holds), so that a bad
// plan can only switch sharing off, never send a kernel out of bounds.
// Block-wide; every thread returns the verdict.
__device__ bool plan_valid(const int32_t *__restrict__ w, int32_t N, int32_t G, int32_t B, int32_t Hk,
                           int32_t max_blocks, int *s_flag, int *s_count) {
    if (threadIdx.x == 0) {
        const int32_t groups = w[4], M = w[5], V = w[6];
        const int32_t R = w[7];
        bool ok = w[0] == kPlanMagic && w[1] == N && w[2] == G && w[3] == B && groups >= 0 && groups <= N &&
                  M >= 0 && M <= N && V >= 0 && V <= N && plan_rows_ok(R) && Hk % plan_stage_heads(R) == 0 &&
                  G <= 8 && 8 % G == 0 && PlanView::words(N, groups, M, V) <= 7 * (int64_t)N + 16;
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
        ok = ok && S >= 1 && passes == (S * G + pv.R - 1) / pv.R && pv.group_prefix[g] >= 1 &&
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
                                                           int32_t *__restrict__ start_s,
                                                           int32_t *__restrict__ rowseq, int32_t plan_in_smem,
                                                           int32_t tc) {
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
    const bool plan_ok = plan && plan_valid(plan, N, G, B, Hk, max_len / B, &s_flag, &s_count);
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
        // CTAs for the shared prefixes, in proportion to the stages each side
        // streams (a shared-prefix stage holds plan_stage_heads(R) KV heads,
        // an own-block stage NH).  Measured on the prefix workload: with
        // mma.sync consumers a stage takes about the same time on either
        // side, whatever the heads in it, since its consumers' work (16 query
        // rows per warp), not its bytes, sets it; a one-head stage of the
        // tcgen05 CTAs weighs kTcStageWeight of an own-block stage.
        int32_t cs = 0;
        if (plan_ok) {
            const double w = tc && pv.R == kPlanSlotRows ? (double)kTcStageWeight : 1.0;
            const double Ws = w * (Hk / plan_stage_heads(pv.R)) * pv.cu_s[pv.V], Wo = (double)NG * carry;
            if (Ws > 0) {
                const double share = Ws / (Ws + Wo);
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
    // The same for the shared-prefix CTAs over the virtual sequences (the
    // list's outer index is the stage's KV heads, plan_stage_heads(R) of them).
    if (s_cs > 0) {
        const int32_t Wv = pv.cu_s[pv.V];
        const int64_t Ws = (int64_t)(Hk / plan_stage_heads(pv.R)) * Wv;
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
        // The sequence of every query row of every virtual sequence (-1 past
        // its group's rows), so that a shared-prefix warp finds its rows'
        // sequences with one load instead of a chain through the plan.
        const int32_t R = pv.R;
        for (int32_t e = threadIdx.x; e < pv.V * R; e += blockDim.x) {
            const int32_t v = e / R, r = e - v * R;
            const int32_t grp = pv.vgroup[v], gb = pv.group_begin[grp];
            const int32_t row = (v - pv.group_vbase[grp]) * R + r;
            rowseq[e] = row < (pv.group_begin[grp + 1] - gb) * G ? pv.members[gb + row / G] : -1;
        }
    }
}

}  // namespace pa
