// Shared-prefix plan for one decode batch (host only).
//
// Sequences forked from one prompt, or matched in the prefix cache, point at
// the same physical blocks ("10 PagedAttention" (PidokuInfra), section 5
// "Copy-on-write sharing": one copy of the prompt's blocks with refcount n;
// "The relationship to prefix caching").  The plan lists groups of such
// sequences and their common prefix, so that decode reads a shared block once
// for every sharer's query heads.  The packed word layout is PlanView's.
//
// Grouping: sequences are bucketed by the physical id of their first block
// (in order of first appearance, so the plan is deterministic).  A bucket of
// two or more sequences is a group; its prefix P is the longest run of
// leading blocks equal in every member's table, cut so that each member keeps
// at least one position after it (P * B < L), and the group is dropped when
// P < min_shared_blocks.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

using namespace pa;

extern "C" size_t pa_shared_plan_ints(int32_t num_seqs) {
    if (num_seqs < 0) return 0;
    // groups <= N / 2, members <= N, V <= 3 N / 4 (PlanView::words)
    return (size_t)7 * (size_t)num_seqs + 16;
}

extern "C" pa_status_t pa_shared_plan_build(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                            const int32_t *seq_lens, int32_t num_seqs, int32_t block_size,
                                            int32_t num_heads, int32_t num_kv_heads, int32_t min_shared_blocks,
                                            int32_t *plan, size_t plan_ints, pa_shared_plan_info_t *info) try {
    const int32_t N = num_seqs;
    if (N < 0 || !plan || block_size <= 0 || max_blocks_per_seq <= 0 || num_kv_heads <= 0 || num_heads <= 0 ||
        num_heads % num_kv_heads != 0 || min_shared_blocks < 1)
        return PA_ERR_INVALID_ARG;
    if (N > 0 && (!block_tables || !seq_lens)) return PA_ERR_INVALID_ARG;
    if ((int64_t)N * max_blocks_per_seq >= ((int64_t)1 << 31) ||
        (int64_t)max_blocks_per_seq * block_size >= ((int64_t)1 << 31))
        return PA_ERR_INVALID_ARG;
    if (plan_ints < pa_shared_plan_ints(N)) return PA_ERR_INVALID_ARG;
    const int64_t max_len = (int64_t)max_blocks_per_seq * block_size;
    for (int32_t i = 0; i < N; ++i)
        if (seq_lens[i] < 0 || seq_lens[i] > max_len) return PA_ERR_INVALID_ARG;
    const int32_t G = num_heads / num_kv_heads;
    const bool sharing_ok = G == 1 || G == 2 || G == 4 || G == 8;

    // Buckets by first physical block, in order of first appearance.
    std::vector<std::vector<int32_t>> buckets;
    if (sharing_ok) {
        std::unordered_map<int32_t, size_t> index;
        for (int32_t i = 0; i < N; ++i) {
            if ((seq_lens[i] - 1) / block_size < 1) continue;  // no full block before its last position
            const int32_t first = block_tables[(int64_t)i * max_blocks_per_seq];
            auto it = index.find(first);
            if (it == index.end()) {
                index.emplace(first, buckets.size());
                buckets.push_back({i});
            } else {
                buckets[it->second].push_back(i);
            }
        }
    }
    struct Group {
        std::vector<int32_t> members;
        int32_t P;
    };
    std::vector<Group> groups;
    for (auto &b : buckets) {
        if (b.size() < 2) continue;
        const int32_t *rep = block_tables + (int64_t)b[0] * max_blocks_per_seq;
        int32_t P = max_blocks_per_seq;
        for (int32_t i : b) P = std::min(P, (seq_lens[i] - 1) / block_size);
        for (size_t k = 1; k < b.size() && P > 0; ++k) {
            const int32_t *t = block_tables + (int64_t)b[k] * max_blocks_per_seq;
            int32_t l = 0;
            while (l < P && t[l] == rep[l]) ++l;
            P = l;
        }
        if (P >= min_shared_blocks) groups.push_back({std::move(b), P});
    }

    const int32_t NGr = (int32_t)groups.size();
    // Rows per pass: the smallest of 16, 32, 64 that holds the largest
    // group's rows (64 for larger groups, which then take several passes).
    // Fewer KV heads per stage for larger R, so one streamed tile serves all
    // of a pass's rows.
    int32_t max_rows = 0;
    for (const auto &g : groups) max_rows = std::max(max_rows, (int32_t)g.members.size() * G);
    const int32_t R = max_rows <= 16 ? 16 : (max_rows <= 32 ? 32 : 64);
    int32_t M = 0, V = 0;
    for (const auto &g : groups) {
        M += (int32_t)g.members.size();
        V += (int32_t)(((int64_t)g.members.size() * G + R - 1) / R);
    }
    if (PlanView::words(N, NGr, M, V) > (int64_t)plan_ints) return PA_ERR_INVALID_ARG;  // cannot happen
    plan[0] = kPlanMagic;
    plan[1] = N;
    plan[2] = G;
    plan[3] = block_size;
    plan[4] = NGr;
    plan[5] = M;
    plan[6] = V;
    plan[7] = R;
    PlanView v = PlanView::at(plan);
    int32_t *seq_group = const_cast<int32_t *>(v.seq_group), *seq_member = const_cast<int32_t *>(v.seq_member);
    int32_t *prefix = const_cast<int32_t *>(v.group_prefix), *vbase = const_cast<int32_t *>(v.group_vbase);
    int32_t *begin = const_cast<int32_t *>(v.group_begin), *members = const_cast<int32_t *>(v.members);
    int32_t *vgroup = const_cast<int32_t *>(v.vgroup), *cu_s = const_cast<int32_t *>(v.cu_s);
    for (int32_t i = 0; i < N; ++i) seq_group[i] = seq_member[i] = -1;
    int64_t shared = 0, saved = 0;
    int32_t m = 0, vv = 0;
    cu_s[0] = 0;
    for (int32_t g = 0; g < NGr; ++g) {
        const auto &grp = groups[g];
        const int32_t S = (int32_t)grp.members.size();
        const int32_t passes = (int32_t)(((int64_t)S * G + R - 1) / R);
        prefix[g] = grp.P;
        vbase[g] = vv;
        begin[g] = m;
        for (int32_t k = 0; k < S; ++k) {
            seq_group[grp.members[k]] = g;
            seq_member[grp.members[k]] = k;
            members[m++] = grp.members[k];
        }
        for (int32_t p = 0; p < passes; ++p) {
            vgroup[vv] = g;
            cu_s[vv + 1] = cu_s[vv] + grp.P;
            ++vv;
        }
        shared += grp.P;
        saved += (int64_t)(S - passes) * grp.P;
    }
    vbase[NGr] = vv;
    begin[NGr] = m;
    if (info) {
        info->num_groups = NGr;
        info->num_members = M;
        info->shared_blocks = shared;
        info->saved_blocks = saved;
    }
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}
