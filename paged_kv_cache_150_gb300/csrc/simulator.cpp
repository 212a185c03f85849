// KV allocation simulator: contiguous max-length reservation against paged
// blocks under one request stream ("10 PagedAttention" (PidokuInfra), section
// 10 exercises B and C: a contiguous and a paged allocator under lognormal
// lengths and Poisson arrivals; peak utilisation, failures, concurrency; a
// block-size sweep).  Host only.
//
// The model, one decode step at a time (t = 0, 1, ...):
//  1. requests whose arrival step is t join the back of a FIFO queue;
//  2. admission, head of the queue first, stopping at the first request that
//     does not fit: contiguous reserves prompt + max_new_tokens slots in one
//     interval (first fit over the free intervals); paged takes
//     ceil(prompt / B) blocks from the block manager;
//  3. every running request, oldest admission first, generates one token; a
//     paged request whose new token starts a block takes one block, and if
//     none is free it is preempted: its blocks are freed, its progress is
//     lost, and it goes back to the front of the queue;
//  4. requests that generated their output length finish and free memory;
//  5. the step adds its held slots (reservations, or blocks x B), its used
//     slots (tokens stored) and its running count to the totals.
// Utilisation = sum of used / sum of held over all steps.
#include <cstdint>
#include <deque>
#include <map>
#include <new>
#include <vector>

#include "pa.h"

namespace {

struct Req {
    int32_t prompt, output;
    int32_t generated = 0;
    int32_t seq = -1;       // block-manager sequence (paged)
    int64_t start = -1;     // reservation start (contiguous)
    int64_t reserved = 0;   // reservation length (contiguous)
};

// Free intervals of the contiguous pool, keyed by start.
struct Intervals {
    std::map<int64_t, int64_t> free;  // start -> length
    bool take(int64_t len, int64_t *start) {
        for (auto it = free.begin(); it != free.end(); ++it) {
            if (it->second >= len) {
                *start = it->first;
                const int64_t rest = it->second - len, nstart = it->first + len;
                free.erase(it);
                if (rest > 0) free[nstart] = rest;
                return true;
            }
        }
        return false;
    }
    void give(int64_t start, int64_t len) {
        auto next = free.lower_bound(start);
        if (next != free.end() && start + len == next->first) {
            len += next->second;
            next = free.erase(next);
        }
        if (next != free.begin()) {
            auto prev = std::prev(next);
            if (prev->first + prev->second == start) {
                prev->second += len;
                return;
            }
        }
        free[start] = len;
    }
};

}  // namespace

extern "C" pa_status_t pa_sim_run(const pa_sim_config_t *cfg, const int32_t *arrival_step,
                                  const int32_t *prompt_len, const int32_t *output_len, int32_t num_requests,
                                  pa_sim_result_t *out) try {
    if (!cfg || !out || num_requests < 0 || (num_requests > 0 && (!arrival_step || !prompt_len || !output_len)))
        return PA_ERR_INVALID_ARG;
    if (cfg->policy != PA_SIM_CONTIGUOUS && cfg->policy != PA_SIM_PAGED) return PA_ERR_INVALID_ARG;
    if (cfg->total_slots <= 0 || cfg->max_steps <= 0) return PA_ERR_INVALID_ARG;
    const bool paged = cfg->policy == PA_SIM_PAGED;
    const int32_t B = cfg->block_size;
    if (paged && (B <= 0 || cfg->total_slots / B >= INT32_MAX)) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < num_requests; ++i) {
        if (prompt_len[i] < 1 || output_len[i] < 1 || (i > 0 && arrival_step[i] < arrival_step[i - 1]))
            return PA_ERR_INVALID_ARG;
        if (!paged && output_len[i] > cfg->max_new_tokens) return PA_ERR_INVALID_ARG;
    }
    std::vector<Req> reqs((size_t)num_requests);
    for (int32_t i = 0; i < num_requests; ++i) {
        reqs[i].prompt = prompt_len[i];
        reqs[i].output = output_len[i];
    }
    pa_bm_t *bm = nullptr;
    Intervals iv;
    if (paged) {
        bm = pa_bm_create((int32_t)(cfg->total_slots / B), B, nullptr);
        if (!bm) return PA_ERR_INVALID_ARG;
    } else {
        iv.free[0] = cfg->total_slots;
    }
    *out = pa_sim_result_t{};
    std::deque<int32_t> queue;
    std::vector<int32_t> running;  // oldest admission first
    int32_t next_arrival = 0, done = 0;
    int32_t scratch_slot = 0, cs = 0, cd = 0;
    int64_t t = 0;
    for (; t < cfg->max_steps && done < num_requests; ++t) {
        while (next_arrival < num_requests && arrival_step[next_arrival] <= t) queue.push_back(next_arrival++);
        while (!queue.empty()) {
            Req &r = reqs[queue.front()];
            bool ok;
            if (paged) {
                ok = pa_bm_new_seq(bm, r.prompt, &r.seq) == PA_OK;
            } else {
                r.reserved = (int64_t)r.prompt + cfg->max_new_tokens;
                ok = iv.take(r.reserved, &r.start);
            }
            if (!ok) {
                out->blocked_steps += 1;
                break;
            }
            running.push_back(queue.front());
            queue.pop_front();
            out->admitted += 1;
        }
        std::vector<int32_t> keep;
        keep.reserve(running.size());
        std::vector<int32_t> preempted;
        for (int32_t id : running) {
            Req &r = reqs[id];
            if (paged && pa_bm_append_token(bm, r.seq, &scratch_slot, &cs, &cd) != PA_OK) {
                pa_bm_free_seq(bm, r.seq);
                r.seq = -1;
                r.generated = 0;
                preempted.push_back(id);
                out->preemptions += 1;
                continue;
            }
            r.generated += 1;
            if (r.generated == r.output) {
                if (paged)
                    pa_bm_free_seq(bm, r.seq);
                else
                    iv.give(r.start, r.reserved);
                done += 1;
                out->completed += 1;
                continue;
            }
            keep.push_back(id);
        }
        for (auto it = preempted.rbegin(); it != preempted.rend(); ++it) queue.push_front(*it);
        running.swap(keep);
        int64_t used = 0, held = 0;
        for (int32_t id : running) {
            const Req &r = reqs[id];
            used += r.prompt + r.generated;
            held += paged ? (int64_t)(r.prompt + r.generated + B - 1) / B * B : r.reserved;
        }
        out->sum_used += used;
        out->sum_held += held;
        out->sum_running += (int64_t)running.size();
        if ((int64_t)running.size() > out->peak_running) out->peak_running = (int64_t)running.size();
    }
    out->steps = t;
    out->utilization = out->sum_held > 0 ? (double)out->sum_used / (double)out->sum_held : 0.0;
    if (bm) pa_bm_destroy(bm);
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}
