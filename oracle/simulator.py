"""Plain-Python model of the KV allocation simulator, used to check the
library's C++ simulator.  TEST INFRASTRUCTURE ONLY.

It follows the step rules stated with pa_sim_run ("10 PagedAttention",
section 10, exercises B and C): FIFO admission of the queue head while it
fits (contiguous: prompt + max_new_tokens slots in one interval, first fit;
paged: ceil(prompt / B) blocks), one generated token per running request per
step (a paged request takes a block when its token starts one, or is
preempted back to the queue front when none is free), then completions, then
the step's totals.  The paged side uses the oracle's block-manager model.
"""
from .block_manager import OracleBlockManager


def simulate(policy, total_slots, block_size, max_new_tokens, max_steps, arrival_step, prompt_len, output_len):
    paged = policy == "paged"
    n = len(prompt_len)
    gen = [0] * n
    seq = [None] * n
    start = [None] * n
    reserved = [0] * n
    free_iv = [[0, int(total_slots)]]  # sorted [start, length]
    bm = OracleBlockManager(int(total_slots) // block_size, block_size) if paged else None
    queue, running = [], []
    nxt = done = 0
    res = dict(steps=0, admitted=0, completed=0, preemptions=0, blocked_steps=0, peak_running=0,
               sum_used=0, sum_held=0, sum_running=0)
    t = 0
    while t < max_steps and done < n:
        while nxt < n and arrival_step[nxt] <= t:
            queue.append(nxt)
            nxt += 1
        while queue:
            i = queue[0]
            if paged:
                s = bm.new_sequence(prompt_len[i])
                ok = s is not None
                if ok:
                    seq[i] = s
            else:
                need = prompt_len[i] + max_new_tokens
                ok = False
                for j, (st, ln) in enumerate(free_iv):
                    if ln >= need:
                        start[i], reserved[i] = st, need
                        if ln == need:
                            del free_iv[j]
                        else:
                            free_iv[j] = [st + need, ln - need]
                        ok = True
                        break
            if not ok:
                res["blocked_steps"] += 1
                break
            running.append(queue.pop(0))
            res["admitted"] += 1
        keep, preempted = [], []
        for i in running:
            if paged and bm.append_token(seq[i]) is None:
                bm.free_seq(seq[i])
                seq[i] = None
                gen[i] = 0
                preempted.append(i)
                res["preemptions"] += 1
                continue
            gen[i] += 1
            if gen[i] == output_len[i]:
                if paged:
                    bm.free_seq(seq[i])
                else:
                    free_iv.append([start[i], reserved[i]])
                    free_iv.sort()
                    merged = []
                    for st, ln in free_iv:
                        if merged and merged[-1][0] + merged[-1][1] == st:
                            merged[-1][1] += ln
                        else:
                            merged.append([st, ln])
                    free_iv = merged
                done += 1
                res["completed"] += 1
                continue
            keep.append(i)
        queue = preempted + queue
        running = keep
        used = sum(prompt_len[i] + gen[i] for i in running)
        if paged:
            held = sum(-(-(prompt_len[i] + gen[i]) // block_size) * block_size for i in running)
        else:
            held = sum(reserved[i] for i in running)
        res["sum_used"] += used
        res["sum_held"] += held
        res["sum_running"] += len(running)
        res["peak_running"] = max(res["peak_running"], len(running))
        t += 1
    res["steps"] = t
    res["utilization"] = res["sum_used"] / res["sum_held"] if res["sum_held"] else 0.0
    return res
