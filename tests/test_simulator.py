"""The allocation simulator: the C++ simulator against the oracle's plain
Python model on the same streams (exact integer totals), and the pages'
qualitative claims: reserving for the longest possible output leaves most
reserved KV memory empty, paging keeps it nearly full; paging fits more
requests at once; per-sequence waste of paging is about B/2 tokens."""
import numpy as np
import pytest

from oracle.simulator import simulate as oracle_simulate
import paged_kv_cache_150_gb300 as pa
from paged_kv_cache_150_gb300 import inputs

KEYS = ("steps", "admitted", "completed", "preemptions", "blocked_steps", "peak_running",
        "sum_used", "sum_held", "sum_running")


@pytest.mark.parametrize("policy,B,slots,rate,seed", [
    ("contiguous", 16, 40000, 0.5, 1), ("paged", 16, 40000, 0.5, 1), ("paged", 1, 20000, 0.8, 2),
    ("paged", 128, 20000, 0.8, 3), ("contiguous", 16, 9000, 2.0, 4), ("paged", 8, 6000, 2.0, 5),
    ("paged", 32, 3000, 1.0, 6)])
def test_simulator_matches_oracle_model(policy, B, slots, rate, seed):
    a, p, o = inputs.request_stream(seed, 300, rate, prompt_median=200, output_median=100, max_prompt=1000,
                                    max_new_tokens=1000)
    got = pa.simulate(policy, a, p, o, slots, block_size=B, max_new_tokens=1000, max_steps=200000)
    want = oracle_simulate(policy, slots, B, 1000, 200000, a.tolist(), p.tolist(), o.tolist())
    assert {k: got[k] for k in KEYS} == {k: want[k] for k in KEYS}
    assert got["utilization"] == pytest.approx(want["utilization"], rel=1e-12)
    assert got["completed"] == 300


def _stream():
    return inputs.request_stream(7, 2000, 1.0, prompt_median=256, output_median=128, max_prompt=2048,
                                 max_new_tokens=2048)


def test_paging_keeps_reserved_memory_full_and_fits_more_requests():
    # "10 PagedAttention" section 2: KV memory holding useful tokens 20.4-38.2%
    # with contiguous reservation versus 96.3% paged; concurrency 2.5-4x.
    a, p, o = _stream()
    cont = pa.simulate("contiguous", a, p, o, 200000, max_new_tokens=2048)
    paged = pa.simulate("paged", a, p, o, 200000, block_size=16, max_new_tokens=2048)
    assert cont["utilization"] < 0.40
    assert paged["utilization"] > 0.95
    assert paged["peak_running"] >= 2.5 * cont["peak_running"]
    assert paged["steps"] < cont["steps"]  # the same queue finishes sooner


def test_paged_waste_is_about_half_a_block_per_sequence():
    # "10 PagedAttention" section 5: average internal fragmentation B/2 tokens per sequence.
    a, p, o = _stream()
    for B in (16, 64):
        r = pa.simulate("paged", a, p, o, 10 ** 7, block_size=B, max_new_tokens=2048)
        waste_per_seq = (r["sum_held"] - r["sum_used"]) / r["sum_running"]
        assert abs(waste_per_seq - (B - 1) / 2) < 0.1 * B


# ---------------------------------------------------------------------------
# Exact pins: tiny streams worked out by hand from the step rules stated with
# pa_sim_run ("10 PagedAttention" (PidokuInfra), section 10 exercises B and C;
# the contiguous-versus-paged contrast of section 2 "The three wastes it
# eliminates").  Each derivation lists, per step, what is admitted, what each
# running request does, and the step's (used, held, running) after
# completions.  A request is (arrival step, prompt, output tokens).

# Paged, B = 4, 16 slots = 4 blocks.  r0 (0, 4, 6), r1 (0, 4, 6), r2 (3, 7, 1).
# t0: admit r0, r1 (1 block each, 2 free).  r0 pos 4 starts a block (1 free),
#     r1 pos 4 likewise (0 free).  Lengths 5, 5: used 10, held 16, running 2.
# t1: lengths 6, 6: (12, 16, 2).     t2: lengths 7, 7: (14, 16, 2).
# t3: r2 arrives; it needs 2 blocks, 0 free: blocked (1).  Lengths 8, 8:
#     (16, 16, 2).
# t4: r2 blocked again (2).  r0 pos 8 needs a block, none free: PREEMPTED
#     (its 2 blocks freed, progress lost, queue front: [r0, r2]).  r1 takes
#     one of them (1 free), length 9: (9, 12, 1).
# t5: admit r0 (1 block, 0 free); r2 blocked behind it (3).  r1 generates its
#     6th token and finishes (3 blocks back, 3 free).  r0 pos 4 starts a
#     block (2 free), length 5: (5, 8, 1).
# t6: admit r2 (2 blocks, 0 free).  r0 length 6; r2 pos 7 stays in its 2nd
#     block and finishes at once (2 free): (6, 8, 1).
# t7..t8: r0 lengths 7, 8: (7, 8, 1), (8, 8, 1).
# t9: r0 pos 8 starts a block (1 free), length 9: (9, 12, 1).
# t10: r0 finishes: (0, 0, 0).  All done after 11 steps.
# admitted r0, r1, r0, r2 = 4; used 10+12+14+16+9+5+6+7+8+9 = 96;
# held 4*16 + 12 + 4*8 + 12 = 120; running 4*2 + 6*1 = 14.
PAGED_PREEMPT = dict(
    policy="paged", B=4, slots=16, max_new=4, max_steps=1000,
    a=[0, 0, 3], p=[4, 4, 7], o=[6, 6, 1],
    want=dict(steps=11, admitted=4, completed=3, preemptions=1, blocked_steps=3, peak_running=2,
              sum_used=96, sum_held=120, sum_running=14))

# The same stream cut at max_steps = 5: steps t0..t4 above, nothing finished.
# used 10+12+14+16+9 = 61, held 4*16 + 12 = 76, running 4*2 + 1 = 9.
PAGED_PREEMPT_CUT = dict(PAGED_PREEMPT, max_steps=5, want=dict(
    steps=5, admitted=2, completed=0, preemptions=1, blocked_steps=2, peak_running=2,
    sum_used=61, sum_held=76, sum_running=9))

# Contiguous, 20 slots, reservation = prompt + 4.  r0 (0, 6, 2) needs 10,
# r1 (0, 8, 3) needs 12, r2 (0, 2, 3) needs 6.
# t0: r0 takes [0, 10); r1 needs 12 > the free [10, 20): blocked (1), and r2,
#     which would fit, waits behind it (head-of-line).  r0 length 7:
#     (7, 10, 1).
# t1: r1 blocked (2).  r0 finishes; [0, 10) merges with [10, 20).  (0, 0, 0).
# t2: r1 takes [0, 12), r2 takes [12, 18).  Lengths 9 and 3: (12, 18, 2).
# t3: lengths 10 and 4: (14, 18, 2).
# t4: both finish: (0, 0, 0).  5 steps.
# used 7+12+14 = 33, held 10+18+18 = 46, running 1+2+2 = 5.
CONTIG_HEAD_OF_LINE = dict(
    policy="contiguous", B=16, slots=20, max_new=4, max_steps=1000,
    a=[0, 0, 0], p=[6, 8, 2], o=[2, 3, 3],
    want=dict(steps=5, admitted=3, completed=3, preemptions=0, blocked_steps=2, peak_running=2,
              sum_used=33, sum_held=46, sum_running=5))

# Contiguous, 26 slots, reservation = prompt + 2: first fit, not best fit.
# r0 (0, 4, 2) 6, r1 (0, 5, 1) 7, r2 (0, 6, 2) 8, r3 (1, 2, 2) 4, r4 (1, 5, 2) 7.
# t0: r0 [0, 6), r1 [6, 13), r2 [13, 21); free [21, 26).  r0 length 5; r1
#     finishes (free [6, 13), [21, 26)); r2 length 7: (12, 14, 2).
# t1: r3 takes the FIRST hole that fits, [6, 10) (best fit would take
#     [21, 25)); r4 needs 7: holes [10, 13) and [21, 26) are too small:
#     blocked (1).  r0 finishes ([0, 6) free); r2 finishes ([13, 21) merges
#     with [10, 13) and [21, 26) into [10, 26)); r3 length 3: (3, 4, 1).
# t2: r4 takes [10, 17).  r3 finishes ([6, 10) joins [0, 6)); r4 length 6:
#     (6, 7, 1).
# t3: r4 finishes: (0, 0, 0).  4 steps.
CONTIG_FIRST_FIT = dict(
    policy="contiguous", B=16, slots=26, max_new=2, max_steps=1000,
    a=[0, 0, 0, 1, 1], p=[4, 5, 6, 2, 5], o=[2, 1, 2, 2, 2],
    want=dict(steps=4, admitted=5, completed=5, preemptions=0, blocked_steps=1, peak_running=2,
              sum_used=21, sum_held=25, sum_running=4))

# Paged, B = 2, 6 slots = 3 blocks, with an idle step.  r0 (0, 3, 1), r1 (2, 1, 2).
# t0: r0 takes 2 blocks; pos 3 stays in its 2nd block and it finishes.
#     (0, 0, 0).   t1: nothing queued or running: (0, 0, 0).
# t2: r1 arrives and takes 1 block; length 2: (2, 2, 1).
# t3: r1 pos 2 starts a block and it finishes: (0, 0, 0).  4 steps.
PAGED_IDLE = dict(
    policy="paged", B=2, slots=6, max_new=4, max_steps=1000,
    a=[0, 2], p=[3, 1], o=[1, 2],
    want=dict(steps=4, admitted=2, completed=2, preemptions=0, blocked_steps=0, peak_running=1,
              sum_used=2, sum_held=2, sum_running=1))

HAND_STREAMS = [PAGED_PREEMPT, PAGED_PREEMPT_CUT, CONTIG_HEAD_OF_LINE, CONTIG_FIRST_FIT, PAGED_IDLE]
_IDS = ["paged-preempt", "paged-preempt-cut", "contig-head-of-line", "contig-first-fit", "paged-idle"]


def _run_oracle(fn, s):
    return fn(s["policy"], s["slots"], s["B"], s["max_new"], s["max_steps"], s["a"], s["p"], s["o"])


@pytest.mark.parametrize("s", HAND_STREAMS, ids=_IDS)
def test_oracle_simulator_hand_worked_streams(s):
    got = _run_oracle(oracle_simulate, s)
    assert {k: got[k] for k in KEYS} == s["want"]
    assert got["utilization"] == pytest.approx(s["want"]["sum_used"] / s["want"]["sum_held"], rel=1e-15)


@pytest.mark.parametrize("s", HAND_STREAMS, ids=_IDS)
def test_library_simulator_hand_worked_streams(s):
    got = pa.simulate(s["policy"], s["a"], s["p"], s["o"], s["slots"], block_size=s["B"],
                      max_new_tokens=s["max_new"], max_steps=s["max_steps"])
    assert {k: got[k] for k in KEYS} == s["want"]


# Plausible one-line mistakes planted in a copy of the oracle (CPU only):
# every one must change the totals of at least one hand-worked stream.
MUTATIONS = {
    "preempted request to the queue tail": [("queue = preempted + queue", "queue = queue + preempted")],
    "preemption keeps progress": [("                gen[i] = 0\n", "                gen[i] = gen[i]\n")],
    "arrival one step late": [("arrival_step[nxt] <= t", "arrival_step[nxt] < t")],
    "any request that fits is admitted": [
        ("        while queue:\n            i = queue[0]\n", "        for i in list(queue):\n"),
        ("                break\n            running.append(queue.pop(0))\n",
         "                continue\n            queue.remove(i)\n            running.append(i)\n")],
    "best fit instead of first fit": [
        ("for j, (st, ln) in enumerate(free_iv):",
         "for j, (st, ln) in sorted(enumerate(free_iv), key=lambda e: e[1][1]):")],
    "no merge of freed intervals": [("free_iv = merged\n", "pass\n")],
    "reservation of the true output length": [
        ("need = prompt_len[i] + max_new_tokens", "need = prompt_len[i] + output_len[i]")],
    "held slots not rounded up to blocks": [
        ("-(-(prompt_len[i] + gen[i]) // block_size) * block_size", "(prompt_len[i] + gen[i])")],
    "one token too many": [("if gen[i] == output_len[i]:", "if gen[i] == output_len[i] + 1:")],
    "step count off by one": [('res["steps"] = t\n', 'res["steps"] = t + 1\n')],
    "blocked steps not counted": [('res["blocked_steps"] += 1\n', 'pass\n')],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_hand_worked_streams_catch_planted_mistakes(name):
    import importlib.util
    import inspect
    import oracle.simulator as mod
    src = inspect.getsource(mod)
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    spec = importlib.util.spec_from_loader("oracle._mutated_simulator", loader=None)
    m = importlib.util.module_from_spec(spec)
    m.__package__ = "oracle"
    exec(compile(src, "<mutated simulator>", "exec"), m.__dict__)
    changed = []
    for s in HAND_STREAMS:
        got = _run_oracle(m.simulate, s)
        changed.append({k: got[k] for k in KEYS} != s["want"])
    assert any(changed), name
