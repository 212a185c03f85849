#!/usr/bin/env python3
"""Benchmark of the paged-KV decode hot path on GB300.

One step = one pass of the whole path over one batch: copy-on-write block
copies (when the batch has any), the slot-mapped KV write of the step's new
tokens, and paged decode attention (plan, attention kernel, split reduce).

Headline workload: 16 sequences x 32768 tokens, 64 query / 8 KV heads,
head_dim 128, bf16, block_size 16, blocks randomly placed in a pool of 1.05x
the need (2,147,483,648 bytes of K and V read per step).  The metric is KV
bytes read per second (GB/s); decode tokens/s and the fraction of the measured
HBM bandwidth are reported beside it.  Other workloads (the mixed-length GQA
batch, block_size 32, MHA, parallel sampling with copy-on-write) are timed
the same way and reported under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same per-GPU workload on its own GPU (weak
scaling, no data-path collective); rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV bytes read GB/s (% of GB300 HBM peak), tokens/s"
EXTRA = [("cfg2", {}), ("cfg4", {"block_size": 32}), ("cfg1", {}), ("cfg3", {"prompt_len": 2008}), ("cfg4", {"block_size": 16}),
         ("cfg4", {"block_size": 16, "layout": "split"}), ("cfg2", {"layout": "split"}), ("prefix", {}),
         ("cfg3", {"prompt_len": 2008, "shared": True}), ("prefix", {"shared": True}),
         ("cfg4", {"block_size": 16, "placement": "contiguous"}), ("cfg2-f32", {}), ("d256", {})]
FLUSH_BYTES = 512 << 20  # > 129 MB L2: written between timed steps
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="time only the headline workload")
    ap.add_argument("--extra-steps", type=int, default=300)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--workload", default="cfg4-b16",
                    help="headline workload: cfg4-b16 (default), cfg4-b32, cfg2, cfg1, cfg3-p2000, cfg3-p2008, "
                         "cfg4-b16-split, cfg2-split, prefix, cfg0 (tiny fp32), cfg2-f32, d256 (head_dim 256)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-write-copy", action="store_true",
                    help="skip timing the cache write and block copy on their own (launch lists of a step)")
    ap.add_argument("--l2", choices=["none", "write"], default="none",
                    help="between timed steps: nothing (every workload's KV is several times the 129 MB L2) "
                         "or write a 512 MiB buffer (leaves dirty lines whose write-back the next step pays)")
    return ap.parse_args()


WORKLOADS = {"cfg4-b16": ("cfg4", {"block_size": 16}), "cfg4-b32": ("cfg4", {"block_size": 32}),
             "cfg2": ("cfg2", {}), "cfg1": ("cfg1", {}), "cfg3-p2000": ("cfg3", {}),
             "cfg3-p2008": ("cfg3", {"prompt_len": 2008}),
             "cfg4-b16-split": ("cfg4", {"block_size": 16, "layout": "split"}),
             "cfg2-split": ("cfg2", {"layout": "split"}), "prefix": ("prefix", {}),
             "cfg4-b16-contiguous": ("cfg4", {"block_size": 16, "placement": "contiguous"}),
             "cfg3-p2008-shared": ("cfg3", {"prompt_len": 2008, "shared": True}),
             "prefix-shared": ("prefix", {"shared": True}), "cfg0": ("cfg0", {}),
             "cfg2-f32": ("cfg2-f32", {}), "d256": ("d256", {})}
# The workloads the 70%-of-HBM goal names (mixed-length GQA batch, long
# contexts at both block sizes): summarised under "targets" at the end of the
# line, with every output checked against the oracle when the CPU leg runs.
TARGETS = ("cfg2", "cfg4-b16", "cfg4-b32")


# ---------------------------------------------------------------- helpers
def make_workload(cfg, kw, seed_offset=0):
    """(workload, cache layout, shared-prefix plan) of a bench name's (cfg,
    options): "layout" and "shared" choose how the CUDA path runs (and mark
    the workload's name); the other options go to inputs.workload."""
    from paged_kv_cache_150_gb300 import inputs

    kw = dict(kw)
    layout = kw.pop("layout", "row")
    shared = kw.pop("shared", False)
    wl = inputs.workload(cfg, **kw)
    wl.seed += seed_offset
    if layout == "split":
        wl.name += "-split"
    if shared:
        wl.name += "-shared"
    return wl, layout, shared


def bench_config(wl, l2, world):
    """The line's "config": the same object for both arms."""
    kv = wl.kv_bytes_read()
    return {"workload": describe(wl), "kv_bytes_per_step": kv, "num_seqs": wl.num_seqs,
            "max_seq_len": int(wl.seq_lens.max()), "block_size": wl.block_size,
            "l2": ("inputs larger than L2: %.2f GB of KV per step vs 129 MB L2, no flush" % (kv / 1e9)
                   if l2 == "none" else "512 MiB buffer written between timed steps"),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def dist_setup(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons of this process's GPU,
    sampled DURING the timed region.  Read-only queries: nothing is set.

    Primary source: NVML through ctypes (the library nvidia-smi reads), polled
    from a thread every 5 ms, so even a timed region of a few milliseconds gets
    samples.  Fallback: an nvidia-smi loop started before the region (and
    allowed to print its first row first, since it needs longer than a short
    region to start).  The GPU is found by UUID, else by its index in
    CUDA_VISIBLE_DEVICES, else by the CUDA index; the record says which, and
    why when nothing could be read."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.005

    def __init__(self, device_index):
        self.notes = []
        self.selectors = []
        try:
            import torch

            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self.selectors.append(u if u.startswith("GPU-") else "GPU-" + u)
        except Exception as e:  # noqa: BLE001
            self.notes.append("no uuid: %s" % str(e)[:60])
        vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        if device_index < len(vis):
            self.selectors.append(vis[device_index])
        self.selectors.append(str(device_index))
        self.samples = []  # (sm_mhz, sm_max_mhz, power_w, reasons)
        self.source, self.selector = None, None
        self._nvml = self._open_nvml()

    # ---------------------------------------------------------------- NVML
    def _open_nvml(self):
        import ctypes

        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
        except Exception as e:  # noqa: BLE001
            self.notes.append("nvml unavailable: %s" % str(e)[:60])
            return None
        h = ctypes.c_void_p()
        for sel in self.selectors:
            if sel.startswith("GPU-") or sel.startswith("MIG-"):
                rc = lib.nvmlDeviceGetHandleByUUID(sel.encode(), ctypes.byref(h))
            elif sel.isdigit():
                rc = lib.nvmlDeviceGetHandleByIndex_v2(int(sel), ctypes.byref(h))
            else:
                continue
            if rc == 0:
                self.selector = sel
                break
            self.notes.append("nvml: no handle for %s (rc %d)" % (sel, rc))
        else:
            return None
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._h = h
        if self._nvml_sample(lib) is None:
            self.notes.append("nvml: clock query failed")
            return None
        return lib

    def _nvml_sample(self, lib):
        import ctypes

        sm, smax, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        lib.nvmlDeviceGetMaxClockInfo(self._h, 1, ctypes.byref(smax))
        lib.nvmlDeviceGetPowerUsage(self._h, ctypes.byref(mw))
        self._reasons_fn(self._h, ctypes.byref(rs))
        return (float(sm.value), float(smax.value), mw.value / 1e3,
                [n for bit, n in self.REASONS.items() if rs.value & bit])

    def _poll(self):
        while not self._stop.is_set():
            s = self._nvml_sample(self._nvml)
            if s is not None:
                self.samples.append(s)
            self._stop.wait(self.PERIOD_S)

    # ----------------------------------------------------------- nvidia-smi
    def _start_smi(self):
        self.path = os.path.join(os.environ.get("PA_CLOCKS_DIR") or tempfile.gettempdir(),
                                 "pa_clocks_r%d.csv" % os.getpid())
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        for sel in self.selectors:
            try:
                probe = subprocess.run(["nvidia-smi", "-i", sel, "--query-gpu=clocks.sm", "--format=csv,noheader"],
                                       capture_output=True, text=True, timeout=20)
            except Exception as e:  # noqa: BLE001
                self.notes.append("nvidia-smi: %s" % str(e)[:60])
                return
            if probe.returncode == 0 and probe.stdout.strip():
                self.selector = sel
                break
            self.notes.append("nvidia-smi -i %s: %s" % (sel, (probe.stderr or probe.stdout).strip()[:60]))
        else:
            return
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen(["nvidia-smi", "-i", self.selector, "--query-gpu=" + self.FIELDS,
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=self.fh, stderr=subprocess.DEVNULL)
        t0 = time.time()
        while time.time() - t0 < 10 and self._smi_rows() == 0:  # its first row, before the region opens
            time.sleep(0.05)

    def _smi_rows(self):
        try:
            return sum(1 for line in open(self.path) if line.count(",") >= 7)
        except OSError:
            return 0

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        out = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
                pw = float(parts[2])
            except ValueError:
                continue
            out.append((sm, smax, pw, [n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")]))
        return out

    # ------------------------------------------------------------------ API
    def start(self):
        import threading

        self.samples, self.proc = [], None
        if self._nvml is not None:
            self.source = "nvml (every %d ms)" % int(self.PERIOD_S * 1e3)
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return
        try:
            self._start_smi()
            if self.proc is not None:
                self.source = "nvidia-smi (every 100 ms)"
        except Exception as e:  # noqa: BLE001
            self.notes.append("nvidia-smi: %s" % str(e)[:60])

    def stop(self):
        if self.source and self.source.startswith("nvml"):
            self._stop.set()
            self._thread.join(timeout=5)
        elif self.proc is not None:
            n0 = self._smi_rows()
            t0 = time.time()
            while time.time() - t0 < 2 and self._smi_rows() <= n0:  # one row after the region closes
                time.sleep(0.02)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
            self.fh.close()
            self.samples = self._read_smi()
        s = self.samples
        rec = {"sm_mhz": statistics.median(x[0] for x in s) if s else None,
               "sm_max_mhz": max(x[1] for x in s) if s else None,
               "reasons": sorted({r for x in s for r in x[3]}), "samples": len(s),
               "power_w_max": round(max(x[2] for x in s), 1) if s else None,
               "source": self.source, "gpu": self.selector}
        if not s:
            rec["why_none"] = "; ".join(self.notes) or "no sample returned"
        return rec


def source_sha():
    h = hashlib.sha256()
    for f in ("decode.cu", "decode_mma_plain.cu", "decode_mma_shared.cu", "decode_simt.cu", "decode_fma.cu",
              "decode_kernels.h", "decode_merge.cuh", "decode_plan.cuh", "decode_simt.cuh", "decode_mma.cuh",
              "decode_fma.cuh", "decode_tc.cuh", "pa_common.cuh"):
        h.update(open(os.path.join(ROOT, "paged_kv_cache_150_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None, None
    e = d.get(workload_name)
    if not e or e.get("source_sha") != source_sha():
        return None, e.get("source_sha") if e else None
    return float(e["dram_bytes_per_launch"]), e["source_sha"]


# ------------------------------------------------------------- the step
class Step:
    """Device-resident state of one workload and its step."""

    def __init__(self, cfg, kw, seed_offset=0):
        import numpy as np
        import torch

        import paged_kv_cache_150_gb300 as pa
        from paged_kv_cache_150_gb300 import inputs

        self.pa = pa
        wl, layout, shared = make_workload(cfg, kw, seed_offset)
        self.shared = shared
        self.wl = wl
        self.layout = layout
        vals = inputs.make_values(wl, device="cuda")
        if layout == "split":  # same values, vLLM split cache layout
            vals["k_cache"], vals["v_cache"] = inputs.to_split_layout(vals["k_cache"], vals["v_cache"])
        self.initial_host = None
        self.vals = vals
        bm = pa.BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
        t0 = time.perf_counter()
        slots, pairs = bm.apply_script(wl.script)
        tables, lens = bm.export(list(range(wl.num_seqs)), wl.max_blocks_per_seq)
        self.bm_ms = (time.perf_counter() - t0) * 1e3
        self.host = {"slots": slots, "pairs": pairs, "tables": tables, "lens": lens}
        # The step's per-call inputs live in one packed device buffer (views), so
        # the end-to-end leg moves them with a single host-to-device copy.
        per_step = {"q": vals["q"], "k": vals["k"], "v": vals["v"], "slots": torch.from_numpy(slots),
                    "tables": torch.from_numpy(tables), "lens": torch.from_numpy(lens),
                    "pairs": torch.from_numpy(pairs)}
        self.plan_ms, self.plan_info = None, None
        if shared:  # shared-prefix plan of this batch, built on the host like the tables
            t1 = time.perf_counter()
            plan, self.plan_info = pa.shared_prefix_plan(tables, lens, wl.block_size, wl.num_q_heads,
                                                         wl.num_kv_heads)
            self.plan_ms = (time.perf_counter() - t1) * 1e3
            per_step["plan"] = plan
        offs, total = {}, 0
        for name, t in per_step.items():
            offs[name] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.packed = torch.empty(max(total, 256), dtype=torch.uint8, device="cuda")
        views = {}
        for name, t in per_step.items():
            nbytes = t.numel() * t.element_size()
            v = self.packed[offs[name]:offs[name] + nbytes].view(t.dtype).view(t.shape)
            v.copy_(t.to("cuda"))
            views[name] = v
        self.packed_bytes = total
        vals["q"], vals["k"], vals["v"] = views["q"], views["k"], views["v"]
        self.slots, self.tables, self.lens, self.pairs = views["slots"], views["tables"], views["lens"], views["pairs"]
        self.plan = views.get("plan")
        self.out = torch.empty_like(vals["q"])
        ws = pa.pa_decode_workspace_bytes(vals["k_cache"], wl.num_seqs, wl.num_q_heads, shared=shared)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
        # block copy when there are pairs, the cache write, and the kernels of the
        # decode call as the library counts them (plan, attention, merges)
        self.kernel_launches = (1 if pairs.shape[0] else 0) + 1 + pa.pa_decode_launch_count(
            vals["k_cache"], wl.num_seqs, wl.num_q_heads, wl.max_blocks_per_seq, shared=shared, host_seq_lens=lens)
        H, D, eb = wl.num_q_heads, wl.head_dim, wl.elem_bytes
        self.kv_bytes = wl.kv_bytes_read()
        # distinct physical blocks the decode reads (shared prefixes counted once)
        used = {int(b) for i, L in enumerate(lens) for b in tables[i, :-(-int(L) // wl.block_size)]}
        self.unique_block_bytes = len(used) * wl.block_size * wl.num_kv_heads * wl.head_dim * 2 * wl.elem_bytes
        nb_used = int(sum(-(-int(L) // wl.block_size) for L in wl.seq_lens))
        # attention kernel's algorithmic bytes: K/V rows, q, out, block-table entries
        self.kernel_bytes = self.kv_bytes + 2 * wl.num_seqs * H * D * eb + 4 * nb_used
        self.tokens = wl.num_seqs

    def keep_initial_host_copy(self):
        from paged_kv_cache_150_gb300 import inputs

        self.initial_host = {k: inputs.to_numpy_elems(v).copy() for k, v in self.vals.items()}

    def run(self, events=None):
        pa, v = self.pa, self.vals
        if self.pairs.shape[0]:
            pa.pa_copy_blocks(v["k_cache"], v["v_cache"], self.pairs)
        pa.pa_reshape_and_cache(v["k"], v["v"], self.slots, v["k_cache"], v["v_cache"])
        # the host copy of the lengths, as a serving loop that builds its tables on the host has it
        pa.pa_decode(v["q"], v["k_cache"], v["v_cache"], self.tables, self.lens, self.wl.scale, out=self.out,
                     workspace=self.workspace, events=events, shared_plan=self.plan,
                     host_seq_lens=self.host["lens"])


def _events(n):
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in ev:  # create the CUDA events outside any timed region
        a.record()
        b.record()
    return ev


def time_steps(step, steps, warmup, world, flush, sampler=None, kernel_steps=None):
    """Per-step device time of whole steps (events around each step, L2 flushed
    before each), then, in a second loop, the attention kernel's own duration
    (events the library records around that kernel on the launching stream)."""
    import torch

    for _ in range(warmup):
        if flush.numel():
            flush.zero_()
        step.run()
    torch.cuda.synchronize()
    step.pa.pa_get_device_error()
    ev = _events(steps)
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    for i in range(steps):
        if flush.numel():
            flush.zero_()
        ev[i][0].record()
        step.run()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    step.pa.pa_get_device_error()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    nk = min(steps, kernel_steps or steps)
    kev = _events(nk)
    torch.cuda.synchronize()
    for i in range(nk):
        if flush.numel():
            flush.zero_()
        step.run(events=kev[i])
    torch.cuda.synchronize()
    step.pa.pa_get_device_error()
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    return step_ms, kern_ms, clocks


def time_e2e(step, steps, graph=False):
    """Through the public API with host buffers: pinned H2D of the step's
    inputs, the step, and a D2H read of the output, synchronised per step.

    graph=True records that same sequence (H2D copy, the library calls, D2H
    copy) once in a CUDA graph and replays it per step, as a serving loop
    does once its batch shape is fixed: each replay still copies the pinned
    inputs in and the output back.  Returns (seconds per step, H2D bytes,
    D2H bytes, mode) where mode says which was timed."""
    import torch

    pinned = step.packed.cpu().pin_memory()  # this step's inputs, packed (q, new K/V, slots, tables, lengths, pairs)
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = pinned.numel()
    d2h = out_host.numel() * out_host.element_size()

    def one_step():
        step.packed.copy_(pinned, non_blocking=True)
        step.run()
        out_host.copy_(step.out, non_blocking=True)

    mode = "eager"
    run = one_step
    if graph:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # warm the calls on the capture stream
                for _ in range(3):
                    one_step()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one_step()
            torch.cuda.synchronize()
            run, mode = g.replay, "cuda_graph"
        except Exception as e:  # report the eager timing instead
            mode = "eager (graph capture failed: %s)" % str(e).splitlines()[0][:80]
            torch.cuda.synchronize()
    times = []
    stream = torch.cuda.current_stream()
    for i in range(steps + 3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run()
        stream.synchronize()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    step.pa.pa_get_device_error()
    return statistics.mean(times), h2d, d2h, mode


def time_write_copy(step, iters, peak):
    """The cache write and the block copy timed on their own (CUDA events
    around each call, median), reported as GB/s of bytes read + written.  A
    512 MiB buffer is READ before each timed call, so the call's source rows
    are not in L2 and no dirty line of the flush is written back inside it."""
    import torch

    pa, v, wl = step.pa, step.vals, step.wl
    row = wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    rows = int((step.host["slots"] >= 0).sum())
    npairs = int(step.host["pairs"].shape[0])
    flush = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    calls = {"cache_write": (lambda: pa.pa_reshape_and_cache(v["k"], v["v"], step.slots, v["k_cache"], v["v_cache"]),
                             2 * 2 * rows * row + 4 * int(step.slots.numel()), rows)}
    if npairs:
        calls["block_copy"] = (lambda: pa.pa_copy_blocks(v["k_cache"], v["v_cache"], step.pairs),
                               2 * 2 * npairs * wl.block_size * row + 8 * npairs, npairs)
    def median_us(fn):
        for _ in range(3):
            fn()
        ev = _events(iters)
        for i in range(iters):
            flush.sum()
            ev[i][0].record()
            fn()
            ev[i][1].record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3

    # The same timing around a kernel that does nothing: what one launch
    # between two events costs on this machine whatever it moves (about 4 us).
    floor_us = median_us(lambda: torch.cuda._sleep(0)) if hasattr(torch.cuda, "_sleep") else None
    out = {}
    for name, (fn, nbytes, units) in calls.items():
        us = median_us(fn)
        pa.pa_get_device_error()
        gbs = nbytes / (us / 1e6) / 1e9
        out[name] = {"us": round(us, 2), "bytes_read_written": nbytes,
                     ("rows" if name == "cache_write" else "pairs"): units,
                     "gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4)}
        if floor_us is not None:
            out[name]["empty_launch_us"] = round(floor_us, 2)
            if us > floor_us:  # bandwidth of the time the call takes beyond an empty launch
                out[name]["gbs_above_empty_launch"] = round(nbytes / ((us - floor_us) / 1e6) / 1e9, 1)
    del flush
    return out


def oracle_baseline(step, max_groups, threads, repeat=1):
    """The CPU oracle, as it stands, on a bounded sample of the workload:
    whole (sequence, KV head) groups, all G query heads of each (timed
    ``repeat`` times over, for samples too small to time once)."""
    import oracle

    wl = step.wl
    if step.initial_host is None:
        raise RuntimeError("initial host copy missing")
    host = step.initial_host
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    kc, vc = host["k_cache"].copy(), host["v_cache"].copy()
    oracle.copy_blocks(kc, vc, r["pairs"])
    oracle.reshape_and_cache(host["k"], host["v"], r["slots"], kc, vc)
    tables = oracle.pad_tables(r["tables"], wl.max_blocks_per_seq)
    G = wl.num_q_heads // wl.num_kv_heads
    groups = [(s, kh) for s in range(wl.num_seqs) for kh in range(wl.num_kv_heads)][:max_groups]
    pairs = [(s, kh * G + j) for s, kh in groups for j in range(G)]
    t0 = time.perf_counter()
    for _ in range(repeat):
        ref = oracle.decode(host["q"], kc, vc, tables, r["lens"], wl.scale, pairs=pairs, num_threads=threads)
    dt = time.perf_counter() - t0
    bytes_ = repeat * sum(int(wl.seq_lens[s]) * wl.head_dim * 2 * wl.elem_bytes for s, _ in groups)
    return ref, pairs, dt, bytes_, len(groups)


def oracle_single_thread():
    """The oracle with one host thread on the three smaller workloads (cfg0
    whole, cfg1 and cfg2 on a sample of (sequence, KV head) groups): a
    per-core figure beside the all-core baseline."""
    import torch

    out = {}
    for cfg, kw, max_groups, repeat in (("cfg0", {}, 10 ** 9, 200), ("cfg1", {}, 10 ** 9, 1), ("cfg2", {}, 768, 1)):
        st = Step(cfg, kw)
        st.keep_initial_host_copy()
        _, _, dt, nbytes, ngroups = oracle_baseline(st, max_groups, 1, repeat)
        out[st.wl.name] = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                           "sample": "%d of %d (sequence, KV head) groups, all query heads, x%d, %.2f s" %
                                     (ngroups, st.wl.num_seqs * st.wl.num_kv_heads, repeat, dt)}
        del st
        torch.cuda.empty_cache()
    return out


def allocation_simulator():
    """Host-side context (not the metric): contiguous max-length reservation
    against paging with a block-size sweep, on one synthetic stream of 2000
    requests (Poisson arrivals, lognormal lengths), 200k token slots."""
    import paged_kv_cache_150_gb300 as pa
    from paged_kv_cache_150_gb300 import inputs

    a, p, o = inputs.request_stream(7, 2000, 1.0, prompt_median=256, output_median=128, max_prompt=2048,
                                    max_new_tokens=2048)
    out = {}
    runs = [("contiguous", 16)] + [("paged", b) for b in (1, 8, 16, 32, 64, 128)]
    for policy, b in runs:
        r = pa.simulate(policy, a, p, o, 200000, block_size=b, max_new_tokens=2048)
        key = policy if policy == "contiguous" else "paged_b%d" % b
        out[key] = {"kv_utilization": round(r["utilization"], 4), "peak_running": r["peak_running"],
                    "steps_to_drain": r["steps"], "preemptions": r["preemptions"],
                    "waste_tokens_per_seq": round((r["sum_held"] - r["sum_used"]) / max(r["sum_running"], 1), 2)}
    return out


def parity_check(step, ref, pairs):
    import numpy as np

    out = step.out.double().cpu().numpy()
    idx = np.asarray(pairs)
    return float(np.abs(out[idx[:, 0], idx[:, 1]] - ref[idx[:, 0], idx[:, 1]]).max())


def uses_mma(wl):
    """Whether pa_decode's automatic choice is the tensor-core kernel (bf16,
    head_dim 64 or 128, block size 16 or 32, at most 8 query heads per KV
    head); else it runs the CUDA-core kernel."""
    G = wl.num_q_heads // wl.num_kv_heads
    return wl.dtype == "bf16" and wl.head_dim in (64, 128) and wl.block_size in (16, 32) and G <= 8


def workload_name(step):
    return step.wl.name


def describe(wl):
    G = wl.num_q_heads // wl.num_kv_heads
    return ("%s: %d seqs (lengths %d..%d, %d tokens), %d q / %d KV heads (group %d), head_dim %d, %s, "
            "block %d, pool %d blocks, seeded random placement; %s"
            % (wl.name, wl.num_seqs, int(wl.seq_lens.min()), int(wl.seq_lens.max()), int(wl.seq_lens.sum()),
               wl.num_q_heads, wl.num_kv_heads, G, wl.head_dim, wl.dtype, wl.block_size, wl.num_blocks, wl.note))


# -------------------------------------------------------------- arms
def run_ours(args, rank, world):
    import torch

    peak, peak_kind = measured_peaks()
    flush = torch.empty(FLUSH_BYTES if args.l2 == "write" else 0, dtype=torch.uint8, device="cuda")
    step = Step(*WORKLOADS[args.workload], seed_offset=1000 * rank)
    do_cpu = rank == 0 and world == 1 and not args.no_cpu
    if do_cpu:
        step.keep_initial_host_copy()
    sampler = ClockSampler(torch.cuda.current_device())
    step_ms, kern_ms, clocks = time_steps(step, args.steps, args.warmup, world, flush, sampler, kernel_steps=1000)
    total_ms = reduce_max(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * step.kv_bytes * args.steps / (total_ms / 1e3) / 1e9
    tokens_per_s = world * step.tokens * args.steps / (total_ms / 1e3)
    kern_avg_ms = statistics.mean(kern_ms)
    achieved = step.kernel_bytes / (kern_avg_ms / 1e3) / 1e9
    traffic, _ = profiled_traffic(workload_name(step))

    write_copy = None if args.no_write_copy else time_write_copy(step, 50, peak)
    if args.no_e2e:
        e2e = None
    else:
        eager_s, h2d, d2h, _ = time_e2e(step, args.e2e_steps)
        e2e_s, _, _, mode = time_e2e(step, args.e2e_steps, graph=True)
        e2e = {"value": round(world * step.kv_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4), "mode": mode,
               "eager": {"value": round(world * step.kv_bytes / eager_s / 1e9, 2),
                         "ms_per_step": round(eager_s * 1e3, 4)}}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": step.wl.dtype, "data": "synthetic",
        "config": bench_config(step.wl, args.l2, world),
        "tokens_per_s": round(tokens_per_s, 1),
        "hbm_frac": round(value / world / peak, 4),
        "roofline": {"bound": "hbm",
                     "kernel": "decode attention (%s kernel)" % ("tensor-core" if uses_mma(step.wl) else "CUDA-core"),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": step.kernel_bytes,
                     "avg_launch_ms": round(kern_avg_ms, 5), "peak_source": peak_kind},
        "e2e": e2e,
        "gpu_launches": step.kernel_launches * args.steps,
        "clocks": clocks,
        "block_manager_ms": round(step.bm_ms, 3),
        "write_copy": write_copy,
    }
    targets = {"goal": "pa_decode >= 0.70 of HBM peak; outputs within 2e-2 of the fp64 oracle",
               "peak_gbs": peak}

    def target(name, st, step_ms, kernel_ms, parity):
        gbs = st.kernel_bytes / (kernel_ms / 1e3) / 1e9
        targets[name] = {"hbm_frac": round(st.kv_bytes / (step_ms / 1e3) / 1e9 / peak, 4),
                         "kernel_gbs": round(gbs, 1), "kernel_frac": round(gbs / peak, 4)}
        if parity is not None:
            targets[name].update(parity)

    def full_parity(st, threads):
        """Every output of the workload against the oracle (CPU leg)."""
        ref, pairs, dt, nbytes, _ = oracle_baseline(st, 10 ** 9, threads)
        return {"max_abs_err": float("%.3g" % parity_check(st, ref, pairs)), "outputs_checked": len(pairs)}

    if do_cpu:
        import oracle

        threads = oracle.available_threads()
        ref, pairs, dt, nbytes, ngroups = oracle_baseline(step, 128, threads)
        line["cpu_baseline"] = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle",
                                "sample": "%d of %d (sequence, KV head) groups of the workload, all query heads, "
                                          "fp64, %.1f s wall" % (ngroups, step.wl.num_seqs * step.wl.num_kv_heads, dt)}
        line["parity"] = {"max_abs_err": parity_check(step, ref, pairs), "pairs_checked": len(pairs),
                          "tolerance": 2e-2 if step.wl.dtype == "bf16" else 1e-5}
    if args.workload in TARGETS:
        par = None
        if do_cpu:
            par = ({"max_abs_err": float("%.3g" % line["parity"]["max_abs_err"]), "outputs_checked": len(pairs)}
                   if len(pairs) == step.wl.num_seqs * step.wl.num_q_heads else full_parity(step, threads))
        target(args.workload, step, ms_per_step, kern_avg_ms, par)
    del step
    torch.cuda.empty_cache()
    if do_cpu:
        line["cpu_baseline"]["single_thread"] = oracle_single_thread()
    if not args.no_extra:
        extra = {}
        for cfg, kw in EXTRA:
            if WORKLOADS[args.workload] == (cfg, kw):
                continue
            torch.cuda.empty_cache()
            st = Step(cfg, kw, seed_offset=1000 * rank)
            tname = next((n for n in TARGETS if WORKLOADS[n] == (cfg, kw)), None)
            if tname and do_cpu:
                st.keep_initial_host_copy()
            sm, km, _ = time_steps(st, args.extra_steps, args.warmup, world, flush, kernel_steps=args.extra_steps)
            mean_ms = reduce_max(statistics.mean(sm), world)
            kms = statistics.mean(km)
            if tname:
                target(tname, st, mean_ms, kms, full_parity(st, threads) if do_cpu else None)
            extra[st.wl.name] = {"kv_gbs": round(st.kv_bytes / (mean_ms / 1e3) / 1e9, 2),
                                 "ms_per_step": round(mean_ms, 5),
                                 "tokens_per_s": round(st.tokens / (mean_ms / 1e3), 1),
                                 "hbm_frac": round(st.kv_bytes / (mean_ms / 1e3) / 1e9 / peak, 4),
                                 "kernel_gbs": round(st.kernel_bytes / (kms / 1e3) / 1e9, 2),
                                 "kernel_ms": round(kms, 5), "kv_bytes": st.kv_bytes,
                                 "cow_pairs": int(st.host["pairs"].shape[0]), "new_tokens": st.wl.num_new_tokens,
                                 "unique_block_bytes": st.unique_block_bytes,
                                 "written_rows": int((st.host["slots"] >= 0).sum()),
                                 "cache_layout": st.layout,
                                 "write_copy": None if args.no_write_copy else time_write_copy(st, 50, peak)}
            if st.unique_block_bytes < st.kv_bytes:  # blocks shared between sequences: the bytes read once
                extra[st.wl.name]["unique_gbs"] = round(st.unique_block_bytes / (mean_ms / 1e3) / 1e9, 2)
                extra[st.wl.name]["unique_hbm_frac"] = round(st.unique_block_bytes / (mean_ms / 1e3) / 1e9 / peak, 4)
            if st.shared:
                extra[st.wl.name]["shared_plan"] = dict(st.plan_info, host_ms=round(st.plan_ms, 3))
            del st
            torch.cuda.empty_cache()
        line["workloads"] = extra
    if rank == 0:
        line["allocation_simulator"] = allocation_simulator()
        line["targets"] = targets  # last: the end of the line is what a log tail keeps
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle as the reference arm, timed on this machine's host cores."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from paged_kv_cache_150_gb300 import inputs

    wl, _, _ = make_workload(*WORKLOADS[args.workload])  # the oracle reads the row layout of the same values
    vals = inputs.make_values(wl, device="cpu")
    host = {k: inputs.to_numpy_elems(v).copy() for k, v in vals.items()}
    r = oracle.run_script(wl.num_blocks, wl.block_size, wl.free_order, wl.script)
    kc, vc = host["k_cache"], host["v_cache"]
    oracle.copy_blocks(kc, vc, r["pairs"])
    oracle.reshape_and_cache(host["k"], host["v"], r["slots"], kc, vc)
    tables = oracle.pad_tables(r["tables"], wl.max_blocks_per_seq)
    threads = oracle.available_threads()
    G = wl.num_q_heads // wl.num_kv_heads
    groups_all = [(s, kh) for s in range(wl.num_seqs) for kh in range(wl.num_kv_heads)]
    # one step = a bounded sample of (sequence, KV head) groups, sized so the
    # whole run stays within a few minutes
    budget_s = 150.0
    for _ in range(2):  # the second call is timed: the first also faults in the caches' pages
        t0 = time.perf_counter()
        oracle.decode(host["q"], kc, vc, tables, r["lens"], wl.scale,
                      pairs=[(0, j) for j in range(G)], num_threads=threads)
        t_group = time.perf_counter() - t0
    per_step = max(1, min(len(groups_all), int(budget_s / max(args.steps + args.warmup, 1) / max(t_group, 1e-6))))
    used = min(threads, per_step * G)  # the oracle's threads split the step's (sequence, head) pairs
    times, nbytes = [], 0
    for i in range(args.warmup + args.steps):
        gs = [groups_all[(i * per_step + j) % len(groups_all)] for j in range(per_step)]
        pairs = [(s, kh * G + j) for s, kh in gs for j in range(G)]
        t0 = time.perf_counter()
        oracle.decode(host["q"], kc, vc, tables, r["lens"], wl.scale, pairs=pairs, num_threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes += sum(int(wl.seq_lens[s]) * wl.head_dim * 2 * wl.elem_bytes for s, _ in gs)
    total = sum(times)
    value = nbytes / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, args.l2, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": "%d groups (%d sequence-head pairs) per step of %d groups; %d host threads"
                                   % (per_step, per_step * G, len(groups_all), threads)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":  # host cores only: rank 0 runs it, other ranks exit without work
        run_reference(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, _ = dist_setup(args)
    import __graft_entry__

    __graft_entry__.build()
    run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
