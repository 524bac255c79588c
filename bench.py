"""Benchmark: restricted-vocabulary MTP draft head + greedy verify on GB300.

One bench step = one MTP3 draft chain on the single-stream decode workload:
three sequential draft-head calls (B = 1, a fresh hidden vector each) on a
65,536-row x 2048 bf16 candidate head drawn from the 248,320-row output head.
`value` is draft steps/s (3 calls per bench step) measured on the device with
CUDA events around each call, with L2 flushed before every call and outside
the timed events (a 256 MiB write, then a 256 MiB read so that the write's
dirty lines go back to HBM before the start event, not inside the timed
call), so every call reads the 268 MB head from HBM.  The same run also measures (reported under "verify", "sweep" and
"nvfp4"): the batched greedy verify (64 x 4 rows against the full head), the
head-size sweep (248,320 / 65,536 / 32,768 rows) and the 4-bit head
(65,536 x 4096, B = 1 and 8).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the only reference implementation
this method has) on the host cores, on the same workload and metric.
Under torchrun each rank runs an independent replica on its own GPU
(no data-path collective); value = all ranks' draft steps / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft steps/s and verify rounds/s; head HBM GB/s as % of GB300 roofline"
UNIT = "draft steps/s"
WORKLOAD = ("draft head: 65,536 sorted candidate rows of a 248,320 x 2048 bf16 head ~N(0,0.02) (seed 2), "
            "B=1 hidden ~N(0,1), 3 sequential draft steps per bench step")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
PREROLL_CYCLES = 200_000  # ~100 us of GPU sleep queued before each timed call


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)

        def pick(*names):
            for n in names:
                if n in d and isinstance(d[n], (int, float)):
                    return float(d[n])
            return None
        hbm = pick("hbm_gbs", "hbm_GBps", "hbm")
        bf = pick("bf16_tflops", "bf16_TFLOPs")
        bfs = pick("bf16_tflops_sustained")
        if hbm and bf:
            return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs or bf}, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ----------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms from before the warm-up
    to the end of the run; mark() brackets the timed region of the headline."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.start = 0
        self.region = None  # (start, end) byte offsets of the timed region in the sample file
        # the raw samples (the JSON line carries their summary); VH_BENCH_LOG_DIR overrides the location
        log_dir = os.environ.get("VH_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"vh_clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            # wait (at most 3 s) for the sampler's first line, then count what follows
            t0 = time.time()
            while time.time() - t0 < 3.0 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
            self.start = os.path.getsize(self.path)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark(self, begin: bool):
        if self.proc is None:
            return
        self.f.flush()
        off = os.path.getsize(self.path)
        self.region = (off, None) if begin else (self.region[0] if self.region else self.start, off)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    @staticmethod
    def _parse(lines):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return sm, mx, reasons

    def summary(self):
        """Median SM clock, the maximum, and every throttle reason seen over
        the whole run (warm-up, timed chains and the other workloads); the
        headline's timed region is also given on its own when it holds
        samples (a run of 20 steps times about 3 ms, less than one
        sampling interval of some tools)."""
        if self.proc is None:
            return None
        try:
            with open(self.path) as f:
                text = f.read()
        except OSError:
            return None
        sm, mx, reasons = self._parse(text[self.start:].splitlines())
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm), "window": "whole run: warm-up, timed chains and every other workload",
               "sample_interval_ms": 20}
        if self.region and self.region[1] is not None:
            r_sm, _, r_reasons = self._parse(text[self.region[0]:self.region[1]].splitlines())
            out["timed_region"] = ({"sm_mhz": statistics.median(r_sm), "samples": len(r_sm),
                                    "reasons": sorted(r_reasons)} if r_sm else {"samples": 0})
        return out


# ----------------------------------------------------------------------------
# device timing helpers

class Timer:
    """Per-call device time with CUDA events on the current stream; L2 is
    flushed before each call, outside the events."""

    def __init__(self, torch, flush=True, clean=True):
        self.torch = torch
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda") if flush else None
        # read after the write: it evicts the write's dirty lines (written back to HBM here, outside the
        # events) and leaves L2 holding clean lines of a buffer the timed call never touches
        self.clean_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda") if flush and clean \
            else None
        self.sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush(self):
        """Evict L2 (256 MiB write, then a 256 MiB read), then queue ~100 us
        of GPU sleep so that the host has enqueued the timed call before its
        start event runs: the events then bracket device time only, not host
        launch latency.  Without the read, up to an L2's worth of the write's
        dirty lines is written back while the timed call streams its head,
        which took the headline chain from 41.8 to 45.5 us per call."""
        if self.flush_buf is not None:
            self.flush_buf.fill_(1)
        if self.clean_buf is not None:
            self.torch.sum(self.clean_buf, dim=0, keepdim=True, out=self.sink)
        self.torch.cuda._sleep(PREROLL_CYCLES)

    def time_calls(self, fn, n, warmup=3):
        torch = self.torch
        for _ in range(warmup):
            self.flush()
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            self.flush()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in evs]  # microseconds


def stats(us):
    us = sorted(us)
    return {"median_us": round(statistics.median(us), 3), "p10_us": round(us[len(us) // 10], 3),
            "p90_us": round(us[(len(us) * 9) // 10], 3), "mean_us": round(sum(us) / len(us), 3)}


KERNEL_HEADERS = ("vh_common.cuh", "vh_kernels.h", "vh_ptx.cuh")  # included by every kernel file


_COMMENTS = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def source_sha(kernel_file: str) -> str:
    """First 16 hex digits of sha256 over the code of a kernel file followed by
    the shared headers it compiles with (the key a profile summary was taken
    on).  Comments, trailing blanks and empty lines are left out, so editing a
    comment does not orphan a profile; any change to the code does."""
    h = hashlib.sha256()
    for name in (kernel_file,) + KERNEL_HEADERS:
        text = open(os.path.join(ROOT, "verify_head_gb300", "csrc", name), encoding="utf-8").read()
        code = "\n".join(ln.rstrip() for ln in _COMMENTS.sub("", text).splitlines() if ln.strip())
        h.update(code.encode("utf-8"))
    return h.hexdigest()[:16]


def profile_traffic(kernel_file: str, summary: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (source_sha of the .cu file and the shared
    headers); else None."""
    try:
        sha = source_sha(kernel_file)
        vals = {}
        for line in open(os.path.join(ROOT, "profiles", summary)):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") == sha and "dram_bytes_per_launch" in vals:
            return float(vals["dram_bytes_per_launch"])
    except (OSError, ValueError):
        pass
    return None


def load_verify_golden():
    """Draft ids (inputs) and the oracle's greedy ids for the batched-verify
    workload, stored by tests/golden/make_verify_golden.py."""
    path = os.path.join(ROOT, "tests", "golden", "verify_b64_k3_248320x2048.txt")
    nid = np.zeros(256, np.int32)
    draft = np.zeros((64, 3), np.int32)
    for line in open(path):
        p = line.split()
        if p and p[0] == "row":
            nid[int(p[1])] = int(p[2])
        elif p and p[0] == "seq":
            draft[int(p[1])] = [int(v) for v in p[2:5]]
    return {"next_ids": nid, "draft": draft}


# ----------------------------------------------------------------------------

def run_ours(args):
    import torch
    import synth
    import verify_head_gb300 as vh

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    vh.lib()
    dev = torch.device("cuda")
    peaks, peak_src = load_peaks()

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- headline workload: draft head 65,536 x 2048, B=1, 3 steps ----
    case = synth.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    W = t_bf16(case.W)
    cand = torch.from_numpy(case.cand_ids).to(dev)
    xs = [t_bf16(h) for h in case.hidden]
    ws = vh.workspace(1)
    ids = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(3)]
    timer = Timer(torch)

    def call(i):
        vh.mtp_draft_head_argmax(xs[i], W, cand, ids=ids[i], maxlogit=mls[i], ws=ws)

    bytes_per_call = case.Vc * case.H * 2 + case.Vc * 4 + case.B * case.H * 2

    sampler = ClockSampler(local)
    sampler.__enter__()  # clocks from the warm-up to the end of the run
    for _ in range(max(3, args.warmup)):
        for i in range(3):
            timer.flush()
            call(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark(True)
    evs = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        timer.flush()
        a.record()
        for i in range(3):  # one MTP3 draft chain: three dependent-launch calls back to back
            call(i)
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    sampler.mark(False)
    per_step = [a.elapsed_time(b) * 1e3 for a, b in evs]
    # warm extra: the same chain with no L2 flush in between (the 268 MB table is twice
    # the L2, so most of it still streams from HBM); reported beside the value, never as it
    warm_evs = []
    for _ in range(max(10, args.steps // 10)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(PREROLL_CYCLES)
        a.record()
        for i in range(3):
            call(i)
        b.record()
        warm_evs.append((a, b))
    torch.cuda.synchronize()
    warm_st = stats([a.elapsed_time(b) * 1e3 / 3 for a, b in warm_evs])
    # the same chain after a write-only flush: the write's dirty lines stay in L2 and go back to HBM
    # while the chain streams its head; reported beside the value for comparison, never as it
    wo_timer = Timer(torch, clean=False)
    wo_st = stats([t / 3 for t in wo_timer.time_calls(lambda: [call(i) for i in range(3)],
                                                      max(10, args.steps // 10))])
    del wo_timer
    total_s = sum(per_step) * 1e-6
    if world > 1:
        t = torch.tensor([total_s], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_s = float(t.item())
        torch.distributed.barrier()
    n_calls = 3 * args.steps
    value = world * n_calls / total_s
    st = stats([t / 3 for t in per_step])
    avg_us = sum(per_step) / n_calls
    achieved = bytes_per_call / (avg_us * 1e-6) / 1e9

    # ---- end to end through the binding: pinned host hidden in, ids out ----
    # One step's three hidden vectors go up in one copy and its three (id,
    # maxlogit) pairs come back in one copy: [ids(3) | maxlogit bits(3)] int32.
    host_x = torch.from_numpy(np.ascontiguousarray(np.stack(case.hidden)).view(np.int16)).pin_memory()
    host_res = torch.empty(6, dtype=torch.int32).pin_memory()
    dx = torch.empty(3, 1, case.H, dtype=torch.bfloat16, device=dev)
    dres = torch.empty(6, dtype=torch.int32, device=dev)
    e_ids = [dres[i:i + 1] for i in range(3)]
    e_mls = [dres[3 + i:4 + i].view(torch.float32) for i in range(3)]
    e2e_us = []
    e2e_steps = max(5, args.steps // 2)
    for it in range(e2e_steps + 2):
        timer.flush()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dx.view(torch.int16).copy_(host_x, non_blocking=True)
        for i in range(3):
            vh.mtp_draft_head_argmax(dx[i], W, cand, ids=e_ids[i], maxlogit=e_mls[i], ws=ws)
        host_res.copy_(dres, non_blocking=True)
        b.record()
        b.synchronize()
        if it >= 2:
            e2e_us.append(a.elapsed_time(b) * 1e3)
    if host_res[:3].tolist() != [int(t.item()) for t in ids]:
        raise RuntimeError("end-to-end ids differ from the device-resident calls")
    e2e_value = world * 3 * len(e2e_us) / (sum(e2e_us) * 1e-6)

    # the same step (copy in, three calls, copy out) captured once as a CUDA graph and replayed
    def e2e_step():
        dx.view(torch.int16).copy_(host_x, non_blocking=True)
        for i in range(3):
            vh.mtp_draft_head_argmax(dx[i], W, cand, ids=e_ids[i], maxlogit=e_mls[i], ws=ws)
        host_res.copy_(dres, non_blocking=True)

    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        e2e_step()
    torch.cuda.current_stream().wait_stream(gs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        e2e_step()
    host_res.zero_()
    g_us = []
    for it in range(e2e_steps + 2):
        timer.flush()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        if it >= 2:
            g_us.append(a.elapsed_time(b) * 1e3)
    if host_res[:3].tolist() != [int(t.item()) for t in ids]:
        raise RuntimeError("graph-replayed end-to-end ids differ from the device-resident calls")
    e2e_graph_value = world * 3 * len(g_us) / (sum(g_us) * 1e-6)
    del graph
    del W

    extra = {}
    if rank == 0 and not args.skip_extra and args.workload == "all":
        extra = measure_extra(torch, vh, synth, timer, peaks, load_verify_golden)
    sampler.__exit__(None, None, None)

    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu, first = cpu_baseline(case, seconds=args.cpu_seconds, threads=args.oracle_threads)
        # the three timed draft steps against the oracle's (ids exact where the top-1 / top-2 gap > 1e-2)
        g_ids = [int(t.item()) for t in ids]
        g_ml = [float(t.item()) for t in mls]
        ok = sum(1 for i, (o_ids, o_ml, o_sec) in enumerate(first)
                 if (g_ids[i] == int(o_ids[0]) or float(o_ml[0]) - float(o_sec[0]) <= 1e-2)
                 and abs(g_ml[i] - float(o_ml[0])) <= 2e-2)
        parity = {"draft_steps_matching_oracle": f"{ok}/3",
                  "max_abs_maxlogit_err": round(max(abs(g_ml[i] - float(first[i][1][0])) for i in range(3)), 6)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(total_s / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generators; no corpus or trained weights)",
        "config": {"workload": WORKLOAD, "Vc": case.Vc, "H": case.H, "B": case.B, "draft_steps_per_step": 3,
                   "l2": "flushed before every chain outside the timed events: a 256 MiB write, then a 256 MiB "
                         "read, so that no dirty flush lines are written back inside the timed region",
                   "timing": "CUDA events around each 3-call chain on the launching stream (L2 flushed before "
                             "each chain); a ~100 us sleep kernel is queued before the start event so host "
                             "launch latency is not timed",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "draft_call_us": st,
        "draft_call_us_warm": {**warm_st, "what": "the same 3-call chain without the L2 flush between chains"},
        "draft_call_us_write_only_flush": {**wo_st, "what": "the same 3-call chain after a 256 MiB write alone "
                                                            "(its dirty lines are written back inside the chain)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_src,
                     "frac_of_8000_spec": round(achieved / 8000.0, 4),
                     "traffic": profile_traffic("gemv_argmax.cu", "draft_gemv_65536x2048.txt"),
                     "algorithmic_bytes_per_launch": bytes_per_call,
                     "kernel": "k_gemv_bf16<1> (split-V streaming GEMV + fused argmax)"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": 3 * case.H * 2,
                "d2h_bytes_per_step": 3 * 8, "copies_per_step": "1 H2D + 1 D2H",
                "median_us_per_step": round(statistics.median(e2e_us), 2),
                "graph_replay": {"value": round(e2e_graph_value, 2), "unit": UNIT,
                                 "median_us_per_step": round(statistics.median(g_us), 2),
                                 "what": "the same step (pinned-host copy in, three calls, copy out) captured "
                                         "once as a CUDA graph and replayed"}},
        "gpu_launches": n_calls,
        "clocks": sampler.summary(),
        "cpu_baseline": cpu,
        "parity": parity,
    }
    line.update(extra)
    line["summary"] = summarize(line)  # last key: a compact digest of every workload
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def summarize(line):
    """One short entry per workload (config 1 tiny, 2 draft, 3 sweep, 4 verify,
    5 4-bit draft; the gather, 4-bit verify and end-to-end figures), so that a
    reader of the end of the line sees every result: [us per call or round,
    fraction of the measured HBM roofline] unless named otherwise."""
    def g(d, *ks):
        for k in ks:
            if not isinstance(d, dict) or k not in d:
                return None
            d = d[k]
        return d

    def pair(d, us_key="median_us", frac_key="hbm_frac"):
        return None if not isinstance(d, dict) else [d.get(us_key), d.get(frac_key)]

    s = {"draft_65536x2048": {"steps_per_s": line["value"], "us": g(line, "draft_call_us", "mean_us"),
                              "hbm_frac": g(line, "roofline", "frac")},
         "e2e_steps_per_s": g(line, "e2e", "value")}
    t = line.get("tiny")
    if t:
        s["tiny_4096x256"] = {"draft_us": g(t, "draft_call_us", "median_us"),
                              "verify_us": g(t, "verify_call_us", "median_us"),
                              "ids": t.get("draft_ids_equal_oracle"), "verify_ids": t.get("verify_next_ids_equal_oracle")}
    if line.get("sweep"):
        s["sweep"] = {k: pair(v, "mean_us") for k, v in line["sweep"].items()}
    v = line.get("verify")
    if v:
        s["verify_256x248320"] = {"rounds_per_s": v.get("rounds_per_s"), "us": v.get("median_us"),
                                  "hbm_frac": v.get("hbm_frac"), "tensor_frac_burst": v.get("tensor_frac_burst"),
                                  "tensor_frac_sustained": v.get("tensor_frac_sustained")}
    if line.get("verify_rows") and "4" in line["verify_rows"]:
        s["verify_batch1_4x248320"] = pair(line["verify_rows"]["4"])
    r = line.get("mtp3_round")
    if r:
        s["mtp3_round_b1"] = {k: [v.get("mean_us"), v.get("rounds_per_s")] for k, v in r.items() if isinstance(v, dict)}
    if line.get("gather"):
        s["gather"] = pair(line["gather"], "mean_us")
    if line.get("draft_batch"):
        s["draft_batch_65536x2048"] = {k: pair(v, "mean_us") for k, v in line["draft_batch"].items()}
    nv = line.get("nvfp4")
    if nv:
        s["nvfp4_65536x4096"] = {**{k: pair(v, "mean_us") for k, v in nv.items() if k.startswith("B")},
                                 **{"row_major_" + k: pair(v, "mean_us") for k, v in nv.get("row_major", {}).items()}}
    if line.get("verify_nvfp4"):
        s["verify_nvfp4"] = {k.replace("head_", "").replace("full_head_", "full_"): pair(v)
                             for k, v in line["verify_nvfp4"].items()}
    s["peaks"] = g(line, "roofline", "peak_source")
    return s


def measure_extra(torch, vh, synth, timer, peaks, load_verify_golden, only="all"):
    dev = torch.device("cuda")
    out = {}
    if only in ("all", "tiny"):
        out["tiny"] = measure_tiny(torch, vh, synth, timer)
    if only in ("all", "verify"):
        out.update(measure_verify(torch, vh, synth, timer, peaks, load_verify_golden, cuda_core=(only == "verify")))
    if only in ("all", "sweep"):
        out["sweep"] = measure_sweep(torch, vh, synth, timer, peaks)
    if only in ("all", "gather"):
        out["gather"] = measure_gather(torch, vh, synth, timer, peaks)
    if only in ("all", "draft_batch"):
        out["draft_batch"] = measure_draft_batch(torch, vh, synth, timer, peaks)
    if only in ("all", "mtp3_round"):
        out["mtp3_round"] = measure_mtp3_round(torch, vh, synth, timer, peaks)
    if only in ("all", "chain"):
        out["chain_graph"] = measure_chain_graph(torch, vh, synth, timer, peaks)
    if only in ("all", "verify_nvfp4"):
        out["verify_nvfp4"] = measure_verify_nvfp4(torch, vh, synth, timer, peaks)
    if only in ("all", "nvfp4"):
        out["nvfp4"] = measure_nvfp4(torch, vh, synth, timer, peaks)
    return out


def measure_tiny(torch, vh, synth, timer):
    """The tiny oracle check (4,096 x 256 head, 1,024 candidates, 3 draft steps,
    verify of 1 x 4 rows): GPU results against the oracle, and call times."""
    import oracle
    oracle.build()
    dev = torch.device("cuda")
    draft, verify, W_full = synth.tiny_case()

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    W, cand = t_bf16(draft.W), torch.from_numpy(draft.cand_ids).to(dev)
    ids_ok = 0
    for h in draft.hidden:
        g_ids, _ = vh.mtp_draft_head_argmax(t_bf16(h), W, cand)
        o_ids, _, _ = oracle.draft_argmax(h, draft.W, draft.cand_ids)
        ids_ok += int(int(g_ids.item()) == int(o_ids[0]))
    _, o_nid, _, _ = oracle.verify_greedy(verify.X, W_full, None, 1, 3)
    d = verify.draft_ids_from(o_nid)
    acc, nid, _ = vh.spec_verify_greedy(t_bf16(verify.X), t_bf16(W_full), torch.from_numpy(d).to(dev), 1, 3)
    o_acc = oracle.accept_len(o_nid[:3], d[0])
    # timed as a decode loop calls it: workspace and outputs allocated once, outside the timed calls
    x0 = t_bf16(draft.hidden[0])
    ws_d, ids_d = vh.workspace(1), torch.empty(1, dtype=torch.int32, device=dev)
    ml_d = torch.empty(1, dtype=torch.float32, device=dev)
    us_d = timer.time_calls(lambda: vh.mtp_draft_head_argmax(x0, W, cand, ids=ids_d, maxlogit=ml_d, ws=ws_d), 20)
    Xv, Wv, dv = t_bf16(verify.X), t_bf16(W_full), torch.from_numpy(d).to(dev)
    ws_v = vh.workspace(4)
    acc_v, nid_v = torch.empty(1, dtype=torch.int32, device=dev), torch.empty(4, dtype=torch.int32, device=dev)
    ml_v = torch.empty(4, dtype=torch.float32, device=dev)
    us_v = timer.time_calls(lambda: vh.spec_verify_greedy(Xv, Wv, dv, 1, 3, accept_len=acc_v, next_ids=nid_v,
                                                          row_maxlogit=ml_v, ws=ws_v), 20)
    return {"workload": "4,096 x 256 head, 1,024 candidates, B=1 x 3 draft steps; verify 1 x 4 rows (seed 1)",
            "draft_ids_equal_oracle": f"{ids_ok}/3",
            "verify_next_ids_equal_oracle": f"{int((nid.cpu().numpy() == o_nid).sum())}/4",
            "accept_len": int(acc.item()), "oracle_accept_len": int(o_acc),
            "draft_call_us": stats(us_d), "verify_call_us": stats(us_v),
            "kernels": "draft and verify k_gemv_mma_bf16 (warp MMAs fed from the weight stream)"}


def measure_verify(torch, vh, synth, timer, peaks, load_verify_golden, cuda_core=True):
    dev = torch.device("cuda")
    out = {}

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- batched greedy verify: 64 x 4 rows vs 248,320 x 2048 ----
    vc = synth.verify_case(B=64, k=3, H=2048, V=synth.V_FULL, seed_w=2, seed=4, with_head=True)
    Wf = t_bf16(vc.W)
    X = t_bf16(vc.X)
    gold = load_verify_golden()
    draft = torch.from_numpy(gold["draft"]).to(dev)
    ws = vh.workspace(256)
    acc = torch.empty(64, dtype=torch.int32, device=dev)
    nid = torch.empty(256, dtype=torch.int32, device=dev)
    ml = torch.empty(256, dtype=torch.float32, device=dev)
    paths = [(vh.VH_PATH_TENSOR, "verify")] + ([(vh.VH_PATH_CUDA_CORE, "verify_cuda_core")] if cuda_core else [])
    for path, name in paths:
        us = timer.time_calls(lambda: vh.spec_verify_greedy(X, Wf, draft, 64, 3, accept_len=acc, next_ids=nid,
                                                            row_maxlogit=ml, ws=ws, path=path),
                              5 if path == vh.VH_PATH_TENSOR else 2, warmup=2 if path == vh.VH_PATH_TENSOR else 1)
        med = statistics.median(us)
        nbytes = vc.W.nbytes + vc.X.nbytes
        flops = 2.0 * 256 * synth.V_FULL * 2048
        a = acc.cpu().numpy()
        out[name] = {
            "workload": "64 seqs x (k+1)=4 rows x 2048 bf16 vs full 248,320 x 2048 bf16 head (seeds 2/4), "
                        "draft ids = oracle greedy ids corrupted w.p. 0.45",
            "rounds_per_s": round(1e6 / med, 2), **stats(us),
            "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
            "tflops": round(flops / (med * 1e-6) / 1e12, 1),
            "tensor_frac_burst": round(flops / (med * 1e-6) / 1e12 / peaks["bf16_tflops"], 4),
            "tensor_frac_sustained": round(flops / (med * 1e-6) / 1e12 / peaks["bf16_tflops_sustained"], 4),
            "accept_hist": np.bincount(a, minlength=4).tolist(), "mean_accept": round(float(a.mean()), 4),
            "matches_stored_oracle_ids": int((nid.cpu().numpy() == gold["next_ids"]).sum()),
            "gpu_launches_per_round": 1 if path == vh.VH_PATH_TENSOR else 32,
        }
        if path == vh.VH_PATH_TENSOR:
            out[name]["kernel"] = "k_verify_tc2 (CTA pair, tcgen05 cta_group::2, fused column argmax + acceptance)"
            out[name]["dram_bytes_per_launch"] = profile_traffic("verify_tc.cu", "verify_tc2_256x248320x2048.txt")
            out[name]["algorithmic_bytes_per_launch"] = nbytes
    # fewer verified rows against the same head: B sequences x 4 positions, AUTO kernel choice
    rows = {}
    for B in (1, 4, 16, 32, 48):
        R = 4 * B
        Xs, ds = X[:R].contiguous(), draft[:B].contiguous()
        ws_r = vh.workspace(R)
        us = timer.time_calls(lambda: vh.spec_verify_greedy(Xs, Wf, ds, B, 3, ws=ws_r), 5, warmup=2)
        med = statistics.median(us)
        nbytes_r = vc.W.nbytes + R * 2048 * 2
        rows[str(R)] = {"rounds_per_s": round(1e6 / med, 1), "median_us": round(med, 2),
                        "hbm_frac": round(nbytes_r / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                        "kernel": ("k_verify_tc (one CTA, eight-stage ring)" if R <= 64 else
                                   "k_verify_tc (one CTA)" if R <= 128 else "k_verify_tc2 (CTA pair)")}
    out["verify_rows"] = rows
    del Wf, X
    return out


def measure_sweep(torch, vh, synth, timer, peaks):
    dev = torch.device("cuda")

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    sweep = {}
    for Vc in (248_320, 65_536, 32_768):
        c = synth.draft_case(Vc=Vc, H=2048, B=1, steps=1, seed=2, cand_seed=3)
        Wc = t_bf16(c.W)
        cc = torch.from_numpy(c.cand_ids).to(dev)
        x = t_bf16(c.hidden[0])
        w1 = vh.workspace(1)
        ids1 = torch.empty(1, dtype=torch.int32, device=dev)
        ml1 = torch.empty(1, dtype=torch.float32, device=dev)

        def chain():  # one MTP3 chain: three draft steps back to back
            for _ in range(3):
                vh.mtp_draft_head_argmax(x, Wc, cc, ids=ids1, maxlogit=ml1, ws=w1)

        us = [t / 3 for t in timer.time_calls(chain, 20)]
        med = statistics.mean(us)
        nbytes = Vc * 2048 * 2 + Vc * 4 + 4096
        sweep[str(Vc)] = {"steps_per_s": round(1e6 / med, 1), "timing": "3-call chains, per call", **stats(us),
                          "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
                          "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
        del Wc
    return sweep


def measure_draft_batch(torch, vh, synth, timer, peaks):
    """The bf16 draft head 65,536 x 2048 for 2 / 4 / 8 / 16 hidden rows per
    call (warp-level MMAs fed from the weight stream) and 64 (the tcgen05
    contraction), one pass each: three draft steps per chain as in the bench
    step, per call = chain / 3."""
    dev = torch.device("cuda")
    c = synth.draft_case(Vc=65_536, H=2048, B=64, steps=3, seed=2)
    Wc = torch.from_numpy(c.W.view(np.int16)).to(dev).view(torch.bfloat16)
    cc = torch.from_numpy(c.cand_ids).to(dev)
    out = {}
    for B in (2, 4, 8, 16, 64):
        xs = [torch.from_numpy(np.ascontiguousarray(h[:B]).view(np.int16)).to(dev).view(torch.bfloat16)
              for h in c.hidden]
        wsb = vh.workspace(B)
        ids = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(3)]
        mls = [torch.empty(B, dtype=torch.float32, device=dev) for _ in range(3)]

        def chain():
            for k in range(3):
                vh.mtp_draft_head_argmax(xs[k], Wc, cc, ids=ids[k], maxlogit=mls[k], ws=wsb)

        us = [t / 3 for t in timer.time_calls(chain, 20)]
        mean = statistics.mean(us)
        nbytes = 65_536 * 2048 * 2 + 65_536 * 4 + B * 2048 * 2
        out[f"B{B}"] = {"timing": "3-call chains, per call", "steps_per_s": round(1e6 / mean, 1), **stats(us),
                        "hbm_frac": round(nbytes / (mean * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                        "kernel": ("k_gemv_mma_bf16 (warp MMAs fed from the weight stream)" if B <= 16 else
                                   "k_verify_tc (tcgen05, one CTA per SM) with candidate-id mapping")}
    del Wc
    return out


def measure_mtp3_round(torch, vh, synth, timer, peaks):
    """One batch-1 MTP3 decode round as the pages run it: three draft steps on
    the 65,536 x 2048 candidate table (B = 1), each writing its id into the
    draft-id buffer, then the greedy verify of the 4 rows against the full
    248,320 x 2048 head, which reads those ids.  AUTO kernels (the tcgen05
    verify) against the same round with the warp-MMA verify."""
    dev = torch.device("cuda")
    c = synth.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    Wc = torch.from_numpy(c.W.view(np.int16)).to(dev).view(torch.bfloat16)
    cc = torch.from_numpy(c.cand_ids).to(dev)
    xs = [torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(dev).view(torch.bfloat16) for h in c.hidden]
    Wf = torch.from_numpy(synth.full_head(2, synth.V_FULL, 2048).view(np.int16)).to(dev).view(torch.bfloat16)
    X = torch.from_numpy(synth.normal_bf16(4, synth.STREAM_VHIDDEN, (4, 2048), 1.0).view(np.int16)).to(dev)
    X = X.view(torch.bfloat16)
    draft = torch.zeros(1, 3, dtype=torch.int32, device=dev)
    mld = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(3)]
    wsd, wsv = vh.workspace(1), vh.workspace(4)
    acc = torch.empty(1, dtype=torch.int32, device=dev)
    nid = torch.empty(4, dtype=torch.int32, device=dev)
    mlv = torch.empty(4, dtype=torch.float32, device=dev)
    out = {}
    for name, path in (("auto", vh.VH_PATH_AUTO), ("warp_mma_verify", vh.VH_PATH_WARP_MMA)):
        def rnd(path=path):
            for k in range(3):
                vh.mtp_draft_head_argmax(xs[k], Wc, cc, ids=draft[0, k:k + 1], maxlogit=mld[k], ws=wsd)
            vh.spec_verify_greedy(X, Wf, draft, 1, 3, accept_len=acc, next_ids=nid, row_maxlogit=mlv, ws=wsv,
                                  path=path)

        us = timer.time_calls(rnd, 20)
        mean = statistics.mean(us)
        nbytes = 3 * (65_536 * 2048 * 2 + 65_536 * 4) + synth.V_FULL * 2048 * 2
        out[name] = {"rounds_per_s": round(1e6 / mean, 1), **stats(us),
                     "hbm_frac": round(nbytes / (mean * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "kernels": "3 x k_gemv_bf16<1> + " + ("k_verify_tc" if name == "auto" else "k_gemv_mma_bf16")}
    out["workload"] = ("B = 1, k = 3: 3 draft calls on 65,536 x 2048 (one id each into the draft buffer) + verify "
                       "of 4 rows against 248,320 x 2048; one round between one pair of CUDA events, L2 flushed")
    del Wc, Wf
    return out


def measure_gather(torch, vh, synth, timer, peaks):
    """Dynamic candidate rows read in place: 32,768 fixed + 16,384 per-step
    rows of the 248,320 x 2048 head, B = 1.  Timed as the bench step is (one
    MTP3 chain of three dependent calls, each step with its own dynamic rows,
    per-call time = chain / 3) and as single calls."""
    dev = torch.device("cuda")
    W = torch.from_numpy(synth.full_head(2, synth.V_FULL, 2048).view(np.int16)).to(dev)
    rows = [torch.from_numpy(synth.gather_row_ids(6, synth.V_FULL, step=k)).to(dev) for k in range(3)]
    xs = [torch.from_numpy(h.view(np.int16)).to(dev) for h in synth.draft_hidden(2, 3, 1, 2048)]
    w1 = vh.workspace(1)
    ids = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(3)]

    def chain():
        for k in range(3):
            vh.mtp_draft_head_argmax_gather(xs[k], W, rows[k], ids=ids[k], maxlogit=mls[k], ws=w1)

    us = [t / 3 for t in timer.time_calls(chain, 20)]
    single = timer.time_calls(lambda: vh.mtp_draft_head_argmax_gather(xs[0], W, rows[0], ws=w1), 20)
    mean = statistics.mean(us)
    n = rows[0].numel()
    nbytes = n * 2048 * 2 + n * 4 + 4096
    return {"workload": "32,768 fixed + 16,384 dynamic rows gathered from 248,320 x 2048 bf16, B=1",
            "timing": "3-call chains (one per MTP3 step, own dynamic rows), per call",
            "steps_per_s": round(1e6 / mean, 1), **stats(us), "hbm_gbs": round(nbytes / (mean * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (mean * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
            "single_call_us": stats(single)}


def measure_chain_graph(torch, vh, synth, timer, peaks):
    """The 3-step draft chain (65,536 x 2048, B = 1) captured once as a CUDA
    graph and replayed (L2 flushed before each replay)."""
    dev = torch.device("cuda")
    case = synth.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    W = torch.from_numpy(case.W.view(np.int16)).to(dev)
    cand = torch.from_numpy(case.cand_ids).to(dev)
    xs = [torch.from_numpy(h.view(np.int16)).to(dev) for h in case.hidden]
    ws = vh.workspace(1)
    ids = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(3)]

    def chain():
        for i in range(3):
            vh.mtp_draft_head_argmax(xs[i], W, cand, ids=ids[i], maxlogit=mls[i], ws=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    us = timer.time_calls(g.replay, 30)
    med = statistics.median(us)
    nbytes = 3 * (case.Vc * case.H * 2 + case.Vc * 4 + case.H * 2)
    return {"workload": "3 draft steps of 65,536 x 2048 bf16, B=1, one graph replay", "us_per_chain": stats(us),
            "draft_steps_per_s": round(3e6 / med, 1), "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}


def measure_verify_nvfp4(torch, vh, synth, timer, peaks):
    """Greedy verify over 4-bit heads: 64 sequences x 4 positions against the
    full 248,320 x 2048 head (CTA-pair kernel), and 4 x 4 rows against the
    65,536 x 4096 head (16-row kernel)."""
    dev = torch.device("cuda")
    out = {}
    # full head, 256 rows
    q, s, g = synth.nvfp4_head(seed=2, V=synth.V_FULL, H=2048)
    X = synth.verify_case(B=64, k=3, H=2048, V=synth.V_FULL, seed=4, with_head=False).X
    dq, ds = torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev)
    dX = torch.from_numpy(X.view(np.int16)).to(dev)
    d = torch.from_numpy(synth.corrupt_ids(11, synth.STREAM_CORRUPT, np.zeros((64, 3), np.int32), synth.V_FULL,
                                           1.0)).to(dev)
    ws = vh.verify_nvfp4_workspace(256, 2048)
    us = timer.time_calls(lambda: vh.spec_verify_greedy_nvfp4(dX, dq, ds, g, d, 64, 3, ws=ws), 10)
    med = statistics.median(us)
    nbytes = q.nbytes + s.nbytes + X.nbytes
    flops = 2.0 * 256 * synth.V_FULL * 2048
    out["full_head_256_rows"] = {
        "workload": "64 seqs x 4 rows x 2048 bf16 vs the full 248,320 x 2048 4-bit head (seed 2; hidden seed 4; "
                    "draft ids uniform, so acceptance is not reported)",
        "kernel": "k_hidden_f16 + k_verify_fp4_pair<256> (CTA pair, exact f16 dequantisation in shared memory, tcgen05 cta_group::2)", "gpu_launches_per_round": 2,
        "rounds_per_s": round(1e6 / med, 1), **stats(us),
        "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
        "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
        "tflops": round(flops / (med * 1e-6) / 1e12, 1),
        "tensor_frac_burst": round(flops / (med * 1e-6) / 1e12 / peaks["bf16_tflops"], 4),
        "algorithmic_bytes_per_launch": nbytes,
        "dram_bytes_per_launch": profile_traffic("verify_fp4_tc.cu", "verify_fp4_pair_256x248320x2048.txt")}
    del dq, ds, dX
    # 16 rows vs the 65,536 x 4096 head
    c = synth.nvfp4_case(Vc=65_536, H=4096, B=1, steps=1, seed=5)
    q = torch.from_numpy(c.q).to(dev)
    s = torch.from_numpy(c.s).to(dev)
    X = torch.from_numpy(synth.normal_bf16(7, synth.STREAM_VHIDDEN, (16, 4096), 1.0).view(np.int16)).to(dev)
    d = torch.zeros((4, 3), dtype=torch.int32, device=dev)
    ws = vh.verify_nvfp4_workspace(16, 4096)
    us = timer.time_calls(lambda: vh.spec_verify_greedy_nvfp4(X, q, s, c.g, d, 4, 3, ws=ws), 20)
    med = statistics.median(us)
    nbytes = c.q.nbytes + c.s.nbytes + 16 * 4096 * 2
    out["head_65536x4096_16_rows"] = {
        "workload": "4 seqs x 4 rows x 4096 bf16 vs 65,536 x 4096 4-bit head", "kernel": "k_nvfp4_tc",
        "rounds_per_s": round(1e6 / med, 1), **stats(us), "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
        "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    # the same 16 and 4 rows against the tiled copy of the head
    P = vh.nvfp4_pack(q, s)
    for R in (16, 4):
        Xr, dr = X[:R].contiguous(), d[:R // 4].contiguous()
        wsr = vh.workspace(R)
        us = timer.time_calls(lambda: vh.spec_verify_greedy_nvfp4_packed(Xr, P, c.g, dr, R // 4, 3, 65_536, ws=wsr), 20)
        med = statistics.median(us)
        nbytes = c.q.nbytes + c.s.nbytes + R * 4096 * 2
        out[f"tiled_65536x4096_{R}_rows"] = {
            "workload": f"{R // 4} seqs x 4 rows x 4096 bf16 vs the tiled 65,536 x 4096 4-bit head",
            "kernel": "k_nvfp4_packed<%d>" % (2 if R > 8 else 1),
            "rounds_per_s": round(1e6 / med, 1), **stats(us), "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    del P
    # 4 rows (one MTP3 sequence) vs the same head
    X4, d1 = X[:4].contiguous(), d[:1].contiguous()
    ws = vh.verify_nvfp4_workspace(4, 4096)
    us = timer.time_calls(lambda: vh.spec_verify_greedy_nvfp4(X4, q, s, c.g, d1, 1, 3, ws=ws), 20)
    med = statistics.median(us)
    nbytes = c.q.nbytes + c.s.nbytes + 4 * 4096 * 2
    out["head_65536x4096_4_rows"] = {
        "workload": "1 seq x 4 rows x 4096 bf16 vs 65,536 x 4096 4-bit head", "kernel": "k_nvfp4_mma",
        "rounds_per_s": round(1e6 / med, 1), **stats(us), "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
        "hbm_frac": round(nbytes / (med * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
    return out


def measure_nvfp4(torch, vh, synth, timer, peaks):
    """4-bit draft head 65,536 x 4096 at B = 1, 8 and 16: three draft steps
    per chain as in the bench step (per call = chain / 3), and single calls.
    The head is converted once to the tiled layout (vh_nvfp4_pack, as a model
    loader would) and scored with mtp_draft_head_argmax_nvfp4_packed, which
    reads the same bytes per call; the row-major call is timed beside it."""
    dev = torch.device("cuda")

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    nv, rm = {}, {}
    c = synth.nvfp4_case(Vc=65_536, H=4096, B=16, steps=3, seed=5)
    q = torch.from_numpy(c.q).to(dev)
    s = torch.from_numpy(c.s).to(dev)
    cc = torch.from_numpy(c.cand_ids).to(dev)
    P = vh.nvfp4_pack(q, s)
    for B in (1, 8, 16):
        xs = [t_bf16(h[:B]) for h in c.hidden]
        wsb = vh.workspace(B)
        ids = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(3)]
        mls = [torch.empty(B, dtype=torch.float32, device=dev) for _ in range(3)]
        nbytes = c.q.nbytes + c.s.nbytes + 65_536 * 4 + B * 4096 * 2
        for layout in ("tiled", "row_major"):
            if layout == "row_major" and B == 16:
                continue

            def one(k, layout=layout):
                if layout == "tiled":
                    vh.mtp_draft_head_argmax_nvfp4_packed(xs[k], P, c.g, cc, ids=ids[k], maxlogit=mls[k], ws=wsb)
                else:
                    vh.mtp_draft_head_argmax_nvfp4(xs[k], q, s, c.g, cc, ids=ids[k], maxlogit=mls[k], ws=wsb)

            def chain():
                for k in range(3):
                    one(k)

            us = [t / 3 for t in timer.time_calls(chain, 20)]
            single = timer.time_calls(lambda: one(0), 20)
            mean = statistics.mean(us)
            entry = {"timing": "3-call chains, per call", "steps_per_s": round(1e6 / mean, 1), **stats(us),
                     "hbm_gbs": round(nbytes / (mean * 1e-6) / 1e9, 1),
                     "hbm_frac": round(nbytes / (mean * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "single_call_us": stats(single),
                     "kernel": ("k_nvfp4_packed<%d> (tiled layout, warp-level MMAs)" % (1 if B <= 8 else 2))
                     if layout == "tiled" else ("k_gemv_nvfp4_xs" if B == 1 else "k_nvfp4_mma")}
            if layout == "tiled":
                entry["algorithmic_bytes_per_launch"] = nbytes
                nv[f"B{B}"] = entry
            else:
                rm[f"B{B}"] = entry
    nv["row_major"] = rm
    return nv

def run_single(args):
    """One of the extra measurements on its own (a short profiling target)."""
    import torch
    import synth
    import verify_head_gb300 as vh
    vh.lib()
    peaks, _ = load_peaks()
    timer = Timer(torch)
    out = measure_extra(torch, vh, synth, timer, peaks, load_verify_golden, only=args.workload)
    print(json.dumps(out), flush=True)


def cpu_baseline(case, seconds: float = 10.0, threads: int | None = None):
    """The oracle, as it stands, on the host cores: whole draft steps of the
    same workload until about `seconds` of CPU time have passed."""
    import oracle
    oracle.build()
    threads = threads or oracle.threads()
    n = 0
    first = []
    t0 = time.perf_counter()
    while True:
        r = oracle.draft_argmax(case.hidden[n % 3], case.W, case.cand_ids, nthreads=threads)
        if n < 3:
            first.append(r)
        n += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    # the same oracle on one thread, over a shorter sample
    n1, t1 = 0, time.perf_counter()
    while True:
        oracle.draft_argmax(case.hidden[n1 % 3], case.W, case.cand_ids, nthreads=1)
        n1 += 1
        if time.perf_counter() - t1 > min(3.0, seconds / 3):
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(n / dt, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} whole draft steps (65,536 x 2048 bf16 head, B=1) in {dt:.1f} s",
            "single_thread": {"value": round(n1 / dt1, 3), "unit": UNIT, "cores": 1,
                              "sample": f"{n1} whole draft steps in {dt1:.1f} s"}}, first


def run_reference(args):
    """The CPU oracle timed on this workload (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    threads = args.oracle_threads or oracle.threads()
    case = synth.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    for _ in range(max(1, min(args.warmup, 2))):
        oracle.draft_argmax(case.hidden[0], case.W, case.cand_ids, nthreads=threads)
    per_step = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for i in range(3):
            oracle.draft_argmax(case.hidden[i], case.W, case.cand_ids, nthreads=threads)
        per_step.append(time.perf_counter() - t0)
    total = sum(per_step)
    value = 3 * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "Vc": case.Vc, "H": case.H, "B": case.B},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} bench steps x 3 whole draft steps"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-extra", action="store_true", help="omit the verify / sweep / 4-bit measurements")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle baseline")
    ap.add_argument("--workload", default="all",
                    choices=["all", "tiny", "draft", "verify", "sweep", "nvfp4", "gather", "chain", "verify_nvfp4",
                             "draft_batch", "mtp3_round"],
                    help="all = the bench line; others run one measurement only (for profiling)")
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5],
                    help="one workload by number: 1 tiny oracle check, 2 draft head 65,536 x 2048, "
                         "3 head-size sweep, 4 batched verify, 5 4-bit draft head")
    ap.add_argument("--oracle-threads", type=int, default=None, help="host threads for the CPU oracle")
    args = ap.parse_args()
    if args.config is not None:
        args.workload = {1: "tiny", 2: "draft", 3: "sweep", 4: "verify", 5: "nvfp4"}[args.config]
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "ours" and args.workload not in ("all", "draft"):
        run_single(args)
        return
    if args.impl == "reference":
        args.steps = max(1, min(args.steps, 50))  # bounded: ~0.1-0.5 s of CPU per draft step
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
