#!/usr/bin/env python
"""Throughput of the branch-packed scoring hot path on one or more GB300s.

Workload (default): the Wikinews-shaped job -- 24 contents of 400-540 tokens
sharing 56 two-option questions of 8-16 tokens, plus one floor per question,
packed into two 16384-token passes; Gemma-12B-class attention (16 query heads,
8 kv heads, d_head 256) and lm head (d_model 3840, vocabulary 262144, bf16).
Inputs are synthetic (seeded) and resident in HBM before the timed region.

One step = the whole job: per pass, tree-masked attention (one layer) and slot
scoring (gather, lm head with full-vocabulary log-sum-exp, option log-probs),
then the token log-probs to the host and the per-option collect.  The layout
(planner output) is part of the resident input; the planner, the descriptor
upload and every host<->device copy of the activations are inside the ``e2e``
number, measured through the public API with host buffers.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same job and extrapolates to the whole job.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
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

METRIC = "packed tokens/s and scored questions/s per GB300; % of tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) of one score_main_kernel launch of the step (every pass's slot
# rows in one sweep), from one ncu capture of the current kernel.  Keyed by (workload, fp8);
# any other case reports null.
NCU_SCORE_TRAFFIC = {("wikinews", False): 2024229376 + 14412032}
# DRAM bytes (read + write) per step of the attention kernel (both passes of the job), from
# ncu captures of the current kernel; any other workload reports null.
NCU_ATTN_TRAFFIC = {"wikinews": None}   # pass 0 only was captured: see per-pass figure below
# DRAM bytes (read + write) of one attention launch on the Wikinews-shaped pass 0, from one ncu
# capture of the current kernel (408.1 MB read, 105.6 MB written)
NCU_ATTN_TRAFFIC_PASS0 = {"wikinews": 408090624 + 105582848}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _burst_peaks():
    """(bf16 TFLOP/s, HBM GB/s, label): the burst bf16 GEMM figure, since every kernel here is
    timed inside steps of a few milliseconds (a sub-second region), not a seconds-long loop."""
    peaks, src = _peaks()
    bf16 = _peak_value(peaks, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    hbm = _peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    return bf16, hbm, f"{src} bf16_tflops (burst; x2 for e4m3) and hbm_gbs"


def _peak_value(d, *names):
    for n in names:
        for k, v in d.items():
            if k == n and isinstance(v, (int, float)):
                return float(v)
    for n in names:   # nested forms, e.g. {"bf16_tflops": {"value": ...}}
        v = d.get(n)
        if isinstance(v, dict):
            for kk in ("value", "median", "max"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


class ClockSampler:
    """SM clock and clock-event reasons during the timed region: NVML (the driver's
    libnvidia-ml, read-only queries) polled every 2 ms from a thread, else nvidia-smi at 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of the NVML API
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, index):
        self.index = index
        self.f = None
        self.p = None
        self.nvml = None
        self.thread = None
        self.samples = []
        self.stop_flag = False
        try:
            self.nvml = self._nvml_handle(index)
        except Exception:
            self.nvml = None

    @staticmethod
    def _nvml_handle(index):
        import ctypes

        import torch

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        prop = torch.cuda.get_device_properties(index)
        bus = f"{prop.pci_domain_id:08X}:{prop.pci_bus_id:02X}:{prop.pci_device_id:02X}.0".encode()
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _poll(self):
        import ctypes

        lib, h, reasons = self.nvml
        mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
        while not self.stop_flag:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and reasons(h, ctypes.byref(bits)) == 0:
                self.samples.append((mhz.value, mx.value, bits.value))
            time.sleep(0.002)

    def start(self):
        if self.nvml is not None:
            import threading

            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 1.0:   # the first sample precedes the region
                time.sleep(0.001)
            return
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=1.0)
            sm = [s[0] for s in self.samples]
            reasons = {n for _, _, b in self.samples for bit, n in self.REASONS.items() if b & bit}
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": max(s[1] for s in self.samples) if sm else None,
                    "samples": len(sm), "source": "nvml, 2 ms", "reasons": sorted(reasons)}
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "source": "nvidia-smi, 200 ms", "reasons": sorted(reasons)}


def max_over_ranks(ms, world, device):
    """The slowest rank's step time (the only collective of the replica path)."""
    if world <= 1:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_value(tokens_per_replica, world, ms):
    """Whole-job throughput: every rank runs its own replica of the job (weak scaling)."""
    return world * tokens_per_replica / (ms * 1e-3)


def build_job(workload, device, spinf, sv, wl, w_dtype):
    f, shape = wl.WORKLOADS[workload]
    inputs = f()
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    passes = []
    for p in range(plan.num_passes):
        info = plan.pass_info(p)
        keys = sv.path_keys(info.tok, info.parent, info.T)
        q, k, v = sv.qkv(keys, info.T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
        h = sv.hidden(keys, info.T_pad, shape.d_model, rows=info.slot_row.tolist())
        passes.append({"info": info, "host": (q, k, v, h)})
    w = sv.lm_head(shape.vocab, shape.d_model, device=device)
    w_scale = None
    if w_dtype == spinf.DTYPE_E4M3:
        w, w_scale = sv.e4m3_rows(w)
    return inputs, shape, plan, passes, w, w_scale


def work_counts(inputs, plan, passes, shape):
    """Tokens, user questions, unmasked attention pairs and scoring FLOPs of the job."""
    import numpy as np

    tokens = sum(p["info"].T for p in passes)
    questions = sum(len(qs) for _, qs in inputs)
    pairs = 0
    flops_score = 0
    for p in passes:
        info = p["info"]
        T = info.T
        end = info.end[:T].astype(np.int64)
        pairs += int((end - np.arange(T)).sum())     # key k is seen by rows [k, end[k])
        flops_score += 2 * info.M * shape.vocab * shape.d_model
    flops_attn = 4 * shape.d_head * shape.n_q_heads * pairs
    bytes_attn = sum(p["info"].T for p in passes) * (2 * shape.n_q_heads + 2 * shape.n_kv_heads) * shape.d_head * 2
    return tokens, questions, pairs, flops_attn, bytes_attn, flops_score


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import branch_packed_scoring_gb300 as spinf
    from synth import values as sv
    from synth import workloads as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    w_dtype = spinf.DTYPE_E4M3 if args.fp8 else spinf.DTYPE_BF16
    inputs, shape, plan, passes, w, w_scale = build_job(args.workload, dev, spinf, sv, wl, w_dtype)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for pi, p in enumerate(passes):
            info = p["info"]
            q, k, v, h = (t.to(dev) for t in p["host"])
            p["dev"] = (q, k, v, h)
            p["o"] = torch.empty_like(q)
            plan.upload(pi, stream)
            nbytes = spinf.score_workspace_bytes(plan, pi, shape.vocab, shape.d_model, w_dtype)
            p["ws"] = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            p["lse"] = torch.empty(max(info.M, 1), device=dev)
            p["tlp"] = torch.empty(max(info.G, 1), device=dev)
            p["tlp_host"] = torch.empty(max(info.G, 1), dtype=torch.float32, pin_memory=True)
    all_passes = list(range(len(passes)))
    ws_all = torch.empty(spinf.score_passes_workspace_bytes(plan, all_passes, shape.vocab, shape.d_model, w_dtype),
                         dtype=torch.uint8, device=dev)
    stream.synchronize()
    tokens, questions, pairs, flops_attn, bytes_attn, flops_score = work_counts(inputs, plan, passes, shape)
    sched_tiles = sum(int(p["info"].n_sched) for p in passes)
    # the KV tiles the attention kernel executes: 64-key halves at d_head 256, else 128 keys
    key_tile, q_rows = exec_tiling(shape)
    exec_tiles = sum(len(plan.tile_schedule(pi, 0, key_tile, q_rows)[1]) for pi in range(len(passes)))

    ev = {"attn": [], "score": []}

    for p in passes:   # two host buffers: step r + 1's copy lands while step r's results are collected
        p["tlp_host2"] = [p["tlp_host"], torch.empty_like(p["tlp_host"]).pin_memory()]

    def launch(r, record=False):
        """Step r's GPU work: the attention of every pass, one scoring sweep over all passes'
        slot rows, the token lps to host buffer r % 2; returns the event of its end."""
        for pi, p in enumerate(passes):
            q, k, v, h = p["dev"]
            if record:
                a0, a1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
                a0.record(stream)
            spinf.branch_attention(plan, pi, q, k, v, p["o"], shape.n_q_heads, shape.n_kv_heads, shape.d_head,
                                   stream=stream)
            if record:
                a1.record(stream)
                ev["attn"].append((a0, a1))
        if record:
            s0, s1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            s0.record(stream)
        spinf.score_passes(plan, all_passes, [p["dev"][3] for p in passes], w, w_scale, w_dtype, shape.d_model,
                           shape.vocab, [p["lse"] for p in passes], [p["tlp"] for p in passes], ws_all, stream=stream)
        if record:
            s1.record(stream)
            ev["score"].append((s0, s1))
        for p in passes:
            p["tlp_host2"][r % 2].copy_(p["tlp"], non_blocking=True)
        done = torch.cuda.Event()
        done.record(stream)
        return done

    def finish(r, done):
        """Step r's collect on the host, once its GPU work is done."""
        done.synchronize()
        return plan.collect([p["tlp_host2"][r % 2][:p["info"].G].numpy() for p in passes])

    def run_steps(n, record=False):
        # step r + 1's GPU work is enqueued before step r's results are collected, so the GPU
        # is not idle while the host collects (two steps in flight, as a server would run them)
        prev = launch(0, record)
        for r in range(1, n):
            cur = launch(r, record)
            finish(r - 1, prev)
            prev = cur
        return finish(n - 1, prev)

    run_steps(args.warmup)
    plan.device_status(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    res = run_steps(args.steps, record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end) / args.steps
    plan.device_status(stream)
    assert np.isfinite(res["option_lp"]).all()
    ms = max_over_ranks(ms, world, dev)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev["attn"]) * len(passes)
    score_ms = statistics.mean(a.elapsed_time(b) for a, b in ev["score"])

    def per_step_stats(pairs, per_step):
        """median and min over steps of the per-step sum of ``per_step`` intervals (ms)."""
        t = [a.elapsed_time(b) for a, b in pairs]
        steps = [sum(t[i:i + per_step]) for i in range(0, len(t), per_step)]
        return {"median": statistics.median(steps), "min": min(steps)}

    attn_stats, score_stats = per_step_stats(ev["attn"], len(passes)), per_step_stats(ev["score"], 1)
    # The step's kernels again, back to back with no host work between steps (still cold: the
    # scoring sweep reads the 2 GB lm head between attention calls).  Reported beside the timed
    # region's own figures, which the roofline uses: the pipelined steps keep the host ahead of the
    # GPU, so those events time the kernels alone too, and this longer unbroken run can meet the
    # power cap's lower clocks, which the clock samples of the timed region do not see.
    bev = {"attn": [], "score": []}
    clocks_b2b = ClockSampler(torch.cuda.current_device())
    clocks_b2b.start()
    with torch.cuda.stream(stream):
        for r in range(max(4, args.steps) + 1):
            for pi, p in enumerate(passes):
                q, k, v, h = p["dev"]
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                spinf.branch_attention(plan, pi, q, k, v, p["o"], shape.n_q_heads, shape.n_kv_heads, shape.d_head,
                                       stream=stream)
                a1.record(stream)
                if r:
                    bev["attn"].append((a0, a1))
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            spinf.score_passes(plan, all_passes, [p["dev"][3] for p in passes], w, w_scale, w_dtype, shape.d_model,
                               shape.vocab, [p["lse"] for p in passes], [p["tlp"] for p in passes], ws_all,
                               stream=stream)
            s1.record(stream)
            if r:
                bev["score"].append((s0, s1))
    torch.cuda.synchronize()
    clk_b2b = clocks_b2b.stop()
    plan.device_status(stream)
    attn_b2b = per_step_stats(bev["attn"], len(passes))["median"]
    score_b2b = per_step_stats(bev["score"], 1)["median"]
    # for comparison: the same scoring as one spinf_score call per pass (each pads its own last
    # 128-row tile and reads the whole lm head)
    pev = []
    with torch.cuda.stream(stream):
        for r in range(max(3, args.steps // 2) + 1):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for pi, p in enumerate(passes):
                spinf.score(plan, pi, p["dev"][3], w, w_scale, w_dtype, shape.d_model, shape.vocab, p["lse"],
                            p["tlp"], p["ws"], stream=stream)
            a1.record(stream)
            if r:
                pev.append((a0, a1))
    torch.cuda.synchronize()
    score_per_pass_ms = statistics.median(a.elapsed_time(b) for a, b in pev)
    # the attention call again right after itself on the same pass (its q/k/v partly in L2): the
    # step's figure is the cold one (every pass's inputs exceed L2 and the lm head flushes it)
    warm = []
    with torch.cuda.stream(stream):
        for pi, p in enumerate(passes):
            q, k, v, _h = p["dev"]
            for r in range(4):
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                spinf.branch_attention(plan, pi, q, k, v, p["o"], shape.n_q_heads, shape.n_kv_heads, shape.d_head,
                                       stream=stream)
                a1.record(stream)
                if r:
                    warm.append((a0, a1))
    torch.cuda.synchronize()
    attn_warm_ms = statistics.median(a.elapsed_time(b) for a, b in warm) * len(passes)
    # workloads whose alternate layers use a sliding window: the windowed attention call is
    # timed too (outside the step; the step holds one unwindowed layer)
    attn_win_ms = None
    if shape.window > 0:
        wev = []
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.steps)):
                for pi, p in enumerate(passes):
                    q, k, v, _h = p["dev"]
                    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a0.record(stream)
                    spinf.branch_attention(plan, pi, q, k, v, p["o"], shape.n_q_heads, shape.n_kv_heads,
                                           shape.d_head, window=shape.window, stream=stream)
                    a1.record(stream)
                    wev.append((a0, a1))
        torch.cuda.synchronize()
        plan.device_status(stream)
        attn_win_ms = statistics.mean(a.elapsed_time(b) for a, b in wev) * len(passes)

    layer = None if args.no_layer else layer_timing(args, spinf, shape, plan, passes, dev, stream)
    per_workload = None if args.no_per_workload else per_workload_timing(args, spinf, wl, dev, stream)
    extract = None if args.no_extract else extract_timing(args, spinf, sv, wl, inputs, shape, w, w_scale, w_dtype,
                                                          dev, stream)

    # end to end through the public API with host buffers
    e2e = run_e2e(args, spinf, inputs, shape, passes, w, w_scale, w_dtype, dev, res) if not args.no_e2e else None

    bf16_peak, hbm_peak, peak_label = _burst_peaks()
    mma_peak = bf16_peak * (2.0 if args.fp8 else 1.0)
    # average launch durations over the timed region (CUDA events on the launching stream)
    score_tflops = flops_score / (score_ms * 1e-3) / 1e12
    attn_tflops = flops_attn / (attn_ms * 1e-3) / 1e12
    attn_gbs = bytes_attn / (attn_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC,
        "value": replica_value(tokens, world, ms),
        "unit": "packed tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if not args.fp8 else "e4m3",
        "data": "synthetic",
        "scored_questions_per_s": world * questions / (ms * 1e-3),
        "config": {**_config(args, inputs, len(passes), tokens, questions, shape, world),
                   "value_covers": "per step: attention per pass + one scoring sweep over every pass's slot rows, "
                                   "token-lp D2H, collect on the host; step r+1's GPU work is enqueued before "
                                   "step r's collect (two steps in flight); layout resident"},
        "roofline": {"kernel": "spinf_score_passes (gather + tcgen05 lm head + lse + combine, all passes)",
                     "timing": "CUDA events per launch on the launching stream over the timed region, mean "
                               "(kernel_ms_per_step.score); launches back to back in a separate loop: "
                               "kernel_ms_per_step.score_back_to_back",
                     "bound": "tensor",
                     "achieved": score_tflops, "peak": mma_peak, "unit": "TFLOP/s",
                     "frac": score_tflops / mma_peak,
                     "traffic": NCU_SCORE_TRAFFIC.get((args.workload, bool(args.fp8))),
                     "peak_source": peak_label},
        "roofline_attention": {"kernel": "spinf_branch_attention", "tensor_tflops_unmasked": attn_tflops,
                               "tensor_frac": attn_tflops / bf16_peak, "hbm_gbs": attn_gbs,
                               "hbm_frac": attn_gbs / hbm_peak, "unmasked_pairs": pairs,
                               "tile_occupancy": pairs / (exec_tiles * q_rows * key_tile), "q_rows": q_rows,
                               "key_tile": key_tile, "executed_kv_tiles": exec_tiles,
                               "tile_occupancy_128x128": pairs / (sched_tiles * 128 * 128),
                               "traffic": NCU_ATTN_TRAFFIC.get(args.workload),
                               "traffic_pass0": NCU_ATTN_TRAFFIC_PASS0.get(args.workload),
                               "compulsory_bytes_pass0": passes[0]["info"].T_pad * (2 * shape.n_q_heads
                                                                                     + 2 * shape.n_kv_heads)
                               * shape.d_head * 2,
                               "compulsory_bytes": bytes_attn,
                               "peak_source": peak_label},
        # per kernel: packed tokens per attention-kernel second
        # (one layer call per pass) and user questions per scoring second (gather + main + combine)
        "per_kernel": {"attention_packed_tokens_per_s": world * tokens / (attn_ms * 1e-3),
                       "scoring_questions_per_s": world * questions / (score_ms * 1e-3),
                       "timing": "CUDA events per launch over the timed region (the host ahead of the GPU)",
                       "user_questions": questions, "packed_tokens": tokens},
        "kernel_ms_per_step": {"attention": attn_ms, "score": score_ms,
                               "attention_median": attn_stats["median"], "attention_min": attn_stats["min"],
                               "score_median": score_stats["median"], "score_min": score_stats["min"],
                               "score_one_call_per_pass": score_per_pass_ms,
                               "attention_back_to_back": attn_b2b, "score_back_to_back": score_b2b,
                               "clocks_back_to_back": clk_b2b,
                               "attention_l2_warm": attn_warm_ms,
                               **({"attention_windowed": attn_win_ms, "window": shape.window} if attn_win_ms else {})},
        "searched_slots": extract,
        "layer_projections": layer,
        "per_workload": per_workload,
        "clocks": clk,
        "gpu_launches": (len(passes) + 3) * args.steps,   # attention per pass; gather, lm head, combine
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, inputs, shape, plan, passes, w, w_scale, budget_s=args.cpu_seconds)
    return out


def layer_timing(args, spinf, shape, plan, passes, dev, stream):
    """The projections around the attention call on every pass of the job (outside the
    step): the QKV projection with the rotary turn fused (spinf_qkv_rope) and the output
    projection (spinf_linear), bf16 and e4m3 with static scales, seeded random weights of
    the workload's shapes.  Tensor-bound: 2 * T_pad * in * out FLOPs per call."""
    import torch

    Hq, Hkv, d, D = shape.n_q_heads, shape.n_kv_heads, shape.d_head, shape.d_model
    n_qkv, n_o = (Hq + 2 * Hkv) * d, Hq * d
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    w_qkv = (torch.randn(n_qkv, D, generator=g, device=dev) / D ** 0.5).to(torch.bfloat16)
    w_o = (torch.randn(D, n_o, generator=g, device=dev) / n_o ** 0.5).to(torch.bfloat16)

    def e4m3(w):
        s_w = (w.float().abs().amax(dim=1) / 448.0).clamp_min(1e-12)
        return (w.float() / s_w[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8), s_w

    wq8, sq8 = e4m3(w_qkv)
    wo8, so8 = e4m3(w_o)
    x_scale, o_scale = 5.0 / 448, 4.0 / 448   # static activation scales (calibration stand-ins)
    bufs = []
    for pi, p in enumerate(passes):
        Tp = p["info"].T_pad
        x = torch.randn(Tp, D, generator=g, device=dev).to(torch.bfloat16)
        bufs.append({"x": x, "x8": torch.empty(Tp, D, dtype=torch.uint8, device=dev),
                     "o8": torch.empty(Tp, n_o, dtype=torch.uint8, device=dev),
                     "q": torch.empty(Tp, Hq, d, dtype=torch.bfloat16, device=dev),
                     "k": torch.empty(Tp, Hkv, d, dtype=torch.bfloat16, device=dev),
                     "v": torch.empty(Tp, Hkv, d, dtype=torch.bfloat16, device=dev),
                     "y": torch.empty(Tp, D, dtype=torch.bfloat16, device=dev)})
    torch.cuda.synchronize()
    reps = max(3, args.steps // 2)

    def timed(fn):
        for pi, b in enumerate(bufs):   # warm-up
            fn(pi, b)
        ev = []
        for _ in range(reps):
            for pi, b in enumerate(bufs):
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                fn(pi, b)
                a1.record(stream)
                ev.append((a0, a1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * len(bufs)

    def qkv16(pi, b):
        spinf.qkv_rope(plan, pi, b["x"], w_qkv, b["q"], b["k"], b["v"], Hq, Hkv, d, stream=stream)

    def o16(pi, b):
        spinf.linear(plan, b["q"].view(-1, n_o), w_o, b["y"], stream=stream)

    def quant(pi, b):
        spinf.quantize_static(b["x"], x_scale, b["x8"], stream=stream)

    def qkv8(pi, b):
        spinf.qkv_rope(plan, pi, b["x8"], wq8, b["q"], b["k"], b["v"], Hq, Hkv, d, w_scale=sq8, x_scale=x_scale,
                       w_dtype=spinf.DTYPE_E4M3, stream=stream)

    def o8(pi, b):
        spinf.linear(plan, b["o8"], wo8, b["y"], w_scale=so8, x_scale=o_scale, w_dtype=spinf.DTYPE_E4M3,
                     stream=stream)

    with torch.cuda.stream(stream):
        for b in bufs:   # the e4m3 output projection reads codes of the attention output's shape
            spinf.quantize_static(b["q"].view(-1, n_o), o_scale, b["o8"], stream=stream)
        ms = {"qkv_rope_bf16": timed(qkv16), "o_proj_bf16": timed(o16), "quantize_x": timed(quant),
              "qkv_rope_e4m3": timed(qkv8), "o_proj_e4m3": timed(o8)}
    plan.device_status(stream)
    rows = sum(p["info"].T_pad for p in passes)
    fl_qkv, fl_o = 2.0 * rows * D * n_qkv, 2.0 * rows * n_o * D
    bf16_peak = _burst_peaks()[0]
    tf = {k: (fl_qkv if k.startswith("qkv") else fl_o) / (v * 1e-3) / 1e12 for k, v in ms.items() if k != "quantize_x"}
    return {"shapes": f"rows {rows} (all passes), QKV {D}->{n_qkv}, O {n_o}->{D}",
            "ms": ms, "tflops": tf,
            "frac": {k: v / (bf16_peak * (2.0 if k.endswith("e4m3") else 1.0)) for k, v in tf.items()}}


def exec_tiling(shape):
    """(keys per KV tile, rows per Q tile) the attention kernel executes for these heads:
    64-key tiles at d_head 256, on 64-row Q tiles when each kv head serves two query heads
    (both heads stacked in the MMA's 128 rows)."""
    if shape.d_head != 256:
        return 128, 128
    return 64, (64 if shape.n_q_heads == 2 * shape.n_kv_heads else 128)


def pass_pairs(info, window=0):
    """Unmasked (row, key) pairs of one pass: key k is seen by the rows [k, end[k]) whose depth
    is within the window (pos[q] - pos[k] < window; 0: no window)."""
    import numpy as np

    T = info.T
    end = info.end[:T].astype(np.int64)
    if window <= 0:
        return int((end - np.arange(T)).sum())
    pos = info.pos[:T].astype(np.int64)
    return int(sum(int((pos[k:end[k]] - pos[k] < window).sum()) for k in range(T)))


def per_workload_timing(args, spinf, wl, dev, stream, reps=3):
    """The other workloads of the scope table, timed outside the headline step: the
    moderation-shaped job (plus its 1024-token windowed layer), the many-questions stress job
    at Qwen-class shapes (plus a window that bites), one packing of the batch-invariance
    pass (2000 short inputs + the 470-token target) with the e4m3 per-row-scaled lm head, and
    the Wikinews job asked as placeholder grids (with the host planning time of the grid
    request and of the same questions written out).
    Values are seeded N(0, 1) bf16 drawn on the device (the path-keyed values change no
    amount of work); one attention call per pass and one scoring sweep over every pass's
    slot rows, ``reps`` times."""
    import torch

    bf16_peak, hbm_peak, _ = _burst_peaks()
    cases = [("moderation", False), ("stress", False), ("invariance_e4m3", True), ("wikinews_grid", False)]
    out = {}
    g = torch.Generator(device=dev)
    g.manual_seed(11)

    def plan_ms(inputs, vocab, n=5):
        """median host time to marshal and plan a request (ms)"""
        ts = []
        for _ in range(n):
            t0 = time.perf_counter()
            spinf.Plan(inputs, vocab=vocab).close()
            ts.append((time.perf_counter() - t0) * 1e3)
        return statistics.median(ts)

    for name, fp8 in cases:
        extra = {}
        if name == "invariance_e4m3":
            inputs, _ = wl.invariance_packing(1)
            shape = wl.GEMMA
        elif name == "wikinews_grid":   # the Wikinews job with its questions as one grid per content
            inputs, shape = wl.wikinews_grid(), wl.GEMMA
            extra = {"grid": "per content: 2 placeholders of 7 and 8 values -> 56 cells, 2 single-token options",
                     "host_plan_ms": plan_ms(inputs, shape.vocab),
                     "host_plan_ms_written_out": plan_ms(wl.written_out(inputs), shape.vocab)}
        else:
            f, shape = wl.WORKLOADS[name]
            inputs = f()
        plan = spinf.Plan(inputs, vocab=shape.vocab)
        w_dtype = spinf.DTYPE_E4M3 if fp8 else spinf.DTYPE_BF16
        w = (torch.randn(shape.vocab, shape.d_model, generator=g, device=dev) / shape.d_model ** 0.5).to(torch.bfloat16)
        w_scale = None
        if fp8:
            w, w_scale = _e4m3_rows_dev(w)
        bufs = []
        Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.d_head
        for pi in range(plan.num_passes):
            info = plan.pass_info(pi)
            Tp = info.T_pad
            mk = lambda *sz: torch.randn(*sz, generator=g, device=dev).to(torch.bfloat16)  # noqa: E731
            b = {"info": info, "q": mk(Tp, Hq, d), "k": mk(Tp, Hkv, d), "v": mk(Tp, Hkv, d), "h": mk(Tp, shape.d_model),
                 "lse": torch.empty(max(info.M, 1), device=dev), "tlp": torch.empty(max(info.G, 1), device=dev)}
            b["o"] = torch.empty_like(b["q"])
            plan.upload(pi, stream)
            bufs.append(b)
        all_p = list(range(len(bufs)))
        ws = torch.empty(spinf.score_passes_workspace_bytes(plan, all_p, shape.vocab, shape.d_model, w_dtype),
                         dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

        def timed(fn, per_pass=True):
            """mean ms of one call per pass (summed over the passes), or of one call for all"""
            units = list(enumerate(bufs)) if per_pass else [(None, None)]
            for pi, b in units:   # warm-up
                fn(pi, b)
            ev = []
            for _ in range(reps):
                for pi, b in units:
                    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a0.record(stream)
                    fn(pi, b)
                    a1.record(stream)
                    ev.append((a0, a1))
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in ev) * len(units)

        def attn(window):
            return lambda pi, b: spinf.branch_attention(plan, pi, b["q"], b["k"], b["v"], b["o"], Hq, Hkv, d,
                                                        window=window, stream=stream)

        def score(_pi, _b):   # one sweep over every pass's slot rows
            spinf.score_passes(plan, all_p, [b["h"] for b in bufs], w, w_scale, w_dtype, shape.d_model, shape.vocab,
                               [b["lse"] for b in bufs], [b["tlp"] for b in bufs], ws, stream=stream)

        with torch.cuda.stream(stream):
            t_attn, t_score = timed(attn(0)), timed(score, per_pass=False)
            t_win = timed(attn(shape.window)) if shape.window > 0 else None
        plan.device_status(stream)
        key_tile, q_rows = exec_tiling(shape)
        tokens = sum(b["info"].T for b in bufs)
        rows = sum(b["info"].M for b in bufs)
        questions = plan.counts()[0]
        pairs = sum(pass_pairs(b["info"]) for b in bufs)
        tiles = sum(len(plan.tile_schedule(pi, 0, key_tile, q_rows)[1]) for pi in range(len(bufs)))
        fl_attn = 4 * d * Hq * pairs
        by_attn = tokens * (2 * Hq + 2 * Hkv) * d * 2
        fl_score = 2 * rows * shape.vocab * shape.d_model
        mma_peak = bf16_peak * (2.0 if fp8 else 1.0)
        e = {**extra, "inputs": len(inputs), "user_questions": questions, "passes": len(bufs), "packed_tokens": tokens,
             "scoring_rows": rows, "shape": f"Hq={Hq} Hkv={Hkv} d_head={d} d_model={shape.d_model} V={shape.vocab}",
             "lm_head": "e4m3 per-row scaled" if fp8 else "bf16",
             "ms": {"attention": t_attn, "score": t_score, "step": t_attn + t_score},
             "packed_tokens_per_s": tokens / ((t_attn + t_score) * 1e-3),
             "scored_questions_per_s": questions / (t_score * 1e-3),
             "tile_occupancy": pairs / (tiles * q_rows * key_tile), "key_tile": key_tile, "q_rows": q_rows,
             "roofline": {"attention_tensor_frac": fl_attn / (t_attn * 1e-3) / 1e12 / bf16_peak,
                          "attention_hbm_frac": by_attn / (t_attn * 1e-3) / 1e9 / hbm_peak,
                          "score_tensor_frac": fl_score / (t_score * 1e-3) / 1e12 / mma_peak,
                          "score_peak_tflops": mma_peak}}
        if t_win is not None:
            pw = sum(pass_pairs(b["info"], shape.window) for b in bufs)
            tw = sum(len(plan.tile_schedule(pi, shape.window, key_tile, q_rows)[1]) for pi in range(len(bufs)))
            e["windowed"] = {"window": shape.window, "attention_ms": t_win, "unmasked_pairs": pw,
                             "tile_occupancy": pw / (tw * q_rows * key_tile),
                             "attention_tensor_frac": 4 * d * Hq * pw / (t_win * 1e-3) / 1e12 / bf16_peak}
        out[name] = e
        del bufs, w, w_scale, ws
        torch.cuda.empty_cache()
    return out


def _e4m3_rows_dev(w):
    """Per-row e4m3 codes and scales of a device lm head (absmax / 448, round to nearest even)."""
    import torch

    s_w = w.float().abs().amax(dim=1)
    s_w = torch.where(s_w == 0, torch.ones_like(s_w), s_w / 448.0)
    codes = (w.float() / s_w[:, None]).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, s_w.contiguous()


def extract_timing(args, spinf, sv, wl, inputs, shape, w, w_scale, w_dtype, dev, stream, n_slots=2):
    """Scoring with searched slots: every input also gets ``n_slots`` searched slots ({*} over
    any token, {n} over a 1% token set).  Times the scoring call of the same plan with and
    without the searched-slot answers (outside the step)."""
    import numpy as np
    import torch

    inputs_x = wl.with_searched_slots(inputs, n_slots, vocab=shape.vocab, n_sets=1)
    plan = spinf.Plan(inputs_x, vocab=shape.vocab)
    sets = wl.token_sets(shape.vocab, n_sets=1)
    words = np.zeros((1, -(-shape.vocab // 32) * 32), dtype=bool)
    words[:, :shape.vocab] = sets
    packed = np.packbits(words.reshape(1, -1, 8), axis=2, bitorder="little").reshape(1, -1).view(np.int32)
    sets_dev = torch.from_numpy(packed.copy()).to(dev)
    k = plan.extract_counts()[1]
    bufs = []
    with torch.cuda.stream(stream):
        for p in range(plan.num_passes):
            info = plan.pass_info(p)
            keys = sv.path_keys(info.tok, info.parent, info.T)
            h = sv.hidden(keys, info.T_pad, shape.d_model, rows=info.slot_row.tolist()).to(dev)
            plan.upload(p, stream)
            nb = spinf.score_workspace_bytes(plan, p, shape.vocab, shape.d_model, w_dtype)
            bufs.append({"h": h, "ws": torch.empty(nb, dtype=torch.uint8, device=dev),
                         "lse": torch.empty(max(info.M, 1), device=dev), "tlp": torch.empty(max(info.G, 1), device=dev),
                         "ex": {"token_sets": sets_dev,
                                "top_tok": torch.empty((max(info.X, 1), k), dtype=torch.int32, device=dev),
                                "top_lp": torch.empty((max(info.X, 1), k), device=dev)}})
    stream.synchronize()

    def run(with_x):
        evs = []
        for _ in range(max(3, args.steps // 2)):
            for p, b in enumerate(bufs):
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                spinf.score(plan, p, b["h"], w, w_scale, w_dtype, shape.d_model, shape.vocab, b["lse"], b["tlp"],
                            b["ws"], stream=stream, extract=b["ex"] if with_x else None)
                a1.record(stream)
                evs.append((a0, a1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs) * len(bufs)

    run(True)
    ms_plain, ms_x = run(False), run(True)
    plan.device_status(stream)
    n_x = plan.extract_counts()[0]

    # one decoding step of beam 4 on the pass with the most searched slots: every slot's 4 best
    # first tokens become decode rows (their q/k/v drawn like any token's), attention on the
    # pass's cached K/V, then the next-token answers at those rows
    pd = max(range(plan.num_passes), key=lambda p: plan.pass_info(p).X)
    info = plan.pass_info(pd)
    kp = sv.path_keys(info.tok, info.parent, info.T)
    q_p, k_p, v_p = (t.to(dev) for t in sv.qkv(kp, info.T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head))
    top = bufs[pd]["ex"]["top_tok"][:info.X, :4].cpu().numpy()
    anchor = np.repeat(info.slot_row[info.x_m], 4)
    dkeys = [sv.extend_key(kp[a], t) for a, t in zip(anchor, top.reshape(-1))]
    qd, kd, vd = (t.to(dev) for t in sv.qkv(dkeys, len(dkeys), shape.n_q_heads, shape.n_kv_heads, shape.d_head))
    hd = sv.hidden(dkeys, len(dkeys), shape.d_model).to(dev)
    nd = len(dkeys)
    i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32)).to(dev)  # noqa: E731
    anchor, parent, rows = i32(anchor), i32(np.full(nd, -1)), i32(np.arange(nd))
    tsets = i32(np.repeat(info.x_set, 4))
    od_ = torch.empty_like(qd)
    sws = torch.empty(spinf.lib().spinf_score_rows_workspace_bytes(nd, shape.vocab, shape.d_model, w_dtype, k),
                      dtype=torch.uint8, device=dev)
    lse_d = torch.empty(nd, device=dev)
    tt_d = torch.empty(nd, k, dtype=torch.int32, device=dev)
    tl_d = torch.empty(nd, k, device=dev)

    def step():
        spinf.decode_attention(plan, pd, qd, k_p, v_p, kd, vd, anchor, parent, rows, od_, shape.n_q_heads,
                               shape.n_kv_heads, shape.d_head, stream=stream)
        spinf.score_rows(plan, hd, w, w_scale, w_dtype, shape.d_model, shape.vocab, k, lse_d, tt_d, tl_d,
                         token_set=tsets, token_sets=sets_dev, workspace=sws, stream=stream)

    with torch.cuda.stream(stream):
        step()
        ev = []
        for _ in range(max(3, args.steps // 2)):
            a0, a1, a2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a0.record(stream)
            spinf.decode_attention(plan, pd, qd, k_p, v_p, kd, vd, anchor, parent, rows, od_, shape.n_q_heads,
                                   shape.n_kv_heads, shape.d_head, stream=stream)
            a1.record(stream)
            spinf.score_rows(plan, hd, w, w_scale, w_dtype, shape.d_model, shape.vocab, k, lse_d, tt_d, tl_d,
                             token_set=tsets, token_sets=sets_dev, workspace=sws, stream=stream)
            a2.record(stream)
            ev.append((a0, a1, a2))
    torch.cuda.synchronize()
    plan.device_status(stream)
    dec_attn = statistics.median(a.elapsed_time(b) for a, b, _ in ev)
    dec_score = statistics.median(b.elapsed_time(c) for _, b, c in ev)
    return {"workload": f"every input + {n_slots} searched slots ({{*}} any token, {{n}} 1% token set), k={k}",
            "slots": n_x, "score_ms_plain": ms_plain, "score_ms_with_answers": ms_x,
            "overhead_ms": ms_x - ms_plain, "slots_per_s": n_x / (ms_x * 1e-3),
            "decode_step": {"rows": nd, "beam": 4, "pass": pd, "attention_ms": dec_attn, "score_rows_ms": dec_score,
                            "note": "attention on the pass's cached K/V (no re-read of the questions' layout), "
                                    "next-token top-k over the whole vocabulary per row"}}


# requests in flight in the end-to-end leg (buffer sets of activations and descriptors)
E2E_DEPTH = 3


def run_e2e(args, spinf, inputs, shape, passes, w, w_scale, w_dtype, dev, resident):
    """Same job through the public API from pinned host buffers: plan, upload, H2D, kernels, D2H, collect.

    Requests are pipelined the way a server would run them, E2E_DEPTH in flight: request i is
    planned on the host, its descriptors (from pinned staging, so the call does not wait for the
    copy engine) and then its activations go up on the copy stream into buffer set i % E2E_DEPTH
    while earlier requests compute; its kernels start pass by pass as each pass's copies land,
    and its token log-probs come back and are collected two requests later.  Every request
    copies every byte again and reads its results back; the timed region covers n whole requests.
    """
    import numpy as np
    import torch

    depth = E2E_DEPTH
    # per pass: q, k, v and the hidden states of its scoring rows only (the lm head reads no other row)
    host = [tuple(t.pin_memory() for t in (*p["host"][:3], p["host"][3][torch.as_tensor(p["info"].slot_row).long()]))
            for p in passes]
    copy_stream = torch.cuda.Stream()
    stream = torch.cuda.Stream()
    sets = [[tuple(torch.empty_like(t, device=dev) for t in hp) for hp in host] for _ in range(depth)]
    obufs = [torch.empty_like(db[0]) for db in sets[0]]
    h2d = sum(t.numel() * t.element_size() for hp in host for t in hp)
    ws = [None]
    tl_host = [[torch.empty(max(p["info"].G, 1), dtype=torch.float32, pin_memory=True) for p in passes]
               for _ in range(depth)]
    tl_dev = [torch.empty(max(p["info"].G, 1), device=dev) for p in passes]
    lse_dev = [torch.empty(max(p["info"].M, 1), device=dev) for p in passes]
    # descriptor memory and its pinned staging kept across requests (per-plan allocations and
    # frees would synchronise the device every request), one set per request in flight
    probe = spinf.Plan(inputs, vocab=shape.vocab)
    dbytes = [(probe.descriptor_bytes(pi) + 255) // 256 * 256 + (1 << 20) for pi in range(probe.num_passes)]
    probe.close()
    dsc = [[torch.empty(b, dtype=torch.uint8, device=dev) for b in dbytes] for _ in range(depth)]
    stg = [[torch.empty(b, dtype=torch.uint8).pin_memory() for b in dbytes] for _ in range(depth)]
    freed = [None] * depth   # per buffer set: compute of the request that last read it is done
    plan_ms = []             # host time to marshal and plan each request

    def launch(i):
        b = i % depth
        t_plan = time.perf_counter()
        plan = spinf.Plan(inputs, vocab=shape.vocab)       # marshal the token lists and plan
        plan_ms.append((time.perf_counter() - t_plan) * 1e3)
        ready = []
        with torch.cuda.stream(copy_stream):
            if freed[b] is not None:   # the kernels that last read this set's memory are done
                copy_stream.wait_event(freed[b])
            for pi in range(plan.num_passes):
                plan.upload(pi, copy_stream, buffer=dsc[b][pi], staging=stg[b][pi])
            for pi in range(len(passes)):
                for src, dst in zip(host[pi], sets[b][pi]):
                    dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                ready.append(ev)
        all_p = list(range(plan.num_passes))
        if ws[0] is None:
            ws[0] = torch.empty(spinf.score_passes_workspace_bytes(plan, all_p, shape.vocab, shape.d_model, w_dtype),
                                dtype=torch.uint8, device=dev)
        for pi in all_p:
            stream.wait_event(ready[pi])
            q, k, v, h = sets[b][pi]
            spinf.branch_attention(plan, pi, q, k, v, obufs[pi], shape.n_q_heads, shape.n_kv_heads,
                                   shape.d_head, stream=stream)
        spinf.score_passes(plan, all_p, [sets[b][pi][3] for pi in all_p], w, w_scale, w_dtype, shape.d_model,
                           shape.vocab, [lse_dev[pi] for pi in all_p], [tl_dev[pi] for pi in all_p], ws[0],
                           stream=stream, slot_rows=True)
        with torch.cuda.stream(stream):
            for pi in all_p:
                tl_host[b][pi].copy_(tl_dev[pi], non_blocking=True)
        done = torch.cuda.Event()
        done.record(stream)
        freed[b] = done
        return plan, done

    def finish(i, plan, done):
        done.synchronize()
        res = plan.collect([tl_host[i % depth][pi][:passes[pi]["info"].G].numpy() for pi in range(plan.num_passes)])
        plan.close()
        return res

    def run(n):
        inflight, res = [], None
        for i in range(n):
            inflight.append((i, *launch(i)))
            if len(inflight) == depth:
                res = finish(*inflight.pop(0))
        while inflight:
            res = finish(*inflight.pop(0))
        return res

    run(max(depth, args.warmup))
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    t0 = time.perf_counter()
    res = run(n)
    ms = (time.perf_counter() - t0) * 1e3 / n
    assert res["option_lp"].size > 0
    # the same kernels on the same values as the resident step: the results must agree bit for bit
    same = all(np.array_equal(res[k], resident[k], equal_nan=True) for k in res)
    tokens = sum(p["info"].T for p in passes)
    return {"value": tokens / (ms * 1e-3), "unit": "packed tokens/s", "ms_per_step": ms,
            "results_bitwise_equal_to_resident_step": bool(same),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": sum(p["info"].G for p in passes) * 4,
            "host_plan_ms_median": statistics.median(plan_ms[-n:]),
            "covers": "per request: plan (marshalling of the request's token lists + C planner) + descriptor "
                      "upload from pinned staging into kept device memory + H2D q/k/v and the scoring rows' "
                      "hidden states (copy stream, overlapping earlier requests' kernels) + attention per pass "
                      "(each pass as its copies land) + one scoring sweep + D2H token lps + collect; "
                      f"{depth} requests in flight"}


# The oracle sample both CPU legs time (the repo arm's cpu_baseline and --impl reference),
# so that the two agree: per step, the oracle planner on the whole job, the oracle attention
# on ORACLE_ATTN_ROWS rows of pass 0 (all heads), and one oracle scoring call on
# ORACLE_SCORE_ROWS whole slot rows of pass 0 (full vocabulary, every option token of them).
ORACLE_ATTN_ROWS = 48
ORACLE_SCORE_ROWS = 32


class OracleSample:
    """The fp64 oracle, as it stands, on a bounded sample of the job; each ``step()`` times one
    sample and extrapolates it to the whole job: planner + attention per row x packed tokens +
    one scoring call per ORACLE_SCORE_ROWS scoring rows of every pass (the oracle run over the
    job in blocks of that many rows, which bounds its fp64 logits at 64 MB per block)."""

    def __init__(self, inputs, shape, pass0_host, w, w_scale):
        import numpy as np

        from oracle import plan as op

        self.inputs, self.shape = inputs, shape
        self.P = op.plan(inputs, vocab=shape.vocab)
        self.lay = self.P.passes[0]
        q, k, v, h = pass0_host
        self.q, self.k, self.v = (t.float().numpy() for t in (q, k, v))
        self.h = h.float().numpy()[self.lay.slot_row]
        self.wkw = ({"w": _BF16Rows(w.cpu())} if w_scale is None
                    else {"w_codes": w.cpu().numpy(), "w_scale": w_scale.cpu().numpy()})
        self.tokens = sum(p.T for p in self.P.passes)
        self.blocks = sum(-(-len(p.slot_row) // ORACLE_SCORE_ROWS) for p in self.P.passes)
        self.rows_total = sum(len(p.slot_row) for p in self.P.passes)
        self.g = np.random.default_rng(0)

    def step(self):
        """(seconds this sample took, seconds the whole job is estimated to take)."""
        import numpy as np

        from oracle import attention as oa
        from oracle import collect as oc
        from oracle import plan as op
        from oracle import score as osc

        lay, sh = self.lay, self.shape
        t_start = time.perf_counter()
        op.plan(self.inputs, vocab=sh.vocab)
        t_plan = time.perf_counter() - t_start
        rows = self.g.choice(lay.T, size=min(lay.T, ORACLE_ATTN_ROWS), replace=False)
        t0 = time.perf_counter()
        oa.attention_rows(lay, self.q, self.k, self.v, sh.n_q_heads, sh.n_kv_heads, rows)
        t_attn_row = (time.perf_counter() - t0) / len(rows)
        n = min(ORACLE_SCORE_ROWS, len(lay.slot_row))
        m0 = int(self.g.integers(0, len(lay.slot_row) - n + 1))
        ms = np.arange(m0, m0 + n)
        sel = np.isin(lay.gather_m, ms)
        t0 = time.perf_counter()
        _, lp = osc.score_rows(self.h[ms], lay.gather_m[sel] - m0, lay.gather_tok[sel], **self.wkw)
        oc.option_stats(lp[:2])
        t_block = time.perf_counter() - t0
        sample_s = time.perf_counter() - t_start
        job_s = t_plan + t_attn_row * self.tokens + t_block * self.blocks
        return sample_s, job_s

    def describe(self):
        return (f"per sample: oracle planner on the whole job, oracle attention on {ORACLE_ATTN_ROWS} rows of "
                f"pass 0 (all heads), one oracle scoring call on {ORACLE_SCORE_ROWS} whole slot rows of pass 0 "
                f"(full vocabulary); extrapolated to {self.tokens} packed tokens and {self.rows_total} scoring "
                f"rows ({self.blocks} calls of {ORACLE_SCORE_ROWS} rows)")


def cpu_baseline(args, inputs, shape, plan, passes, w, w_scale, budget_s=20.0):
    """The fp64 oracle on the host cores: the same sample as --impl reference, repeated within a
    time budget, its job estimate averaged."""
    sample = OracleSample(inputs, shape, passes[0]["host"], w, w_scale)
    t0 = time.perf_counter()
    est = []
    while not est or (time.perf_counter() - t0 < budget_s and len(est) < 5):
        est.append(sample.step()[1])
    job_s = statistics.mean(est)
    return {"value": sample.tokens / job_s, "unit": "packed tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": sample.describe() + f"; {len(est)} samples averaged",
            "job_seconds_estimate": job_s}


class _BF16Rows:
    """Lazy fp64 view of a bf16 torch matrix, row slices converted on demand (bounded host memory)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, sl):
        return self.t[sl].float().numpy()


def run_reference(args):
    """--impl reference: the oracle, as it stands, on the host cores; one bounded sample of the
    job per step (the same sample as the repo arm's cpu_baseline).  ``ms_per_step`` is the
    measured time of one sample; ``value`` is the job's packed tokens over the job time the
    samples extrapolate to."""
    from synth import values as sv
    from synth import workloads as wl
    from oracle import plan as op

    f, shape = wl.WORKLOADS[args.workload]
    inputs = f()
    lay = op.plan(inputs, vocab=shape.vocab).passes[0]
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    q, k, v = sv.qkv(keys, lay.T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    h = sv.hidden(keys, lay.T_pad, shape.d_model, rows=lay.slot_row.tolist())
    w = sv.lm_head(shape.vocab, shape.d_model, device="cpu") if shape.vocab * shape.d_model < (1 << 28) \
        else _cpu_lm_head(shape)
    w_scale = None
    if args.fp8:
        w, w_scale = sv.e4m3_rows(w)
    sample = OracleSample(inputs, shape, (q, k, v, h), w, w_scale)
    for _ in range(args.warmup):
        sample.step()
    runs = [sample.step() for _ in range(args.steps)]
    step_s = statistics.mean(r[0] for r in runs)
    job_s = statistics.mean(r[1] for r in runs)
    value = sample.tokens / job_s
    questions = sum(len(x) for _, x in inputs)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "packed tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64" if not args.fp8 else "f64 (e4m3 codes)",
        "data": "synthetic",
        "config": _config(args, inputs, len(sample.P.passes), sample.tokens, questions, shape, 1),
        "job_seconds_estimate": job_s,
        "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": value, "unit": "packed tokens/s",
                         "sample": sample.describe() + "; one sample per step"},
        "e2e": {"value": value, "unit": "packed tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _config(args, inputs, n_passes, tokens, questions, shape, world):
    """The ``config`` of both arms' JSON lines (the same words for the same workload)."""
    return {"workload": f"{args.workload}: {len(inputs)} contents, {questions} questions, "
                        f"{n_passes} passes of <=16384 tokens ({tokens} tokens)",
            "attention": f"Hq={shape.n_q_heads} Hkv={shape.n_kv_heads} d_head={shape.d_head} (1 layer)",
            "lm_head": f"d_model={shape.d_model} vocab={shape.vocab} "
                       f"{'e4m3 per-row scaled' if args.fp8 else 'bf16'}, fp32 logits",
            "l2": "inputs larger than L2 (per pass q/k/v/o ~0.4 GB, lm head 2 GB)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def _cpu_lm_head(shape):
    import torch

    g = torch.Generator().manual_seed(0x1E4D)
    return (torch.randn(shape.vocab, shape.d_model, generator=g) / math.sqrt(shape.d_model)).to(torch.bfloat16)


def run_ncu_case(args):
    """Pass 0 of the workload, one boundary call repeated: the small case for ncu captures."""
    import torch

    import branch_packed_scoring_gb300 as spinf
    from synth import values as sv
    from synth import workloads as wl

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    f, shape = wl.WORKLOADS[args.workload]
    inputs = f()
    if args.ncu_case == "decode":   # two searched slots per input, as in the searched-slot timing
        inputs = wl.with_searched_slots(inputs, 2, vocab=shape.vocab, n_sets=1)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    info = plan.pass_info(0)
    keys = sv.path_keys(info.tok, info.parent, info.T)
    plan.upload(0)
    w_dtype = spinf.DTYPE_E4M3 if args.fp8 else spinf.DTYPE_BF16
    if args.ncu_case == "decode":
        # one decoding step of beam 4 on pass 0: every searched slot's row extended by 4 tokens
        # (token ids 0-3 stand in for its best four), attention on the pass's cached K/V
        import numpy as np

        q_p, k_p, v_p = (t.to(dev) for t in sv.qkv(keys, info.T_pad, shape.n_q_heads, shape.n_kv_heads,
                                                   shape.d_head))
        anchor = np.repeat(info.slot_row[info.x_m], 4)
        dkeys = [sv.extend_key(keys[a], t) for a, t in zip(anchor, np.tile(np.arange(4), len(info.x_m)))]
        qd, kd, vd = (t.to(dev) for t in sv.qkv(dkeys, len(dkeys), shape.n_q_heads, shape.n_kv_heads,
                                                shape.d_head))
        nd = len(dkeys)
        i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32)).to(dev)  # noqa: E731
        anchor, parent, rows = i32(anchor), i32(np.full(nd, -1)), i32(np.arange(nd))
        od = torch.empty_like(qd)

        def call():
            spinf.decode_attention(plan, 0, qd, k_p, v_p, kd, vd, anchor, parent, rows, od, shape.n_q_heads,
                                   shape.n_kv_heads, shape.d_head)
    elif args.ncu_case == "qkv":   # the fused QKV projection + rotary of pass 0, seeded random inputs
        Hq, Hkv, d, D = shape.n_q_heads, shape.n_kv_heads, shape.d_head, shape.d_model
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        x = torch.randn(info.T_pad, D, generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn((Hq + 2 * Hkv) * d, D, generator=g, device=dev) / D ** 0.5).to(torch.bfloat16)
        q = torch.empty(info.T_pad, Hq, d, dtype=torch.bfloat16, device=dev)
        k = torch.empty(info.T_pad, Hkv, d, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        kw = {}
        if args.fp8:
            s_w = (w.float().abs().amax(dim=1) / 448.0).clamp_min(1e-12)
            w = (w.float() / s_w[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            x8 = torch.empty(info.T_pad, D, dtype=torch.uint8, device=dev)
            spinf.quantize_static(x, 5.0 / 448, x8)
            x = x8
            kw = {"w_scale": s_w, "x_scale": 5.0 / 448, "w_dtype": spinf.DTYPE_E4M3}

        def call():
            spinf.qkv_rope(plan, 0, x, w, q, k, v, Hq, Hkv, d, **kw)
    elif args.ncu_case == "attention":
        q, k, v = (t.to(dev) for t in sv.qkv(keys, info.T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head))
        o = torch.empty_like(q)

        def call():
            spinf.branch_attention(plan, 0, q, k, v, o, shape.n_q_heads, shape.n_kv_heads, shape.d_head,
                                   window=args.window)
    elif args.ncu_case == "score_passes":   # the step's scoring launch: every pass's slot rows in one sweep
        all_p = list(range(plan.num_passes))
        hs, lses, tlps = [], [], []
        for pi in all_p:
            inf = plan.pass_info(pi)
            kk = sv.path_keys(inf.tok, inf.parent, inf.T)
            hs.append(sv.hidden(kk, inf.T_pad, shape.d_model, rows=inf.slot_row.tolist()).to(dev))
            lses.append(torch.empty(max(inf.M, 1), device=dev))
            tlps.append(torch.empty(max(inf.G, 1), device=dev))
            plan.upload(pi)
        w = sv.lm_head(shape.vocab, shape.d_model, device=dev)
        w_scale = None
        if args.fp8:
            w, w_scale = sv.e4m3_rows(w)
        ws = torch.empty(spinf.score_passes_workspace_bytes(plan, all_p, shape.vocab, shape.d_model, w_dtype),
                         dtype=torch.uint8, device=dev)

        def call():
            spinf.score_passes(plan, all_p, hs, w, w_scale, w_dtype, shape.d_model, shape.vocab, lses, tlps, ws)
    else:
        h = sv.hidden(keys, info.T_pad, shape.d_model, rows=info.slot_row.tolist()).to(dev)
        w = sv.lm_head(shape.vocab, shape.d_model, device=dev)
        w_scale = None
        if args.fp8:
            w, w_scale = sv.e4m3_rows(w)
        ws = torch.empty(spinf.score_workspace_bytes(plan, 0, shape.vocab, shape.d_model, w_dtype),
                         dtype=torch.uint8, device=dev)
        lse = torch.empty(info.M, device=dev)
        tlp = torch.empty(info.G, device=dev)

        def call():
            spinf.score(plan, 0, h, w, w_scale, w_dtype, shape.d_model, shape.vocab, lse, tlp, ws)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    plan.device_status()
    print(json.dumps({"ncu_case": args.ncu_case, "workload": args.workload, "T": info.T, "M": info.M,
                      "calls": args.warmup + args.steps}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wikinews", choices=["wikinews", "moderation", "stress", "invariance"])
    ap.add_argument("--fp8", action="store_true", help="e4m3 lm head with per-row scales")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extract", action="store_true", help="skip the searched-slot scoring timing")
    ap.add_argument("--no-layer", action="store_true", help="skip the projection timing")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the moderation / stress / e4m3 invariance-pass timings")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ncu-case", choices=["score", "score_passes", "attention", "qkv", "decode"], default=None,
                    help="run one boundary call on pass 0 only (small case for profiler captures)")
    ap.add_argument("--window", type=int, default=0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.ncu_case:
        run_ncu_case(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch

    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    out = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
