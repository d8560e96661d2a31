#!/usr/bin/env python
"""Benchmark of the candidate-set scoring head on GB300.

One step = one pass of the whole path over one batch.  The headline workload
(default) is the large batch: 16 requests x 64 candidates of 8-32 tokens,
about 20k scored positions, d=4096, V=152064, full vocabulary: pre-pass,
tcgen05 head, split merge, set rules.  The line's ``per_config`` block times
the other workloads the same way: the binary batch (256 questions, d=2560,
V=248320) in full-vocabulary mode, in restricted mode over its 26-code union
(latency-bound: reported, not a roofline target), and both passes in one step;
the binary batch with its rows read in place from a right-padded source, the
multi-token choice batch, the wide-schema batch, the large batch with each
distinct hidden row projected once (the row-dedup pass inside the step), and
the large batch with W in the library's default row-major layout (every other
entry streams W packed once by jet_tile_weights).
The ``ops`` block times the widened ops at the same steps: row dedup of the
large batch's rows, temperature fitting, layer sensitivity, and restricted
mode over unions of 600 and 4096 codes.  The metric is scored candidate
tokens per second (of the first pass where a step holds two).

Printed: one JSON line (rank 0).  Timing: CUDA events on the launching stream,
after warm-up, synchronised on both sides; W (0.8-1.3 GB) is larger than L2, so
consecutive steps do not hit in L2 for the dominant stream.  Kernel-level
times come from event pairs the library records around its own launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload large|binary|multitoken|wideschema|tiny]
                  [--per-config binary,binary-restricted,binary-both,binary-gather,multitoken,wideschema,
                                large-dedup,large-rowmajor|none]
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "candidate tokens scored/sec (full-vocab log-softmax) and % of roofline, 1 GB300"
UNIT = "tokens/s"

WORKLOADS = {
    # name: (generator, modes per step, default steps, description)
    "binary": ("binary_batch", ("full",), 6000,
               "binary single-token batch: 256 questions x {A,B} codes, d=2560, V=248320; full vocabulary (T=1)"),
    "binary-restricted": ("binary_batch", ("restricted",), 6000,
                          "binary single-token batch: 256 questions x {A,B} codes, d=2560; restricted 26-code "
                          "union (T=2.179)"),
    "binary-gather": ("binary_batch", ("full",), 6000,
                      "binary single-token batch: 256 questions x {A,B} codes, d=2560, V=248320; full vocabulary "
                      "(T=1); hidden rows read in place from a right-padded [256, 8, d] source "
                      "(jet_score_sets_gather)"),
    "binary-both": ("binary_batch", ("full", "restricted"), 6000,
                    "binary single-token batch: 256 questions x {A,B} codes, d=2560, V=248320; full vocabulary "
                    "(T=1) then the restricted 26-code union (T=2.179) in one step"),
    "multitoken": ("multi_token_choice", ("full",), 300,
                   "multi-token choice: 64 questions x K=8, 1-12 tokens, d=1536, V=262144, T=1"),
    "wideschema": ("wide_schema", ("full",), 60,
                   "wide schema: 16 requests x 32 fields, enum K 2-26 / ordinal K=5, d=2560, V=248320, T=2.179"),
    "large": ("large_choice", ("full",), 40,
              "large choice: 16 requests x K=64, 8-32 tokens, d=4096, V=152064, T=1"),
    "large-dedup": ("large_choice", ("full",), 40,
                    "large choice: 16 requests x K=64, 8-32 tokens, d=4096, V=152064, T=1; each distinct hidden "
                    "row projected once (jet_dedup_rows inside the step)"),
    "large-rowmajor": ("large_choice", ("full",), 40,
                       "large choice: 16 requests x K=64, 8-32 tokens, d=4096, V=152064, T=1; W read in the "
                       "library's default row-major [V, d] layout (no jet_tile_weights)"),
    "tiny": ("tiny", ("full",), 2000, "tiny: d=64, V=1000, 3 sets"),
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# the head kernel's own sources (the ABI header it also includes supplies only
# the status codes, so declarations added there leave the kernel unchanged)
HEAD_SOURCES = ("candidate_answer_scoring_gb300/csrc/k_head.cu", "candidate_answer_scoring_gb300/csrc/jet_head.cuh",
                "candidate_answer_scoring_gb300/csrc/jet_wait.cuh")


def head_source_hash():
    h = hashlib.sha256()
    for f in HEAD_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload):
    """DRAM bytes per head launch from a committed ncu summary, if it was taken
    on the current head-kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "head_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("source_hash") != head_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 200 ms; the
    statistics cover the samples received during the marked timed passes (or,
    for a pass shorter than the sampling period, the first sample after its
    start)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.rows = []        # (host receive time, fields)
        self.windows = []     # (start, end) host times of the timed passes
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((time.monotonic(), parts))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        picked = []
        for t0, t1 in self.windows:
            inside = [r for t, r in self.rows if t0 <= t <= t1]
            after = [r for t, r in self.rows if t > t0][:1]
            picked += inside if inside else after
        rows = picked if picked else [r for _, r in self.rows]
        num = lambda v: v.replace(".", "").isdigit()
        sm = [float(r[0]) for r in rows if num(r[0])]
        mx = [float(r[1]) for r in rows if num(r[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        pw = [float(r[2]) for r in rows if num(r[2])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "window_s": sum(t1 - t0 for t0, t1 in self.windows), "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The largest value of x over the ranks (x itself with one rank): every
    rank's timed region counts, the slowest one sets the job's time."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step, steps, world, ms):
    """Whole-job tokens/s: every replica scores tokens_per_step each step."""
    return world * tokens_per_step * steps / (ms / 1e3)


_GENERATED = {}


def make_workload(name, rank=0):
    import workloads as wk
    gen_name = WORKLOADS[name][0]
    if gen_name not in _GENERATED:         # a batch serving several workloads is generated once
        _GENERATED[gen_name] = getattr(wk, gen_name)()
    base = _GENERATED[gen_name]
    steps = []
    for mode in WORKLOADS[name][1]:
        if mode == "full":
            steps.append(base)
        else:
            steps.append(wk.binary_restricted(base=base))
    return steps[0], steps


def roofline_terms(wl, peaks, sustained, n_rows=None):
    """Algorithmic work of one full-vocabulary head launch over n_rows hidden
    rows (default: all of the workload's rows) and the roofline time."""
    N, d, V, n_tok = (wl.N if n_rows is None else n_rows), wl.d, wl.V, wl.n_tok
    flops = 2.0 * N * d * V
    bytes_ = 2.0 * V * d + 2.0 * N * d + 8.0 * n_tok
    tc = (peaks["bf16_sustained"] if sustained else peaks["bf16"]) * 1e12
    t_tc = flops / tc
    t_hbm = bytes_ / (peaks["hbm"] * 1e9)
    return flops, bytes_, t_tc, t_hbm


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def _subset(wl, n_cand):
    """The workload cut to its first n_cand candidates (whole sets, then the
    leading candidates of the next set, which becomes a choice set), with only
    the hidden rows those candidates' tokens read.  The oracle's cost is one
    full-vocabulary row per distinct row, so a candidate-granular cut keeps a
    sample of a few hundred rows bounded even where one set holds a thousand."""
    import numpy as np
    import workloads as wk
    c1 = max(1, min(int(n_cand), wl.n_cand))
    so = wl.set_offsets.astype(np.int64)
    k = int(np.searchsorted(so, c1, side="left"))      # sets [0, k) start before c1
    set_off = np.minimum(so[:k + 1], c1).astype(np.int32)
    set_off[k] = c1
    kind = wl.kind[:k].copy()
    if so[k] != c1:                                    # the last set was cut short
        kind[k - 1] = wk.KIND_CHOICE
    t1 = int(wl.cand_offsets[c1])
    rows, new_row = np.unique(wl.tok_row[:t1], return_inverse=True)
    return wk.Workload(wl.name + f"-first{c1}c", wl.d, wl.V, np.ascontiguousarray(wl.H[rows]), wl.W,
                       new_row.astype(np.int32), wl.tok_ids[:t1].copy(), wl.cand_offsets[:c1 + 1].copy(),
                       set_off, kind, wl.T, wl.mode, wl.union_ids, dict(wl.info))


def time_oracle(steps_wl, n_cand, repeats=1):
    """Run the oracle on the first n_cand candidates of each step workload;
    returns (seconds per step, full-mode tokens per step, threads)."""
    import oracle
    subs = [_subset(w, n_cand) for w in steps_wl]
    t0 = time.perf_counter()
    for _ in range(repeats):
        for s in subs:
            oracle.score_workload(s)
    dt = (time.perf_counter() - t0) / repeats
    return dt, subs[0].n_tok, oracle.max_threads()


def cpu_sample_cands(steps_wl, target_s):
    """Number of leading candidates whose oracle run takes about target_s
    seconds of wall time on this host.  The oracle runs rows in parallel, so
    the probe takes enough candidates for about two rows per thread."""
    import numpy as np
    import oracle
    wl = steps_wl[0]
    rows_per_cand = max(1.0, wl.N / max(1, wl.n_cand))
    probe = int(min(wl.n_cand, max(1, np.ceil(2 * oracle.max_threads() / rows_per_cand))))
    dt, _, _ = time_oracle(steps_wl, probe)
    return max(1, min(wl.n_cand, int(probe * target_s / max(dt, 1e-4)))), probe


def reference_arm(args, world, rank):
    if rank != 0:
        return 0
    name = args.workload
    wl, steps_wl = make_workload(name)
    import oracle
    oracle.build()
    # size one step to about 2 s of oracle work, then cap the whole run at ~3 min
    n_cand, _ = cpu_sample_cands(steps_wl, target_s=2.0)
    K = args.steps if args.steps is not None else 5
    W = args.warmup if args.warmup is not None else 1
    budget = 180.0
    step_est = 2.0
    k_run = max(1, min(K, int(budget / max(step_est, 1e-3)) - W))
    for _ in range(W):
        time_oracle(steps_wl, n_cand)
    t0 = time.perf_counter()
    tokens = 0
    threads = 1
    for _ in range(k_run):
        dt, ntok, threads = time_oracle(steps_wl, n_cand)
        tokens += ntok
    el = time.perf_counter() - t0
    value = tokens / el
    sub = _subset(wl, n_cand)
    sample = (f"first {n_cand} of {wl.n_cand} candidates per step ({sub.n_tok} full-vocab tokens over {sub.N} "
              f"hidden rows{', plus the same candidates restricted' if len(steps_wl) > 1 else ''}); "
              "fp64 C oracle, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": k_run, "steps_requested": K, "warmup": W, "ms_per_step": 1e3 * el / k_run,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[name][3], "d": wl.d, "V": wl.V, "N": wl.N, "n_tok": wl.n_tok,
                   "n_cand": wl.n_cand, "n_sets": wl.n_sets, "modes": list(WORKLOADS[name][1]),
                   "parallelism": "rank 0 (host cores)", "accumulate": "fp64 (oracle)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def gpu_uuid_of(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def measure_workload(name, args, dev, world, peaks, K, W, keep=False):
    """Time K steps of one workload on the device (inputs resident, after W
    warm-up steps), then the same K steps with the library's per-launch event
    pairs for the kernel times.  Returns the measurements and, with keep, the
    scorer and device inputs for the end-to-end leg."""
    import numpy as np
    import torch

    import candidate_answer_scoring_gb300 as jet

    wl, steps_wl = make_workload(name)
    dedup = bool(args.dedup) or name.endswith("-dedup")
    gather_rows = args.gather_rows or (8 if name.endswith("-gather") else 0)
    w_layout = "rowmajor" if name.endswith("-rowmajor") else args.w_layout
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    Wd = t(wl.W.view(np.int16)).view(torch.bfloat16)
    ins = []
    for s in steps_wl:
        ins.append(dict(H=t(s.H.view(np.int16)).view(torch.bfloat16), tok_row=t(s.tok_row), tok_ids=t(s.tok_ids),
                        cand_offsets=t(s.cand_offsets), set_offsets=t(s.set_offsets), kind=t(s.kind),
                        union_ids=None if s.union_ids is None else t(s.union_ids), T=s.T, mode=s.mode, wl=s))
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok, device=dev.index)
    if w_layout == "tiled":
        # the output embedding is stored once in the head's tiled layout (as a
        # model loader would), outside the timed region
        Wd = sc.tile_weights(Wd)
        torch.cuda.synchronize(dev)
    outs = [sc.alloc_outputs(s.N, s.n_tok, s.n_cand, s.n_sets) for s in steps_wl]
    if gather_rows:
        # rows read in place from a right-padded [N, L, d] source at each
        # sequence's last valid position (lengths uniform in 1..L)
        L = gather_rows
        grng = np.random.default_rng(20261202 + 77)
        lengths = grng.integers(1, L + 1, size=wl.N)
        from workloads import to_bf16_bits as wk_to_bf16
        src = wk_to_bf16(grng.standard_normal((wl.N * L, wl.d)).astype(np.float32))
        row_index = (np.arange(wl.N) * L + lengths - 1).astype(np.int32)
        src[row_index] = wl.H
        for x in ins:
            x["H_src"] = t(src.view(np.int16)).view(torch.bfloat16)
            x["row_index"] = t(row_index)
    stream = torch.cuda.Stream(dev)
    n_rows_scored = wl.N
    if dedup:
        # candidate-preserving readout: score each distinct hidden row once
        Hu_buf = [torch.empty_like(x["H"]) for x in ins]
        with torch.cuda.stream(stream):
            n_rows_scored = int(sc.dedup_rows(ins[0]["H"], ins[0]["tok_row"], H_unique=Hu_buf[0])[0].shape[0])

    # the plain step: each pass one C call with its arguments marshalled once,
    # as a C caller holding these buffers makes it (the Python wrapper's
    # per-call checks cost more host time than a restricted pass's GPU time)
    bound = []
    if gather_rows and not dedup:
        with torch.cuda.stream(stream):
            bound = [sc.bind_gather_call(x["H_src"], x["row_index"], Wd, x["tok_row"], x["tok_ids"],
                                         x["cand_offsets"], x["set_offsets"], x["kind"], x["T"], x["mode"],
                                         x["union_ids"], out=o)[0] for x, o in zip(ins, outs)]
    elif not dedup:
        with torch.cuda.stream(stream):
            bound = [sc.bind_call(x["H"], Wd, x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"],
                                  x["kind"], x["T"], x["mode"], x["union_ids"], out=o)[0] for x, o in zip(ins, outs)]

    def step():
        if bound:
            for call in bound:
                call()
            return
        for i, (x, o) in enumerate(zip(ins, outs)):
            H, tok_row = x["H"], x["tok_row"]
            if dedup:
                H, tok_row, _ = sc.dedup_rows(H, tok_row, H_unique=Hu_buf[i])
            if gather_rows:
                sc.score_sets_gather(x["H_src"], x["row_index"], Wd, tok_row, x["tok_ids"], x["cand_offsets"],
                                     x["set_offsets"], x["kind"], x["T"], x["mode"], x["union_ids"], out=o,
                                     sync=False)
                continue
            sc.score_sets(H, Wd, tok_row, x["tok_ids"], x["cand_offsets"], x["set_offsets"], x["kind"],
                          x["T"], x["mode"], x["union_ids"], out=o, sync=False)

    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
        rc = sc.sync_status()
        if rc != 0:
            raise RuntimeError(f"{name}: device status {rc} ({jet.status_string(rc)}) after warm-up")
        torch.cuda.synchronize(dev)

        clocks = ClockSampler(gpu_uuid_of(dev))
        clocks.start()
        time.sleep(0.3)

        def timed(K_):
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K_):
                step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            return e0.elapsed_time(e1)

        # (1) the step as a user runs it: no event records between kernels,
        # so each kernel's launch overlaps the previous one's tail
        h0 = time.monotonic()
        ms = timed(K)
        clocks.mark(h0, time.monotonic())
        # (2) the same loop with the library's per-launch event pairs, for the
        # kernel-level roofline (events between kernels remove that overlap)
        sc.profile(True)
        h0 = time.monotonic()
        ms_prof = timed(K)
        clocks.mark(h0, time.monotonic())
        prof = sc.profile_read()
        sc.profile(False)
        clk = clocks.stop()
        rc = sc.sync_status()
        if rc != 0:
            raise RuntimeError(f"{name}: device status {rc} ({jet.status_string(rc)}) in the timed region")
    ms = max_over_ranks(ms, world, dev)
    tokens_per_step = steps_wl[0].n_tok
    ms_step = ms / K

    if wl.mode == 1:
        return restricted_record(name, wl, steps_wl, sc, prof, ms, K, W, world, peaks, clk, ms_prof, keep,
                                 Wd, ins, outs, stream)
    # kernel roofline: the full-vocabulary head
    head = prof["head"]
    head_ms = head["ms"] / max(1, head["launches"])
    flops, bytes_, t_tc, t_hbm = roofline_terms(wl, peaks, sustained=True, n_rows=n_rows_scored)
    _, _, t_tc_burst, _ = roofline_terms(wl, peaks, sustained=False, n_rows=n_rows_scored)
    # the bound by the roofline formula with the burst tensor peak
    bound = "hbm" if t_hbm >= t_tc_burst else "tensor"
    tflops = flops / (head_ms / 1e3) / 1e12
    gbs = bytes_ / (head_ms / 1e3) / 1e9
    if bound == "hbm":
        achieved, peak, unit = gbs, peaks["hbm"], "GB/s"
    else:
        # the burst peak: the head is timed in a loop well under a second
        # long, not the seconds-long loop the sustained figure comes from
        achieved, peak, unit = tflops, peaks["bf16"], "TFLOP/s"
    launches = sum(v["launches"] for k, v in prof.items() if isinstance(v, dict))   # = launches of pass (1)
    t_roof = max(t_tc_burst, t_hbm)
    note = "of measured" if peaks["source"] == "measured" else "of fallback"
    rec = {
        "name": name, "wl": wl, "steps_wl": steps_wl, "K": K, "W": W, "ms": ms, "ms_step": ms_step, "dedup": dedup,
        "gather_rows": gather_rows, "w_layout": w_layout,
        "value": job_throughput(tokens_per_step, K, world, ms), "tokens_per_step": tokens_per_step,
        "n_rows_scored": n_rows_scored, "plan": sc.plan_info(n_rows_scored), "clocks": clk,
        "gpu_launches": int(launches), "ms_prof": ms_prof, "prof": prof, "head_ms": head_ms,
        "step_roofline_us": t_roof * 1e6, "step_roofline_frac": t_roof / (ms_step / 1e3),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak,
                     "frac_vs_burst_tensor": t_tc_burst / (head_ms / 1e3),
                     "frac_vs_sustained_tensor": t_tc / (head_ms / 1e3),
                     "frac_vs_hbm": t_hbm / (head_ms / 1e3),
                     # the committed capture is of the default launch (all rows, row-major
                     # problem rows, tiled W); other configurations report none
                     "traffic": committed_traffic(name.split("-")[0]) if not (dedup or gather_rows
                                                                             or w_layout != "tiled") else None,
                     "kernel": "head_lse_gather (tcgen05)", "kernel_ms": head_ms,
                     "achieved_tflops": tflops, "achieved_gbs": gbs,
                     "algorithmic_bytes": bytes_, "algorithmic_flops": flops,
                     "t_tensor_us_sustained": t_tc * 1e6, "t_tensor_us_burst": t_tc_burst * 1e6,
                     "t_hbm_us": t_hbm * 1e6, "peak_note": note},
    }
    if keep:
        rec.update(sc=sc, Wd=Wd, stream=stream)
    else:
        sc.close()
        del Wd, ins, outs
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return rec


def restricted_record(name, wl, steps_wl, sc, prof, ms, K, W, world, peaks, clk, ms_prof, keep, Wd, ins, outs,
                      stream):
    """Measurements of a restricted-mode-only workload: the projection onto the
    union is the dominant kernel; its algorithmic work is 2|U|d + 2Nd bytes
    and 2Nd|U| flops, far below a microsecond at the peaks, so the pass is
    bound by launch and memory latency (reported, not a roofline target)."""
    import torch
    n_u = int(wl.union_ids.size)
    k = prof["head"] if prof["head"]["launches"] else prof["restricted"]
    proj_ms = k["ms"] / max(1, k["launches"])
    bytes_ = 2.0 * n_u * wl.d + 2.0 * wl.N * wl.d
    flops = 2.0 * wl.N * wl.d * n_u
    t_roof = max(bytes_ / (peaks["hbm"] * 1e9), flops / (peaks["bf16"] * 1e12))
    ms_step = ms / K
    rec = {
        "name": name, "wl": wl, "steps_wl": steps_wl, "K": K, "W": W, "ms": ms, "ms_step": ms_step,
        "value": job_throughput(wl.n_tok, K, world, ms), "tokens_per_step": wl.n_tok,
        "n_rows_scored": wl.N, "plan": None, "clocks": clk,
        "gpu_launches": int(sum(v["launches"] for v in prof.values() if isinstance(v, dict))),
        "ms_prof": ms_prof, "prof": prof, "head_ms": proj_ms,
        "step_roofline_us": t_roof * 1e6, "step_roofline_frac": t_roof / (ms_step / 1e3),
        "roofline": {"bound": "latency", "achieved": bytes_ / (proj_ms / 1e3) / 1e9, "peak": peaks["hbm"],
                     "unit": "GB/s", "frac": bytes_ / (proj_ms / 1e3) / 1e9 / peaks["hbm"],
                     "kernel": ("head_lse_gather (tcgen05) over the staged union" if prof["head"]["launches"]
                                else "restricted_head (mma.sync) over the union"),
                     "kernel_ms": proj_ms, "algorithmic_bytes": bytes_, "algorithmic_flops": flops,
                     "n_union": n_u, "t_roof_us": t_roof * 1e6, "traffic": None,
                     "peak_note": "of measured" if peaks["source"] == "measured" else "of fallback"},
    }
    if keep:
        rec.update(sc=sc, Wd=Wd, stream=stream)
    else:
        sc.close()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return rec


def config_block(rec, args):
    wl = rec["wl"]
    return {"workload": WORKLOADS[rec["name"]][3], "d": wl.d, "V": wl.V, "N": wl.N, "n_tok": wl.n_tok,
            "n_cand": wl.n_cand, "n_sets": wl.n_sets, "modes": list(WORKLOADS[rec["name"]][1]),
            "rows_scored": rec["n_rows_scored"], "plan": rec["plan"],
            "row_dedup": bool(rec.get("dedup")),
            "weights_layout": ("tiled (jet_tile_weights once, before timing)" if rec["w_layout"] == "tiled"
                               else "row-major"),
            "row_gather": (f"rows read in place from a right-padded [N, {rec['gather_rows']}, d] source "
                           "(one compaction launch, then the head's tiled loads)") if rec.get("gather_rows") else None,
            "l2": "inputs larger than L2 (W = %.2f GB > 129 MB L2)" % (wl.W.nbytes / 1e9),
            "step_roofline_us": rec["step_roofline_us"], "step_roofline_frac": rec["step_roofline_frac"],
            "kernel_ms_per_step": {k: v["ms"] / rec["K"] for k, v in rec["prof"].items() if isinstance(v, dict)},
            "ms_per_step_with_kernel_events": rec["ms_prof"] / rec["K"]}


def _round(x, sig=5):
    """Floats to sig significant digits (the line stays short enough for a
    bounded log tail); everything else unchanged, recursively."""
    if isinstance(x, float):
        return float(f"{x:.{sig}g}")
    if isinstance(x, dict):
        return {k: _round(v, sig) for k, v in x.items()}
    if isinstance(x, list):
        return [_round(v, sig) for v in x]
    return x


def compact_config(rec, K, W):
    """One per_config entry: the workload's sizes, throughput, step and head
    time, the roofline of its dominant kernel and the clocks seen."""
    wl, rf = rec["wl"], rec["roofline"]
    keep = ("bound", "achieved", "peak", "unit", "frac", "frac_vs_burst_tensor", "frac_vs_sustained_tensor",
            "traffic", "kernel_ms", "n_union")
    clk = rec["clocks"] or {}
    out = {"d": wl.d, "V": wl.V, "N": wl.N, "n_tok": wl.n_tok, "rows_scored": rec["n_rows_scored"],
           "value": rec["value"], "unit": UNIT, "steps": K, "warmup": W, "ms_per_step": rec["ms_step"],
           "head_ms": rec["head_ms"], "step_roofline_frac": rec["step_roofline_frac"],
           "gpu_launches": rec["gpu_launches"],
           "roofline": {k: rf[k] for k in keep if k in rf},
           "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}}
    return _round(out)


def compact_op(rec):
    """One ops entry: its rate, time per call and roofline note."""
    out = {k: rec[k] for k in ("metric", "value", "unit", "ms", "T") if k in rec}
    if "roofline" in rec:
        out["roofline"] = {k: rec["roofline"][k] for k in ("bound", "achieved", "unit", "frac", "note")
                           if k in rec["roofline"]}
    if "per_union" in rec:
        out["per_union"] = {u: {"path": v["path"], "us_per_call": v["us_per_call"],
                                "projection_us": v["projection_us"], "roofline_us": v["roofline_us"]}
                            for u, v in rec["per_union"].items()}
    return _round(out)


def gpu_arm(args, world, rank, local):
    import numpy as np
    import torch

    from candidate_answer_scoring_gb300 import build as libbuild

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    libbuild.build()
    peaks = load_peaks()

    name = args.workload
    K = args.steps if args.steps is not None else WORKLOADS[name][2]
    W = max(3, args.warmup if args.warmup is not None else 10)
    rec = measure_workload(name, args, dev, world, peaks, K, W, keep=True)
    wl, steps_wl, sc, Wd, stream = rec["wl"], rec["steps_wl"], rec["sc"], rec["Wd"], rec["stream"]
    tokens_per_step = rec["tokens_per_step"]

    cfg = config_block(rec, args)
    cfg.update({"parallelism": f"replicas x{world}", "accumulate": "fp32 (tcgen05 bf16 x bf16 -> fp32 TMEM)",
                "peaks": peaks["source"]})
    line = {
        "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": rec["ms_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": cfg, "gpu_launches": rec["gpu_launches"],
        "roofline": rec["roofline"], "clocks": rec["clocks"],
    }

    # end to end through the public API with host buffers (pinned)
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        hins = []
        h2d = d2h = 0
        for s in steps_wl:
            hi = dict(H=pin(s.H.view(np.int16)).view(torch.bfloat16), tok_row=pin(s.tok_row), tok_ids=pin(s.tok_ids),
                      cand_offsets=pin(s.cand_offsets), set_offsets=pin(s.set_offsets), kind=pin(s.kind),
                      union_ids=None if s.union_ids is None else pin(s.union_ids), T=s.T, mode=s.mode)
            hins.append(hi)
            h2d += sum(v.numel() * v.element_size() for k, v in hi.items() if isinstance(v, torch.Tensor))
            ho = {k: torch.empty(n, dtype=torch.int32 if k == "decision" else torch.float32).pin_memory()
                  for k, n in (("q", s.n_cand), ("decision", s.n_sets), ("expected", s.n_sets),
                               ("confidence", s.n_sets), ("mass", s.n_sets))}
            hi["out"] = ho
            d2h += sum(v.numel() * 4 for v in ho.values())
        Ke = max(3, min(K, 500))
        with torch.cuda.stream(stream):
            # the C-ABI call itself, arguments marshalled once (as a C caller holding these buffers);
            # pipelined: each step's input copy overlaps the previous step's kernels
            calls = [sc.bind_host_call(hi["H"], Wd, hi["tok_row"], hi["tok_ids"], hi["cand_offsets"],
                                       hi["set_offsets"], hi["kind"], hi["T"], hi["mode"], hi["union_ids"],
                                       out=hi["out"], pipelined=True)[0] for hi in hins]
            for _ in range(3):
                for call in calls:
                    call()
            if sc.host_wait() != 0:
                raise RuntimeError("end-to-end warm-up calls failed on the device")
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            for _ in range(Ke):
                for call in calls:
                    call()
            rc = sc.host_wait()      # every step's results are in the host buffers
            el = time.perf_counter() - t0
            if rc != 0:
                raise RuntimeError(f"end-to-end calls: device status {rc}")
        el = max_over_ranks(el, world, dev)
        line["e2e"] = {"value": job_throughput(tokens_per_step, Ke, world, el * 1e3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                       "ms_per_step": 1e3 * el / Ke,
                       "note": "jet_score_sets_host_async (the C call, arguments marshalled once) per mode, "
                               "jet_host_wait at the end: every step copies its pinned host inputs to the device "
                               "(overlapping the previous step's kernels) and its results back to pinned host "
                               "buffers; W resident on the device like any model weight"}
    sc.close()
    del Wd, rec
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()

    # the other full-vocabulary workloads, each timed the same way
    others = [w for w in (args.per_config.split(",") if args.per_config not in ("", "none") else [])
              if w != name]
    if others:
        line["per_config"] = {}
        for other in others:
            r = measure_workload(other, args, dev, world, peaks, K, W)
            line["per_config"][other] = compact_config(r, K, W)

    # the widened ops and restricted mode over larger unions, at the same steps
    if world == 1 and args.ops not in ("", "none"):
        line["ops"] = {}
        for op in args.ops.split(","):
            line["ops"][op] = compact_op(run_op(op, args, K, W, "600,4096"))

    # CPU oracle baseline on a bounded sample (rank 0, one GPU only)
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        n_cand, _ = cpu_sample_cands(steps_wl, target_s=15.0)
        dt, ntok, threads = time_oracle(steps_wl, n_cand)
        sub = _subset(wl, n_cand)
        line["cpu_baseline"] = {
            "value": ntok / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {n_cand} of {wl.n_cand} candidates ({ntok} full-vocab tokens over {sub.N} hidden "
                      f"rows{', plus the restricted pass' if len(steps_wl) > 1 else ''}); {dt:.1f} s",
        }
    line["per_config_workloads"] = {w: WORKLOADS[w][3] for w in line.get("per_config", {})}
    if rank == 0:
        print(json.dumps(_round(line, 7)), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# the widened rows: row dedup, temperature fitting, layer sensitivity
# ---------------------------------------------------------------------------
def time_op(fn, K, W):
    import torch
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def op_arm(args):
    """One JSON line for a widened op (not the headline scoring metric)."""
    from candidate_answer_scoring_gb300 import build as libbuild
    libbuild.build()
    K = args.steps if args.steps is not None else 50
    W = max(3, args.warmup if args.warmup is not None else 5)
    line = run_op(args.op, args, K, W, args.unions)
    print(json.dumps(line), flush=True)
    return 0


def run_op(op, args, K, W, unions):
    """Time one widened op (row dedup, temperature fit, layer sensitivity) or
    restricted mode over the given union sizes; returns its record."""
    import numpy as np
    import torch

    import candidate_answer_scoring_gb300 as jet
    import workloads as wk
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    line = {"op": op, "n_gpus": 1, "steps": K, "warmup": W, "data": "synthetic"}
    if op == "dedup":
        wl = make_workload("large")[0]
        sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
        H = t(wl.H.view(np.int16)).view(torch.bfloat16)
        tok_row = t(wl.tok_row)
        Hu = torch.empty_like(H)
        # the bare C call, arguments marshalled once (as a C caller holding these buffers)
        fn = sc.bind_dedup_rows(H, tok_row, Hu, torch.empty_like(tok_row))
        n_u = fn()
        ms = time_op(fn, K, W)
        nbytes = 2.0 * wl.N * wl.d + 2.0 * 2 * n_u * wl.d + 8.0 * wl.n_tok   # hash read, copy read+write
        line.update(metric="hidden rows deduplicated per second", value=wl.N / (ms / 1e3), unit="rows/s",
                    ms=ms, config={"workload": "large choice H: %d rows x d=%d, %d distinct" % (wl.N, wl.d, n_u)},
                    roofline={"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": peaks["hbm"],
                              "unit": "GB/s", "frac": nbytes / (ms / 1e3) / 1e9 / peaks["hbm"],
                              "note": "synchronous C call (arguments marshalled once): includes the count "
                                      "read-back"})
    elif op == "fit_temperature":
        # scores s(c) of the wide-schema batch from the library's own scoring
        # call; gold labels drawn from q = softmax(s / T0) with T0 = 2.179, so
        # the fit has an interior optimum near T0
        wl = make_workload("wideschema")[0]
        scorer = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
        Wd = t(wl.W.view(np.int16)).view(torch.bfloat16)
        out = scorer.score_sets(t(wl.H.view(np.int16)).view(torch.bfloat16), Wd, t(wl.tok_row), t(wl.tok_ids),
                                t(wl.cand_offsets), t(wl.set_offsets), t(wl.kind), wl.T, wl.mode, None)
        s = out["s"].cpu().numpy().astype(np.float32)
        scorer.close()
        del Wd, out
        torch.cuda.empty_cache()
        T0 = 2.179
        rng = np.random.default_rng(0)
        gold = np.empty(wl.n_sets, np.int32)
        for k in range(wl.n_sets):
            a = s[wl.set_offsets[k]:wl.set_offsets[k + 1]].astype(np.float64) / T0
            q = np.exp(a - a.max())
            gold[k] = rng.choice(q.size, p=q / q.sum())
        sc = jet.JetScorer(64, 100, 4, wl.n_tok)
        args_ = [t(s), t(wl.tok_ids), t(wl.cand_offsets), t(wl.set_offsets), t(gold)]
        fn = sc.bind_fit_temperature(*args_)
        T, nll = fn()
        ms = time_op(fn, K, W)
        line.update(metric="temperature fits per second", value=1e3 / ms, unit="fits/s", ms=ms, T=T, nll=nll,
                    config={"workload": "wide schema: %d sets, %d candidates; gold drawn from q at T0 = %.3f"
                                        % (wl.n_sets, wl.n_cand, T0)},
                    roofline={"bound": "latency", "note": "one CTA, bracketed Newton on 1/T; synchronous C call "
                                                          "(arguments marshalled once)"})
    elif op == "restricted":
        # restricted mode on the binary batch's shape (256 questions, one row
        # each, d=2560, V=248320) over unions of several sizes: each question a
        # binary pair of codes drawn from the union
        line.update(metric="restricted-mode candidate tokens scored per second", unit="tokens/s", per_union={})
        W_dev = None
        for n_union in [int(x) for x in unions.split(",")]:
            wl = wk.union_choice(256, n_union)
            if W_dev is None:
                W_dev = t(wl.W.view(np.int16)).view(torch.bfloat16)
            sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
            Wt = sc.tile_weights(W_dev) if args.w_layout == "tiled" else W_dev
            x = [t(a) for a in (wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets, wl.kind, wl.union_ids)]
            H = t(wl.H.view(np.int16)).view(torch.bfloat16)
            # the bare C call, arguments marshalled once (as a C caller holding these buffers)
            fn = sc.bind_call(H, Wt, x[0], x[1], x[2], x[3], x[4], wl.T, wl.mode, x[5])[0]
            ms = time_op(fn, K, W)
            sc.profile(True)
            time_op(fn, K, 0)
            prof = sc.profile_read()
            sc.profile(False)
            rc = sc.sync_status()
            if rc != 0:
                raise RuntimeError(f"restricted |U|={n_union}: status {rc}")
            kern = {k: v["ms"] * 1e3 / K for k, v in prof.items() if isinstance(v, dict) and v["launches"]}
            path = "tcgen05 head over the staged union" if prof["head"]["launches"] else "mma.sync union kernel"
            proj_us = kern.get("head", kern.get("restricted", 0.0))
            nbytes = 2.0 * n_union * wl.d + 2.0 * wl.N * wl.d
            flops = 2.0 * wl.N * wl.d * n_union
            line["per_union"][str(n_union)] = {
                "path": path, "us_per_call": ms * 1e3, "tokens_per_s": wl.n_tok / (ms / 1e3),
                "kernel_us": kern, "projection_us": proj_us,
                "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                "projection_gbs": nbytes / (proj_us / 1e6) / 1e9 if proj_us else None,
                "projection_tflops": flops / (proj_us / 1e6) / 1e12 if proj_us else None,
                "roofline_us": max(nbytes / (peaks["hbm"] * 1e9), flops / (peaks["bf16"] * 1e12)) * 1e6}
            sc.close()
            del Wt
        line["config"] = {"workload": "256 questions x binary pair of codes from the union, d=2560, V=248320, "
                                      "one row per question, T=2.179; asynchronous calls back to back",
                          "weights_layout": args.w_layout, "peaks": peaks["source"]}
    elif op == "layer_sensitivity":
        rng = np.random.default_rng(0)
        n, L, m = 4096, 64, 64
        offsets = np.arange(0, n * m + 1, m, dtype=np.int32)
        z = rng.normal(-20, 6, size=n * m).astype(np.float32)
        z_skip = (z[None, :] + rng.normal(size=(L, n * m)) * 0.1).astype(np.float32)
        sc = jet.JetScorer(64, 100, 4, 4)
        a = [t(z), t(z_skip), t(offsets)]
        fn = sc.bind_layer_sensitivity(*a, 8, torch.empty((L, n), dtype=torch.float32, device=dev),
                                       torch.empty(L, dtype=torch.float32, device=dev),
                                       torch.empty(8, dtype=torch.int32, device=dev))
        ms = time_op(fn, K, W)
        nbytes = 4.0 * (L + 1) * n * m + 4.0 * L * n
        line.update(metric="layer-input sensitivities per second", value=L * n / (ms / 1e3), unit="1/s", ms=ms,
                    config={"workload": "%d inputs x %d logits x %d layers" % (n, m, L)},
                    roofline={"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": peaks["hbm"],
                              "unit": "GB/s", "frac": nbytes / (ms / 1e3) / 1e9 / peaks["hbm"],
                              "note": "synchronous C call (arguments marshalled once): includes the status "
                                      "read-back"})
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="large", choices=sorted(WORKLOADS),
                    help="the headline workload (default: the large 20k-row batch, the largest)")
    ap.add_argument("--per-config",
                    default="binary,binary-restricted,binary-both,binary-gather,multitoken,wideschema,large-dedup,"
                            "large-rowmajor",
                    help="other workloads timed the same way into the line's per_config block ('none': skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--w-layout", default="tiled", choices=["rowmajor", "tiled"],
                    help="layout of the resident output embedding (tiled: jet_tile_weights once, the default)")
    ap.add_argument("--gather-rows", type=int, default=0, metavar="L",
                    help="read H in place from a right-padded [N, L, d] source (jet_score_sets_gather)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dedup", action="store_true",
                    help="score each distinct hidden row once (jet_dedup_rows before every step)")
    ap.add_argument("--op", default=None, choices=["dedup", "fit_temperature", "layer_sensitivity", "restricted"],
                    help="time one of the widened ops, or restricted mode over larger unions, instead of the "
                         "scoring path")
    ap.add_argument("--unions", default="26,256,600,4096", help="union sizes for --op restricted")
    ap.add_argument("--ops", default="dedup,fit_temperature,layer_sensitivity,restricted",
                    help="widened ops timed into the line's ops block ('none': skip; restricted: 600 and 4096 codes)")
    return ap.parse_args(argv)


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.op is not None:
        return op_arm(args)
    if args.impl == "reference":
        return reference_arm(args, world, rank)
    return gpu_arm(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
