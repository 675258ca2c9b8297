#!/usr/bin/env python3
"""Benchmark of one verification step (plan + verify) on synthetic data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workload (default ``adaptive_hc``): BS=256 requests, K=7 drafted slots each,
V=129280, bf16 logits, temperatures over {0, 0.7, 1.0}, T=256 non-draft tokens,
cost(n) = 1 + 0.004*ceil16(n) -- the adaptive high-concurrency setup, the
configuration that exercises every stage of the path (the planner chooses B,
greedy and sampled requests mix).

One step = sd_plan + sd_verify on device-resident inputs.  Two input sets, each larger than the 129 MB L2, alternate between
steps, so no step reads data the previous one left in L2.  Metric: verified
draft tokens/s (sum of n_i over requests, per second).  Also reported:
achieved HBM bandwidth of the sampling kernel against the measured copy peak,
planner latency, acceptance statistics, an end-to-end figure through the C
ABI from pinned host buffers, and the CPU oracle as a reported baseline.

Under torchrun (N > 1) every rank runs its own independent batch (different
seed): the step shards by request with no data-path collective (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import sdsynth as S  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
PEAKS = ROOT / "MEASURED_PEAKS.json"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="adaptive_hc", choices=sorted(S.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=2026)
    ap.add_argument("--blocks", type=int, default=0, help="sampler CTAs (0 = one per SM)")
    ap.add_argument("--early-exit", action="store_true",
                    help="skip rows of slots after a request's first rejection")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-plan-graph", action="store_true",
                    help="skip the planner CUDA-graph timing (1000 launches)")
    ap.add_argument("--no-detail", action="store_true",
                    help="skip the per-workload blocks and the early-exit comparison")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(elapsed_ms, units, device, world):
    """Weak scaling over replicas: the job takes as long as the slowest rank
    (max of the elapsed times) and does the work of all ranks (sum of the
    units).  Returns (max elapsed ms, total units); one rank returns its own."""
    if world <= 1:
        return float(elapsed_ms), float(units)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units)], device=device, dtype=torch.float64)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def whole_job_rate(total_units, steps, elapsed_ms):
    """Units per second of the whole job: every rank's units of every step over
    the slowest rank's time."""
    return total_units * steps / (elapsed_ms / 1e3)


def hbm_peak():
    try:
        d = json.loads(PEAKS.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("sampler.cu", "sd_device.cuh", "sd_internal.h")
TRAFFIC = ROOT / "profiles" / "dram_traffic.json"


def kernel_sources_hash():
    import hashlib
    src = ROOT / "speculative_decoding_verification_sd_gb300" / "csrc"
    return hashlib.sha256(b"".join((src / n).read_bytes() for n in KERNEL_SOURCES)).hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes (read + write) per sampling launch, from the ncu capture
    recorded in profiles/dram_traffic.json for this workload, or None when
    the kernel sources have changed since those counters were taken (or no
    capture exists)."""
    try:
        d = json.loads(TRAFFIC.read_text())
    except (OSError, ValueError):
        return None
    e = d.get("workloads", {}).get(workload)
    if not e or e.get("kernel_sources_sha256_16") != kernel_sources_hash():
        return None
    return int(e["traffic_bytes_per_launch"])


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.win = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def window(self, t0, t1):
        """Restrict the summary to samples taken between t0 and t1 (monotonic)."""
        self.win = (t0, t1)

    def __exit__(self, *a):
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        win = self.win
        if win is not None:
            inside = [x for x in lines if win[0] <= x[0] <= win[1]]
            lines = inside if inside else lines
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle arms


def oracle_step(w, seed, pi, vi_fn, budget_s, cu=None):
    """Times the oracle (single thread) on a bounded sample of one step:
    the full plan plus the sampling stage for as many requests as fit in
    ``budget_s`` seconds.  Returns (verified draft tokens/s, sample text)."""
    import oracle
    t0 = time.perf_counter()
    pl = oracle.plan(pi["conf"], pi["draft_lens"], w.k_max, pi["cost"], pi["T"], pi["mode"],
                     budget_conf=pi["budget_conf"], budget_draft_lens=pi["budget_draft_lens"])
    t_plan = time.perf_counter() - t0
    cu = pl["cu_seqlens"]
    n = np.diff(cu) - 1
    vi = vi_fn(cu)
    done, tokens, t_ver = 0, 0, 0.0
    for i in range(w.bs):
        t1 = time.perf_counter()
        oracle.verify(vi["target"], vi["draft"] if len(vi["draft"]) else None, w.dtype, w.V,
                      vi["draft_ids"], vi["uniforms"], vi["temps"], cu, w.k_max, requests=[i])
        t_ver += time.perf_counter() - t1
        done += 1
        tokens += int(n[i])
        if t_ver + t_plan >= budget_s:
            break
    # per-request rate scaled to the whole step: plan once + all requests
    per_req = t_ver / done
    step_time = t_plan + per_req * w.bs
    value = float(n.sum()) / step_time
    sample = (f"oracle plan of all {w.bs} requests ({t_plan*1e3:.1f} ms) + sampling stage of "
              f"{done} of {w.bs} requests ({t_ver:.2f} s), scaled to one full step "
              f"({step_time:.2f} s)")
    return value, sample, step_time


def _oracle_share(job):
    """Worker of oracle_all_cores: times the oracle's sampling stage on its
    share of the requests, with the inputs of those requests regenerated from
    the seed (the same bytes as the full step's)."""
    name, seed, reqs, budget_s = job
    import oracle
    w = S.WORKLOADS[name]
    pi = S.plan_inputs(w, seed, 0)
    pl = oracle.plan(pi["conf"], pi["draft_lens"], w.k_max, pi["cost"], pi["T"], pi["mode"],
                     budget_conf=pi["budget_conf"], budget_draft_lens=pi["budget_draft_lens"])
    cu = pl["cu_seqlens"]
    vi = S.verify_inputs(w, seed, 0, cu, pi["draft_lens"], requests=reqs)
    done, t = 0, 0.0
    for i in reqs:
        t0 = time.perf_counter()
        oracle.verify(vi["target"], vi["draft"] if len(vi["draft"]) else None, w.dtype, w.V,
                      vi["draft_ids"], vi["uniforms"], vi["temps"], cu, w.k_max, requests=[i])
        t += time.perf_counter() - t0
        done += 1
        if t >= budget_s:
            break
    return done, t, len(reqs)


def oracle_all_cores(w, seed, budget_s, workers=None):
    """The same oracle on every host core: the requests are dealt round-robin
    to one spawned process per core, each timing its share for up to
    ``budget_s`` seconds.  One step = the plan (one core) + the slowest share
    scaled to all of its requests.  Returns a cpu_baseline-style dict."""
    import multiprocessing as mp
    import oracle
    if workers is None:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    pi = S.plan_inputs(w, seed, 0)
    t0 = time.perf_counter()
    pl = oracle.plan(pi["conf"], pi["draft_lens"], w.k_max, pi["cost"], pi["T"], pi["mode"],
                     budget_conf=pi["budget_conf"], budget_draft_lens=pi["budget_draft_lens"])
    t_plan = time.perf_counter() - t0
    n = np.diff(pl["cu_seqlens"]) - 1
    shares = [list(range(r, w.bs, workers)) for r in range(min(workers, w.bs))]
    with mp.get_context("spawn").Pool(len(shares)) as pool:
        res = pool.map(_oracle_share, [(w.name, seed, sh, budget_s) for sh in shares])
    slowest = max(t / done * total for done, t, total in res)
    step = t_plan + slowest
    sampled = sum(done for done, _, _ in res)
    return {"value": float(n.sum()) / step, "unit": "verified draft tokens/s",
            "cores": len(shares), "kind": "oracle",
            "sample": (f"oracle plan of all {w.bs} requests on one core ({t_plan*1e3:.1f} ms) + "
                       f"sampling stage with the requests dealt to {len(shares)} processes, "
                       f"{sampled} of {w.bs} requests timed, the slowest share scaled to "
                       f"its requests ({slowest:.2f} s)")}


def all_cores_or_error(w, seed, budget_s):
    """oracle_all_cores, or the reason it could not run (the bench line
    is printed either way)."""
    try:
        return oracle_all_cores(w, seed, budget_s)
    except Exception as e:  # noqa: BLE001 -- reported in the JSON line instead
        return {"error": f"{type(e).__name__}: {e}"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    pi = S.plan_inputs(w, args.seed, 0)

    cache = {}

    def vi_fn(cu):
        # the plan is the same every step: build the logits once
        key = cu.tobytes()
        if key not in cache:
            cache.clear()
            cache[key] = S.verify_inputs(w, args.seed, 0, cu, pi["draft_lens"])
        return cache[key]

    vals, times = [], []
    # each step samples whole requests until its share of about two minutes
    # is used up (at least one request per step)
    per_step = min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup))
    for k in range(args.warmup + args.steps):
        v, sample, st = oracle_step(w, args.seed, pi, vi_fn, per_step)
        if k >= args.warmup:
            vals.append(v)
            times.append(st)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": "verified draft tokens/s", "value": value,
        "unit": "verified draft tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "verified draft tokens/s", "cores": 1,
                         "kind": "oracle", "sample": sample,
                         "all_cores": all_cores_or_error(w, args.seed, per_step)},
        "e2e": {"value": value, "unit": "verified draft tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "bs": w.bs, "k_max": w.k_max, "V": w.V,
            "logits": "fp32" if w.dtype == S.F32 else "bf16", "T": w.T,
            "mode": {S.MODE_ADAPTIVE: "adaptive", S.MODE_ALL_SLOTS: "all_slots",
                     S.MODE_UNIFORM_K: "uniform_k"}[w.mode],
            "parallelism": "replicas (independent batch per GPU)",
            "l2": "two alternating input sets, each larger than L2"}


# ---------------------------------------------------------------------------
# GPU arm


class GpuStep:
    """One workload's step on the device: sd_plan + sd_verify on inputs
    already resident in HBM (two input sets, each larger than L2, alternating
    between steps), with the bytes the sampling stage must read."""

    def __init__(self, w, seed, dev, stream, step=0):
        import torch
        import speculative_decoding_verification_sd_gb300 as sd
        self.sd, self.torch, self.w, self.dev, self.stream = sd, torch, w, dev, stream
        bs, k = w.bs, w.k_max
        self.dtype = sd.SD_F32 if w.dtype == S.F32 else sd.SD_BF16
        tdt = torch.float32 if w.dtype == S.F32 else torch.int16
        self.rows_cap = bs * (k + 1)

        def host(a, t):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a, t))

        pi = S.plan_inputs(w, seed, step)
        self.pi = pi
        self.d_lens = host(pi["draft_lens"], np.int32).to(dev)
        self.d_conf = host(pi["conf"], np.float32).to(dev) if pi["conf"] is not None else None
        self.d_cost = host(pi["cost"], np.float32).to(dev) if pi["cost"] is not None else None
        self.cost_len = 0 if pi["cost"] is None else len(pi["cost"])
        # the previous step's confidences and lengths, where the budget comes from them
        self.d_bconf = host(pi["budget_conf"], np.float32).to(dev) if pi["budget_conf"] is not None else None
        self.d_blens = host(pi["budget_draft_lens"], np.int32).to(dev) if pi["budget_draft_lens"] is not None else None
        self.bs_budget = 0 if pi["budget_draft_lens"] is None else len(pi["budget_draft_lens"])
        self.d_B = torch.zeros(1, dtype=torch.int32, device=dev)
        self.d_mask = torch.zeros((bs, max(k, 1)), dtype=torch.uint8, device=dev)
        self.d_nv = torch.zeros(bs, dtype=torch.int32, device=dev)
        self.d_cu = torch.zeros(bs + 1, dtype=torch.int32, device=dev)
        self.d_err = torch.zeros(1, dtype=torch.int32, device=dev)
        # The plan fixes the compacted layout the "target forward" would have
        # produced; the logits rows are built in that layout.
        self.plan()
        torch.cuda.synchronize()
        cu = self.d_cu.cpu().numpy()
        self.cu = cu
        self.n = np.diff(cu) - 1
        t0 = time.perf_counter()
        vi = S.verify_inputs(w, seed, step, cu, pi["draft_lens"])
        self.gen_s = time.perf_counter() - t0
        self.vi = vi
        self.temps = vi["temps"]
        self.B = int(cu[-1]) - bs
        self.rows_t = int(cu[-1])
        self.sets = []
        for _ in range(2):
            tgt = torch.empty((self.rows_cap, w.V), dtype=tdt, device=dev)
            dft = torch.empty((max(bs * k, 1), w.V), dtype=tdt, device=dev)
            tgt[: self.rows_t].copy_(torch.from_numpy(vi["target"].view(np.int16) if w.dtype == S.BF16 else vi["target"]))
            if self.B > 0:
                dft[: self.B].copy_(torch.from_numpy(vi["draft"].view(np.int16) if w.dtype == S.BF16 else vi["draft"]))
            self.sets.append((tgt, dft))
        self.d_ids = torch.zeros(max(bs * k, 1), dtype=torch.int32, device=dev)
        if self.B > 0:
            self.d_ids[: self.B] = torch.from_numpy(vi["draft_ids"]).to(dev)
        self.d_u = torch.from_numpy(vi["uniforms"]).to(dev)
        self.d_t = torch.from_numpy(self.temps).to(dev)
        self.d_acc = torch.zeros(bs, dtype=torch.int32, device=dev)
        self.d_out = torch.zeros((bs, k + 1), dtype=torch.int32, device=dev)
        self.ws_bytes = sd.sd_verify_workspace_bytes(bs, k, w.V, self.dtype)
        self.d_ws = sd.verify_workspace(bs, k, w.V, self.dtype, dev)

    def plan(self, stream=None):
        w = self.w
        self.sd.sd_plan(self.d_conf, self.d_bconf, self.d_blens, self.bs_budget, self.d_lens, w.bs,
                        w.k_max, self.d_cost,
                        self.cost_len, w.T, w.mode, self.d_B, self.d_mask, self.d_nv, self.d_cu,
                        self.d_err, None, 0, stream if stream is not None else self.stream)

    def step(self, s, cfg, ev=None):
        tgt, dft = self.sets[s & 1]
        w = self.w
        if ev:
            ev[0].record(self.stream)
        self.plan()
        if ev:
            ev[1].record(self.stream)
        self.sd.sd_verify_ex(tgt, dft, self.dtype, w.V, self.d_ids, self.d_u, self.d_t, self.d_cu,
                             w.bs, w.k_max, self.d_acc, self.d_out, None, self.d_err, self.d_ws,
                             self.ws_bytes, cfg=cfg, stream=self.stream)
        if ev:
            ev[2].record(self.stream)

    def run(self, steps, warmup, cfg, barrier=None):
        """Times `steps` steps after `warmup`; returns (elapsed ms, per-step
        plan ms, per-step verify ms)."""
        torch = self.torch
        for s in range(warmup):
            self.step(s, cfg)
        (barrier or torch.cuda.synchronize)()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for s in range(steps):
            self.step(s, cfg, evs[s])
        t1.record(self.stream)
        (barrier or torch.cuda.synchronize)()
        return (t0.elapsed_time(t1), [e[0].elapsed_time(e[1]) for e in evs],
                [e[1].elapsed_time(e[2]) for e in evs])

    def bytes_alg(self):
        """Algorithmic bytes of one sampling launch: every target row
        (n_i + 1 of request i) and the draft rows of sampling requests, each
        read once in full, plus the small inputs and outputs."""
        w, n = self.w, self.n
        sampled = self.temps > 0
        rows_read = int((n + 1).sum() + n[sampled].sum())
        small = ((w.bs + 1) * 4 + w.bs * 4 + self.B * 4 + w.bs * (w.k_max + 1) * 4 + w.bs * 4
                 + w.bs * (w.k_max + 1) * 4 + 32 * rows_read)
        return rows_read * w.V * w.elem + small, rows_read

    def bytes_needed(self):
        """Bytes of the rows a request needs once its first rejection is
        known (early exit): target rows up to the accepted length, the draft
        rows of the slots tested, from the outputs of the last step."""
        w, n = self.w, self.n
        acc = self.d_acc.cpu().numpy()
        sampled = self.temps > 0
        t_rows = int((np.minimum(acc, n) + 1).sum())
        d_rows = int(np.minimum(acc + 1, n)[sampled].sum())
        return (t_rows + d_rows) * w.V * w.elem, t_rows + d_rows

    def free(self):
        self.sets = None
        self.d_ws = None
        self.torch.cuda.empty_cache()


def workload_block(gs, steps, warmup, cfg, peak, elapsed=None):
    """ms per step, launch microseconds, algorithmic bytes and the roofline
    fraction of one workload (its sampling kernel against the copy peak)."""
    el, plan_ms, rows_ms = gs.run(steps, warmup, cfg) if elapsed is None else elapsed
    bytes_alg, rows_read = gs.bytes_alg()
    verify_us = 1e3 * statistics.median(rows_ms)
    avg_ms = sum(rows_ms) / len(rows_ms)
    return {"ms_per_step": el / steps, "verify_us_median": verify_us,
            "plan_us_median": 1e3 * statistics.median(plan_ms), "bytes_alg_per_launch": bytes_alg,
            "rows_read": rows_read, "achieved_gbs": bytes_alg / (avg_ms / 1e3) / 1e9,
            "frac": bytes_alg / (avg_ms / 1e3) / 1e9 / peak,
            "verified_draft_tokens_per_s": float(gs.n.sum()) * steps / (el / 1e3),
            "device_err_flag": int(gs.d_err.item())}


def detail_workloads(args, sd, dev, stream, peak):
    """The other workloads, each timed the same way (fewer steps); varlen is
    the mean over its 20 plan steps; early exit beside the all-rows kernel at
    adaptive_hc and stress."""
    out = {}
    steps, warmup = 100, 5
    for name in ("stress", "dense_fixed_k", "uniform_hc"):
        w = S.WORKLOADS[name]
        gs = GpuStep(w, args.seed, dev, stream)
        blk = workload_block(gs, steps, warmup, {"blocks": args.blocks, "flags": 0}, peak)
        if name == "stress":
            ee = workload_block(gs, steps, warmup, {"blocks": args.blocks,
                                                    "flags": sd.SD_VERIFY_EARLY_EXIT}, peak)
            need, rows_need = gs.bytes_needed()
            blk["early_exit"] = {"ms_per_step": ee["ms_per_step"], "verify_us_median": ee["verify_us_median"],
                                 "bytes_needed_per_launch": need, "rows_needed": rows_need,
                                 "speedup_vs_all_rows": blk["verify_us_median"] / ee["verify_us_median"]}
        blk["config"] = config_of(w)
        out[name] = blk
        gs.free()
    w = S.WORKLOADS["varlen_mixed"]
    per = []
    for step in range(20):
        gs = GpuStep(w, args.seed, dev, stream, step=step)
        per.append(workload_block(gs, 20, 3, {"blocks": args.blocks, "flags": 0}, peak))
        gs.free()
    out["varlen_mixed"] = {
        "steps": 20, "ms_per_step": statistics.mean(b["ms_per_step"] for b in per),
        "verify_us_mean": statistics.mean(b["verify_us_median"] for b in per),
        "bytes_alg_per_launch_mean": statistics.mean(b["bytes_alg_per_launch"] for b in per),
        "frac_mean": statistics.mean(b["frac"] for b in per),
        "device_err_flags": sorted({b["device_err_flag"] for b in per}),
        "config": config_of(w)}
    return out


def run_ours(args, w, rank, world, local):
    import torch
    import speculative_decoding_verification_sd_gb300 as sd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    seed = args.seed + 1000 * rank
    stream = torch.cuda.current_stream()
    cfg = {"blocks": args.blocks, "flags": sd.SD_VERIFY_EARLY_EXIT if args.early_exit else 0}
    gs = GpuStep(w, seed, dev, stream)
    bs, k = w.bs, w.k_max
    n = gs.n

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for s in range(args.warmup):
        gs.step(s, cfg)
    barrier()
    with ClockSampler(local) as clk:
        barrier()
        w0 = time.monotonic()
        elapsed_ms, plan_ms, rows_ms = gs.run(args.steps, 0, cfg, barrier)
        clk.window(w0, time.monotonic())
    err = int(gs.d_err.item())
    acc = gs.d_acc.cpu().numpy()

    verified = int(n.sum())
    sampled = gs.temps > 0
    bytes_alg, rows_read = gs.bytes_alg()
    elapsed_ms, total_verified = reduce_over_ranks(elapsed_ms, verified, dev, world)
    value = whole_job_rate(total_verified, args.steps, elapsed_ms)
    rows_avg_ms = sum(rows_ms) / len(rows_ms)
    achieved = bytes_alg / (rows_avg_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()

    # Planner alone: 1000 launches in a CUDA graph.
    plan_graph_us = None
    try:
        if args.no_plan_graph:
            raise RuntimeError("disabled by --no-plan-graph")
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            gs.plan(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                for _ in range(1000):
                    gs.plan(side)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g.replay()
        torch.cuda.synchronize()
        a0.record(stream)
        g.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        plan_graph_us = 1e3 * a0.elapsed_time(a1) / 1000.0
    except Exception as ex:  # graph capture unsupported -> report the event time only
        print(f"# planner graph timing skipped: {ex}", file=sys.stderr)

    # Early exit beside the all-rows kernel on the same inputs.
    ee = None
    if not args.early_exit and not args.no_detail:
        ee_blk = workload_block(gs, min(args.steps, 200), 5,
                                {"blocks": args.blocks, "flags": sd.SD_VERIFY_EARLY_EXIT}, peak)
        need, rows_need = gs.bytes_needed()
        ee = {"verify_us_median": ee_blk["verify_us_median"], "ms_per_step": ee_blk["ms_per_step"],
              "bytes_needed_per_launch": need, "rows_needed": rows_need,
              "speedup_vs_all_rows": (1e3 * statistics.median(rows_ms)) / ee_blk["verify_us_median"]}

    # End to end through the C ABI from pinned host buffers.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, sd, dev, stream, gs.pi, gs.vi, gs.cu, gs.ws_bytes, cfg, gs.rows_cap)
        if world > 1 and e2e is not None:
            e2e_ms, _ = reduce_over_ranks(e2e["_ms"], 0, dev, world)
            e2e["value"] = whole_job_rate(total_verified, args.steps, e2e_ms)
        if e2e is not None:
            e2e.pop("_ms", None)

    workloads = None
    if rank == 0 and not args.no_detail and args.workload == "adaptive_hc":
        gs.free()
        workloads = detail_workloads(args, sd, dev, stream, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        vi = gs.vi
        v, sample, _ = oracle_step(w, seed, gs.pi, lambda c: vi, args.cpu_seconds)
        cpu = {"value": v, "unit": "verified draft tokens/s", "cores": 1, "kind": "oracle",
               "sample": sample, "all_cores": all_cores_or_error(w, seed, args.cpu_seconds)}

    accepted = int(acc.sum())
    pos = np.zeros(k)
    for j in range(k):
        pos[j] = float((acc > j).mean())
    line = {
        "metric": "verified draft tokens/s", "value": value, "unit": "verified draft tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == S.BF16 else "f32",
        "data": "synthetic", "config": config_of(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                     "kernel": "sampler_kernel (sd_verify)", "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "bytes_per_launch": bytes_alg, "avg_launch_ms": rows_avg_ms},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,  # sd_plan and sd_verify per step
        "clocks": clk.summary(),
        "detail": {
            "B": gs.B, "verified_draft_tokens_per_step": verified, "target_rows": gs.rows_t,
            "draft_rows_read": int(n[sampled].sum()), "bytes_alg_per_step": bytes_alg,
            "bytes_per_verified_token": bytes_alg / max(verified, 1),
            "plan_us_event": 1e3 * statistics.median(plan_ms),
            "plan_us_graph": plan_graph_us,
            "verify_us_median": 1e3 * statistics.median(rows_ms),
            "accepted_draft_tokens_per_step": accepted,
            "emitted_tokens_per_s": (accepted + bs) * args.steps / (elapsed_ms / 1e3),
            "mean_acceptance_length": 1.0 + accepted / bs,
            "per_position_cumulative_acceptance": [round(x, 4) for x in pos],
            "device_err_flag": err, "input_generation_s": gs.gen_s,
            "launch": sd.sd_verify_launch_info(w.V, gs.dtype, bs, args.blocks, cfg["flags"]),
            "early_exit": ee,
            "workloads": workloads,
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, w, sd, dev, stream, pi, vi, cu, ws_bytes, cfg, rows_cap):
    """Same step from pinned host buffers: H2D of every input, plan, verify,
    D2H of accepted lengths and tokens, all inside the timed region."""
    import torch
    bs, k = w.bs, w.k_max
    dtype = sd.SD_F32 if w.dtype == S.F32 else sd.SD_BF16
    tdt = torch.float32 if w.dtype == S.F32 else torch.int16
    rows_t = int(cu[-1])
    B = rows_t - bs

    def pin(a, t=None):
        x = torch.from_numpy(np.ascontiguousarray(a if t is None else a.astype(t)))
        return x.pin_memory()

    h_conf = pin(pi["conf"], np.float32) if pi["conf"] is not None else None
    h_lens = pin(pi["draft_lens"], np.int32)
    h_cost = pin(pi["cost"], np.float32) if pi["cost"] is not None else None
    h_tgt = pin(vi["target"].view(np.int16) if w.dtype == S.BF16 else vi["target"])
    h_dft = pin(vi["draft"].view(np.int16) if w.dtype == S.BF16 else vi["draft"])
    h_ids = pin(vi["draft_ids"], np.int32)
    h_u = pin(vi["uniforms"], np.float32)
    h_t = pin(vi["temps"], np.float32)
    h_acc = torch.empty(bs, dtype=torch.int32).pin_memory()
    h_out = torch.empty((bs, k + 1), dtype=torch.int32).pin_memory()
    d_conf = torch.empty_like(h_conf, device=dev) if h_conf is not None else None
    d_lens = torch.empty_like(h_lens, device=dev)
    d_cost = torch.empty_like(h_cost, device=dev) if h_cost is not None else None
    d_tgt = torch.empty((rows_cap, w.V), dtype=tdt, device=dev)
    d_dft = torch.empty((max(bs * k, 1), w.V), dtype=tdt, device=dev)
    d_ids = torch.zeros(max(bs * k, 1), dtype=torch.int32, device=dev)
    d_u = torch.empty_like(h_u, device=dev)
    d_t = torch.empty_like(h_t, device=dev)
    d_B = torch.zeros(1, dtype=torch.int32, device=dev)
    d_mask = torch.zeros((bs, max(k, 1)), dtype=torch.uint8, device=dev)
    d_nv = torch.zeros(bs, dtype=torch.int32, device=dev)
    d_cu = torch.zeros(bs + 1, dtype=torch.int32, device=dev)
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    d_acc = torch.zeros(bs, dtype=torch.int32, device=dev)
    d_out = torch.zeros((bs, k + 1), dtype=torch.int32, device=dev)
    d_ws = sd.verify_workspace(bs, k, w.V, dtype, dev)
    h2d = 0
    for h in (h_conf, h_lens, h_cost, h_tgt, h_dft, h_ids, h_u, h_t):
        if h is not None:
            h2d += h.numel() * h.element_size()
    d2h = h_acc.numel() * 4 + h_out.numel() * 4

    def step():
        if h_conf is not None:
            d_conf.copy_(h_conf, non_blocking=True)
        d_lens.copy_(h_lens, non_blocking=True)
        if h_cost is not None:
            d_cost.copy_(h_cost, non_blocking=True)
        d_tgt[:rows_t].copy_(h_tgt, non_blocking=True)
        if B > 0:
            d_dft[:B].copy_(h_dft, non_blocking=True)
            d_ids[:B].copy_(h_ids, non_blocking=True)
        d_u.copy_(h_u, non_blocking=True)
        d_t.copy_(h_t, non_blocking=True)
        sd.sd_plan(d_conf, None, None, 0, d_lens, bs, k, d_cost,
                   0 if h_cost is None else h_cost.numel(), w.T, w.mode, d_B, d_mask, d_nv, d_cu,
                   d_err, None, 0, stream)
        sd.sd_verify_ex(d_tgt, d_dft, dtype, w.V, d_ids, d_u, d_t, d_cu, bs, k, d_acc, d_out, None,
                        d_err, d_ws, ws_bytes, cfg=cfg, stream=stream)
        h_acc.copy_(d_acc, non_blocking=True)
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(min(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    n = np.diff(cu) - 1
    return {"value": float(n.sum()) * args.steps / (ms / 1e3), "unit": "verified draft tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms / args.steps, "_ms": ms}


def main():
    args = parse()
    rank, world, local = dist_env()
    w = S.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    run_ours(args, w, rank, world, local)


if __name__ == "__main__":
    main()
