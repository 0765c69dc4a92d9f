#!/usr/bin/env python
"""Benchmark of the MoE expert-parallel hot path on GB300.

One step = one pass of the whole hot path on one batch of synthetic routing:
fresh routing plan -> BF16 dispatch (row scatter, zero padding) -> combine
(identity expert: the dispatched rows are the expert outputs), on the
workload P=8 ranks, E=64 experts, S=2048 tokens/rank (T=16384), hidden 7168,
top-6, expert_alignment 128.

Prints ONE JSON line (rank 0).  `value` is the HBM-ledger throughput of the
whole step in GB/s (bytes the method must move: routing plan + dispatch +
combine, see `ledger`) over device time with inputs resident in HBM; the same
line carries tokens/s, the roofline of the dominant kernel, the end-to-end
number through the C ABI with host buffers, the CPU oracle baseline and the
SM clocks seen during the timed region.

`--impl reference` times the CPU oracle (the reference arm) instead.
With --gpus N > 1 (torchrun, one rank per GPU) every rank runs an
independent replica: the path does not shard across GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine GB/s and tokens/s on 1×GB300; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and max over ranks)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(use_cuda: bool):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if use_cuda else "gloo")
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    """Max of a host float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_bytes: float, per_rank_tokens: float, local_ms: float, world: int, steps: int):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    t_ms = max_over_ranks(local_ms)
    per_step_s = t_ms / 1e3 / steps
    return {
        "ms_per_step": t_ms / steps,
        "gbs": world * per_rank_bytes / per_step_s / 1e9,
        "tokens_per_s": world * per_rank_tokens / per_step_s,
    }


# ---------------------------------------------------------------------------
# ledger (algorithmic HBM bytes)
# ---------------------------------------------------------------------------

def ledger(w, n_exp: int, n_valid: int, n_recv: int, fp8: bool = False) -> dict:
    """Bytes the method must move on one device (reads deduplicated, padding
    rows included, the dense S*P*H window not counted)."""
    T, P, E, K, H = w.T, w.P, w.E, w.K, w.H
    plan = (T * K * 8 + T * P + T * P * 4 + T * K * 4 + n_recv * 4 + n_exp * 4
            + 4 * (4 * P * P + 2 * P * P * 16 + 3 * E + P))
    if fp8:
        dispatch = T * H * 2 + n_exp * (H + 4 * H // 128) + T * K * 4
    else:
        dispatch = T * H * 2 + n_exp * H * 2 + T * K * 4
    combine = n_valid * H * 2 + T * K * (4 + 4) + T * H * 2
    return {"plan": plan, "dispatch": dispatch, "combine": combine, "total": plan + dispatch + combine}


def step_ledger(w, n_exp: int, n_valid: int, n_recv: int) -> dict:
    """Ledger of one step of a workload: plan, its dispatches, one combine."""
    led = ledger(w, n_exp, n_valid, n_recv, fp8=w.fp8)
    n_disp = 1 + w.cached_steps
    led["dispatches"] = n_disp
    led["total"] = led["plan"] + n_disp * led["dispatch"] + led["combine"]
    return led


# The source pages' own throughput figures, reported beside ours as context
# only: per-rank bus bandwidth of an interconnect-bound Ascend supernode, FP8
# dispatch and BF16 combine at hidden 7168, top-6, 256 experts; not a target
# for, and not comparable with, one GPU's HBM traffic.
PAGES_CONTEXT = {
    "hardware": "Ascend 950DT 128-card supernode, per-rank bus bandwidth over its interconnect",
    "dispatch_fp8_gbs_per_rank": {"EP8": "373-375", "EP16": "348-352", "EP32": "335-340", "EP128": "313"},
    "combine_bf16_gbs_per_rank": {"EP8": "345-347", "EP128": "272"},
    "dispatch_efficiency": "90-95 % of the physical payload bandwidth limit, EP up to 32",
    "comparable_here": "payload_gbs (received token rows times per-token bytes, no padding)",
}


def payload_ledger(w, n_recv: int) -> int:
    """The pages' 'physical payload' form: received (token, destination) rows
    times the per-token bytes of x, topk_idx and topk_weights, no padding."""
    return n_recv * (w.H * 2 + w.K * 8 + w.K * 4)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if any(a - 0.1 <= r[0] <= b + 0.1 for a, b in self.windows)]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {
            "sm_mhz": statistics.median(r[1] for r in use) if use else None,
            "sm_max_mhz": max(r[2] for r in use) if use else None,
            "reasons": reasons,
            "samples": len(inside),
        }


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel_file: str) -> str:
    with open(os.path.join(ROOT, "combine_ep_plan_gb300", "csrc", kernel_file), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if the kernel source has not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            quoted = re.search(r"`([^`]*)`", v)
            vals[k.strip()] = quoted.group(1) if quoted else v.strip()
    if vals.get("source_sha256") != source_digest(kernel_file):
        return None
    try:  # the number, before any note in parentheses
        return float(vals["dram_bytes_per_launch"].split()[0])
    except (KeyError, ValueError, IndexError):
        return None


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_pass(w, idx, wts, x):
    """One step of the workload by the CPU oracle (cached dispatches reuse x)."""
    import oracle
    pl = oracle.plan(idx, w.S, w.P, w.E, w.A)
    for _ in range(1 + w.cached_steps):
        if w.fp8:
            q, sc = oracle.dispatch_fp8(x, pl, True)
        else:
            y = oracle.dispatch_bf16(x, pl, True)
    if w.expert == "dequant":
        y = oracle.expert_dequant(q, sc)
    elif w.expert == "scale":
        y = oracle.expert_scale(y, pl)
    oracle.combine(y, pl, wts)
    return pl


def oracle_sample(w, min_seconds: float, parallel: bool = False):
    """Whole-workload oracle passes until min_seconds of CPU work -> GB/s.
    parallel: the OpenMP build of the same source (all host threads)."""
    import oracle
    from combine_ep_plan_gb300.inputs import draw_hidden, draw_topk, hidden_seed
    idx, wts = draw_topk(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    times = []
    pl = None
    with oracle.parallel(parallel):
        threads = oracle.threads()
        t_start = time.perf_counter()
        while not times or time.perf_counter() - t_start < min_seconds:
            t0 = time.perf_counter()
            pl = oracle_pass(w, idx, wts, x)
            times.append(time.perf_counter() - t0)
    n_valid = int(np.sum(pl.slot >= 0))
    led = step_ledger(w, pl.num_expanded, n_valid, pl.num_recv_total)
    t = statistics.mean(times)
    return {"gbs": led["total"] / t / 1e9, "tokens_per_s": w.T / t, "seconds_per_pass": t, "passes": len(times),
            "threads": threads}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores
    (its OpenMP build, every host thread)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from combine_ep_plan_gb300.inputs import draw_hidden, draw_topk, hidden_seed
    full = pick_workload(args)
    parallel = oracle.omp_available()
    with oracle.parallel(parallel):
        threads = oracle.threads()
    # each step is a bounded sample of the workload: fewer tokens per rank, so
    # that warmup + steps take about two minutes of CPU time (a full bf16 pass
    # takes about 4 s on one core; the split loops scale with the threads)
    per_thread = 4.0 / min(threads, 8) if parallel else 4.0
    est_full_s = per_thread * full.T / 16384 * full.H / 7168 * full.K / 6 * (1 + 0.2 * full.cached_steps)
    budget = 120.0 / max(1, args.steps + args.warmup)
    S = int(max(8, min(full.S, full.S * budget / est_full_s)))
    w = full.scaled(S=S)
    idx, wts = draw_topk(w)
    x = draw_hidden(w.T, w.H, hidden_seed(w))
    with oracle.parallel(parallel):
        for _ in range(args.warmup):
            oracle_pass(w, idx, wts, x)
        t0 = time.perf_counter()
        pl = None
        for _ in range(args.steps):
            pl = oracle_pass(w, idx, wts, x)
        dt = time.perf_counter() - t0
    n_valid = int(np.sum(pl.slot >= 0))
    led = step_ledger(w, pl.num_expanded, n_valid, pl.num_recv_total)
    gbs = led["total"] * args.steps / dt / 1e9
    build = f"OpenMP C oracle, {threads} threads" if parallel else "single-threaded C oracle"
    sample = f"{args.workload} workload with S={S} tokens/rank (T={w.T}) per step, {build}"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "tokens_per_s": w.T * args.steps / dt,
        "config": workload_config(full, sample_S=S),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def pick_workload(args):
    """The workload of --workload, with --tokens-per-rank tokens per rank if given."""
    from combine_ep_plan_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.tokens_per_rank:
        w = w.scaled(S=args.tokens_per_rank, name=f"{w.name}_S{args.tokens_per_rank}")
    return w


def step_description(w) -> str:
    disp = "FP8 E4M3 dispatch (quantised inside, zero padding)" if w.fp8 else "BF16 dispatch (zero padding)"
    if w.cached_steps:
        disp += f" -> {w.cached_steps} cached-handle dispatches with new x"
    expert = {"identity": "identity expert (the dispatched rows)",
              "dequant": "expert outputs = dequantised rows (prepared once, outside the timing)",
              "scale": "expert outputs = rows scaled by 1+e/E (prepared once, outside the timing)"}[w.expert]
    return f"fresh plan -> {disp} -> {expert} -> combine"


def workload_config(w, sample_S=None) -> dict:
    c = {"workload": f"{w.name}: P={w.P} ranks, E={w.E} experts, S={w.S} tokens/rank (T={w.T}), "
                     f"H={w.H} bf16, top-{w.K} {w.routing}, expert_alignment={w.A}; {step_description(w)}",
         "ranks": w.P, "experts": w.E, "tokens": w.T, "hidden": w.H, "topk": w.K, "expert_alignment": w.A,
         "l2": "no flush: inputs larger than L2 (x %.0f MB, expanded rows ~%.2f GB per step)" % (
             w.T * w.H * 2 / 1e6, w.T * w.K * w.H * 2 / 1e9)}
    if sample_S is not None and sample_S != w.S:  # a sample smaller than the workload
        c["sample_tokens_per_rank"] = sample_S
    return c


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Bench:
    """One workload on the device: inputs resident in HBM, one handle
    re-planned from topk_idx every step (ep_replan recomputes every plan array
    without allocating), outputs sized for the worst case (no host sync), and
    the expert outputs the combine reads, prepared once outside any timing."""

    def __init__(self, ep, w, dev, stream):
        import torch
        from combine_ep_plan_gb300.inputs import bits_to_bf16_tensor, draw_hidden, draw_topk, hidden_seed
        self.ep, self.w, self.dev, self.stream = ep, w, dev, stream
        self.idx_np, self.w_np = draw_topk(w)
        self.x_nps = [draw_hidden(w.T, w.H, hidden_seed(w, i)) for i in range(1 + w.cached_steps)]
        self.idx_t = torch.from_numpy(self.idx_np).to(dev)
        self.wts_t = torch.from_numpy(self.w_np).to(dev)
        self.x_ts = [bits_to_bf16_tensor(xn).to(dev) for xn in self.x_nps]
        self.out_dtype = "fp8" if w.fp8 else "bf16"
        self.cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
        self.recv = torch.empty((self.cap, w.H), dtype=torch.float8_e4m3fn if w.fp8 else torch.bfloat16, device=dev)
        self.recv_sc = torch.empty((self.cap, w.H // 128), dtype=torch.float32, device=dev) if w.fp8 else None
        self.out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        self.h = ep.plan(self.idx_t, w.P, w.E, w.A, stream=stream)
        ep.dispatch(self.h, self.x_ts[0], self.out_dtype, True, recv_x=self.recv, recv_scales=self.recv_sc,
                    stream=stream)
        self.n_exp, self.n_recv = self.h.sizes(stream)
        self.h.check(stream)
        self.n_valid = int((self.idx_t >= 0).sum().item())
        self.led = step_ledger(w, self.n_exp, self.n_valid, self.n_recv)
        if w.expert == "identity":
            self.y = self.recv
        elif w.expert == "dequant":
            self.y = (self.recv.float() * self.recv_sc.repeat_interleave(128, dim=1)).to(torch.bfloat16)
        else:
            e_of_row = torch.repeat_interleave(torch.arange(w.E, device=dev),
                                               torch.diff(self.h.field("expert_offsets").long()))
            self.y = torch.zeros((self.cap, w.H), dtype=torch.bfloat16, device=dev)
            self.y[: len(e_of_row)] = (self.recv[: len(e_of_row)].float()
                                       * (1.0 + e_of_row.float() / w.E)[:, None]).to(torch.bfloat16)
        torch.cuda.synchronize()

    def step(self, ev=None, hh=None, xs=None, idx=None, wts=None, o=None, st=None):
        """Plan -> the fresh dispatch -> the cached dispatches -> combine.  ev:
        five events, recorded at the start, after the plan, after the fresh
        dispatch, after the last dispatch and after the combine."""
        ep = self.ep
        st = st or self.stream
        hh = hh or self.h
        xs = xs if xs is not None else self.x_ts
        if ev is not None:
            ev[0].record(st)
        hh.replan(self.idx_t if idx is None else idx, stream=st)
        if ev is not None:
            ev[1].record(st)
        for i, xi in enumerate(xs):
            ep.dispatch(hh, xi, self.out_dtype, True, recv_x=self.recv, recv_scales=self.recv_sc, stream=st)
            if ev is not None and i == 0:
                ev[2].record(st)
        if ev is not None:
            ev[3].record(st)
        ep.combine(hh, self.y, self.wts_t if wts is None else wts, out=self.out if o is None else o, stream=st)
        if ev is not None:
            ev[4].record(st)

    def capture(self):
        """One step captured in a CUDA graph (the library's launches of
        replan, dispatch and combine), replayed on the bench stream."""
        import torch
        side = torch.cuda.Stream()
        side.wait_stream(self.stream)
        with torch.cuda.stream(side):
            self.step(st=side)
        self.stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(st=torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g

    def timed(self, steps: int, warmup: int, sampler=None, every: int = 4, graph: bool = False) -> dict:
        """warmup untimed steps, then `steps` timed ones between two events.
        Per-phase times come from events recorded between the kernels of every
        `every`-th timed step: an event between two kernels serialises them (the
        next launch can no longer overlap the end of the previous grid), so the
        other steps carry none.  graph: the timed steps replay one captured step
        (no host launch cost between kernels); the per-phase events then come
        from a separate pass of directly launched steps."""
        import torch
        st = self.stream
        if graph:
            return self._timed_graph(steps, warmup, sampler, every)
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        barrier()
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] if i % every == 0 else None
                  for i in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_wall0 = time.time()
        start.record(st)
        for i in range(steps):
            self.step(events[i])
        end.record(st)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        barrier()
        if sampler is not None:
            sampler.mark(t_wall0, t_wall1)
        sampled = [e for e in events if e is not None]
        return {"local_ms": start.elapsed_time(end), "phases": self._phases(sampled), "sampled": len(sampled),
                "launch": "direct"}

    def _phases(self, sampled) -> dict:
        n_cached = self.w.cached_steps
        ph = {
            "plan": [e[0].elapsed_time(e[1]) for e in sampled],
            "dispatch": [e[1].elapsed_time(e[2]) for e in sampled],
            "combine": [e[3].elapsed_time(e[4]) for e in sampled],
            "step": [e[0].elapsed_time(e[4]) for e in sampled],
        }
        if n_cached:
            ph["cached_dispatch"] = [e[2].elapsed_time(e[3]) / n_cached for e in sampled]
        return ph

    def _timed_graph(self, steps, warmup, sampler, every) -> dict:
        import torch
        st = self.stream
        g = self.capture()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        start.record(st)
        for _ in range(steps):
            g.replay()
        end.record(st)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        barrier()
        if sampler is not None:
            sampler.mark(t_wall0, t_wall1)
        local_ms = start.elapsed_time(end)
        sampled = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(max(3, steps // every))]
        for e in sampled:
            self.step(e)
        torch.cuda.synchronize()
        del g
        return {"local_ms": local_ms, "phases": self._phases(sampled), "sampled": len(sampled), "launch": "graph"}

    def roofline(self, phases: dict) -> dict:
        """The dominant kernel's algorithmic bytes per launch over its median
        event time, against the measured copy bandwidth."""
        w, led = self.w, self.led
        peak, peak_src = hbm_peak()
        disp_ms = statistics.median(phases["cached_dispatch"] if w.cached_steps else phases["dispatch"])
        comb_ms = statistics.median(phases["combine"])
        if disp_ms >= comb_ms:
            kname = "ep_dispatch_fp8_kernel" if w.fp8 else "ep_dispatch_copy_kernel"
            kfile, kbytes, kms = "ep_dispatch_kernels.cu", led["dispatch"], disp_ms
        else:
            kname, kfile, kbytes, kms = "ep_combine_kernel", "ep_combine_kernels.cu", led["combine"], comb_ms
        achieved = kbytes / (kms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic(kname, kfile, w.name), "algorithmic_bytes": kbytes}

    def close(self):
        import torch
        self.h.destroy(self.stream)
        torch.cuda.synchronize()


def phase_stats(ph: dict) -> dict:
    """Median and max (ms) of each phase over the sampled steps."""
    out = {}
    for k, v in ph.items():
        out[k] = round(statistics.median(v), 5)
        out[k + "_max"] = round(max(v), 5)
    return out


def workload_line(b: Bench, r: dict, world: int, steps: int) -> dict:
    """A workload's numbers for the `workloads` object of the JSON line."""
    w = b.w
    peak, _ = hbm_peak()
    agg = aggregate(b.led["total"], w.T, r["local_ms"], world, steps)
    return {
        "config": workload_config(w)["workload"], "steps": steps, "sampled_steps": r["sampled"],
        "launch": "one captured step replayed from a CUDA graph" if r["launch"] == "graph"
        else "direct launches from the host",
        "ms_per_step": round(agg["ms_per_step"], 5), "gbs": round(agg["gbs"], 2),
        "tokens_per_s": round(agg["tokens_per_s"], 1), "hbm_roofline_frac": round(agg["gbs"] / world / peak, 4),
        "phases_ms": phase_stats(r["phases"]), "ledger_bytes_per_step": b.led,
        "roofline": b.roofline(r["phases"]),
    }


def run_ours(args):
    import torch

    import combine_ep_plan_gb300 as ep
    from combine_ep_plan_gb300 import build as ep_build
    from combine_ep_plan_gb300.inputs import WORKLOADS, bits_to_bf16_tensor

    rank, world, local = dist_init(use_cuda=True)
    torch.cuda.set_device(local)
    ep_build.build()
    ep.load_library()
    if args.kernels:
        return run_kernel_table(ep, args, local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()

    b = Bench(ep, pick_workload(args), dev, stream)
    w, led, n_recv = b.w, b.led, b.n_recv
    r = b.timed(args.steps, args.warmup, sampler, graph=args.launch == "graph")
    agg = aggregate(led["total"], w.T, r["local_ms"], world, args.steps)
    phases = phase_stats(r["phases"])
    roofline = b.roofline(r["phases"])

    # End to end through the public API with host buffers: every step copies
    # its inputs (x for each dispatch, topk_idx, topk_weights) from pinned host
    # memory to the device and its combined output back to pinned host memory,
    # inside the timed region.  Steps are pipelined as a serving loop would run
    # them: the H2D copies of step i+1 and the D2H copy of step i-1 run on
    # their own streams (copy engines) while step i computes; device buffers
    # are double buffered and every reuse waits on the event of the step that
    # used it.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    x_pin = [[bits_to_bf16_tensor(xn).pin_memory() for xn in b.x_nps] for _ in range(2)]
    idx_pin = torch.from_numpy(b.idx_np).pin_memory()
    w_pin = torch.from_numpy(b.w_np).pin_memory()
    out_pin = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xss = [b.x_ts, [torch.empty_like(xt) for xt in b.x_ts]]
    idxs = [b.idx_t, torch.empty_like(b.idx_t)]
    wtss = [b.wts_t, torch.empty_like(b.wts_t)]
    outs = [b.out, torch.empty_like(b.out)]
    hs = [b.h, ep.plan(b.idx_t, w.P, w.E, w.A, stream=stream)]
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def run_e2e(n):
        ev_done = [None, None]    # compute on buffer i finished
        ev_out = [None, None]     # output of buffer i copied back
        for i in range(n):
            j = i & 1
            with torch.cuda.stream(s_h2d):
                if ev_done[j] is not None:
                    s_h2d.wait_event(ev_done[j])
                for dst, src in zip(xss[j], x_pin[j]):
                    dst.copy_(src, non_blocking=True)
                idxs[j].copy_(idx_pin, non_blocking=True)
                wtss[j].copy_(w_pin, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_h2d)
            stream.wait_event(ev_in)
            if ev_out[j] is not None:
                stream.wait_event(ev_out[j])
            b.step(hh=hs[j], xs=xss[j], idx=idxs[j], wts=wtss[j], o=outs[j])
            ev_done[j] = torch.cuda.Event()
            ev_done[j].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[j])
                out_pin[j].copy_(outs[j], non_blocking=True)
                ev_out[j] = torch.cuda.Event()
                ev_out[j].record(s_d2h)
        return ev_out

    run_e2e(min(4, e2e_steps))
    torch.cuda.synchronize()
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    s2.record(s_h2d)
    last = run_e2e(e2e_steps)
    for ev in last:
        if ev is not None:
            s_d2h.wait_event(ev)
    e2.record(s_d2h)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    sampler.mark(t_wall0, t_wall1)
    agg_e2e = aggregate(led["total"], w.T, s2.elapsed_time(e2), world, e2e_steps)
    for hh in hs:
        status = hh.sync_status(stream)
        if status != ep.EP_OK:
            raise RuntimeError(f"device status {status} after the timed steps")
    hs[1].destroy(stream)
    h2d = sum(xp.numel() * 2 for xp in x_pin[0]) + idx_pin.numel() * 8 + w_pin.numel() * 4
    d2h = out_pin[0].numel() * 2
    del x_pin, out_pin, xss, idxs, wtss, outs

    overlap = run_overlap(ep, w, b.idx_t, b.x_ts[0], b.wts_t, stream, args) if args.overlap else None
    cta_profile = run_cta_profile(ep, w, b.idx_t, b.x_ts[0], b.wts_t, b.y, stream, b.recv, b.recv_sc,
                                  b.out_dtype) if args.cta_profile else None
    b.close()
    del b
    torch.cuda.empty_cache()

    # every other workload, device-timed: fewer steps each
    workloads = {}
    if not args.no_workloads:
        wl_steps = max(4, min(args.steps, args.workload_steps))
        wl_warm = max(3, min(args.warmup, 5))
        for name in WORKLOADS:
            if name == args.workload:
                continue
            bw = Bench(ep, WORKLOADS[name], dev, stream)
            rw = bw.timed(wl_steps, wl_warm, sampler, graph=args.workload_launch == "graph")
            if bw.h.sync_status(stream) != ep.EP_OK:
                raise RuntimeError(f"device status after the {name} steps")
            workloads[name] = workload_line(bw, rw, world, wl_steps)
            bw.close()
            del bw
            torch.cuda.empty_cache()
    clocks = sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        single = oracle_sample(w, min_seconds=6.0, parallel=False)
        multi = oracle_sample(w, min_seconds=6.0, parallel=True) if oracle.omp_available() else None
        best = multi or single
        cpu = {"value": round(best["gbs"], 4), "unit": "GB/s", "cores": best["threads"], "kind": "oracle",
               "sample": f"full {w.name} workload (T={w.T}, H={w.H}), {best['passes']} pass(es) of the step, "
                         + (f"OpenMP build of the C oracle on {best['threads']} threads (the scatter, "
                            "expert and combine row loops split; the plan sequential)" if multi
                            else "single-threaded C oracle"),
               "tokens_per_s": round(best["tokens_per_s"], 1),
               "single_thread": {"value": round(single["gbs"], 4), "unit": "GB/s", "cores": 1,
                                 "passes": single["passes"], "tokens_per_s": round(single["tokens_per_s"], 1)}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(agg["gbs"], 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(agg["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Gumbel-top-k routing, N(0,1) bf16 hidden states)",
            "tokens_per_s": round(agg["tokens_per_s"], 1),
            "hbm_roofline_frac": round(agg["gbs"] / world / hbm_peak()[0], 4),
            "config": workload_config(w),
            "launch": "one captured step replayed from a CUDA graph" if r["launch"] == "graph"
            else "direct launches from the host",
            "phases_ms": {**phases, "sampled_steps": r["sampled"],
                          "stat": "median and max over the sampled steps"},
            "ledger_bytes_per_step": led,
            "payload_gbs": round(world * payload_ledger(w, n_recv) / (agg["ms_per_step"] / 1e3) / 1e9, 2),
            "pages_context": PAGES_CONTEXT,
            "roofline": roofline,
            "e2e": {"value": round(agg_e2e["gbs"], 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(agg_e2e["ms_per_step"], 4),
                    "tokens_per_s": round(agg_e2e["tokens_per_s"], 1), "steps": e2e_steps,
                    "api": "C ABI ep_replan/ep_dispatch/ep_combine via the Python binding",
                    "pipeline": "per step: pinned H2D of inputs, plan, dispatch, combine, D2H of the output; "
                                "copies on their own streams overlap the neighbouring steps' compute"},
            "gpu_launches": (2 + 1 + w.cached_steps) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "workloads": workloads,
        }
        if overlap is not None:
            line["overlap"] = overlap
        if cta_profile is not None:
            line["cta_profile"] = cta_profile
        print(json.dumps(line), flush=True)
    barrier()
    return 0


def run_cpu_table(args):
    """The CPU oracle on every workload, whole passes of the step: the
    single-threaded build and the OpenMP build on all host threads.  Prints
    one JSON line (rank 0 only)."""
    import oracle
    from combine_ep_plan_gb300.inputs import WORKLOADS
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    res = {}
    for name, w in WORKLOADS.items():
        row = {}
        for par in ([False, True] if oracle.omp_available() else [False]):
            smp = oracle_sample(w, min_seconds=args.cpu_seconds, parallel=par)
            row["omp" if par else "single"] = {"gbs": round(smp["gbs"], 4), "threads": smp["threads"],
                                               "seconds_per_pass": round(smp["seconds_per_pass"], 3),
                                               "passes": smp["passes"], "tokens_per_s": round(smp["tokens_per_s"], 1)}
        res[name] = row
    print(json.dumps({"cpu_table": res, "unit": "GB/s of the step's ledger",
                      "timing": f"whole passes of the step until {args.cpu_seconds} s of CPU time"}), flush=True)
    return 0


def run_kernel_table(ep, args, local):
    """Each kernel of the library alone, launched back to back on the
    workload: plan, BF16 dispatch, quantising FP8 dispatch, dispatch of
    pre-quantised FP8 input, dispatch metadata, combine, dispatch backward and
    combine backward.  Per kernel: the average time of --steps launches
    between two events (after --warmup untimed ones), its algorithmic bytes
    and their rate against the measured copy bandwidth.  Prints one JSON line."""
    import torch
    from combine_ep_plan_gb300.inputs import bits_to_bf16_tensor, draw_hidden, draw_topk, hidden_seed
    w = pick_workload(args)
    dev = torch.device("cuda", local)
    st = torch.cuda.current_stream()
    idx_np, w_np = draw_topk(w)
    idx = torch.from_numpy(idx_np).to(dev)
    wts = torch.from_numpy(w_np).to(dev)
    x = bits_to_bf16_tensor(draw_hidden(w.T, w.H, hidden_seed(w))).to(dev)
    h = ep.plan(idx, w.P, w.E, w.A, stream=st)
    n_exp, n_recv = h.sizes(st)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    T, K, H = w.T, w.K, w.H
    n_valid = int((idx >= 0).sum().item())
    n_pad = n_exp - n_valid
    G = H // 128
    # pre-quantised input for the pass-through dispatch (scaffolding, not timed)
    xs = (x.float().view(T, G, 128).abs().amax(dim=2) / 448.0).contiguous()
    xq = (x.float().view(T, G, 128) / xs.clamp_min(1e-30)[:, :, None]).view(T, H).to(torch.float8_e4m3fn)
    recv = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
    recv8 = torch.empty((cap, H), dtype=torch.float8_e4m3fn, device=dev)
    sc8 = torch.empty((cap, G), dtype=torch.float32, device=dev)
    rw = torch.empty(cap, dtype=torch.float32, device=dev)
    rm = torch.empty((cap, 2), dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    gy = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
    gw = torch.empty((T, K), dtype=torch.float32, device=dev)
    ep.dispatch(h, x, "bf16", True, recv_x=recv, stream=st)
    row8 = H + 4 * G
    kernels = {
        "ep_plan_kernel": (lambda: h.replan(idx, stream=st), step_ledger(w, n_exp, n_valid, n_recv)["plan"]),
        "ep_dispatch_copy_kernel (bf16)": (
            lambda: ep.dispatch(h, x, "bf16", True, recv_x=recv, stream=st), T * H * 2 + n_exp * H * 2 + T * K * 4),
        "ep_dispatch_fp8_kernel": (
            lambda: ep.dispatch(h, x, "fp8", True, recv_x=recv8, recv_scales=sc8, stream=st),
            T * H * 2 + n_exp * row8 + T * K * 4),
        "ep_dispatch_copy_kernel (fp8 input)": (
            lambda: ep.dispatch(h, xq, "fp8", True, recv_x=recv8, recv_scales=sc8, stream=st, x_scales=xs),
            T * row8 + n_exp * row8 + T * K * 4),
        "ep_dispatch_metadata_kernel": (
            lambda: ep.dispatch_metadata(h, wts, recv_weights=rw, recv_meta=rm, capacity=cap, stream=st),
            T * K * 8 + n_exp * 12),
        "ep_combine_kernel": (lambda: ep.combine(h, recv, wts, out=out, stream=st),
                              n_valid * H * 2 + T * K * 8 + T * H * 2),
        "ep_combine_kernel (dispatch backward)": (lambda: ep.dispatch_backward(h, recv, grad_x=out, stream=st),
                                                  n_valid * H * 2 + T * K * 4 + T * H * 2),
        "ep_combine_backward_kernel": (
            lambda: ep.combine_backward(h, out, recv, wts, zero_pad=True, grad_y=gy, grad_weights=gw, stream=st),
            T * H * 2 + 2 * n_valid * H * 2 + T * K * 12 + n_pad * H * 2),
    }
    peak, _ = hbm_peak()
    res = {}
    for name, (fn, nbytes) in kernels.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.steps):
            fn()
        e.record(st)
        torch.cuda.synchronize()
        us = a.elapsed_time(e) * 1e3 / args.steps
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 2), "bytes": int(nbytes), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    if h.sync_status(st) != ep.EP_OK:
        raise RuntimeError("device status after the kernel table")
    h.destroy(st)
    print(json.dumps({"kernels": res, "workload": workload_config(w)["workload"], "launches_each": args.steps,
                      "timing": "back-to-back launches between two CUDA events, after warm-up; "
                                "bytes: algorithmic, per launch", "peak_gbs": peak}), flush=True)
    return 0


def run_overlap(ep, w, idx_t, x_t, wts_t, stream, args):
    """The pattern of an overlapped shared expert: a fresh dispatch issued on
    the handle's communication stream under an SM budget while a shared-expert
    FFN (two bf16 GEMMs, hidden -> 2048 -> hidden, through torch) runs on the
    compute stream; then the combine adds the shared output as its bias.
    Times per step: both in series on one stream, and overlapped, for several
    SM budgets, plus each part alone."""
    import torch
    F = 2048
    g = torch.Generator(device=x_t.device).manual_seed(11)
    w_up = (torch.randn((w.H, F), device=x_t.device, generator=g) / w.H ** 0.5).to(torch.bfloat16)
    w_down = (torch.randn((F, w.H), device=x_t.device, generator=g) / F ** 0.5).to(torch.bfloat16)
    cap = ep.worst_expanded_rows(w.T, w.K, w.E, w.A)
    recv = torch.empty((cap, w.H), dtype=torch.bfloat16, device=x_t.device)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=x_t.device)
    hid = torch.empty((w.T, F), dtype=torch.bfloat16, device=x_t.device)
    shared = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=x_t.device)
    h = ep.plan(idx_t, w.P, w.E, w.A, stream=stream)

    def shared_expert():
        torch.matmul(x_t, w_up, out=hid)
        torch.matmul(hid, w_down, out=shared)

    def serial():
        h.replan(idx_t, stream=stream)
        ep.dispatch(h, x_t, "bf16", True, recv_x=recv, stream=stream)
        shared_expert()
        ep.combine(h, recv, wts_t, out=out, stream=stream, bias=shared)

    def overlapped():
        pend = ep.dispatch_async(h, x_t, "bf16", True, recv_x=recv, topk_idx=idx_t, stream=stream)
        shared_expert()
        pend.wait(counts=False)  # worst-case capacity: no count readback needed
        ep.combine(h, recv, wts_t, out=out, stream=stream, bias=shared)

    def dispatch_only():
        h.replan(idx_t, stream=stream)
        ep.dispatch(h, x_t, "bf16", True, recv_x=recv, stream=stream)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    n = max(5, min(50, args.steps // 4))
    res = {"shared_expert": f"x[{w.T},{w.H}] @ [{w.H},{F}] @ [{F},{w.H}], bf16 torch matmul",
           "steps": n, "dispatch_alone_ms": round(timed(dispatch_only, n), 4),
           "shared_expert_alone_ms": round(timed(shared_expert, n), 4)}
    h.set_num_sms(0)
    res["serial_ms"] = round(timed(serial, n), 4)
    best = None
    res["overlapped_ms"] = {}
    for sms in (0, 8, 16, 32, 64):
        h.set_num_sms(sms)
        t = timed(overlapped, n)
        res["overlapped_ms"][str(sms)] = round(t, 4)
        if best is None or t < best[1]:
            best = (sms, t)
    h.set_num_sms(0)
    hideable = min(res["dispatch_alone_ms"], res["shared_expert_alone_ms"])
    res["best_num_sms"] = best[0]
    res["hidden_frac"] = round((res["serial_ms"] - best[1]) / hideable, 3) if hideable > 0 else None
    if h.sync_status(stream) != ep.EP_OK:
        raise RuntimeError("device status after the overlap runs")
    h.destroy(stream)
    return res


def run_cta_profile(ep, w, idx_t, x_t, wts_t, y, stream, recv, recv_sc, out_dtype):
    """One step (plan, dispatch, combine) with per-CTA profile records."""
    import torch
    h = ep.plan(idx_t, w.P, w.E, w.A, stream=stream)
    h.profile_begin(1 << 21)
    h.replan(idx_t, stream=stream)
    ep.dispatch(h, x_t, out_dtype, True, recv_x=recv, recv_scales=recv_sc, stream=stream)
    ep.combine(h, y, wts_t, out=torch.empty((w.T, w.H), dtype=torch.bfloat16, device=x_t.device),
               stream=stream)
    rec, dropped = h.profile_end(stream)
    if h.sync_status(stream) != ep.EP_OK or dropped:
        raise RuntimeError("profiled step failed or dropped records")
    h.destroy(stream)
    rows = []
    for r in ep.summarize_profile(rec):
        row = {k.replace("_ns", "_us"): (round(v / 1e3, 3) if "_ns" in k else v) for k, v in r.items()}
        row["gbs"] = round(r["gbs"], 1)
        rows.append(row)
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=800)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads (the `workloads` object of the line)")
    ap.add_argument("--workload-steps", type=int, default=40,
                    help="timed steps of each other workload (at most --steps)")
    ap.add_argument("--launch", choices=["direct", "graph"], default="graph",
                    help="timed steps of the headline workload: direct launches, or one captured step "
                         "replayed from a CUDA graph")
    ap.add_argument("--workload-launch", choices=["direct", "graph"], default="graph",
                    help="the same for the other workloads")
    ap.add_argument("--cpu-table", action="store_true",
                    help="instead of the step: the CPU oracle's rate on every workload (no GPU)")
    ap.add_argument("--cpu-seconds", type=float, default=6.0)
    ap.add_argument("--kernels", action="store_true",
                    help="instead of the step: time each kernel of the library alone on the workload")
    ap.add_argument("--overlap", action="store_true",
                    help="also time dispatch issued on the communication stream under an SM budget, "
                         "overlapped with a shared-expert FFN on the compute stream")
    ap.add_argument("--cta-profile", action="store_true",
                    help="also run one step with per-CTA profile records and summarise them")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="run the workload with this many tokens per rank instead of its own (a smaller "
                         "case of the same kernels, e.g. for a profiler capture); it is then named "
                         "<workload>_S<n>")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps, reported as used
    if args.impl == "reference":
        return run_reference(args)
    if args.cpu_table:
        return run_cpu_table(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
