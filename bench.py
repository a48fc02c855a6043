#!/usr/bin/env python3
"""Benchmark of the MoE routing hot path on GB300: route -> dispatch -> permute -> combine.

One step = one pass of the whole path over one batch of synthetic tokens
(default workload skewed_zipf_n65536_h4096_e64_k2: N=65536, H=4096, E=64, K=2
with a Zipf-like per-expert logit bias -- the largest of the five workloads),
inputs resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W untimed warm-up steps, then K timed steps.  Before every timed step
a 256 MiB buffer is written to flush the 129 MB L2; each step is bracketed by
CUDA events on the launching stream (the flush is outside the brackets); for
the per-kernel figures every call of the step is also timed alone, the L2
flushed before each call.  Under torchrun each rank
runs its own replica on its own token batch (weak scaling, no collective on
the data path); the reported time is the max over ranks.  Every rank shares one gate weight
(the replica layout: tokens differ per rank, W_gate does not).

--impl reference times the CPU oracle (oracle/, fp64 C) on the same workload on
this machine's host cores: the only other implementation of this path here.
Each of its steps is a bounded sample of the workload (its first T tokens, T
sized so that the whole run takes about REF_BUDGET_S seconds).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading

import numpy as np
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "route+dispatch+combine tokens/s on 1 GB300; % of HBM roofline per kernel"
NOMINAL_HBM_GBS = 8000.0   # "about 8 TB/s": the nominal figure the per-kernel fractions are also quoted against
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
E2E_UNIT = 64          # pipelined end-to-end steps per CUDA graph
E2E_BUFFERS = 2        # buffer sets of the pipelined end-to-end steps (3 or 4 measured no faster)
L2_FLUSH_BYTES = 256 << 20
REF_BUDGET_S = 120.0   # wall time of the reference arm's warm-up + timed steps


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=mi.BENCH_WORKLOAD, choices=sorted(mi.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--record-traffic", metavar="NCU_CSV", default=None,
                   help="parse an ncu --csv launch log of this workload's step (metrics dram__bytes_read.sum, "
                        "dram__bytes_write.sum) and write its per-call DRAM bytes into profiles/dram_traffic.csv, "
                        "with the digest of each kernel's current source; runs nothing on a GPU")
    p.add_argument("--tokens", type=int, default=0,
                   help="run the workload's shape with this many tokens instead of its N (for profiler "
                        "captures on a smaller case; the line then names the workload NAME@N=T)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--e2e-buffers", type=int, default=E2E_BUFFERS, help="buffer sets of the pipelined e2e steps")
    p.add_argument("--no-torch-naive", action="store_true", help="skip the stock-PyTorch comparison figure")
    p.add_argument("--route-stats", action="store_true",
                   help="route with the router statistics (moe_route_stats: logsumexp + expert histogram) and "
                        "add moe_load_stats (max/mean, p95/mean, z-loss) to every step")
    p.add_argument("--scale-format", default="fp32", choices=["fp32", "ue8m0"],
                   help="E4M3 block-scale output of fp8 workloads: fp32 scales or UE8M0 exponent bytes")
    p.add_argument("--ep-size", type=int, default=0,
                   help="dispatch as moe_dispatch_ep with this many EP ranks (dedup'd send rows, expand_idx)")
    p.add_argument("--apart", action="store_true",
                   help="route and dispatch as two calls even where moe_route_dispatch runs them as one launch")
    p.add_argument("--residual", action="store_true",
                   help="combine with the residual connection (forward_aggregate: moe_combine_residual)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


KERNEL_SOURCES = {"route": "route_tc.cu", "dispatch": "dispatch.cu", "combine": "combine.cu",
                  "route_dispatch": "route_tc.cu"}
# ncu DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum), one row
# per (kernel, workload), with a digest of the kernel's source at capture time
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.csv")


def code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace runs collapsed (string and
    character literals kept), so that a digest changes with the code, not its comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def source_digest(kernel: str) -> str:
    import hashlib
    path = os.path.join(ROOT, "combine_moe_route_02_gb300", "csrc", KERNEL_SOURCES[kernel])
    with open(path, encoding="utf-8") as f:
        return hashlib.sha256(code_only(f.read()).encode()).hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, path: str = None):
    """DRAM bytes per launch (read + write) from the ncu capture table, or None when
    there is no row for this kernel/workload or the kernel's source has changed since
    the capture (each row records a digest of the source)."""
    import csv
    try:
        with open(path or TRAFFIC_FILE, newline="") as f:
            rows = list(csv.DictReader(f))
    except OSError:
        return None
    for r in rows:
        if r.get("kernel") == kernel and r.get("workload") == workload:
            try:
                value = float(r["dram_bytes_per_launch"])
            except (KeyError, TypeError, ValueError):
                continue
            return value if r.get("source_digest") == source_digest(kernel) else None
    return None


NCU_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}


def ncu_launches(path: str):
    """The launches of an ncu --csv log in launch order: [(kernel name, dram bytes read,
    dram bytes written)], bytes converted from ncu's units."""
    import csv
    import io
    with open(path, newline="") as f:
        lines = f.read().splitlines()
    start = next(i for i, ln in enumerate(lines) if ln.startswith('"ID"'))
    per = {}
    order = []
    for r in csv.DictReader(io.StringIO("\n".join(lines[start:]))):
        key = r["ID"]
        if key not in per:
            per[key] = {"name": r["Kernel Name"]}
            order.append(key)
        name = r["Metric Name"]
        if name in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            per[key][name] = float(r["Metric Value"].replace(",", "")) * NCU_UNITS.get(r["Metric Unit"], 1)
    return [(per[k]["name"], per[k].get("dram__bytes_read.sum"), per[k].get("dram__bytes_write.sum"))
            for k in order]


def record_traffic(ncu_csv: str, w: mi.Workload, path: str = None) -> dict:
    """Per-call DRAM bytes of the step from an ncu launch log, written into the traffic table.

    Each call's figure is the smallest over its captured launches (they agree to a fraction
    of a percent); the dispatch call is its counting-sort launch plus, where the row copy runs
    apart, the permute launch that follows it.  Returns {call: (read, write)}."""
    import csv
    path = path or TRAFFIC_FILE
    calls = {}

    def add(call, rd, wr):
        if rd is None or wr is None:
            return
        if call not in calls or rd + wr < sum(calls[call]):
            calls[call] = (rd, wr)

    launches = ncu_launches(ncu_csv)
    i = 0
    while i < len(launches):
        name, rd, wr = launches[i]
        if "route_tc_kernel" in name:
            add("route_dispatch" if ", 1, 1>" in name else "route", rd, wr)
        elif "dispatch_fused_kernel" in name:
            if i + 1 < len(launches) and "permute_kernel" in launches[i + 1][0]:
                _, rd2, wr2 = launches[i + 1]
                if None not in (rd, wr, rd2, wr2):
                    add("dispatch", rd + rd2, wr + wr2)
                i += 1
            else:
                add("dispatch", rd, wr)
        elif "combine_kernel" in name:
            add("combine", rd, wr)
        i += 1
    kb = kernel_bytes(w)
    with open(path, newline="") as f:
        rows = list(csv.DictReader(f))
    fields = ["kernel", "workload", "dram_bytes_per_launch", "source_digest", "read", "write",
              "algorithmic_bytes", "capture"]
    rows = [r for r in rows if not (r["workload"] == w.name and r["kernel"] in calls)]
    for call, (rd, wr) in sorted(calls.items()):
        rows.append({"kernel": call, "workload": w.name, "dram_bytes_per_launch": int(rd + wr),
                     "source_digest": source_digest(call), "read": int(rd), "write": int(wr),
                     "algorithmic_bytes": kb[call],
                     "capture": os.path.basename(ncu_csv) + " (bench.py --record-traffic)"})
    with open(path, "w", newline="") as f:
        wtr = csv.DictWriter(f, fieldnames=fields, lineterminator="\n")
        wtr.writeheader()
        wtr.writerows(rows)
    return calls


def max_over_ranks(value: float, dist_mod=None, device=None) -> float:
    """The largest `value` over all ranks (the job is as slow as its slowest rank)."""
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(counts, dist_mod=None):
    """The job-wide expert histogram: every rank's counts added up (an all-reduce of E
    integers, for the load statistics only -- nothing on the data path exchanges tokens)."""
    if dist_mod is None:
        return counts
    import torch
    t = counts.to(torch.int64)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.SUM)
    return t.to(counts.dtype)


def weak_scaling_tokens_per_s(world: int, tokens_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank routes its own tokens_per_rank each step."""
    return world * tokens_per_rank * steps / (total_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- algorithmic bytes per launch

def kernel_bytes(w: mi.Workload, residual: bool = False, ue8m0: bool = False, ep_rows=None):
    N, H, E, K = w.N, w.H, w.E, w.K
    route = N * 2 * H + H * E * 2 + N * K * 8 + (E * 4 if w.skew else 0)
    meta = N * K * 4 * 3                      # read topk_idx, write row_map and src_slot
    permute = N * 2 * H + N * K * 2 * H       # read X once, write K rows (bf16)
    if w.fp8:
        permute += N * K * H + N * K * (H // 128) * (1 if ue8m0 else 4)
    combine = N * K * 2 * H + N * 2 * H + N * K * 8
    if residual:
        combine += N * 2 * H                  # read the residual row
    if ep_rows is not None:
        # EP dispatch: read topk_idx, write row_map, slot_send_row, expand_idx and
        # send_token, read X once and write one row per (token, rank)
        return {"route": route, "dispatch": N * K * 4 * 4 + ep_rows * 4 + N * 2 * H + ep_rows * 2 * H,
                "combine": combine}
    # route + dispatch in one launch: X is read once by the algorithm (the row copy
    # takes it again from L2)
    return {"route": route, "dispatch": meta + permute, "combine": combine,
            "route_dispatch": route + meta + permute - N * 2 * H}


# ----------------------------------------------------------------- clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-i={self.gpu}", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, val in zip(names, r[3][5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ----------------------------------------------------------------- CPU oracle baseline

def oracle_pass(oracle, Xb, Wb, bias, w: mi.Workload, Y, R=None, ue8m0=False, ep_size=0, stats=False):
    """One pass of the oracle over the workload: route, dispatch, permute, combine
    (with the residual R when given; UE8M0 block scales when ue8m0; the EP
    metadata and dedup'd send rows when ep_size; the router statistics when stats)."""
    if stats:
        idx, tw, L = oracle.route(Xb, Wb, bias, w.K, w.renorm, want_logits=True)
        counts = np.bincount(idx.ravel(), minlength=w.E).astype(np.int32)
        oracle.load_stats(counts, oracle.logsumexp(L), 1e-3)
    else:
        idx, tw = oracle.route(Xb, Wb, bias, w.K, w.renorm)
    if ep_size:
        ep = oracle.dispatch_ep(idx, w.E, ep_size)
        row_map = ep["row_map"]
        np.take(Xb, ep["send_token"], axis=0)      # the dedup'd send rows (a library gather)
    else:
        counts, offsets, row_map, src_slot = oracle.dispatch(idx, w.E)
        if w.fp8 and ue8m0:
            oracle.permute(Xb, row_map, w.K)
            oracle.permute_ue8m0(Xb, row_map, w.K)
        else:
            oracle.permute(Xb, row_map, w.K, fp8=w.fp8)
    if R is None:
        oracle.combine(Y, row_map, tw)
    else:
        oracle.combine_residual(Y, row_map, tw, R)
    return idx


def residual_rows(w: mi.Workload, rank: int = 0):
    """Synthetic residual stream [N,H] bf16 for the forward_aggregate variant."""
    return mi.random_bf16((w.N, w.H), seed=1000 + rank)


def oracle_sample(w: mi.Workload, T: int, X=None, W=None, bias=None):
    """The first T tokens of the workload as the oracle takes them: (Xb, Wb, bias,
    Y), with the expert outputs Y of that sample built by the oracle (untimed)."""
    import oracle
    if X is None:
        X, W, bias = mi.make_workload_inputs(w)
    Xb, Wb = mi.bf16_bits(X[:T]), mi.bf16_bits(W)
    b = None if bias is None else bias.numpy()
    Y = oracle.run_path(Xb, Wb, b, w.K, w.renorm, w.fp8)["Y"]
    return Xb, Wb, b, Y


def oracle_seconds_per_token(w: mi.Workload, Xb, Wb, b, Y, probe_tokens: int, **kw) -> float:
    """Host seconds per token of one oracle pass, measured on the first probe_tokens tokens."""
    import oracle
    T = min(probe_tokens, Xb.shape[0])
    sw = mi.Workload(w.name, T, w.H, w.E, w.K, w.renorm, w.fp8, w.skew)
    Ys = Y if T == Xb.shape[0] else oracle.run_path(Xb[:T], Wb, b, w.K, w.renorm, w.fp8)["Y"]
    t0 = time.perf_counter()
    oracle_pass(oracle, Xb[:T], Wb, b, sw, Ys, **kw)
    return (time.perf_counter() - t0) / T


def cpu_baseline(w: mi.Workload, seconds: float, max_reps: int = 1000, residual: bool = False,
                 ue8m0: bool = False, ep_size: int = 0, stats: bool = False):
    """The oracle on the host cores over a bounded sample of the workload: passes over
    its first T tokens (T sized for about one second per pass) for `seconds`, then on
    one host thread over a smaller sample for about seconds / 2."""
    import oracle
    X, W, bias = mi.make_workload_inputs(w)
    kw = dict(ue8m0=ue8m0, ep_size=ep_size, stats=stats)
    cores = oracle.num_threads()

    def run(threads, per_pass_s, limit_s):
        oracle.set_num_threads(threads)
        probe = mi.Workload(w.name, min(w.N, 1024), w.H, w.E, w.K, w.renorm, w.fp8, w.skew)
        pXb, pWb, pb, pY = oracle_sample(probe, probe.N, X, W, bias)
        spt = oracle_seconds_per_token(w, pXb, pWb, pb, pY, probe.N, **kw)
        T = int(max(64, min(w.N, per_pass_s / max(spt, 1e-12))))
        sw = mi.Workload(w.name, T, w.H, w.E, w.K, w.renorm, w.fp8, w.skew)
        Xb, Wb, b, Y = oracle_sample(sw, T, X, W, bias)
        R = mi.bf16_bits(residual_rows(w)[:T]) if residual else None
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle_pass(oracle, Xb, Wb, b, sw, Y, R, **kw)
            reps += 1
            el = time.perf_counter() - t0
            if el >= limit_s or reps >= max_reps:
                return T, reps, el

    try:
        T, reps, el = run(cores, min(1.0, seconds / 5), seconds)
        T1, reps1, el1 = run(1, min(1.0, seconds / 10), seconds / 2)
    finally:
        oracle.set_num_threads(cores)
    return {"value": reps * T / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the first {T} of the {w.N} tokens of {w.name}, {reps} passes of route+dispatch+permute+"
                      f"combine in fp64 C, {el:.1f} s",
            "single_thread": {"value": reps1 * T1 / el1, "unit": UNIT, "cores": 1,
                              "sample": f"the first {T1} tokens, {reps1} passes of the same, {el1:.1f} s"},
            "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name as lscpu prints it (else what the platform module knows)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def torch_naive(Xd, Wd, bd, w: mi.Workload, Y, flush, reps: int = 100):
    """The same step as a chain of stock PyTorch ops on the same GPU (a context figure, not
    a product path): fp32 logits through HBM, softmax, topk, renorm, stable argsort of the
    expert ids, index_select for the permute (+ a per-block E4M3 cast for fp8 workloads),
    and an index_select + weighted sum for the combine."""
    import torch

    N, H, E, K = w.N, w.H, w.E, w.K
    ar = torch.arange(N * K, device=Xd.device)

    def step():
        L = Xd.float() @ Wd.float()
        if bd is not None:
            L = L + bd
        p = torch.softmax(L, dim=1)
        idx = torch.topk(L, K, dim=1).indices
        tw = p.gather(1, idx)
        if w.renorm:
            tw = tw / tw.sum(dim=1, keepdim=True)
        flat = idx.flatten()
        order = torch.argsort(flat, stable=True)              # row -> slot
        torch.bincount(flat, minlength=E)
        Xp = Xd.index_select(0, order // K)
        if w.fp8:
            blk = Xp.float().view(N * K, H // 128, 128)
            t = blk.abs().amax(dim=-1, keepdim=True).clamp_min(1e-4) / 448.0
            s = torch.exp2(torch.ceil(torch.log2(t)))
            (blk / s).to(torch.float8_e4m3fn)
        row_map = torch.empty_like(order)
        row_map[order] = ar
        (Y.index_select(0, row_map).view(N, K, H).float() * tw.unsqueeze(-1)).sum(dim=1).to(torch.bfloat16)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    m = statistics.fmean(ms)
    return {"value": N / (m * 1e-3), "unit": UNIT, "ms_per_step": m, "steps": reps,
            "what": "stock PyTorch ops on the same GPU: fp32 matmul, softmax, topk, renorm, stable argsort, "
                    "index_select permute (+ E4M3 cast), index_select + weighted sum; L2 flushed between steps"}


def run_reference(args, rank, world):
    """The reference arm: the oracle on this machine's host cores, rank 0 only.  Each
    step is one pass over the first T tokens of the workload, T sized so that the
    warm-up and timed steps take about REF_BUDGET_S seconds (all N tokens when they fit)."""
    if rank != 0:
        return
    import oracle
    w = mi.WORKLOADS[args.workload]
    X, W, bias = mi.make_workload_inputs(w)
    ue8m0 = args.scale_format == "ue8m0"
    kw = dict(ue8m0=ue8m0, ep_size=args.ep_size, stats=args.route_stats)
    probe = mi.Workload(w.name, min(w.N, 1024), w.H, w.E, w.K, w.renorm, w.fp8, w.skew)
    pXb, pWb, pb, pY = oracle_sample(probe, probe.N, X, W, bias)
    spt = oracle_seconds_per_token(w, pXb, pWb, pb, pY, probe.N, **kw)
    T = int(max(64, min(w.N, REF_BUDGET_S / max(1, args.steps + args.warmup) / max(spt, 1e-12))))
    sw = mi.Workload(w.name, T, w.H, w.E, w.K, w.renorm, w.fp8, w.skew)
    Xb, Wb, b, Y = oracle_sample(sw, T, X, W, bias)
    R = mi.bf16_bits(residual_rows(w)[:T]) if args.residual else None
    for _ in range(args.warmup):
        oracle_pass(oracle, Xb, Wb, b, sw, Y, R, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(oracle, Xb, Wb, b, sw, Y, R, **kw)
    el = time.perf_counter() - t0
    value = args.steps * T / el
    sample = (f"the first {T} of the {w.N} tokens of {w.name} per step (all of them when T == N), "
              "route+dispatch+permute+combine in fp64 C")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(w.as_dict(), **combine_config(args)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample, "tokens_per_step": T},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def fused_step(args) -> bool:
    """Whether the step makes route and dispatch one call (moe_route_dispatch): not for E4M3
    output, the EP metadata, the router statistics, or when --apart asks for three calls."""
    return not (args.apart or args.ep_size or args.route_stats or mi.WORKLOADS[args.workload].fp8)


def combine_config(args):
    c = {"dispatch": f"moe_dispatch_ep, ep_size {args.ep_size}"} if args.ep_size else {}
    c["combine"] = ("forward_aggregate: weighted sum + residual, one bf16 rounding" if args.residual
                    else "weighted sum")
    if args.route_stats:
        c["route"] = "moe_route_stats (logsumexp + expert histogram) and moe_load_stats every step"
    if mi.WORKLOADS[args.workload].fp8:
        c["fp8_scales"] = args.scale_format
    if fused_step(args):
        c["calls"] = "moe_route_dispatch (route + dispatch + row copy, one launch where split-K) + moe_combine"
    else:
        c["calls"] = "moe_route, moe_dispatch, moe_combine"
    return c


# ----------------------------------------------------------------- the GPU arm

def run_ours(args, rank, world, local):
    import torch

    import combine_moe_route_02_gb300 as moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    moe.build()
    moe.lib()

    w = mi.WORKLOADS[args.workload]
    X, W, bias = mi.make_replica_inputs(w, rank)   # each rank its own tokens, one shared gate
    Xd, Wd = X.to(dev), W.to(dev)
    bd = None if bias is None else bias.to(dev)
    N, H, E, K = w.N, w.H, w.E, w.K

    idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    tw = torch.empty((N, K), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    d = moe.dispatch(moe.route(Xd, Wd, K, bd, w.renorm, topk_idx=idx, topk_w=tw)[0], E, Xd, fp8=w.fp8,
                     scale_format=args.scale_format)
    # expert outputs for the combine: synthetic stand-in built once (untimed)
    expert = torch.repeat_interleave(torch.arange(E, device=dev), d.expert_counts.to(torch.int64))
    scale = torch.tensor([np.float32(1.0 + e / E) for e in range(E)], dtype=torch.float32, device=dev)
    Y = (d.X_perm.float() * scale[expert][:, None]).to(torch.bfloat16)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    R = residual_rows(w, rank).to(dev) if args.residual else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    # The timed loop calls the C ABI directly with pointers marshalled once, so
    # that host-side Python work stays far below the GPU time of a step.
    L = moe.lib()
    ws = moe.dispatch_workspace(E, dev, stream)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    sp = ctypes.c_void_p(stream.cuda_stream)
    fmt = moe.SCALE_UE8M0 if args.scale_format == "ue8m0" else moe.SCALE_FP32
    ep_rows = None
    de = None
    if args.ep_size:
        de = moe.dispatch_ep(idx, E, args.ep_size, Xd)
        torch.cuda.synchronize()
        ep_rows = int(de.rank_offsets[-1])
    disp_fn = L.moe_dispatch_ep if args.ep_size else L.moe_dispatch_ex
    route_fn = L.moe_route_stats if args.route_stats else L.moe_route_ex
    lse_buf = torch.empty(N, dtype=torch.float32, device=dev) if args.route_stats else None
    cnt_buf = torch.empty(E, dtype=torch.int32, device=dev) if args.route_stats else None
    stats_buf = torch.empty(4, dtype=torch.float32, device=dev) if args.route_stats else None
    comb_fn = L.moe_combine if R is None else L.moe_combine_residual
    # route and dispatch as one call (one launch where the router runs split-K)
    fuse = fused_step(args)
    fused_launches = ctypes.c_int(0)

    def call_args(xd, o, spp, wsp):
        """Arguments of the three C-ABI calls of one step: tokens from xd, output to o, on stream spp."""
        if args.route_stats:
            ra = (vp(xd), vp(Wd), vp(bd), N, H, E, K, int(w.renorm), vp(idx), vp(tw), vp(lse_buf), vp(cnt_buf),
                  vp(st), moe.ROUTE_AUTO, spp)
        else:
            ra = (vp(xd), vp(Wd), vp(bd), N, H, E, K, int(w.renorm), vp(idx), vp(tw), vp(st), moe.ROUTE_AUTO, spp)
        if de is not None:
            da = (vp(idx), vp(xd), N, H, E, K, args.ep_size, vp(de.expert_counts), vp(de.expert_offsets),
                  vp(de.row_map), vp(de.rank_counts), vp(de.rank_offsets), vp(de.send_token),
                  vp(de.slot_send_row), vp(de.expand_idx), vp(de.send_meta), vp(de.X_send), vp(st), vp(wsp),
                  wsp.numel(), spp)
        else:
            da = (vp(idx), vp(xd), N, H, E, K, vp(d.expert_counts), vp(d.expert_offsets), vp(d.row_map),
                  vp(d.src_slot), vp(d.X_perm), vp(d.X_fp8), vp(d.X_scale), fmt, vp(st), vp(wsp), wsp.numel(), spp)
        if R is None:
            ca = (vp(Y), vp(d.row_map), vp(tw), N, H, K, vp(o), vp(st), spp)
        else:
            ca = (vp(Y), vp(d.row_map), vp(tw), vp(R), N, H, K, vp(o), vp(st), spp)
        fa = (vp(xd), vp(Wd), vp(bd), N, H, E, K, int(w.renorm), vp(idx), vp(tw), vp(d.expert_counts),
              vp(d.expert_offsets), vp(d.row_map), vp(d.src_slot), vp(d.X_perm), vp(st), vp(wsp), wsp.numel(),
              ctypes.byref(fused_launches), spp)
        return ra, da, ca, fa

    def issue(a, spp):
        """The C-ABI calls of one step on stream spp; returns the OR of their status codes."""
        ra, da, ca, fa = a
        if fuse:
            return L.moe_route_dispatch(*fa) | comb_fn(*ca)
        rc = route_fn(*ra) | disp_fn(*da) | comb_fn(*ca)
        if stats_buf is not None:          # load statistics of the step (one small kernel)
            rc |= L.moe_load_stats(vp(cnt_buf), E, vp(lse_buf), N, ctypes.c_float(1e-3), vp(stats_buf), spp)
        return rc

    step_args = call_args(Xd, out, sp, ws)
    route_args, disp_args, comb_args, fused_args = step_args

    def step():
        rc = issue(step_args, sp)
        if rc:
            raise RuntimeError(f"a library call failed: {moe.status_string(rc)}")

    def timed_calls(fn, n):
        """Event times (ms) of n calls of fn, each alone: the L2 flushed before it, an
        event pair around it on the launching stream, no other kernel in between."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        rc = 0
        for i in range(n):
            flush.zero_()
            evs[i][0].record(stream)
            rc |= fn()
            evs[i][1].record(stream)
        if rc:
            raise RuntimeError(f"a library call failed: {moe.status_string(rc)}")
        return evs

    # route + dispatch + combine; moe_dispatch copies rows in a launch of their own
    # once the copy moves 256 MiB or more (moe_dispatch_ep likewise for its send rows)
    copy_bytes = N * (2 * H + 2 * K * H + (K * (H + H // 32) if w.fp8 else 0))
    ep_copy_bytes = N * 2 * H + N * min(K, args.ep_size or 1) * 2 * H
    if args.ep_size:       # two counting-sort passes, a fix-up, and the send-row copy apart when large
        kernels_per_step = 2 + 3 + (1 if ep_copy_bytes >= (256 << 20) else 0)
    else:
        kernels_per_step = 4 if copy_bytes >= (256 << 20) else 3
    if args.route_stats:   # moe_load_stats; moe_route_stats also clears the counts (a memset)
        kernels_per_step += 1
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert st.item() == 0, moe.status_string(st.item())
    if fuse:   # kernels of the one route + dispatch call (1 when fused), then the combine
        kernels_per_step = fused_launches.value + 1

    # ---- timed region: K whole steps, each bracketed by an event pair (the L2
    # flush in between is outside the brackets; no events between the kernels
    # of a step, so consecutive launches may overlap their prologues)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t1 = time.time()
    assert st.item() == 0, moe.status_string(st.item())
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]
    total_ms = max_over_ranks(sum(step_ms), pg, dev)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_tokens_per_s(world, N, args.steps, total_ms)

    # ---- per-kernel durations for the roofline: every call of the step timed in a
    # loop of its own (L2 flushed before each call, one event pair around it: the
    # kernel's time plus its own launch latency).  Timing the calls interleaved
    # inside whole steps instead read the router at the E=128 layer ~4 us slower
    # than the router alone, an effect of the previous step's traffic rather than
    # of the router's work.
    names = ["route", "dispatch", "combine"]
    ksteps = min(args.steps, 1000)
    calls = {"route": lambda: route_fn(*route_args), "dispatch": lambda: disp_fn(*disp_args),
             "combine": lambda: comb_fn(*comb_args)}
    if stats_buf is not None:
        calls["load_stats"] = lambda: L.moe_load_stats(vp(cnt_buf), E, vp(lse_buf), N, ctypes.c_float(1e-3),
                                                       vp(stats_buf), sp)
    if fuse:
        calls["route_dispatch"] = lambda: L.moe_route_dispatch(*fused_args)
    kevs = {n: timed_calls(f, ksteps) for n, f in calls.items()}
    # ---- hot L2: the same steps with no flush in between (what fits in the
    # 129 MB L2 stays there from one step to the next)
    hevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(ksteps)]
    for i in range(ksteps):
        hevs[i][0].record(stream)
        step()
        hevs[i][1].record(stream)
    torch.cuda.synchronize()
    hot_ms = statistics.fmean(ev[0].elapsed_time(ev[1]) for ev in hevs)
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    t2 = time.time()
    per = {n: [ev[0].elapsed_time(ev[1]) for ev in evs] for n, evs in kevs.items()}

    # ---- the same step replayed from a CUDA graph (launch overhead removed)
    graph = None
    try:
        gs = torch.cuda.Stream()
        gsp = ctypes.c_void_p(gs.cuda_stream)
        g_ws = moe.dispatch_workspace(E, dev, gs)
        g_args = call_args(Xd, out, gsp, g_ws)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for _ in range(2):  # warm the graph stream's workspace and plans
                issue(g_args, gsp)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            rc = issue(g_args, gsp)
        if rc:
            raise RuntimeError(moe.status_string(rc))
        gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(ksteps)]
        for i in range(ksteps):
            flush.zero_()
            gevs[i][0].record(stream)
            cg.replay()
            gevs[i][1].record(stream)
        torch.cuda.synchronize()
        g_ms = statistics.fmean(ev[0].elapsed_time(ev[1]) for ev in gevs)
        graph = {"ms_per_step": g_ms, "tokens_per_s": N / (g_ms * 1e-3), "steps": ksteps}
    except Exception as exc:  # graph capture is reported, not required
        graph = {"error": str(exc)[:200]}

    # ---- end to end through the public API: every step uploads its tokens from
    # pinned host memory and reads its output back.  Steps are pipelined over
    # E2E_BUFFERS buffer sets: the upload of step i+1 and the read-back of step i-1
    # run on their own streams while step i computes (the C-ABI calls go on the
    # compute stream).  The value is steps / elapsed time.  The serial latency of one
    # step (upload, compute, read-back, nothing overlapped, L2 flushed before) is
    # reported beside it.
    Xh = X.pin_memory()
    NB = max(2, args.e2e_buffers)
    outh = [torch.empty((N, H), dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    cs, hs, ds = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    c_ws = moe.dispatch_workspace(E, dev, cs)
    Xb = [Xd] + [torch.empty_like(Xd) for _ in range(NB - 1)]
    Ob = [out] + [torch.empty_like(out) for _ in range(NB - 1)]
    cargs = [call_args(Xb[b], Ob[b], ctypes.c_void_p(cs.cuda_stream), c_ws) for b in range(NB)]
    ev_h = [torch.cuda.Event() for _ in range(NB)]
    ev_c = [torch.cuda.Event() for _ in range(NB)]
    ev_d = [torch.cuda.Event() for _ in range(NB)]

    def pipelined(n):
        for i in range(n):
            b = i % NB
            if i >= NB:
                hs.wait_event(ev_c[b])              # step i-NB has finished reading Xb[b]
            with torch.cuda.stream(hs):
                Xb[b].copy_(Xh, non_blocking=True)
            ev_h[b].record(hs)
            cs.wait_event(ev_h[b])
            if i >= NB:
                cs.wait_event(ev_d[b])              # Ob[b] of step i-NB has been read back
            rc = issue(cargs[b], ctypes.c_void_p(cs.cuda_stream))
            if rc:
                raise RuntimeError("a library call failed")
            ev_c[b].record(cs)
            ds.wait_event(ev_c[b])
            with torch.cuda.stream(ds):
                outh[b].copy_(Ob[b], non_blocking=True)
            ev_d[b].record(ds)

    pipelined(2 * NB)
    torch.cuda.synchronize()
    # The pipelined steps are issued two ways and both are timed: from the host
    # (one Python iteration per step) and as units of E2E_UNIT steps captured in
    # one CUDA graph (forked from and joined back to the upload stream) and
    # replayed, so that the host issues one launch per unit.  Small steps are
    # host-bound and gain from the graph; copy-bound large ones overlap their
    # copies better when issued from the host.  `value` is the faster of the two.
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(hs)
    pipelined(args.e2e_steps)
    p1.record(ds)
    torch.cuda.synchronize()
    host_ms = p0.elapsed_time(p1) / args.e2e_steps
    graph_ms = None
    try:
        units = max(1, args.e2e_steps // E2E_UNIT)
        cg2 = torch.cuda.CUDAGraph()
        hs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(cg2, stream=hs):
            cs.wait_stream(hs)
            ds.wait_stream(hs)
            pipelined(E2E_UNIT)
            hs.wait_stream(cs)
            hs.wait_stream(ds)
        rs = torch.cuda.current_stream()           # replay() launches on the current stream
        cg2.replay()
        torch.cuda.synchronize()
        p0.record(rs)
        for _ in range(units):
            cg2.replay()
        p1.record(rs)
        torch.cuda.synchronize()
        graph_ms = p0.elapsed_time(p1) / (units * E2E_UNIT)
    except Exception:                              # capture refused: the host-issued figure stands
        torch.cuda.synchronize()
    best = host_ms if graph_ms is None or host_ms <= graph_ms else graph_ms
    e2e_mode = "host-issued" if best == host_ms else f"CUDA graph, {E2E_UNIT}-step units"
    e2e_mean = max_over_ranks(best, pg, dev)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lat_ms = []
    for _ in range(min(args.e2e_steps, 50)):
        flush.zero_()
        e0.record(stream)
        Xd.copy_(Xh, non_blocking=True)
        step()
        outh[0].copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        lat_ms.append(e0.elapsed_time(e1))
    e2e_latency = max_over_ranks(statistics.fmean(lat_ms), pg, dev)

    # untimed: the expert counts of every rank's step added up, then moe_load_stats on them
    job_counts = sum_over_ranks(d.expert_counts, pg)
    if rank != 0:
        pg.destroy_process_group()
        return

    load = moe.load_stats(job_counts).cpu().tolist()
    naive = torch_naive(Xd, Wd, bd, w, Y, flush, reps=min(args.steps, 100)) if not args.no_torch_naive else None
    peak, peak_src = measured_peaks()
    kb = kernel_bytes(w, args.residual, args.scale_format == "ue8m0", ep_rows)
    kern = {}
    for n in names + (["route_dispatch"] if fuse else []):
        ms = statistics.fmean(per[n])
        kern[n] = {"ms": ms, "median_ms": statistics.median(per[n]), "algorithmic_bytes": kb[n],
                   "gbs": kb[n] / (ms * 1e-3) / 1e9,
                   "frac_of_" + peak_src + "_hbm": kb[n] / (ms * 1e-3) / 1e9 / peak,
                   "frac_of_nominal_8000": kb[n] / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                   "traffic": ncu_traffic(n, w.name)}
    if fuse:
        kern["route_dispatch"]["launches"] = fused_launches.value
    if "load_stats" in per:
        kern["load_stats"] = {"ms": statistics.fmean(per["load_stats"]),
                              "median_ms": statistics.median(per["load_stats"])}
    # the roofline is that of the longest kernel of the timed step (the route +
    # dispatch call counts as a kernel only where it was one launch)
    step_kernels = ["route_dispatch", "combine"] if fuse and fused_launches.value == 1 else names
    dom = max(step_kernels, key=lambda n: kern[n]["ms"])
    roof = {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["gbs"], "peak": peak, "unit": "GB/s",
            "frac": kern[dom]["gbs"] / peak, "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"
            if peak_src == "measured" else "fallback 6800 GB/s",
            "traffic": ncu_traffic(dom, w.name), "algorithmic_bytes_per_launch": kb[dom],
            "traffic_source": "profiles/dram_traffic.csv (ncu dram__bytes_read.sum + dram__bytes_write.sum per "
                              "launch; null when absent or taken on an older source of the kernel)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(w.as_dict(), **combine_config(args),
                       l2="256 MiB buffer written before every timed step (L2 flush)",
                       accumulate="fp32", parallelism="replicas: each GPU routes its own tokens, no collective"),
        "roofline": roof, "kernels": kern, "gpu_launches": kernels_per_step * args.steps,
        "e2e": {"value": world * N / (e2e_mean / 1e3), "unit": UNIT, "h2d_bytes_per_step": N * H * 2,
                "d2h_bytes_per_step": N * H * 2, "ms_per_step": e2e_mean, "steps": args.e2e_steps,
                "issue": e2e_mode, "host_issued_ms_per_step": host_ms, "graph_ms_per_step": graph_ms,
                "latency_ms": e2e_latency,
                "path": "pinned host X -> device, route, dispatch, permute, combine, out -> pinned host, "
                        f"every step; steps pipelined over {NB} buffer sets (copies on their own streams); "
                        "latency_ms: one step alone, nothing overlapped, L2 flushed before"},
        "clocks": sampler.summary(t0, t2) if sampler else None,
        "graph": graph,
        "hot_l2": {"ms_per_step": hot_ms, "tokens_per_s": N / (hot_ms * 1e-3), "steps": ksteps,
                   "what": "the same step with no L2 flush between steps"},
        "kernel_sum": {"tokens_per_s": N / (sum(kern[n]["median_ms"] for n in names) * 1e-3),
                       "ms": sum(kern[n]["median_ms"] for n in names),
                       "what": "N / (median route + median dispatch + median combine), each call timed alone "
                               "with an event pair, L2 flushed before each call"},
        "load": {"max_over_mean": load[0], "p95_over_mean": load[1], "mean_slots_per_expert": load[3],
                 "over_ranks": world},
        "torch_naive": naive,
        "timing": ("value: K steps, one event pair per step; kernels: each call of the step (route, dispatch, "
                   "combine as separate calls; route_dispatch: the one call the step makes when fused) timed "
                   "alone in a loop of min(K,1000) calls, L2 flushed before each call, one event pair per call"),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, residual=args.residual,
                                            ue8m0=args.scale_format == "ue8m0", ep_size=args.ep_size,
                                            stats=args.route_stats)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    args = parse_args()
    if args.tokens:
        import dataclasses
        w = mi.WORKLOADS[args.workload]
        name = f"{w.name}@N={args.tokens}"
        mi.WORKLOADS[name] = dataclasses.replace(w, name=name, N=args.tokens)
        args.workload = name
    if args.record_traffic:
        calls = record_traffic(args.record_traffic, mi.WORKLOADS[args.workload])
        print(json.dumps({"recorded": args.workload, "calls": calls}))
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
