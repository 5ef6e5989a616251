#!/usr/bin/env python3
"""Benchmark of the GB300 skinny BF16 GEMM (Y[M,N] = X[M,K] . W[N,K]^T, fp32 out).

One *step* is one pass of the whole hot path over one batch of the workload:
every call of the workload, each through the C ABI.  The default workload is
the decode projections (M in {1,2,3,8,16} x (N,K) in {(2112,7168),
(24576,1536),(7168,14336)}, ldy = N+64, 15 calls: 30-206 MB weights, where the
bandwidth roofline applies).  The router workloads (M=1 K=7168 N=256; the
dot-product regime M 1-4; the split-K regime M 5-16) are timed the same way
in the same run and reported under ``per_config``.

Timing rules followed here:
* W is a weight resident in HBM; every step reads a different replica of the
  whole workload's W / X / Y, and the replicas together exceed 2x the L2 size,
  so every call reads W from HBM (L2-cold without a flush kernel).
* a step is replayed from a CUDA graph captured from the public C-ABI calls
  (as a decode step is); W untimed warm-up steps, then exactly K timed steps
  bracketed by a barrier and cuda synchronize, timed with CUDA events on the
  launching stream; the max over ranks is reported.
* per-launch durations for the roofline: for each call shape, a CUDA graph of
  back-to-back launches over rotating W copies (L2-cold), PDL off, CUDA events
  around whole replays; cross-checked by a flush kernel (a write of 2x the L2
  size) before each isolated call, with a CUDA-event pair around the call alone.
* clocks are sampled with nvidia-smi while the GPU is under load.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(test infrastructure, single thread) on the same workload instead.
"""
from __future__ import annotations

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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import skinny_inputs as si  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of roofline) for bf16 skinny GEMM, M=1–16"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_DESC = {
    "router_small": "router GEMM M=1, K=7168, N=256",
    "dotprod": "dot-product regime: M in {1,2,3,4} x (K,N) in {(7168,256),(7168,384),(2880,128)}, 12 calls",
    "splitk": "split-K regime: M in {5,8,12,16} x (K,N) in {(7168,256),(7168,384),(4096,256)}, 12 calls",
    "projection": "decode projections: M in {1,2,3,8,16} x (N,K) in {(2112,7168),(24576,1536),(7168,14336)}, "
                  "ldy=N+64, 15 calls",
    "midm": "medium-M decode regime (tensor cores): M in {17,24,32,40,64} x (K,N) in {(7168,256),(4096,384)}, "
            "M in {17,32,64} x (N,K) in {(2112,7168),(24576,1536)}, M in {17,32} x (7168,14336), 18 calls",
}
# the sources that define each kernel family (a committed DRAM-traffic figure
# is used only while they are unchanged)
KERNEL_SOURCES = {"dotprod": ["dotprod.cu"], "dotmma": ["dotmma.cu"], "splitk": ["splitk.cu"],
                  "stream": ["stream.cu"], "tmem_gemm": ["tmem_gemm.cu", "tma.cuh"]}
COMMON_SOURCES = ["common.cuh", "internal.h"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", choices=sorted(WORKLOAD_DESC), default="projection")
    p.add_argument("--no-per-config", action="store_true", help="skip the router workloads' figures")
    p.add_argument("--pdl", type=int, choices=[0, 1, 2], default=1)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget (s)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--only", default=None, help="comma list of case indices of the workload to keep (profiling)")
    p.add_argument("--profile-mode", action="store_true",
                   help="short run for ncu: no clock soak, no CPU baseline, few extra passes")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(elapsed_s: float, units_local: float, group=None):
    """Max elapsed time and summed work over ranks (no data-path collective:
    the GEMM replicas are independent; this only reduces two scalars)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units_local
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ peaks, clocks, traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no measured peak file)"


def kernel_sources_digest(family: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family] + COMMON_SOURCES:
        with open(os.path.join(ROOT, "latency_skinny_bf16_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(family: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{family}_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sources_sha256_16") != kernel_sources_digest(family):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        return self.summary()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ the GPU workload

def select_cases(args):
    cases = si.workload(args.workload)
    if args.only:
        cases = [cases[int(i)] for i in args.only.split(",")]
    return cases


class Replica:
    """Device buffers for one copy of the whole workload."""

    def __init__(self, cases, host_inputs, torch, src=None):
        self.x, self.w, self.y = [], [], []
        for j, (c, (X, W)) in enumerate(zip(cases, host_inputs)):
            if src is None:
                x = torch.from_numpy(X.reshape(-1).view(np.int16).copy()).cuda()
                w = torch.from_numpy(W.reshape(-1).view(np.int16).copy()).cuda()
            else:
                x, w = src.x[j].clone(), src.w[j].clone()
            self.x.append(x)
            self.w.append(w)
            self.y.append(torch.zeros(c.M * c.ly, dtype=torch.float32, device="cuda"))


def launch_step(sk, cases, rep, stream_handle, counter=None):
    for c, x, w, y in zip(cases, rep.x, rep.w, rep.y):
        st = sk.skinny_gemm_bf16(x.data_ptr(), c.lx, w.data_ptr(), c.lw, y.data_ptr(), c.ly, c.M, c.N, c.K,
                                 stream_handle)
        if st != sk.SKINNY_OK:
            raise sk.SkinnyError(st, c.name)
        if counter is not None:
            counter[0] += 1


class Workload:
    """A workload's device replicas (together > 2x L2, so every call reads its W
    from HBM), its plans, and CUDA graphs of `steps_per_graph` whole steps over
    consecutive replicas (graph j starts at replica j * steps_per_graph), so a
    workload of a few short calls is not timed as graph-launch overhead."""

    def __init__(self, sk, torch, cases, l2, stream, steps_per_graph=1):
        self.cases = cases
        self.G = steps_per_graph
        self.host_inputs = [si.make_inputs(c) for c in cases]
        self.step_bytes = sum(c.algorithmic_bytes for c in cases)
        self.step_w_bytes = sum(2 * c.N * c.K for c in cases)
        self.n_rep = max(1, math.ceil(2 * l2 / self.step_w_bytes))
        self.reps = [Replica(cases, self.host_inputs, torch)]
        for _ in range(self.n_rep - 1):
            self.reps.append(Replica(cases, self.host_inputs, torch, src=self.reps[0]))
        self.pool_mb = self.n_rep * self.step_w_bytes / 1e6
        self.plans = [sk.skinny_query_plan(x.data_ptr(), c.lx, w.data_ptr(), c.lw, y.data_ptr(), c.ly, c.M, c.N, c.K)
                      for c, x, w, y in zip(cases, self.reps[0].x, self.reps[0].w, self.reps[0].y)]
        sh = stream.cuda_stream
        with torch.cuda.stream(stream):        # eager warm-up: first launches, module load
            for r in self.reps:
                launch_step(sk, cases, r, sh)
        torch.cuda.synchronize()
        self.graphs = []
        for j in range(self.n_rep):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for t in range(self.G):
                    launch_step(sk, cases, self.reps[(j * self.G + t) % self.n_rep], sh)
            self.graphs.append(g)
        # L2-warm: the same replica every step
        self.warm_graph = self.graphs[0]
        if self.G > 1:
            self.warm_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.warm_graph, stream=stream):
                for t in range(self.G):
                    launch_step(sk, cases, self.reps[0], sh)
        torch.cuda.synchronize()

    def replay(self, i):
        """Replays graph i: steps i * G .. i * G + G - 1."""
        self.graphs[i % self.n_rep].replay()


def time_steps(torch, stream, wl, steps, warmup, soak_s=0.0, use_barrier=True):
    """Exactly `steps` graph replays (rotating replicas) after `warmup` untimed
    ones, bracketed by a barrier and a synchronize; seconds."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            wl.replay(i)
        t_end = time.time() + soak_s          # keep the GPU loaded so the clock samples see it
        i = 0
        while time.time() < t_end:
            for _ in range(50):
                wl.replay(i)
                i += 1
            stream.synchronize()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if use_barrier:
        barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            wl.replay(i)
        ev1.record(stream)
    torch.cuda.synchronize()
    if use_barrier:
        barrier()
    return ev0.elapsed_time(ev1) / 1e3


def time_warm(torch, stream, wl, steps):
    """L2-warm: the same replica every step; us per call."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            wl.warm_graph.replay()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(steps):
            wl.warm_graph.replay()
        w1.record(stream)
    torch.cuda.synchronize()
    return w0.elapsed_time(w1) * 1e3 / (steps * wl.G * len(wl.cases))


def time_isolated(sk, torch, stream, wl, l2, iters, pdl=0):
    """Per call shape: a CUDA graph of back-to-back launches over enough copies
    of that shape's W to exceed 2x L2 (L2-cold), PDL off (or in the given PDL
    mode: the sustained rate of a chain of that call), CUDA events around whole
    replays; us per launch."""
    out = []
    sh = stream.cuda_stream
    with sk.options(pdl=pdl):
        for j, c in enumerate(wl.cases):
            n_j = max(8, math.ceil(2 * l2 / (2 * c.N * c.K)))
            ws = [wl.reps[i % wl.n_rep].w[j] if i < wl.n_rep else wl.reps[0].w[j].clone() for i in range(n_j)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i, w in enumerate(ws):
                    r = wl.reps[i % wl.n_rep]
                    st = sk.skinny_gemm_bf16(r.x[j].data_ptr(), c.lx, w.data_ptr(), c.lw, r.y[j].data_ptr(),
                                             c.ly, c.M, c.N, c.K, sh)
                    if st != sk.SKINNY_OK:
                        raise sk.SkinnyError(st, c.name)
            with torch.cuda.stream(stream):
                g.replay()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                for _ in range(iters):
                    g.replay()
                b_.record(stream)
            torch.cuda.synchronize()
            out.append(a_.elapsed_time(b_) * 1e3 / (iters * n_j))
            del g, ws
    return out


def time_flushed(sk, torch, stream, wl, l2, samples):
    """Cross-check of the L2-cold figures: before each call a flush kernel
    reads a buffer of 2x the L2 size (outside the event pair; a read leaves
    clean lines, where a write would leave dirty ones whose write-back the
    timed call would pay), then a CUDA event pair brackets the call alone;
    PDL off.  (median, p10, p90) us per call shape."""
    flush = torch.ones(max(1, 2 * l2 // 4), dtype=torch.float32, device="cuda")
    sink = torch.empty(1, dtype=torch.float32, device="cuda")
    sh = stream.cuda_stream
    out = []
    with sk.options(pdl=0):
        for j, c in enumerate(wl.cases):
            r = wl.reps[0]
            evs = []
            with torch.cuda.stream(stream):
                for s in range(samples + 2):
                    torch.sum(flush, dim=0, keepdim=True, out=sink)
                    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a_.record(stream)
                    st = sk.skinny_gemm_bf16(r.x[j].data_ptr(), c.lx, r.w[j].data_ptr(), c.lw, r.y[j].data_ptr(),
                                             c.ly, c.M, c.N, c.K, sh)
                    b_.record(stream)
                    if st != sk.SKINNY_OK:
                        raise sk.SkinnyError(st, c.name)
                    if s >= 2:
                        evs.append((a_, b_))
            torch.cuda.synchronize()
            t = sorted(a_.elapsed_time(b_) * 1e3 for a_, b_ in evs)
            out.append((statistics.median(t), t[len(t) // 10], t[(9 * len(t)) // 10]))
    del flush
    return out


def family_of(plan):
    return {1: "dotmma" if plan["consumer"] == 2 else "dotprod", 2: "splitk", 3: "stream",
            4: "tmem_gemm"}[plan["backend"]]


def shape_rows(wl, iso, peak, flushed=None, chained=None):
    rows = []
    for j, (c, p, us) in enumerate(zip(wl.cases, wl.plans, iso)):
        row = {"M": c.M, "N": c.N, "K": c.K, "kernel": family_of(p), "consumer": p["consumer"],
               "split_k": p["split_k"], "block_n": p["block_n"], "grid": [p["grid_x"], p["grid_y"]],
               "us_per_launch": round(us, 3), "gbs": round(c.algorithmic_bytes / us / 1e3, 1),
               "frac_of_peak": round(c.algorithmic_bytes / us / 1e3 / peak, 4)}
        if chained is not None:
            # the same chain with PDL in mode 1 (the plan's own attribute)
            row["chained_pdl"] = {"us_per_launch": round(chained[j], 3),
                                  "frac_of_peak": round(c.algorithmic_bytes / chained[j] / 1e3 / peak, 4)}
        if flushed is not None:
            med, p10, p90 = flushed[j]
            row["flush_us"] = {"median": round(med, 3), "p10": round(p10, 3), "p90": round(p90, 3)}
        rows.append(row)
    return rows


def run_native(args):
    import torch
    import torch.distributed as dist
    import latency_skinny_bf16_gb300 as sk

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    st = sk.skinny_init(local)
    if st != sk.SKINNY_OK:
        raise sk.SkinnyError(st, "skinny_init")
    sk.skinny_set_option(sk.SKINNY_OPT_PDL, args.pdl)
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    peak, _ = hbm_peak()

    cases = select_cases(args)
    wl = Workload(sk, torch, cases, l2, stream)

    clocks = ClockSampler(local) if not (args.no_clocks or args.profile_mode) else None
    if clocks:
        clocks.start()
    # ---- timed region: exactly `steps` graph replays, L2-cold (rotating replicas)
    elapsed = time_steps(torch, stream, wl, args.steps, args.warmup, soak_s=1.5 if clocks else 0.0)
    clock_summary = clocks.stop() if clocks else None
    launches = args.steps * len(cases)
    warm_us_per_call = time_warm(torch, stream, wl, 3 if args.profile_mode else max(50, min(args.steps, 2000)))
    per_launch = time_isolated(sk, torch, stream, wl, l2, 2 if args.profile_mode else 10)
    chained = None if args.profile_mode else time_isolated(sk, torch, stream, wl, l2, 10, pdl=1)
    flushed = None if args.profile_mode else time_flushed(sk, torch, stream, wl, l2, 100)

    # ---- the router workloads, timed the same way (outside the headline's timed region)
    per_config = None
    if not (args.profile_mode or args.no_per_config):
        per_config = {}
        for name, tag in (("router_small", "c0"), ("dotprod", "c1"), ("splitk", "c2")):
            if name == args.workload:
                continue
            pc_cases = si.workload(name)
            # graphs of at least 12 calls: a one-call step is otherwise timed as graph-launch latency
            G = max(1, -(-12 // len(pc_cases)))
            wc = Workload(sk, torch, pc_cases, l2, stream, steps_per_graph=G)
            replays = -(-min(args.steps, 1000) // G)
            k = replays * G
            el = time_steps(torch, stream, wc, replays, max(3, min(args.warmup, 20)), use_barrier=False)
            iso = time_isolated(sk, torch, stream, wc, l2, 10)
            iso_pdl = time_isolated(sk, torch, stream, wc, l2, 10, pdl=1)
            per_config[tag] = {
                "workload": WORKLOAD_DESC[name], "calls_per_step": len(wc.cases), "steps": k,
                "steps_per_graph": G,
                "us_per_call": round(el / k / len(wc.cases) * 1e6, 3),
                "gbs": round(wc.step_bytes * k / el / 1e9, 1),
                "us_per_call_l2_warm": round(time_warm(torch, stream, wc, 200), 3),
                "l2": f"cold: {wc.n_rep} rotating replicas ({wc.pool_mb:.0f} MB)",
                "isolated_us_max": round(max(iso), 3),
                "chained_pdl_us_max": round(max(iso_pdl), 3),
                "per_shape": shape_rows(wc, iso, peak, chained=iso_pdl),
            }
            del wc
            torch.cuda.synchronize()

    # ---- PDL chain: one CUDA graph of 64 back-to-back calls M=4, K=7168,
    # N=256 (same X and W, so L2-warm; a Y per call), total us per replay with
    # programmatic dependent launch on and off (outside the timed region)
    chain = None
    if not args.profile_mode:
        cc = si.pdl_chain_case()
        Xc, Wc = si.make_inputs(cc)
        xc = torch.from_numpy(Xc.reshape(-1).view(np.int16).copy()).cuda()
        wc = torch.from_numpy(Wc.reshape(-1).view(np.int16).copy()).cuda()
        ycs = [torch.zeros(cc.M * cc.N, dtype=torch.float32, device="cuda") for _ in range(64)]
        chain = {"calls": 64, "M": cc.M, "N": cc.N, "K": cc.K,
                 "method": "one CUDA graph of the 64 calls, mean over 20 replays after 2 untimed ones"}
        for pdl in (1, 0):
            with sk.options(pdl=pdl):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for y in ycs:
                        st = sk.skinny_gemm_bf16(xc.data_ptr(), cc.K, wc.data_ptr(), cc.K, y.data_ptr(), cc.N,
                                                 cc.M, cc.N, cc.K, sh)
                        if st != sk.SKINNY_OK:
                            raise sk.SkinnyError(st, cc.name)
            with torch.cuda.stream(stream):
                g.replay()
                g.replay()
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                for _ in range(20):
                    g.replay()
                c1.record(stream)
            torch.cuda.synchronize()
            chain["us_total_pdl_on" if pdl else "us_total_pdl_off"] = round(c0.elapsed_time(c1) * 1e3 / 20, 2)
            del g

    # ---- e2e: host -> device X, the calls, device -> host Y, per step, through the C ABI
    h2d = sum(2 * c.M * c.K for c in cases)
    d2h = sum(4 * c.M * c.N for c in cases)
    x_host = torch.empty(h2d // 2, dtype=torch.int16).pin_memory()
    y_host = torch.empty(sum(c.M * c.ly for c in cases), dtype=torch.float32).pin_memory()
    off = 0
    for c, (X, _) in zip(cases, wl.host_inputs):
        x_host[off:off + c.M * c.K] = torch.from_numpy(X.reshape(-1).view(np.int16).copy())
        off += c.M * c.K
    x_dev = torch.empty_like(x_host, device="cuda")
    # zeros like the replicas' Y, so the never-written gaps of a strided Y compare equal
    y_dev = torch.zeros(y_host.numel(), dtype=torch.float32, device="cuda")
    e2e_graphs = []
    for r in wl.reps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            x_dev.copy_(x_host, non_blocking=True)
            xo = yo = 0
            for c, w in zip(cases, r.w):
                st = sk.skinny_gemm_bf16(x_dev.data_ptr() + 2 * xo, c.K, w.data_ptr(), c.lw,
                                         y_dev.data_ptr() + 4 * yo, c.ly, c.M, c.N, c.K, sh)
                if st != sk.SKINNY_OK:
                    raise sk.SkinnyError(st, c.name)
                xo += c.M * c.K
                yo += c.M * c.ly
            y_host.copy_(y_dev, non_blocking=True)
        e2e_graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            e2e_graphs[i % wl.n_rep].replay()
    torch.cuda.synchronize()
    barrier()
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            e2e_graphs[i % wl.n_rep].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_elapsed = e0.elapsed_time(e1) / 1e3
    barrier()
    # correctness spot check of the e2e output against the device-only path
    ref_y = torch.cat([y.view(-1) for y in wl.reps[(args.steps - 1) % wl.n_rep].y]).cpu()
    if not torch.equal(ref_y, y_host):
        raise RuntimeError("e2e output differs from the device-resident output")

    elapsed_max, units = aggregate(elapsed, float(wl.step_bytes * args.steps))
    e2e_max, _ = aggregate(e2e_elapsed, 0.0)
    return dict(cases=cases, wl=wl, elapsed=elapsed_max, units=units, launches=launches,
                warm_us_per_call=warm_us_per_call, per_launch=per_launch, chained=chained, flushed=flushed,
                clocks=clock_summary,
                e2e_elapsed=e2e_max, h2d=h2d, d2h=d2h, l2=l2, world=world, rank=rank, chain=chain,
                per_config=per_config, peak=peak)


# ------------------------------------------------------------------ oracle timing

def oracle_step_sample(cases, seconds: float, max_steps: int | None = None, threads: int = 1):
    """Time the oracle (test infrastructure) on whole steps of the workload,
    column-sampled when one step would exceed ~`seconds`/4.  threads > 1 splits
    each call's output columns into that many contiguous ranges computed
    concurrently (the oracle's C routine runs without the interpreter lock)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(threads) if threads > 1 else None

    def call(X, W, c, n):
        if pool is None:
            oracle.gemm(X, W[:n], c.M, n, c.K)
            return
        bounds = [n * t // threads for t in range(threads + 1)]
        futs = [pool.submit(oracle.gemm, X, W[a:b], c.M, b - a, c.K)
                for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        for f in futs:
            f.result()

    inputs = [si.make_inputs(c) for c in cases]
    full_macs = sum(c.M * c.N * c.K for c in cases)
    # probe: one call of the smallest case
    t0 = time.perf_counter()
    c0 = min(cases, key=lambda c: c.M * c.N * c.K)
    call(inputs[cases.index(c0)][0], inputs[cases.index(c0)][1], c0, c0.N)
    rate = max(c0.M * c0.N * c0.K / max(time.perf_counter() - t0, 1e-6), 1e6)   # MAC/s
    frac = min(1.0, (seconds / 4) * rate / full_macs)
    bytes_done = 0.0
    steps = 0
    t0 = time.perf_counter()
    while True:
        for c, (X, W) in zip(cases, inputs):
            n = max(1, int(round(c.N * frac)))
            call(X, W, c, n)
            bytes_done += 2 * n * c.K + 2 * c.M * c.K + 4 * c.M * n
        steps += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and steps >= max_steps) or (max_steps is None and el >= seconds):
            break
    who = "single thread" if threads == 1 else f"{threads} threads over output columns"
    sample = (f"{steps} step(s) of the whole workload, each call on the first {frac:.1%} of its N columns "
              f"(all of M and K), {who}" if frac < 1 else
              f"{steps} whole step(s) of the workload, {who}")
    if pool is not None:
        pool.shutdown()
    return bytes_done / el, el / steps, sample


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    cases = select_cases(args)
    step_bytes = sum(c.algorithmic_bytes for c in cases)
    # untimed warm-up steps, then exactly `steps` timed steps, each a bounded sample
    budget = min(120.0, max(5.0, 0.2 * args.steps))
    per_step_budget = budget / max(args.steps, 1)
    if args.warmup:
        oracle_step_sample(cases, per_step_budget, max_steps=args.warmup)
    gbs, s_per_step, sample = oracle_step_sample(cases, per_step_budget * 4, max_steps=args.steps)
    us_per_call = s_per_step / len(cases) * 1e6
    value = gbs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s_per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "us_per_call": round(us_per_call, 2),
        "config": line_config(args, len(cases)),
        "method": {"parallelism": "single host thread"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


# ------------------------------------------------------------------ main

L2_NOTE = "cold: every call reads its W from DRAM (rotating W replicas larger than 2x the L2 size)"


def line_config(args, ncalls):
    """The config object, identical in both arms."""
    return {"workload": WORKLOAD_DESC[args.workload], "calls_per_step": ncalls, "l2": L2_NOTE}


def roofline_of(wl, per_launch, peak, peak_src, workload):
    """The dominant kernel family (largest total isolated-launch time) of the
    workload: its algorithmic bytes per launch over its mean launch time."""
    fam_time, fam_bytes, fam_n = {}, {}, {}
    for c, p, us in zip(wl.cases, wl.plans, per_launch):
        fam = family_of(p)
        fam_time[fam] = fam_time.get(fam, 0.0) + us
        fam_bytes[fam] = fam_bytes.get(fam, 0.0) + c.algorithmic_bytes
        fam_n[fam] = fam_n.get(fam, 0) + 1
    dom = max(fam_time, key=fam_time.get)
    achieved = fam_bytes[dom] / (fam_time[dom] * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": f"{dom}_kernel", "achieved": round(achieved, 1),
            "peak": round(peak, 1), "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": peak_src,
            "traffic": committed_traffic(dom, workload),
            "time_share": round(fam_time[dom] / sum(fam_time.values()), 3),
            "launches_per_step": fam_n[dom],
            "method": "per call shape: CUDA graph of back-to-back launches over rotating W copies (L2-cold), "
                      "PDL off, CUDA events around the replays; achieved = the family's algorithmic bytes "
                      "(2NK + 2MK + 4MN per launch) over its launch time",
            "avg_launch_us": round(fam_time[dom] / fam_n[dom], 3),
            "algorithmic_bytes_per_launch": round(fam_bytes[dom] / fam_n[dom])}


def cpu_baselines(args, cases, per_config):
    """The oracle (single host thread, and split over all host threads) on
    bounded samples of the headline workload; single-thread ms per call for
    every router config too."""
    gbs, s_step, sample = oracle_step_sample(cases, args.cpu_seconds)
    cpu = {"value": round(gbs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
           "ms_per_call": round(s_step / len(cases) * 1e3, 3)}
    cpu_threads = None
    nthr = os.cpu_count() or 1
    if nthr > 1:
        gbs, s_step, sample = oracle_step_sample(cases, args.cpu_seconds, threads=nthr)
        cpu_threads = {"value": round(gbs / 1e9, 4), "unit": "GB/s", "cores": nthr, "kind": "oracle",
                       "sample": sample, "ms_per_call": round(s_step / len(cases) * 1e3, 3)}
    for tag, name in (("c0", "router_small"), ("c1", "dotprod"), ("c2", "splitk")):
        if per_config is None or tag not in per_config:
            continue
        cc = si.workload(name)
        gbs, s_step, sample = oracle_step_sample(cc, max(1.0, args.cpu_seconds / 4))
        per_config[tag]["cpu_baseline"] = {"value": round(gbs / 1e9, 4), "unit": "GB/s", "cores": 1,
                                           "kind": "oracle", "sample": sample,
                                           "ms_per_call": round(s_step / len(cc) * 1e3, 3)}
    return cpu, cpu_threads


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
        return 0
    r = run_native(args)
    if r["rank"] != 0:
        return 0
    wl = r["wl"]
    cases = wl.cases
    n = r["world"]
    step_s = r["elapsed"] / args.steps
    value_gbs = r["units"] / r["elapsed"] / 1e9
    us_per_call = step_s / len(cases) * 1e6
    peak, peak_src = hbm_peak()
    roofline = roofline_of(wl, r["per_launch"], peak, peak_src, args.workload)

    cpu = cpu_threads = None
    if not (args.no_cpu_baseline or args.profile_mode):
        cpu, cpu_threads = cpu_baselines(args, cases, r["per_config"])

    e2e_gbs = wl.step_bytes * args.steps * n / r["e2e_elapsed"] / 1e9
    line = {
        "metric": METRIC, "value": round(value_gbs, 2), "unit": "GB/s", "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": line_config(args, len(cases)),
        "method": {"l2": f"{wl.n_rep} rotating replicas of every W ({wl.pool_mb:.0f} MB > 2x L2 "
                         f"{r['l2'] / 1e6:.0f} MB)",
                   "graph": "each step replayed from a CUDA graph of the C-ABI calls",
                   "pdl": args.pdl, "parallelism": f"replicas x{n}" if n > 1 else "single GPU"},
        "us_per_call": round(us_per_call, 3),
        "us_per_call_l2_warm": round(r["warm_us_per_call"], 3),
        "pct_of_roofline_step": round(value_gbs / n / peak, 4),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "cpu_baseline_threads": cpu_threads,
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "us_per_call": round(r["e2e_elapsed"] / args.steps / len(cases) * 1e6, 3),
                "note": "W resident (weights); X copied in and Y copied out every step, inside the graph"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "pdl_chain": r["chain"],
        "per_shape": shape_rows(wl, r["per_launch"], peak, r["flushed"], r["chained"]),
        "flush_method": None if r["flushed"] is None else
        "per call shape: 100 isolated calls, each after a flush kernel reading 2x L2 (outside the event pair), "
        "a CUDA-event pair around the call alone, PDL off; median / p10 / p90",
        "per_config": r["per_config"],
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
