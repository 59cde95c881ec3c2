#!/usr/bin/env python
"""Benchmark of the expert-cache MoE decode step on one GB300 (or N replicas).

Workload (default): decode at T=1 through 48 MoE layers of E=128 experts,
top-8, hidden 2048, expert ffn 768, BF16 records in a 58 GB page-locked host
pool, 1536 cache slots shared by all layers, AR(1) router logits
(rho 0.8, sigma 0.6), B_P = 52.7, B_H = 120.  One step = one decode token
through all 48 layers: for every layer the control pass (routing, dedup,
hit/miss, q, fill set, LRU victims, map update), the fills, the expert
gate/up + SwiGLU and down + gated merge with the CPU-set partial sum.

Timing: W eager warm-up steps, then R consecutive windows of exactly K steps
of the same AR(1) sequence (R = ceil(256 / K), at least 3: the windows cover
the workload's 256 steps from a cache that started empty).  The K steps are captured from the library calls
into one CUDA graph (no profiling nodes in it), instantiated and uploaded
before timing; before each window the window's inputs are copied into the
graph's input buffers (untimed).  Each window is bracketed by a barrier and a
device synchronisation and timed with CUDA events on the library's compute
stream; `value` comes from the median window (max over ranks), and the line
reports the spread.  Every step streams about 3.6 GB of expert weights, far
more than the 129 MB L2, so no L2 flush is needed.  Per-kernel device times
come from one further window of the same K-step graph captured with the
library's per-launch event records.  Clocks are sampled by the GPU's UUID
and summarised over the windows' time span.

The JSON line carries compact objects for the other workloads ("legs"); with
FT_BENCH_DETAIL=<path> the full per-leg detail is also written there as JSON.

--impl reference times the CPU oracle (exact-integer control + float64
expert numerics) on this machine's host cores on bounded samples of the same
workload; it never touches the GPU.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = synth.DECODE_T1
METRIC = "decode MoE-layer tokens/s"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def headline_config(world: int = 1) -> dict:
    """The workload of the bench line (identical in both arms)."""
    return {"workload": "decode T=1: 48 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, 1536 slots, "
                        "AR(1) rho=0.8, B_P=52.7, B_H=120",
            "l2": "no flush: each step streams ~3.6 GB of expert weights (> 129 MB L2)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


# --------------------------------------------------------------- utilities

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (one all-reduce; only timing plumbing)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def gpu_query_id(device) -> str:
    """nvidia-smi's -i argument for a torch device: the GPU's UUID (the CUDA
    ordinal is not nvidia-smi's index once CUDA_VISIBLE_DEVICES remaps it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        if u and u != "None":
            return u if u.startswith(("GPU-", "MIG-")) else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    idx = device.index if hasattr(device, "index") and device.index is not None else 0
    if vis:
        ent = [v.strip() for v in vis.split(",") if v.strip()]
        if idx < len(ent):
            return ent[idx]
    return str(idx)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 200 ms) while the
    timed windows run; stop() summarises the samples that fall inside the
    given host-time span."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str, tag: str = "0"):
        self.proc = None
        # raw samples go to FT_CLOCKS_DIR (default: the system temporary
        # directory); the JSON line carries their summary
        import tempfile
        self.path = os.path.join(os.environ.get("FT_CLOCKS_DIR", tempfile.gettempdir()), f"ft_clocks_rank{tag}.csv")
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _epoch(ts: str):
        ts = ts.strip()
        try:
            main, _, frac = ts.partition(".")
            base = time.mktime(time.strptime(main, "%Y/%m/%d %H:%M:%S"))
            return base + (float("0." + frac) if frac else 0.0)
        except ValueError:
            return None

    def stop(self, t0: float | None = None, t1: float | None = None) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, pw, reasons, n_all = [], [], [], set(), 0
        for line in open(self.path):
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            n_all += 1
            t = self._epoch(c[0])
            if t0 is not None and t is not None and not (t0 - 0.1 <= t <= t1 + 0.1):
                continue
            try:
                sm.append(float(c[1]))
                mx.append(float(c[2]))
                pw.append(float(c[3]))
            except ValueError:
                continue
            for n, v in zip(self.REASONS, c[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ CUDA graphs

class RawGraph:
    """Stream capture -> instantiate -> upload -> launch, through the CUDA
    runtime the library itself uses (torch's graph API differs across
    versions).  Capture mode: relaxed."""

    def __init__(self, stream_ptr: int):
        import ctypes
        self.ct = ctypes
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.s = ctypes.c_void_p(stream_ptr)
        self.graph = ctypes.c_void_p()
        self.exec = ctypes.c_void_p()

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed ({rc})")

    def capture(self, fn):
        ct = self.ct
        self._ok(self.rt.cudaStreamBeginCapture(self.s, ct.c_int(2)), "cudaStreamBeginCapture")
        try:
            fn()
        finally:
            rc = self.rt.cudaStreamEndCapture(self.s, ct.byref(self.graph))
        self._ok(rc, "cudaStreamEndCapture")
        self._ok(self.rt.cudaGraphInstantiate(ct.byref(self.exec), self.graph, ct.c_ulonglong(0)),
                 "cudaGraphInstantiate")
        self._ok(self.rt.cudaGraphUpload(self.exec, self.s), "cudaGraphUpload")
        self._ok(self.rt.cudaStreamSynchronize(self.s), "cudaStreamSynchronize")

    def launch(self):
        self._ok(self.rt.cudaGraphLaunch(self.exec, self.s), "cudaGraphLaunch")

    def close(self):
        if self.exec:
            self.rt.cudaGraphExecDestroy(self.exec)
        if self.graph:
            self.rt.cudaGraphDestroy(self.graph)
        self.exec = self.ct.c_void_p()
        self.graph = self.ct.c_void_p()


# ------------------------------------------------------------- host pool

def whole_job_rate(units_per_rank: float, seconds_per_rank: float, world: int, device=None) -> float:
    """Whole-job throughput of N replicas: the units all ranks processed over
    the slowest rank's time (max over ranks)."""
    return world * units_per_rank / max_over_ranks(seconds_per_rank, world, device)


def shared_pool_file(shape: synth.Shape, seed: int, world: int, rank: int) -> tuple:
    """The host pool of N replicas on one node as one shared file
    (FT_POOL_DIR, default /dev/shm): rank 0 writes every record once, the
    others wait at a barrier and map it.  Returns (memmap, path)."""
    nbytes = shape.L * shape.E * shape.record_bytes
    path = os.path.join(os.environ.get("FT_POOL_DIR", "/dev/shm"), f"ft_pool_{shape.L}x{shape.E}_{seed}.bin")
    if rank == 0:
        mm = np.memmap(path, dtype=np.uint8, mode="w+", shape=(nbytes,))
        synth.fill_host_pool(mm, shape, seed)
        mm.flush()
        del mm
    barrier(world)
    return np.memmap(path, dtype=np.uint8, mode="r+", shape=(nbytes,)), path


def host_pool(shape: synth.Shape, seed: int, world: int, rank: int):
    """Page-locked host pool with every record.  One process: a pinned torch
    tensor.  N replicas on one node: the shared file of `shared_pool_file`,
    registered page-locked by every rank, so the node holds one copy."""
    import torch
    nbytes = shape.L * shape.E * shape.record_bytes
    if world == 1:
        pool = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        synth.fill_host_pool(pool.numpy(), shape, seed)
        return pool, None
    mm, path = shared_pool_file(shape, seed, world, rank)
    t = torch.from_numpy(mm)
    rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), nbytes, 0)
    if int(rc) != 0:
        raise RuntimeError(f"cudaHostRegister of the shared host pool failed ({rc})")
    return t, (mm, path)


def repeated_pool(sh: synth.Shape, seed: int, distinct: int = 16):
    """Pinned pool of L*E records that repeats the encodings of `distinct`
    drawn experts of layer 0 (the kernels' time and the routing do not depend
    on the values).  Returns (pool, per-record NVFP4 globals or None)."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    rb = sh.record_bytes
    enc = {synth.FMT_BF16: lambda s, l, e, H, F: synth.record_bf16(s, l, e, H, F),
           synth.FMT_NVFP4: synth.record_nvfp4, synth.FMT_MXFP4: synth.record_mxfp4,
           synth.FMT_FP8: synth.record_fp8}[sh.fmt]
    with ThreadPoolExecutor(min(distinct, os.cpu_count() or 1)) as ex:
        got = list(ex.map(lambda e: enc(seed, 0, e, sh.H, sh.F), range(distinct)))
    recs = [g[0] for g in got] if sh.fmt == synth.FMT_NVFP4 else got
    n = sh.L * sh.E
    pool = torch.empty(n * rb, dtype=torch.uint8, pin_memory=True)
    pn = pool.numpy().reshape(n, rb)
    for i in range(n):
        pn[i] = recs[i % distinct]
    glob = (np.array([got[i % distinct][1] for i in range(n)], dtype=np.float32)
            if sh.fmt == synth.FMT_NVFP4 else None)
    return pool, glob


# ------------------------------------------------------------ accounting

def kernel_bytes(shape: synth.Shape, T: int, dcnt: dict) -> dict:
    """Algorithmic bytes moved by each decode kernel over a run.

    expert_ffn (with the fused fill):
        link: every fill copies one record over the host link;
        hbm:  the fills written to HBM + the whole record of every resident
              GPU expert read (a fill is computed from the bytes in flight) +
              x read + h written and read once (fp32) + partial_C read + y
              written.
    route_ctl: logits + ids/gates written (small; reported for completeness).
    """
    H, F, E, k = shape.H, shape.F, shape.E, shape.k
    calls = dcnt["calls"]
    rb = shape.record_bytes
    link = dcnt["fills"] * rb
    hbm = link + dcnt["hits"] * rb + calls * T * H * 2 + 2 * dcnt["assign"] * F * 4 + calls * T * H * 4 * 2
    return {"expert_ffn": {"link": link, "hbm": hbm}, "route_ctl": {"hbm": calls * (T * E * 4 + 2 * T * k * 4)}}


def kernel_table(prof: dict, kb: dict, launches: int, peaks: dict, link_peak: float | None) -> dict:
    """Per-kernel launches, time, share, and achieved GB/s against the HBM
    peak (and the host link for the fills)."""
    total_ms = sum(v["ms"] for v in prof.values()) or 1.0
    out = {}
    for name, v in prof.items():
        us = 1e3 * v["ms"] / max(1, v["launches"])
        ent = {"launches": v["launches"], "ms_total": round(v["ms"], 3), "us_per_launch": round(us, 3),
               "share": round(v["ms"] / total_ms, 4)}
        for kind, byts in kb.get(name, {}).items():
            bpl = byts / max(1, launches)
            gbs = bpl / (us * 1e-6) / 1e9 if us > 0 else 0.0
            peak = link_peak if kind == "link" else peaks["hbm_gbs"]
            ent[kind] = {"bytes_per_launch": int(bpl), "achieved_GBps": round(gbs, 1),
                         "peak_GBps": round(peak, 1) if peak else None,
                         "frac": round(gbs / peak, 4) if peak else None}
        out[name] = ent
    return out


def roofline_entry(dom: str, kernels: dict, peaks: dict, link_peak: float | None, traffic=None) -> dict:
    """Roofline of the dominant kernel against the measured HBM peak.  When
    the kernel also copies fills over the host link, `link` gives that side
    and `binding` names whichever side's bytes at its peak take longer."""
    ent = kernels[dom]
    hbm = ent["hbm"]
    out = {"kernel": dom, "bound": "hbm", "achieved": hbm["achieved_GBps"], "peak": peaks["hbm_gbs"],
           "unit": "GB/s", "frac": hbm["frac"], "traffic": traffic,
           "bytes_per_launch": hbm["bytes_per_launch"], "us_per_launch": ent["us_per_launch"],
           "peak_source": peaks["source"]}
    link = ent.get("link")
    if link and link["bytes_per_launch"] > 0 and link_peak:
        t_link = link["bytes_per_launch"] / (link_peak * 1e9)
        t_hbm = hbm["bytes_per_launch"] / (peaks["hbm_gbs"] * 1e9)
        out["link"] = {"achieved": link["achieved_GBps"], "peak": round(link_peak, 1), "frac": link["frac"]}
        out["binding"] = "link" if t_link >= t_hbm else "hbm"
    return out


def traffic_from_profiles(kernel: str, scale_to: float | None = None):
    """DRAM bytes per launch from a committed ncu capture, if one matches the
    current kernel source (profiles/traffic.json keyed by kernel and source
    hash); else None.  A capture that records the algorithmic HBM bytes of
    its launch (`alg_bytes`) is scaled to `scale_to` algorithmic bytes: the
    traffic of these kernels grows in proportion to the bytes they move."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
        if not d:
            return None
        import hashlib
        h = hashlib.sha256()
        for src in d["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest()[:16] != d["source_sha"]:
            return None
        if "alg_bytes" in d:
            if scale_to is None:
                return None
            return int(d["dram_bytes"] / d["alg_bytes"] * scale_to)
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def measure_h2d_peak(device) -> float:
    import torch
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=device)
    best = 0.0
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize(device)
        best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del h, d
    return best


# ------------------------------------------------------------ our arm

class Decoder:
    """One decode context of the headline workload and the K-step graph that
    reads its inputs from fixed window buffers."""

    def __init__(self, ft, pool, device, K: int, s, ts):
        import torch
        wl = WORKLOAD
        sh = wl.shape
        self.ft, self.sh, self.wl, self.K, self.s, self.device = ft, sh, wl, K, s, device
        self.T, self.L = wl.T, sh.L
        self.ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, pool, T_max=wl.T, compute_stream=s.cuda_stream,
                              transfer_stream=ts.cuda_stream)
        T, L, E, H = self.T, self.L, sh.E, sh.H
        self.lg = torch.empty(K, L, T, E, dtype=torch.float32, device=device)
        self.x = torch.empty(K, L, T, H, dtype=torch.int16, device=device)
        self.pc = torch.from_numpy(np.stack([synth.random_f32(wl.seed, (l,), (T, H), 0.1) for l in range(L)])).to(
            device)
        self.y = torch.empty(L, T, H, dtype=torch.float32, device=device)

    def graph(self):
        import torch
        g = RawGraph(self.s.cuda_stream)
        xb = self.x.view(torch.bfloat16)

        def steps():
            for i in range(self.K):
                for l in range(self.L):
                    self.ctx.route_ctl(l, self.T, logits=self.lg[i, l], B_P=self.wl.B_P, B_H=self.wl.B_H)
                    self.ctx.moe_forward(xb[i, l], self.pc[l], self.y[l])
        with torch.cuda.stream(self.s):
            g.capture(steps)
        return g


def decode_inputs(n_steps: int):
    """AR(1) logits [n, L, T, E] and bf16 tokens [n, L, T, H] of the headline
    workload's first n steps."""
    wl = WORKLOAD
    sh = wl.shape
    lg = synth.ar1_logits(wl.seed, n_steps, sh.L, wl.T, sh.E, wl.rho, wl.sigma)
    xs = np.stack([np.stack([synth.tokens_bf16(wl.seed, s, l, wl.T, sh.H) for l in range(sh.L)])
                   for s in range(n_steps)]).view(np.int16)
    return lg, xs


def run_ours(args, rank, world, local_rank):
    import torch
    import moe_expert_cache_gb300 as ft

    ft.load()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    wl = WORKLOAD
    sh = wl.shape
    T, L, E, H = wl.T, sh.L, sh.E, sh.H
    W, K = args.warmup, args.steps
    peaks = read_peaks()

    t0 = time.time()
    pool, shared = host_pool(sh, wl.seed, world, rank)
    t_pool = time.time() - t0

    s = torch.cuda.Stream(device)
    ts = torch.cuda.Stream(device)
    dec = Decoder(ft, pool, device, K, s, ts)

    # ---- warm-up: W eager steps
    lg_w, x_w = decode_inputs(W)
    lg_wd = torch.from_numpy(lg_w).to(device)
    x_wd = torch.from_numpy(x_w).to(device).view(torch.bfloat16)
    with torch.cuda.stream(s):
        for i in range(W):
            for l in range(L):
                dec.ctx.route_ctl(l, T, logits=lg_wd[i, l], B_P=wl.B_P, B_H=wl.B_H)
                dec.ctx.moe_forward(x_wd[i, l], dec.pc[l], dec.y[l])
    torch.cuda.synchronize(device)
    # windows: enough to cover the workload's configured steps (256 decode
    # steps at T=1), at least 3
    R = args.windows or int(min(50, max(3, math.ceil(wl.steps / K))))
    R = int(max_over_ranks(float(R), world, device))
    n_steps = W + (R + 1) * K  # R timed windows + one profiled window
    lg_all, x_all = decode_inputs(n_steps)
    lg_all_d = torch.from_numpy(lg_all).to(device)
    x_all_d = torch.from_numpy(x_all).to(device)

    def stage(win: int):
        a = W + win * K
        with torch.cuda.stream(s):
            dec.lg.copy_(lg_all_d[a:a + K])
            dec.x.copy_(x_all_d[a:a + K])

    t0 = time.time()
    g = dec.graph()
    t_capture = time.time() - t0
    link_before = measure_h2d_peak(device) if rank == 0 else None
    c0 = dec.ctx.counters()
    clocks = ClockSampler(gpu_query_id(device), str(local_rank))
    win_ms = []
    span0 = time.time()
    for r in range(R):
        stage(r)
        torch.cuda.synchronize(device)
        barrier(world, device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            ev0.record(s)
            g.launch()
            ev1.record(s)
        torch.cuda.synchronize(device)
        barrier(world, device)
        win_ms.append(ev0.elapsed_time(ev1))
    span1 = time.time()
    clk = clocks.stop(span0, span1)
    c1 = dec.ctx.counters()
    g.close()
    assert dec.ctx.status() == ft.FT_OK
    link_after = measure_h2d_peak(device) if rank == 0 else None
    dcnt = {k_: c1[k_] - c0[k_] for k_ in c1}

    # ---- per-kernel times: one more window of the same K steps, captured
    # with the library's event records around every launch
    stage(R)
    dec.ctx.profile_enable(True)
    gp = dec.graph()
    p0 = dec.ctx.counters()
    with torch.cuda.stream(s):
        gp.launch()
    torch.cuda.synchronize(device)
    prof = dec.ctx.profile_read()
    dec.ctx.profile_enable(False)
    p1 = dec.ctx.counters()
    gp.close()
    pcnt = {k_: p1[k_] - p0[k_] for k_ in p1}
    link_fill_gbps = dec.ctx.measure_link(16, 3)
    assert dec.ctx.status() == ft.FT_OK
    dec.ctx.close()

    med = statistics.median(win_ms)
    t_med_max = max_over_ranks(med, world, device)
    value = world * T * K / (t_med_max * 1e-3)
    link_peak = max(x for x in (link_before, link_after) if x) if rank == 0 else None
    kb = kernel_bytes(sh, T, pcnt)
    kernels = kernel_table(prof, kb, pcnt["calls"], peaks, link_peak)
    dom = max(prof, key=lambda n: prof[n]["ms"])
    traffic = (traffic_from_profiles(dom, kernels[dom]["hbm"]["bytes_per_launch"]) if dom == "expert_ffn" else None)
    roofline = roofline_entry(dom, kernels, peaks, link_peak, traffic)
    fills = pcnt["fills"] / max(1, pcnt["calls"])
    floor_ms = fills * L * sh.record_bytes / (link_peak * 1e9) * 1e3 if link_peak else None

    # ---- end to end: every step's inputs copied from pinned host memory and
    # its y read back, inside the timed graph
    e2e_ms = run_e2e(ft, pool, device, W, K, R, lg_all, x_all, world)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(t_med_max / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded AR(1) logits, N(0,0.02) bf16 weights)",
        "gpu_launches": int(2 * L * K),
        "config": headline_config(world),
        "roofline": roofline,
        "repeats": {"windows": R, "of_steps": K, "median_ms": round(med, 3), "min_ms": round(min(win_ms), 3),
                    "max_ms": round(max(win_ms), 3),
                    "link_GBps": [round(x, 1) if x else None for x in (link_before, link_after)],
                    "B_P_fill_path": round(link_fill_gbps, 1)},
        "decode": {"hit_rate": round(dcnt["hits"] / max(1, dcnt["unique"]), 4),
                   "fills_per_layer_step": round(dcnt["fills"] / max(1, dcnt["calls"]), 3),
                   "link_floor_ms_step": round(floor_ms, 3) if floor_ms else None,
                   "route_ctl_us": kernels.get("route_ctl", {}).get("us_per_launch")},
        "clocks": clk,
        "e2e": {"value": round(world * T * K / (e2e_ms * 1e-3), 2), "unit": UNIT,
                "h2d_bytes_per_step": L * T * (E * 4 + H * 2 + H * 4), "d2h_bytes_per_step": L * T * H * 4},
    }
    detail = {"kernels": kernels, "windows_ms": [round(x, 3) for x in win_ms], "counters": dcnt,
              "profile_window_counters": pcnt,
              "setup_s": {"host_pool": round(t_pool, 1), "graph_capture": round(t_capture, 1)}}
    legs, leg_detail = {}, {}
    if rank == 0 and not args.no_t16:
        legs["decode_t16"], leg_detail["decode_t16"] = run_decode_t16_bench(pool, device, link_peak)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(pool.numpy() if world == 1 else shared[0], args.cpu_seconds)
    if rank == 0 and not args.no_hbm:
        legs["bf16_q0"], leg_detail["bf16_q0"] = run_bf16_hbm_bench(pool, device, peaks)
    del pool, dec
    if not args.no_prefill:
        legs["prefill"], leg_detail["prefill"] = run_prefill_bench(device, peaks)
    if rank == 0 and not args.no_fp4:
        legs["quant_q0"], leg_detail["quant_q0"] = run_quant_decode_bench(device, peaks)
    if rank == 0 and not args.no_large:
        legs["large_nvfp4"], leg_detail["large_nvfp4"] = run_large_nvfp4_bench(device, peaks, link_peak)
    out["legs"] = legs
    detail["legs"] = leg_detail
    path = os.environ.get("FT_BENCH_DETAIL")
    if path and rank == 0:
        with open(path, "w") as f:
            json.dump({"line": out, "detail": detail}, f, indent=1)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if shared is not None:
        import torch as _t
        _t.cuda.cudart().cudaHostUnregister(_t.from_numpy(shared[0]).data_ptr())
    return out


def run_e2e(ft, pool, device, W, K, R, lg_all, x_all, world) -> float:
    """Median window time of the same K-step windows with every step's
    logits, x and partial_C copied from pinned host memory and y copied back
    inside the timed graph."""
    import torch
    wl = WORKLOAD
    sh = wl.shape
    T, L, E, H = wl.T, sh.L, sh.E, sh.H
    s, ts = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ctx = ft.Context(L, E, sh.k, H, sh.F, wl.S, pool, T_max=T, compute_stream=s.cuda_stream,
                     transfer_stream=ts.cuda_stream)
    lg_h = torch.empty(K, L, T, E, dtype=torch.float32).pin_memory()
    x_h = torch.empty(K, L, T, H, dtype=torch.int16).pin_memory()
    pc_h = torch.from_numpy(np.stack([synth.random_f32(wl.seed, (l,), (T, H), 0.1) for l in range(L)])).pin_memory()
    y_h = torch.empty(K, L, T, H, dtype=torch.float32).pin_memory()
    lg_d = torch.empty(L, T, E, dtype=torch.float32, device=device)
    x_d = torch.empty(L, T, H, dtype=torch.int16, device=device)
    pc_d = torch.empty(L, T, H, dtype=torch.float32, device=device)
    y_d = torch.empty(L, T, H, dtype=torch.float32, device=device)
    xb = x_d.view(torch.bfloat16)
    with torch.cuda.stream(s):
        lgw = torch.from_numpy(lg_all[:W]).to(device)
        xw = torch.from_numpy(x_all[:W]).to(device).view(torch.bfloat16)
        pc_d.copy_(pc_h)
        for i in range(W):
            for l in range(L):
                ctx.route_ctl(l, T, logits=lgw[i, l], B_P=wl.B_P, B_H=wl.B_H)
                ctx.moe_forward(xw[i, l], pc_d[l], y_d[l])
    torch.cuda.synchronize(device)

    def steps():
        for i in range(K):
            lg_d.copy_(lg_h[i], non_blocking=True)
            x_d.copy_(x_h[i], non_blocking=True)
            pc_d.copy_(pc_h, non_blocking=True)
            for l in range(L):
                ctx.route_ctl(l, T, logits=lg_d[l], B_P=wl.B_P, B_H=wl.B_H)
                ctx.moe_forward(xb[l], pc_d[l], y_d[l])
            y_h[i].copy_(y_d, non_blocking=True)

    g = RawGraph(s.cuda_stream)
    with torch.cuda.stream(s):
        g.capture(steps)
    ms = []
    for r in range(R):
        a = W + r * K
        lg_h.numpy()[:] = lg_all[a:a + K]
        x_h.numpy()[:] = x_all[a:a + K]
        torch.cuda.synchronize(device)
        barrier(world, device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.launch()
            e1.record(s)
        torch.cuda.synchronize(device)
        barrier(world, device)
        ms.append(e0.elapsed_time(e1))
    g.close()
    assert ctx.status() == ft.FT_OK
    ctx.close()
    return max_over_ranks(statistics.median(ms), world, device)


def run_decode_t16_bench(pool, device, link_peak):
    """Decode T=16 with resize (same layer shapes and host pool as decode T=1):
    48 layers, 768 slots shrunk to 384 before step 32 and grown back before
    step 64, 128 steps from an empty cache, AR(1) rho=0.7, B_P=25, B_H=90.
    Steps run eagerly (the resizes are host safe points); tokens/s is over the
    steps' CUDA-event time, resize latency is each call's host time."""
    import torch
    import moe_expert_cache_gb300 as ft
    wl = synth.DECODE_T16
    sh = wl.shape
    T, L, E, H = wl.T, sh.L, sh.E, sh.H
    logits = torch.from_numpy(synth.ar1_logits(wl.seed, wl.steps, L, T, E, wl.rho, wl.sigma)).to(device)
    xs = torch.from_numpy(np.stack([synth.tokens_bf16(wl.seed, 0, l, T, H) for l in range(L)]).view(np.int16)).to(
        device).view(torch.bfloat16)
    pc = torch.zeros(T, H, device=device)
    y = torch.empty(T, H, device=device)
    cs = torch.cuda.Stream(device)
    ctx = ft.Context(L, E, sh.k, H, sh.F, wl.S, pool, T_max=T, compute_stream=cs.cuda_stream)
    resize_at = dict(synth.DECODE_T16_RESIZE)
    ms, resize_ms = 0.0, []
    c0 = ctx.counters()
    for s0, s1 in ((0, 32), (32, 64), (64, wl.steps)):
        if s0 in resize_at:
            t0 = time.perf_counter()
            ctx.cache_resize(resize_at[s0])
            resize_ms.append(round((time.perf_counter() - t0) * 1e3, 2))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):
            e0.record(cs)
            for st in range(s0, s1):
                for l in range(L):
                    ctx.route_ctl(l, T, logits=logits[st, l], B_P=wl.B_P, B_H=wl.B_H)
                    ctx.moe_forward(xs[l], pc, y)
            e1.record(cs)
        torch.cuda.synchronize(device)
        ms += e0.elapsed_time(e1)
    c1 = ctx.counters()
    assert ctx.status() == ft.FT_OK
    ctx.close()
    d = {k_: c1[k_] - c0[k_] for k_ in c1}
    calls = max(1, d["calls"])
    floor = d["fills"] / wl.steps * sh.record_bytes / ((link_peak or 211.0) * 1e9) * 1e3
    leg = {"tok_s": round(T * wl.steps / (ms * 1e-3), 1), "ms_step": round(ms / wl.steps, 3),
           "floor_ms": round(floor, 3), "resize_ms": resize_ms}
    detail = dict(leg, workload="decode T=16: 48 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, 768 slots "
                                "(384 during steps 32-63), AR(1) rho=0.7, B_P=25, B_H=90, 128 steps from an empty "
                                "cache; eager library calls, CUDA-event time of the steps",
                  hit_rate=round(d["hits"] / max(1, d["unique"]), 4),
                  fills_per_layer_step=round(d["fills"] / calls, 3),
                  gpu_experts_per_layer_step=round((d["hits"] + d["fills"]) / calls, 2))
    return leg, detail


class L2Flusher:
    """Reads a buffer twice the size of L2 so the next launch reads HBM.  A
    read leaves only clean lines behind: a write would leave L2 full of dirty
    lines whose write-back would steal bandwidth from the timed launch."""

    def __init__(self, device):
        import torch
        self.buf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.out = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        torch.amax(self.buf, dim=0, out=self.out)


def hits_only_times(ctx, T, routes, x, pc, y, flush, stream, device):
    """Expert-kernel device time of each call of `routes` (a list of
    (topk_ids, topk_w) device tensors or (logits,) tuples), every record
    resident (q = 0), L2 flushed before each call.  Returns (median us,
    counters of the calls)."""
    import torch
    c0 = ctx.counters()
    us = []
    for r in routes:
        with torch.cuda.stream(stream):
            flush()
            if len(r) == 1:
                ctx.route_ctl(0, T, logits=r[0], B_P=1.0, B_H=1.0)
            else:
                ctx.route_ctl(0, T, topk_ids=r[0], topk_w=r[1], B_P=1.0, B_H=1.0)
            ctx.profile_enable(True)
            ctx.moe_forward(x, pc, y)
        pr = ctx.profile_read()
        ctx.profile_enable(False)
        us.append(1e3 * pr["expert_ffn"]["ms"] / pr["expert_ffn"]["launches"])
    c1 = ctx.counters()
    d = {k_: c1[k_] - c0[k_] for k_ in c1}
    assert d["fills"] == 0, "a hits-only leg filled"
    return statistics.median(us), d


def one_fill_times(ctx, E, x, pc, y, flush, stream, calls: int = 12, warmup: int = 1):
    """Expert-kernel device time of T=1 calls that route 7 resident experts
    and 1 expert evicted just before (ft_set_ctl_state), so each call makes
    exactly one fill beside 7 hits; L2 flushed before each call; `warmup`
    untimed calls first (the first fill call of a context runs cold).  Returns
    (median us of the timed calls, the standalone fill time of one record in
    us)."""
    import torch
    k = 8
    w = torch.full((1, k), 1.0 / k, device=x.device)
    us = []
    for i in range(warmup + calls):
        sfi, ifs, stp, clk = ctx.ctl_state()
        victim = 8 * (i + 1)  # resident, not among the call's 7 hits
        s_v = int(sfi[victim])
        sfi[victim] = -1
        ifs[s_v] = -1
        stp[s_v] = 0
        ctx.set_ctl_state(sfi, ifs, stp, clk)
        ids = torch.tensor([[0, 1, 2, 3, 4, 5, 6, victim]], dtype=torch.int32, device=x.device)
        c0 = ctx.counters()
        with torch.cuda.stream(stream):
            flush()
            ctx.route_ctl(0, 1, topk_ids=ids, topk_w=w, B_P=1.0, B_H=1.0)
            ctx.profile_enable(True)
            ctx.moe_forward(x[:1], pc[:1], y[:1])
        pr = ctx.profile_read()
        ctx.profile_enable(False)
        c1 = ctx.counters()
        assert c1["fills"] - c0["fills"] == 1 and c1["hits"] - c0["hits"] == 7
        if i >= warmup:
            us.append(1e3 * pr["expert_ffn"]["ms"] / pr["expert_ffn"]["launches"])
    gbps = ctx.measure_link(1, 3)
    return statistics.median(us), None if not gbps else 1e6 * ctx_record_bytes(ctx) / (gbps * 1e9)


def ctx_record_bytes(ctx) -> int:
    import moe_expert_cache_gb300 as ft
    return ft.record_bytes(ctx.H, ctx.F, ctx.fmt)


def run_bf16_hbm_bench(pool, device, peaks, calls: int = 24):
    """BF16 expert kernel with every record resident (q = 0), the HBM-bound
    case: one layer of the decode shapes (E=128, top-8, H=2048, F=768) in 128
    slots, T=1 (disjoint sets of 8 experts in turn) and T=16 (AR(1) rho=0.7
    routing), L2 flushed before every call; achieved GB/s = the call's
    algorithmic bytes / its device time."""
    import torch
    import moe_expert_cache_gb300 as ft
    sh1 = synth.Shape(L=1, E=128, k=8, H=2048, F=768)
    cs = torch.cuda.Stream(device)
    ctx = ft.Context(1, sh1.E, sh1.k, sh1.H, sh1.F, sh1.E, pool, T_max=16, compute_stream=cs.cuda_stream)
    flush = L2Flusher(device)
    x = torch.from_numpy(synth.tokens_bf16(0, 0, 0, 16, sh1.H).view(np.int16)).to(device).view(torch.bfloat16)
    pc = torch.zeros(16, sh1.H, device=device)
    y = torch.empty(16, sh1.H, device=device)
    w8 = torch.full((1, 8), 1.0 / 8, device=device)
    with torch.cuda.stream(cs):  # make every record of layer 0 resident
        for i in range(16):
            ids = torch.arange(8 * i, 8 * i + 8, dtype=torch.int32, device=device).view(1, 8)
            ctx.route_ctl(0, 1, topk_ids=ids, topk_w=w8, B_P=1.0, B_H=1.0)
            ctx.moe_forward(x[:1], pc[:1], y[:1])
    torch.cuda.synchronize(device)
    leg, detail = {}, {}
    r1 = [(torch.arange(8 * (i % 16), 8 * (i % 16) + 8, dtype=torch.int32, device=device).view(1, 8), w8)
          for i in range(calls)]
    lg16 = torch.from_numpy(synth.ar1_logits(3, calls, 1, 16, sh1.E, 0.7)[:, 0]).to(device)
    r16 = [(lg16[i],) for i in range(calls)]
    for T, routes in ((1, r1), (16, r16)):
        us, d = hits_only_times(ctx, T, routes, x[:T], pc[:T], y[:T], flush, cs, device)
        hbm = kernel_bytes(sh1, T, d)["expert_ffn"]["hbm"] / max(1, d["calls"])
        gbs = hbm / (us * 1e-6) / 1e9
        leg[f"t{T}"] = {"us": round(us, 2), "GBps": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                        "traffic": traffic_from_profiles("expert_ffn_q0", hbm)}
        detail[f"t{T}"] = dict(leg[f"t{T}"], hits_per_launch=round(d["hits"] / max(1, d["calls"]), 2),
                               bytes_per_launch=int(hbm), calls=d["calls"])
    assert ctx.status() == ft.FT_OK
    ctx.close()
    detail["workload"] = ("BF16 decode kernel, hits only: 1 layer, E=128, top-8, hidden 2048, ffn 768, 128 slots "
                          "all resident; T=1 over disjoint 8-expert sets, T=16 AR(1) rho=0.7; L2 flushed per call")
    return leg, detail


def run_quant_decode_bench(device, peaks, calls_t1: int = 48, calls_t64: int = 16):
    """Quantised expert kernels (NVFP4, MXFP4 and block-FP8 records) on the
    Large shapes, hits only: one MoE layer of E=256 experts, top-8, H=4096,
    F=2048, every record resident in 256 slots, AR(1) rho=0.8 logits, T=1
    and T=64, L2 flushed before every call.  The bound is HBM: each launch
    reads the records of its routed experts."""
    import torch
    import moe_expert_cache_gb300 as ft
    H, F, E, k = 4096, 2048, 256, 8
    cs = torch.cuda.Stream(device)
    flush = L2Flusher(device)
    leg, detail = {}, {"workload": "Large shapes, hits only: 1 MoE layer, E=256, top-8, hidden 4096, ffn 2048, "
                                   "every record resident, AR(1) rho=0.8 logits, L2 flushed per call; records of "
                                   "16 drawn experts repeated"}
    for name, fmt in (("nvfp4", synth.FMT_NVFP4), ("mxfp4", synth.FMT_MXFP4), ("fp8", synth.FMT_FP8)):
        sh = synth.Shape(L=1, E=E, k=k, H=H, F=F, fmt=fmt)
        pool, glob = repeated_pool(sh, 0)
        ctx = ft.Context(1, E, k, H, F, E, pool, fmt=fmt, T_max=64, nvfp4_global=glob,
                         compute_stream=cs.cuda_stream)
        x = torch.from_numpy(synth.tokens_bf16(0, 0, 0, 64, H).view(np.int16)).to(device).view(torch.bfloat16)
        pc = torch.zeros(64, H, device=device)
        y = torch.empty(64, H, device=device)
        w8 = torch.full((1, 8), 1.0 / 8, device=device)
        with torch.cuda.stream(cs):  # every record resident
            for i in range(E // 8):
                ids = torch.arange(8 * i, 8 * i + 8, dtype=torch.int32, device=device).view(1, 8)
                ctx.route_ctl(0, 1, topk_ids=ids, topk_w=w8, B_P=1.0, B_H=1.0)
                ctx.moe_forward(x[:1], pc[:1], y[:1])
        torch.cuda.synchronize(device)
        res, det = {}, {"record_bytes": sh.record_bytes}
        for T, calls in ((1, calls_t1), (64, calls_t64)):
            lg = torch.from_numpy(synth.ar1_logits(0, calls, 1, T, E, 0.8)[:, 0]).to(device)
            us, d = hits_only_times(ctx, T, [(lg[i],) for i in range(calls)], x[:T], pc[:T], y[:T], flush, cs,
                                    device)
            hbm = kernel_bytes(sh, T, d)["expert_ffn"]["hbm"] / max(1, d["calls"])
            gbs = hbm / (us * 1e-6) / 1e9
            kname = {synth.FMT_NVFP4: "expert_ffn_fp4", synth.FMT_MXFP4: "expert_ffn_mxfp4",
                     synth.FMT_FP8: "expert_ffn_fp8"}[fmt]
            tr = traffic_from_profiles(kname, hbm)
            res[f"t{T}"] = [round(us, 1), round(gbs / peaks["hbm_gbs"], 4), round(tr / hbm, 3) if tr else None]
            det[f"t{T}"] = {"us_per_launch": round(us, 2), "hits_per_launch": round(d["hits"] / max(1, d["calls"]), 2),
                            "hbm_bytes_per_launch": int(hbm), "achieved_GBps": round(gbs, 1),
                            "frac": round(gbs / peaks["hbm_gbs"], 4),
                            "traffic": tr}
        # one fill beside 7 hits: the fill streams inside the expert launch
        us1, fill_us = one_fill_times(ctx, E, x, pc, y, flush, cs)
        res["fill1"] = [round(us1, 1), round(fill_us, 1) if fill_us else None]
        det["t1_one_fill"] = {"us_per_launch": round(us1, 2), "standalone_fill_us": round(fill_us, 2) if fill_us else None,
                              "hits_only_us": det["t1"]["us_per_launch"]}
        assert ctx.status() == ft.FT_OK
        ctx.close()
        del pool
        leg[name] = res
        detail[name] = det
    leg["cols"] = ("t1, t64: [us per launch, frac of HBM, DRAM traffic / algorithmic bytes]; "
                   "fill1: [us per launch with 1 fill + 7 hits, standalone fill us]")
    return leg, detail


def prefill_chunk_times(ft, sh, S, T, pool, glob, device, reps: int):
    """Chunk time (prefill_begin + one prefill_layer per layer) with the
    double buffer, the per-kernel profile, and the same chunk with the copies
    on the compute stream (single buffer in flight)."""
    import torch
    L = sh.L
    xs = [torch.from_numpy(synth.tokens_bf16(0, 900, l, T, sh.H).view(np.int16)).to(device).view(torch.bfloat16)
          for l in range(L)]
    lg = [torch.from_numpy(synth.iid_logits(0, (900, l), T, sh.E)).to(device) for l in range(L)]
    ys = [torch.empty(T, sh.H, dtype=torch.float32, device=device) for _ in range(L)]
    cs, ts = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def measure(two_streams: bool):
        ctx = ft.Context(L, sh.E, sh.k, sh.H, sh.F, S, pool, fmt=sh.fmt, T_max=4, T_prefill_max=T,
                         nvfp4_global=glob, compute_stream=cs.cuda_stream,
                         transfer_stream=ts.cuda_stream if two_streams else 0)

        def chunk():
            ctx.prefill_begin(0)
            for l in range(L):
                ctx.prefill_layer(l & 1, l, l + 1 if l + 1 < L else -1, T, xs[l], lg[l], ys[l])

        with torch.cuda.stream(cs):
            chunk()
        torch.cuda.synchronize(device)
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(cs):
                e0.record(cs)
                chunk()
                e1.record(cs)
            torch.cuda.synchronize(device)
            times.append(e0.elapsed_time(e1))
        ctx.profile_enable(True)
        with torch.cuda.stream(cs):
            chunk()
        prof = ctx.profile_read()
        assert ctx.status() == ft.FT_OK
        ctx.close()
        return statistics.median(times), prof

    t_db, prof = measure(True)
    t_sb, _ = measure(False)
    return t_db, t_sb, prof


def prefill_summary(sh, T, t_db, t_sb, prof, peaks):
    L = sh.L
    h2d = prof["pf_h2d"]["ms"]
    comp = sum(v["ms"] for k_, v in prof.items() if k_ != "pf_h2d")
    g1 = prof["pf_gemm1_swiglu"]["ms"] / L
    g2 = prof["pf_gemm2"]["ms"] / L
    fl1 = 2.0 * T * sh.k * 2 * sh.F * sh.H
    fl2 = 2.0 * T * sh.k * sh.F * sh.H
    tf = (fl1 + fl2) / ((g1 + g2) * 1e-3) / 1e12
    tot = sum(v["ms"] for v in prof.values())
    leg = {"tok_s": round(T * L / (t_db * 1e-3), 1), "ms_chunk": round(t_db, 2),
           "eta": round(max(h2d, comp) / t_db, 4), "h2d_GBps": round(L * sh.E * sh.record_bytes / (h2d * 1e-3) / 1e9, 1),
           "sb_ms": round(t_sb, 2), "gemm_frac": round(tf / peaks["bf16_tflops"], 4),
           "gemm_TFs": [round(fl1 / (g1 * 1e-3) / 1e12, 1), round(fl2 / (g2 * 1e-3) / 1e12, 1)]}
    detail = dict(leg, ms_h2d=round(h2d, 3), ms_compute=round(comp, 3),
                  hidden_fraction=round((h2d + comp - t_db) / min(h2d, comp), 4),
                  double_buffer_speedup=round(t_sb / t_db, 4),
                  roofline_gemm={"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                                 "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                                 "flops_per_layer": fl1 + fl2, "peak_source": peaks["source"],
                                 "traffic": traffic_from_profiles("pf_gemm")},
                  kernels={k_: {"launches": v["launches"], "ms_total": round(v["ms"], 3),
                                "share": round(v["ms"] / tot, 4)} for k_, v in prof.items()})
    return leg, detail


def run_prefill_bench(device, peaks, reps: int = 3):
    """Prefill workload: 4 layers, E=128, top-8, H=2048, F=768, T=8192, 256
    slots, full-layer double buffer.  Chunk = prefill_begin + 4 prefill_layer
    calls, timed with CUDA events on the compute stream; per-kernel device
    times from the library's event records in one further chunk; the same
    chunk with the copies on the compute stream as the single-buffer A/B."""
    import torch
    import moe_expert_cache_gb300 as ft
    wl = synth.PREFILL
    sh = wl.shape
    pool = torch.empty(sh.L * sh.E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
    synth.fill_host_pool(pool.numpy(), sh, wl.seed)
    t_db, t_sb, prof = prefill_chunk_times(ft, sh, wl.S, wl.T, pool, None, device, reps)
    leg, detail = prefill_summary(sh, wl.T, t_db, t_sb, prof, peaks)
    detail["workload"] = ("prefill: 4 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, T=8192, 256 slots, "
                          "full-layer double buffer")
    return leg, detail


def run_large_nvfp4_bench(device, peaks, link_peak):
    """Large NVFP4 workload: 8 MoE layers, E=256, top-8, H=4096, F=2048,
    NVFP4 records (16 drawn experts repeated over the 2048 records), 512
    slots, AR(1) rho=0.8 logits, B_P=52.7, B_H=150: 64 decode steps at T=1
    then 64 at T=64 from an empty cache (eager library calls, CUDA-event time
    of the steps, fills included), then one T=4096 prefill chunk of all 8
    layers through the full-layer double buffer.  The link floor of a decode
    phase is its fills' bytes over the measured host link."""
    import torch
    import moe_expert_cache_gb300 as ft
    wl = synth.LARGE_NVFP4
    sh = wl.shape
    L, E, H = sh.L, sh.E, sh.H
    pool, glob = repeated_pool(sh, 0)
    cs = torch.cuda.Stream(device)
    ctx = ft.Context(L, E, sh.k, H, sh.F, wl.S, pool, fmt=sh.fmt, T_max=64, nvfp4_global=glob,
                     compute_stream=cs.cuda_stream)
    leg, detail = {}, {}
    lp = link_peak or 211.0
    for T, steps in ((1, 64), (64, 64)):
        lg = torch.from_numpy(synth.ar1_logits(wl.seed, steps, L, T, E, wl.rho)).to(device)
        x = torch.from_numpy(np.stack([synth.tokens_bf16(wl.seed, 0, l, T, H) for l in range(L)]).view(np.int16)).to(
            device).view(torch.bfloat16)
        pc = torch.zeros(T, H, device=device)
        y = torch.empty(T, H, device=device)
        c0 = ctx.counters()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):
            e0.record(cs)
            for st in range(steps):
                for l in range(L):
                    ctx.route_ctl(l, T, logits=lg[st, l], B_P=wl.B_P, B_H=wl.B_H)
                    ctx.moe_forward(x[l], pc, y)
            e1.record(cs)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1)
        c1 = ctx.counters()
        d = {k_: c1[k_] - c0[k_] for k_ in c1}
        floor = d["fills"] * sh.record_bytes / (lp * 1e9) * 1e3
        leg[f"t{T}"] = {"tok_s": round(T * steps / (ms * 1e-3), 1), "ms_step": round(ms / steps, 3),
                        "floor_ms_step": round(floor / steps, 3)}
        detail[f"t{T}"] = dict(leg[f"t{T}"], fills_per_layer_step=round(d["fills"] / max(1, d["calls"]), 3),
                               hit_rate=round(d["hits"] / max(1, d["unique"]), 4))
    assert ctx.status() == ft.FT_OK
    ctx.close()
    t_db, t_sb, prof = prefill_chunk_times(ft, sh, wl.S, 4096, pool, glob, device, reps=2)
    pl, pd = prefill_summary(sh, 4096, t_db, t_sb, prof, peaks)
    leg["prefill"] = {k_: pl[k_] for k_ in ("tok_s", "ms_chunk", "eta", "h2d_GBps")}
    detail["prefill"] = pd
    detail["workload"] = ("Large NVFP4: 8 MoE layers, E=256, top-8, hidden 4096, ffn 2048, 512 slots, AR(1) rho=0.8, "
                          "B_P=52.7, B_H=150; 64 steps T=1 then 64 steps T=64 from an empty cache; T=4096 prefill "
                          "chunk of 8 layers (double buffer)")
    del pool
    return leg, detail


# ---------------------------------------------------------- oracle timing

def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def oracle_samples(pool_np, n_samples: int, seconds: float | None = None):
    """Run the oracle on decode samples of the workload: control for every
    layer of a step (exact integers), fp64 numerics for sampled layers, with
    the expert weights read from the host pool.  A sample = one MoE layer of
    one decode step (control + FFN of its T=1 token over its 8 routed experts).
    Returns (samples done, seconds)."""
    from oracle import control as ctl
    from oracle import numerics as nm
    wl = WORKLOAD
    sh = wl.shape
    rb = sh.record_bytes
    steps = max(1, min(wl.steps, (n_samples + sh.L - 1) // sh.L))
    logits = synth.ar1_logits(wl.seed, steps, sh.L, wl.T, sh.E, wl.rho, wl.sigma)
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    done = 0
    t0 = time.perf_counter()
    for s in range(steps):
        for l in range(sh.L):
            ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits[s, l]])
            ctl.route_ctl(st, l, ids, wl.B_P, wl.B_H)
            x = nm.bf16_to_f64(synth.tokens_bf16(wl.seed, s, l, wl.T, sh.H))

            def weights(e, l=l):
                fid = l * sh.E + e
                return nm.record_weights_bf16(pool_np[fid * rb:(fid + 1) * rb], sh.H, sh.F)
            nm.gated_sum(x, ids, gates, lambda t, j: True, weights)
            done += 1
            if done >= n_samples or (seconds is not None and time.perf_counter() - t0 > seconds):
                return done, time.perf_counter() - t0
    return done, time.perf_counter() - t0


def cpu_baseline(pool_np, seconds: float) -> dict:
    done, dt = oracle_samples(pool_np, 10 ** 9, seconds)
    L = WORKLOAD.shape.L
    tok_s = WORKLOAD.T * done / L / dt
    return {"value": round(tok_s, 5), "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} layer-steps (control + fp64 FFN of 8 experts) in {dt:.1f} s; tok/s = layer-steps/{L}/s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm, on this machine's host cores: W
    warm-up and K timed samples, one sample = one MoE layer of one decode
    token of the headline workload."""
    if rank != 0:
        return None
    sh = WORKLOAD.shape
    pool = np.empty(sh.L * sh.E * sh.record_bytes, dtype=np.uint8)
    synth.fill_host_pool(pool, sh, WORKLOAD.seed)
    W, K = args.warmup, args.steps
    oracle_samples(pool, W)
    done, dt = oracle_samples(pool, K)
    L = sh.L
    v = WORKLOAD.T * done / L / dt
    cores = _blas_threads()
    return {"metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(1e3 * dt / max(1, done), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded AR(1) logits, N(0,0.02) bf16 weights)",
            "impl": "reference", "config": headline_config(world),
            "cpu_baseline": {"value": round(v, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{done} layer-steps (one step = one MoE layer of one decode token)"},
            "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------- profiler cases

def run_ncu_case(args):
    """A small single-layer BF16 case for profiler captures (not a bench line).

    One layer of the decode T=1 shape (E=128, top-8, H=2048, F=768) in 128
    slots.  Every call routes the token to experts 0..7-q (resident) plus q
    experts not yet resident, so each expert-kernel launch runs 8-q hits and
    q fused fills.  Six calls; capture e.g. the fifth expert launch with
    `ncu -k regex:expert_ffn -s 4 -c 1`.
    """
    import torch
    import moe_expert_cache_gb300 as ft

    ft.load()
    q = args.ncu_case
    sh = synth.Shape(L=1, E=128, k=8, H=2048, F=768)
    pool = torch.empty(sh.E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
    synth.fill_host_pool(pool.numpy(), sh, 0)
    s = torch.cuda.Stream()
    x = torch.from_numpy(synth.tokens_bf16(0, 0, 0, 1, sh.H).view(np.int16)).cuda().view(torch.bfloat16)
    pc = torch.zeros(1, sh.H, device="cuda")
    y = torch.empty(1, sh.H, device="cuda")
    w = torch.full((1, sh.k), 1.0 / sh.k, device="cuda")
    ctx = ft.Context(1, sh.E, sh.k, sh.H, sh.F, 128, pool, T_max=1, compute_stream=s.cuda_stream)
    with torch.cuda.stream(s):
        for i in range(6):
            ids = list(range(sh.k - q)) + [sh.k + q * i + j for j in range(q)]
            ctx.route_ctl(0, 1, topk_ids=torch.tensor([ids], dtype=torch.int32, device="cuda"), topk_w=w,
                          B_P=1.0, B_H=1.0)
            ctx.moe_forward(x, pc, y)
    torch.cuda.synchronize()
    st = ctx.status()
    ctx.close()
    if st != ft.FT_OK:
        raise SystemExit(f"device status {st}")


def run_ncu_quant(args):
    """A small quantised case for profiler captures (not a bench line).

    One layer of the Large shape (E=256, top-8, H=4096, F=2048) with NVFP4
    (fmt 1), MXFP4 (fmt 2) or block-FP8 (fmt 3) records in 16 slots; T=1
    calls alternate between experts 0..7 and 8..15, so after the first two
    (the fills) every launch reads 8 resident records and the working set
    (two sets of 8 records) exceeds L2.  Twelve calls; capture e.g. the
    seventh expert launch with `ncu -k regex:expert_ffn_fp4 -s 6 -c 1`.
    """
    import torch
    import moe_expert_cache_gb300 as ft

    ft.load()
    fmt = args.ncu_quant
    H, F, E, k = 4096, 2048, 256, 8
    sh = synth.Shape(L=1, E=E, k=k, H=H, F=F, fmt=fmt)
    pool, glob = repeated_pool(sh, 0, distinct=2)
    ctx = ft.Context(1, E, k, H, F, 16, pool, fmt=fmt, T_max=1, nvfp4_global=glob)
    x = torch.from_numpy(synth.tokens_bf16(0, 0, 0, 1, H).view(np.int16)).cuda().view(torch.bfloat16)
    pc = torch.zeros(1, H, device="cuda")
    y = torch.empty(1, H, device="cuda")
    w = torch.full((1, k), 1.0 / k, device="cuda")
    for i in range(12):
        ids = torch.arange(8 * (i & 1), 8 * (i & 1) + 8, dtype=torch.int32, device="cuda").view(1, k)
        ctx.route_ctl(0, 1, topk_ids=ids, topk_w=w, B_P=1.0, B_H=1.0)
        ctx.moe_forward(x, pc, y)
    torch.cuda.synchronize()
    st = ctx.status()
    ctx.close()
    if st != ft.FT_OK:
        raise SystemExit(f"device status {st}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--windows", type=int, default=0,
                    help="timed windows of K steps (0: enough to cover the workload's 256 steps, 3..50)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill measurement")
    ap.add_argument("--no-t16", action="store_true", help="skip the decode T=16 (resize) measurement")
    ap.add_argument("--no-hbm", action="store_true", help="skip the BF16 hits-only (HBM) measurement")
    ap.add_argument("--no-fp4", action="store_true",
                    help="skip the quantised (NVFP4, MXFP4, block-FP8) hits-only decode measurement")
    ap.add_argument("--no-large", action="store_true", help="skip the Large NVFP4 workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--leg", default=None, choices=["prefill", "quant", "hbm", "large"],
                    help="run one leg alone and print its detail object (no bench line)")
    ap.add_argument("--ncu-quant", type=int, default=None, metavar="FMT",
                    help="run the small quantised profiling case (1 NVFP4, 2 MXFP4, 3 block-FP8) and exit")
    ap.add_argument("--ncu-case", type=int, default=None, metavar="Q",
                    help="run the small single-layer BF16 profiling case with Q fills per call (0..8) and exit")
    args = ap.parse_args()
    if args.ncu_quant is not None:
        if args.ncu_quant not in (1, 2, 3):
            raise SystemExit("--ncu-quant takes 1 (NVFP4), 2 (MXFP4) or 3 (block-FP8)")
        run_ncu_quant(args)
        return
    if args.ncu_case is not None:
        if not 0 <= args.ncu_case <= 8:
            raise SystemExit("--ncu-case takes 0..8")
        run_ncu_case(args)
        return
    if args.leg:
        import torch
        torch.cuda.set_device(0)
        import moe_expert_cache_gb300 as ft
        ft.load()
        dev, peaks = torch.device("cuda", 0), read_peaks()
        if args.leg == "prefill":
            r = run_prefill_bench(dev, peaks)
        elif args.leg == "quant":
            r = run_quant_decode_bench(dev, peaks)
        elif args.leg == "large":
            r = run_large_nvfp4_bench(dev, peaks, measure_h2d_peak(dev))
        else:
            sh = WORKLOAD.shape
            pool = torch.empty(sh.E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
            synth.fill_host_pool(pool.numpy(), synth.Shape(L=1, E=sh.E, k=sh.k, H=sh.H, F=sh.F), WORKLOAD.seed)
            r = run_bf16_hbm_bench(pool, dev, peaks)
        print(json.dumps({args.leg: r[1]}), flush=True)
        return
    rank, world, local_rank = dist_env()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out, separators=(",", ":")), flush=True)


if __name__ == "__main__":
    main()
