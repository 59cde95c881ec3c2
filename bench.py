#!/usr/bin/env python
"""Benchmark of the expert-cache MoE decode step on one GB300 (or N replicas).

Workload (default): decode at T=1 through 48 MoE layers of E=128 experts,
top-8, hidden 2048, expert ffn 768, BF16 records in a 58 GB page-locked host
pool, 1536 cache slots shared by all layers, AR(1) router logits
(rho 0.8, sigma 0.6), B_P = 52.7, B_H = 120.  One step = one decode token
through all 48 layers: for every layer the control pass (routing, dedup,
hit/miss, q, fill set, LRU victims, map update), the fills, the expert
gate/up + SwiGLU and down + gated merge with the CPU-set partial sum.

Timed region: K steps after W eager warm-up steps, captured from the library
calls into one CUDA graph (instantiated and uploaded beforehand), bracketed by
a barrier and a device synchronisation, CUDA events on the library's compute
stream, max over ranks.  Every step streams about 3.6 GB of expert weights, far more than the
129 MB L2, so no explicit L2 flush is used.  Per-kernel device times come
from the library's own event records in the same timed region.

The JSON line also carries a "prefill" object: the Prefill workload (4
layers, T=8192, full-layer double buffer) timed per chunk, with overlap and
tensor-core utilisation of the grouped GEMMs.

--impl reference times the CPU oracle (exact-integer control + float64
expert numerics) on this machine's host cores on bounded samples of the same
workload; it never touches the GPU.
"""
from __future__ import annotations

import argparse
import json
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
PROFILE_EVERY = 16
UNIT = "tokens/s"


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


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples go to FT_CLOCKS_DIR (default: the system temporary
        # directory); the JSON line carries their summary
        import tempfile
        self.path = os.path.join(os.environ.get("FT_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"ft_clocks_rank{gpu_index}.csv")
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx.append(float(c[2]))
            except ValueError:
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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


# ------------------------------------------------------------ our arm

def kernel_bytes(shape: synth.Shape, T: int, dcnt: dict) -> dict:
    """Algorithmic bytes moved by each decode kernel over the timed region.

    expert_ffn (with the fused fill):
        link: every fill copies one record over the host link;
        hbm:  the fills written to HBM + the whole record of every resident
              GPU expert read (3*F*H*2 B; a fill is computed from the bytes in
              flight) + x read + h written and read once (fp32) + partial_C
              read + y written.
    route_ctl: logits + ids/gates written (small; reported for completeness).
    """
    H, F, E, L, k = shape.H, shape.F, shape.E, shape.L, shape.k
    calls = dcnt["calls"]
    rb = shape.record_bytes
    link = dcnt["fills"] * rb
    hbm = link + dcnt["hits"] * rb + calls * T * H * 2 + 2 * dcnt["assign"] * F * 4 + calls * T * H * 4 * 2
    return {"expert_ffn": {"link": link, "hbm": hbm}, "route_ctl": {"hbm": calls * (T * E * 4 + 2 * T * k * 4)}}


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
    n_steps = W + K

    t0 = time.time()
    pool, shared = host_pool(sh, wl.seed, world, rank)
    t_pool = time.time() - t0

    logits = synth.ar1_logits(wl.seed, n_steps, L, T, E, wl.rho, wl.sigma)          # [steps, L, T, E]
    xs = np.stack([np.stack([synth.tokens_bf16(wl.seed, s, l, T, H) for l in range(L)]) for s in range(n_steps)])
    pc = np.stack([synth.random_f32(wl.seed, (l,), (T, H), 0.1) for l in range(L)])   # [L, T, H]
    logits_d = torch.from_numpy(logits).to(device)
    xs_d = torch.from_numpy(xs.view(np.int16)).to(device).view(torch.bfloat16)
    pc_d = torch.from_numpy(pc).to(device)
    y_d = torch.empty(L, T, H, dtype=torch.float32, device=device)

    s = torch.cuda.Stream(device)
    ts = torch.cuda.Stream(device)

    def make_ctx():
        return ft.Context(L, E, sh.k, H, sh.F, wl.S, pool, T_max=T, compute_stream=s.cuda_stream,
                          transfer_stream=ts.cuda_stream)

    def step(ctx, si, lg, x, p, y):
        for l in range(L):
            ctx.route_ctl(l, T, logits=lg[si, l], B_P=wl.B_P, B_H=wl.B_H)
            ctx.moe_forward(x[si, l], p[l], y[l])

    # ---- device-resident run: W eager warm-up steps, then the K timed steps
    # captured (with the library's per-kernel event nodes) into one CUDA graph
    # that is instantiated and uploaded before the timed region.
    ctx = make_ctx()
    with torch.cuda.stream(s):
        for i in range(W):
            step(ctx, i, logits_d, xs_d, pc_d, y_d)
    torch.cuda.synchronize(device)
    c0 = ctx.counters()
    ctx.profile_enable(True)
    t0 = time.time()
    g = RawGraph(s.cuda_stream)
    def timed_steps():
        for i in range(W, W + K):
            # per-kernel event records on one timed step in PROFILE_EVERY
            # (an event node costs a few microseconds of GPU time)
            ctx.profile_pause((i - W) % PROFILE_EVERY != 0)
            step(ctx, i, logits_d, xs_d, pc_d, y_d)
        ctx.profile_pause(False)

    with torch.cuda.stream(s):
        g.capture(timed_steps)
    t_capture = time.time() - t0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    clocks = ClockSampler(local_rank)
    with torch.cuda.stream(s):
        ev0.record(s)
        g.launch()
        ev1.record(s)
    torch.cuda.synchronize(device)
    barrier(world, device)
    clk = clocks.stop()
    t_ms = ev0.elapsed_time(ev1)
    prof = ctx.profile_read()
    ctx.profile_enable(False)
    g.close()
    c1 = ctx.counters()
    assert ctx.status() == ft.FT_OK
    dcnt = {k_: c1[k_] - c0[k_] for k_ in c1}
    # B_P as the library measures it (its own fill path, 16 records, best of 3)
    link_fill_gbps = ctx.measure_link(16, 3)
    ctx.close()
    t_max_ms = max_over_ranks(t_ms, world, device)

    # ---- end to end: inputs copied from pinned host memory and y read back every step
    lg_h = torch.from_numpy(logits).pin_memory()
    xs_h = torch.from_numpy(xs.view(np.int16)).pin_memory()
    pc_h = torch.from_numpy(pc).pin_memory()
    y_h = torch.empty(L, T, H, dtype=torch.float32).pin_memory()
    lg_step = torch.empty(1, L, T, E, dtype=torch.float32, device=device)
    x_step = torch.empty(1, L, T, H, dtype=torch.int16, device=device)
    pc_step = torch.empty(L, T, H, dtype=torch.float32, device=device)
    ctx2 = make_ctx()
    with torch.cuda.stream(s):
        for i in range(W):
            step(ctx2, i, logits_d, xs_d, pc_d, y_d)
    torch.cuda.synchronize(device)
    def e2e_steps():
        for i in range(W, W + K):
            lg_step.copy_(lg_h[i:i + 1], non_blocking=True)
            x_step.copy_(xs_h[i:i + 1], non_blocking=True)
            pc_step.copy_(pc_h, non_blocking=True)
            step(ctx2, 0, lg_step, x_step.view(torch.bfloat16), pc_step, y_d)
            y_h.copy_(y_d, non_blocking=True)

    g2 = RawGraph(s.cuda_stream)
    with torch.cuda.stream(s):
        g2.capture(e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(s):
        e0.record(s)
        g2.launch()
        e1.record(s)
    torch.cuda.synchronize(device)
    g2.close()
    barrier(world, device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    assert ctx2.status() == ft.FT_OK
    ctx2.close()
    h2d_bytes = (L * T * E * 4) + (L * T * H * 2) + (L * T * H * 4)
    d2h_bytes = L * T * H * 4

    # ---- roofline of the dominant kernel and per-kernel table
    peaks = read_peaks()
    kb = kernel_bytes(sh, T, dcnt)
    total_ms = sum(v["ms"] for v in prof.values())
    h2d_peak = measure_h2d_peak(device) if rank == 0 else None
    kernels = {}
    launches_total = dcnt["calls"]  # each decode kernel runs once per control pass
    for name, v in prof.items():
        us = 1e3 * v["ms"] / v["launches"]
        ent = {"launches_timed": v["launches"], "ms_total": round(v["ms"], 3), "us_per_launch": round(us, 3),
               "share": round(v["ms"] / total_ms, 4)}
        if name in kb:
            for kind, byts in kb[name].items():
                bpl = byts / max(1, launches_total)
                gbs = bpl / (us * 1e-6) / 1e9
                peak = h2d_peak if kind == "link" else peaks["hbm_gbs"]
                ent[kind] = {"bytes_per_launch": int(bpl), "achieved_GBps": round(gbs, 1),
                             "peak_GBps": round(peak, 1) if peak else None,
                             "frac": round(gbs / peak, 4) if peak else None}
        kernels[name] = ent
    dom = max(prof, key=lambda n: prof[n]["ms"])
    roofline = roofline_entry(dom, kernels, peaks, h2d_peak,
                              dcnt["hits"] / max(1, dcnt["calls"]) if dom == "expert_ffn" else None)
    ex = kernels.get("expert_ffn", {})
    expert_roofline = {"kernel": "expert_ffn", "bound": "hbm",
                       "achieved": ex.get("hbm", {}).get("achieved_GBps"), "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": ex.get("hbm", {}).get("frac"), "peak_source": peaks["source"],
                       "note": "HBM side of the fused kernel; its time also covers the fill over the host link"}

    value = whole_job_rate(T * K, t_ms * 1e-3, world, device)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(t_max_ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; AR(1) router logits, N(0,0.02) bf16 weights)",
        "config": {"workload": "decode T=1: 48 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, "
                               "1536 slots, AR(1) rho=0.8, B_P=52.7, B_H=120",
                   "L": L, "E": E, "k": sh.k, "H": H, "F": sh.F, "S": wl.S, "T": T,
                   "l2": "no flush: each step streams ~3.6 GB of expert weights (> 129 MB L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "token_layers_per_s": round(value * L, 1),
        "hit_rate": round(dcnt["hits"] / max(1, dcnt["unique"]), 4),
        "fills_per_layer_step": round(dcnt["fills"] / max(1, dcnt["calls"]), 4),
        "cpu_set_per_layer_step": round(dcnt["cpu"] / max(1, dcnt["calls"]), 4),
        "roofline": roofline,
        "roofline_expert_kernels": expert_roofline,
        "link_GBps": {"pinned_memcpy": round(h2d_peak, 1) if h2d_peak else None,
                      "fill_path_B_P": round(link_fill_gbps, 1)},
        "kernels": kernels,
        "gpu_launches": int(2 * dcnt["calls"]),
        "kernel_timing": f"library CUDA-event records around each launch of 1 timed step in {PROFILE_EVERY}",
        "clocks": clk,
        "e2e": {"value": round(world * T * K / (e2e_ms * 1e-3), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes},
        "setup_s": {"host_pool": round(t_pool, 1), "graph_capture": round(t_capture, 1)},
        "execution": "the K timed steps run as one CUDA graph (captured from the library calls, uploaded before timing)",
    }
    if rank == 0 and not args.no_t16:
        out["decode_t16"] = run_decode_t16_bench(pool, device)
    if not args.no_prefill:
        out["prefill"] = run_prefill_bench(device, peaks)
    if rank == 0 and not args.no_fp4:
        out["quant_decode"] = run_quant_decode_bench(device, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(pool.numpy() if world == 1 else shared[0], args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if shared is not None:
        torch.cuda.cudart().cudaHostUnregister(pool.data_ptr())
    return out


def run_decode_t16_bench(pool, device) -> dict:
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
    ms, resize_ms = 0.0, {}
    c0 = ctx.counters()
    for s0, s1 in ((0, 32), (32, 64), (64, wl.steps)):
        if s0 in resize_at:
            t0 = time.perf_counter()
            ctx.cache_resize(resize_at[s0])
            resize_ms[f"to_{resize_at[s0]}_before_step_{s0}"] = round((time.perf_counter() - t0) * 1e3, 2)
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
    return {"workload": "decode T=16: 48 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, 768 slots "
                        "(384 during steps 32-63), AR(1) rho=0.7, B_P=25, B_H=90, 128 steps from an empty cache",
            "tokens_per_s": round(T * wl.steps / (ms * 1e-3), 1), "ms_per_step": round(ms / wl.steps, 3),
            "resize_ms": resize_ms, "execution": "eager library calls, CUDA-event time of the steps",
            "hit_rate": round(d["hits"] / max(1, d["unique"]), 4),
            "fills_per_layer_step": round(d["fills"] / calls, 3),
            "gpu_experts_per_layer_step": round((d["hits"] + d["fills"]) / calls, 2),
            "link_floor_ms_per_step": round(d["fills"] / wl.steps * sh.record_bytes / 211e9 * 1e3, 3)}


def _fp4_pool(sh: synth.Shape, seed: int, distinct: int = 16):
    """Pinned pool of one layer whose E records are the encodings of
    `distinct` drawn experts, repeated (the FP4 kernel's time does not depend
    on the values).  Returns (pool, per-record globals or None)."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    rb = sh.record_bytes
    enc = {synth.FMT_NVFP4: synth.record_nvfp4, synth.FMT_MXFP4: synth.record_mxfp4,
           synth.FMT_FP8: synth.record_fp8}[sh.fmt]
    with ThreadPoolExecutor(min(distinct, os.cpu_count() or 1)) as ex:
        got = list(ex.map(lambda e: enc(seed, 0, e, sh.H, sh.F), range(distinct)))
    recs = [g[0] for g in got] if sh.fmt == synth.FMT_NVFP4 else got
    pool = torch.empty(sh.E * rb, dtype=torch.uint8, pin_memory=True)
    pn = pool.numpy()
    for e in range(sh.E):
        pn[e * rb:(e + 1) * rb] = recs[e % distinct]
    glob = (np.array([got[e % distinct][1] for e in range(sh.E)], dtype=np.float32)
            if sh.fmt == synth.FMT_NVFP4 else None)
    return pool, glob


def run_quant_decode_bench(device, peaks, calls_t1: int = 96, calls_t64: int = 24) -> dict:
    """Quantised expert kernels (NVFP4, MXFP4 and block-FP8 records) on the
    Large shapes, hits only: one MoE layer of E=256 experts, top-8, H=4096,
    F=2048, every record resident in 512 slots (a warm-up with B_P = B_H
    fills every miss), AR(1) rho=0.8 logits, T=1 and T=64.  The bound is
    HBM: each launch reads the records of its routed experts.  Per-launch
    device time from the library's CUDA-event records around each launch of
    the expert kernel (both FP8 kernels under one record)."""
    import torch
    import moe_expert_cache_gb300 as ft
    out = {"workload": "Large shapes, hits only: 1 MoE layer, E=256, top-8, hidden 4096, ffn 2048, 512 slots "
                       "holding every record, AR(1) rho=0.8 logits; records of 16 drawn experts repeated",
           "execution": "eager library calls; expert-kernel time from the library's per-launch CUDA events"}
    H, F, E, k = 4096, 2048, 256, 8
    cs = torch.cuda.Stream(device)
    for name, fmt in (("nvfp4", synth.FMT_NVFP4), ("mxfp4", synth.FMT_MXFP4), ("fp8", synth.FMT_FP8)):
        sh = synth.Shape(L=1, E=E, k=k, H=H, F=F, fmt=fmt)
        pool, glob = _fp4_pool(sh, 0)
        ctx = ft.Context(1, E, k, H, F, 512, pool, fmt=fmt, T_max=64, nvfp4_global=glob,
                         compute_stream=cs.cuda_stream)
        res = {"record_bytes": sh.record_bytes}
        with torch.cuda.stream(cs):
            pc = torch.zeros(64, H, device=device)
            y = torch.empty(64, H, device=device)
            warm = torch.from_numpy(synth.iid_logits(1, (77,), 64, E)).to(device)
            for i in range(8):  # fill every expert (q = m when B_P = B_H)
                ctx.route_ctl(0, 64, logits=torch.roll(warm, i * 32, dims=1), B_P=1.0, B_H=1.0)
                ctx.moe_forward(torch.zeros(64, H, dtype=torch.bfloat16, device=device), pc, y)
        torch.cuda.synchronize(device)
        for T, calls in ((1, calls_t1), (64, calls_t64)):
            lg = torch.from_numpy(synth.ar1_logits(0, calls, 1, T, E, 0.8)[:, 0]).to(device)
            x = torch.from_numpy(synth.tokens_bf16(0, 0, 0, T, H).view(np.int16)).to(device).view(torch.bfloat16)
            with torch.cuda.stream(cs):
                for i in range(4):
                    ctx.route_ctl(0, T, logits=lg[i], B_P=52.7, B_H=150.0)
                    ctx.moe_forward(x, pc[:T], y[:T])
            torch.cuda.synchronize(device)
            c0 = ctx.counters()
            ctx.profile_enable(True)
            with torch.cuda.stream(cs):
                for i in range(calls):
                    ctx.route_ctl(0, T, logits=lg[i], B_P=52.7, B_H=150.0)
                    ctx.moe_forward(x, pc[:T], y[:T])
            torch.cuda.synchronize(device)
            prof = ctx.profile_read()
            ctx.profile_enable(False)
            c1 = ctx.counters()
            d = {k_: c1[k_] - c0[k_] for k_ in c1}
            ms = prof["expert_ffn"]["ms"]
            n = prof["expert_ffn"]["launches"]
            hbm = kernel_bytes(sh, T, d)["expert_ffn"]["hbm"]
            gbs = hbm / (ms * 1e-3) / 1e9
            res[f"t{T}"] = {"us_per_launch": round(ms * 1e3 / n, 2), "launches": n,
                            "hits_per_launch": round(d["hits"] / max(1, d["calls"]), 2),
                            "fills": d["fills"], "hbm_bytes_per_launch": int(hbm / n),
                            "achieved_GBps": round(gbs, 1), "peak_GBps": peaks["hbm_gbs"],
                            "frac": round(gbs / peaks["hbm_gbs"], 4),
                            "traffic": traffic_from_profiles("expert_ffn_fp4", d["hits"] / max(1, d["calls"]))
                            if fmt == synth.FMT_NVFP4 else None}
        assert ctx.status() == ft.FT_OK
        ctx.close()
        del pool
        out[name] = res
    return out


def run_prefill_bench(device, peaks, reps: int = 3) -> dict:
    """Prefill workload: 4 layers, E=128, top-8, H=2048, F=768, T=8192, 256
    slots, full-layer double buffer.  Times whole chunks (prefill_begin + 4
    prefill_layer calls) with CUDA events on the compute stream; per-kernel
    device times from the library's event records; the same chunk with the
    copies on the compute stream (one buffer in flight, no overlap) as the
    single-buffer A/B."""
    import torch
    import moe_expert_cache_gb300 as ft
    wl = synth.PREFILL
    sh = wl.shape
    T, L = wl.T, sh.L
    pool = torch.empty(L * sh.E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
    synth.fill_host_pool(pool.numpy(), sh, wl.seed)
    xs = [torch.from_numpy(synth.tokens_bf16(wl.seed, 900, l, T, sh.H).view(np.int16)).to(device).view(torch.bfloat16)
          for l in range(L)]
    lg = [torch.from_numpy(synth.iid_logits(wl.seed, (900, l), T, sh.E)).to(device) for l in range(L)]
    ys = [torch.empty(T, sh.H, dtype=torch.float32, device=device) for _ in range(L)]
    cs, ts = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def measure(two_streams: bool):
        ctx = ft.Context(L, sh.E, sh.k, sh.H, sh.F, wl.S, pool, T_max=4, T_prefill_max=T,
                         compute_stream=cs.cuda_stream, transfer_stream=ts.cuda_stream if two_streams else 0)

        def chunk():
            ctx.prefill_begin(0)
            for l in range(L):
                ctx.prefill_layer(l & 1, l, l + 1 if l + 1 < L else -1, T, xs[l], lg[l], ys[l])

        with torch.cuda.stream(cs):
            chunk()
        torch.cuda.synchronize(device)
        ctx.profile_enable(True)
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(cs):
                e0.record(cs)
                chunk()
                e1.record(cs)
            torch.cuda.synchronize(device)
            times.append(e0.elapsed_time(e1))
        prof = ctx.profile_read()
        assert ctx.status() == ft.FT_OK
        ctx.close()
        return statistics.median(times), prof

    t_db, prof = measure(True)
    t_sb, _ = measure(False)
    n = reps
    h2d = prof["pf_h2d"]["ms"] / n
    comp = sum(v["ms"] for k_, v in prof.items() if k_ != "pf_h2d") / n
    g1 = prof["pf_gemm1_swiglu"]["ms"] / (n * L)
    g2 = prof["pf_gemm2"]["ms"] / (n * L)
    fl1 = 2.0 * T * sh.k * 2 * sh.F * sh.H
    fl2 = 2.0 * T * sh.k * sh.F * sh.H
    tf = (fl1 + fl2) / ((g1 + g2) * 1e-3) / 1e12
    tot = sum(v["ms"] for v in prof.values())
    return {
        "workload": "prefill: 4 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, T=8192, 256 slots, "
                    "full-layer double buffer",
        "expert_tokens_per_s": round(T * L / (t_db * 1e-3), 1),
        "routed_assignments_per_s": round(T * sh.k * L / (t_db * 1e-3), 1),
        "ms_per_chunk": round(t_db, 3),
        "h2d_GBps": round(L * sh.E * sh.record_bytes / (h2d * 1e-3) / 1e9, 1),
        "ms_h2d": round(h2d, 3), "ms_compute": round(comp, 3),
        "overlap_eta": round(max(h2d, comp) / t_db, 4),
        "hidden_fraction": round((h2d + comp - t_db) / min(h2d, comp), 4),
        "single_buffer_ms_per_chunk": round(t_sb, 3),
        "double_buffer_speedup": round(t_sb / t_db, 4),
        "roofline_gemm": {"kernels": ["pf_gemm1_swiglu", "pf_gemm2"], "bound": "tensor",
                          "achieved": round(tf, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                          "frac": round(tf / peaks["bf16_tflops"], 4),
                          "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                          "gemm1_TFLOPs": round(fl1 / (g1 * 1e-3) / 1e12, 1),
                          "gemm2_TFLOPs": round(fl2 / (g2 * 1e-3) / 1e12, 1),
                          "flops_per_layer": fl1 + fl2, "peak_source": peaks["source"],
                          "traffic": traffic_from_profiles("pf_gemm1_swiglu")},
        "kernels": {k_: {"launches": v["launches"], "ms_total": round(v["ms"], 3),
                         "share": round(v["ms"] / tot, 4)} for k_, v in prof.items()},
    }


def roofline_entry(dom, kernels, peaks, h2d_peak, records_per_launch=None):
    """Roofline of the dominant kernel: the side (host link or HBM) whose
    bytes at peak take longer is the bound."""
    ent = kernels[dom]
    link, hbm = ent.get("link"), ent.get("hbm", {})
    t_link = link["bytes_per_launch"] / (h2d_peak * 1e9) if link and h2d_peak else 0.0
    t_hbm = hbm.get("bytes_per_launch", 0) / (peaks["hbm_gbs"] * 1e9)
    if t_link >= t_hbm and link:
        side, bound, src = link, "h2d", "measured live: pinned host->device cudaMemcpyAsync, 1 GiB, best of 4"
    else:
        side, bound, src = hbm, "hbm", peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"
    return {"kernel": dom, "bound": bound, "achieved": side.get("achieved_GBps"), "peak": side.get("peak_GBps"),
            "unit": "GB/s", "frac": side.get("frac"), "peak_source": src,
            "bytes_per_launch": side.get("bytes_per_launch"), "us_per_launch": ent["us_per_launch"],
            "traffic": traffic_from_profiles(dom, records_per_launch)}


def traffic_from_profiles(kernel: str, records_per_launch: float | None = None):
    """DRAM bytes per launch from a committed ncu capture, if one matches the
    current kernel source (profiles/traffic.json keyed by kernel and source
    hash); else None.  A capture that lists the records its launch read is
    scaled to `records_per_launch` (the traffic of these kernels grows with
    the records they read)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
        if not d:
            return None
        import hashlib
        src = os.path.join(ROOT, d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != d["source_sha"]:
            return None
        if "records_read" in d:
            if records_per_launch is None:
                return None
            return int(d["dram_bytes"] / d["records_read"] * records_per_launch)
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
            "sample": f"{done} layer-steps of the workload (control + fp64 FFN of all 8 routed experts, "
                      f"weights read from the host pool) in {dt:.1f} s; tokens/s = layer-steps/{L}/s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm, on this machine's host cores."""
    if rank != 0:
        return None
    import torch
    sh = WORKLOAD.shape
    pool = np.empty(sh.L * sh.E * sh.record_bytes, dtype=np.uint8)
    synth.fill_host_pool(pool, sh, WORKLOAD.seed)
    W, K = args.warmup, args.steps
    # a step of this arm is one sampled layer-step, bounded in total time
    oracle_samples(pool, min(W, 2))
    done, dt = oracle_samples(pool, K, args.cpu_seconds * 4)
    L = sh.L
    v = WORKLOAD.T * done / L / dt
    cores = _blas_threads()
    del torch
    return {"metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": world, "steps": done, "warmup": min(W, 2),
            "ms_per_step": round(1e3 * dt / max(1, done), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": "decode T=1: 48 MoE layers, E=128, top-8, hidden 2048, ffn 768, BF16, "
                                   "1536 slots, AR(1) rho=0.8, B_P=52.7, B_H=120"},
            "cpu_baseline": {"value": round(v, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{done} layer-steps (one step = one MoE layer of one decode token)"},
            "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ncu_case(args):
    """A small single-layer case for profiler captures (not a bench line).

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
    return None


def run_ncu_fp4(args):
    """A small FP4 case for profiler captures (not a bench line).

    One layer of the Large shape (E=256, top-8, H=4096, F=2048) with NVFP4
    (fmt 1) or MXFP4 (fmt 2) records in 16 slots; T=1 calls alternate
    between experts 0..7 and 8..15, so after the first two (the fills) every
    launch reads 8 resident records and the 226 MB working set exceeds L2.
    Twelve calls; capture e.g. the seventh expert launch with
    `ncu -k regex:expert_ffn_fp4 -s 6 -c 1`.
    """
    import torch
    import moe_expert_cache_gb300 as ft

    ft.load()
    fmt = args.ncu_fp4
    H, F, E, k = 4096, 2048, 256, 8
    sh = synth.Shape(L=1, E=E, k=k, H=H, F=F, fmt=fmt)
    pool, glob = _fp4_pool(sh, 0, distinct=2)
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
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill measurement")
    ap.add_argument("--no-t16", action="store_true", help="skip the decode T=16 (resize) measurement")
    ap.add_argument("--no-fp4", action="store_true",
                    help="skip the quantised (NVFP4, MXFP4, block-FP8) decode measurement")
    ap.add_argument("--fp4-only", action="store_true",
                    help="only the quantised decode measurement (one JSON object)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill measurement and print its object (no bench line)")
    ap.add_argument("--ncu-fp4", type=int, default=None, metavar="FMT",
                    help="run the small FP4 profiling case (1 = NVFP4, 2 = MXFP4) and exit")
    ap.add_argument("--ncu-case", type=int, default=None, metavar="Q",
                    help="run the small single-layer profiling case with Q fills per call (0..8) and exit")
    args = ap.parse_args()
    if args.ncu_fp4 is not None:
        if args.ncu_fp4 not in (1, 2):
            raise SystemExit("--ncu-fp4 takes 1 (NVFP4) or 2 (MXFP4)")
        run_ncu_fp4(args)
        return
    if args.ncu_case is not None:
        if not 0 <= args.ncu_case <= 8:
            raise SystemExit("--ncu-case takes 0..8")
        run_ncu_case(args)
        return
    if args.prefill_only:
        import torch
        torch.cuda.set_device(0)
        import moe_expert_cache_gb300 as ft
        ft.load()
        print(json.dumps({"prefill": run_prefill_bench(torch.device("cuda", 0), read_peaks())}), flush=True)
        return
    if args.fp4_only:
        import torch
        torch.cuda.set_device(0)
        import moe_expert_cache_gb300 as ft
        ft.load()
        print(json.dumps({"quant_decode": run_quant_decode_bench(torch.device("cuda", 0), read_peaks())}), flush=True)
        return
    rank, world, local_rank = dist_env()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
