"""GPU parity of the quantised decode and prefill paths for the FP4 record
formats, NVFP4 (e4m3 block-16 scales, fp32 global) and MXFP4 (E8M0 block-32
scales), and for block-FP8 (E4M3 values, fp32 scale per 128 x 128 block):
control bit-exact, outputs within rel-L2 5e-3 of the fp64 oracle on
identically dequantised weights."""
import os

import numpy as np
import pytest

import synth
from oracle import control as ctl
from oracle import numerics as nm
from oracle import fp8 as f8
from oracle import mxfp4 as mx
from oracle import nvfp4 as fp4
from tests import harness as hz

pytestmark = pytest.mark.gpu
NVFP4_REL_L2 = 5e-3


@pytest.fixture(scope="module")
def ft():
    import torch
    assert torch.cuda.is_available()
    import moe_expert_cache_gb300 as ft
    ft.load()
    return ft


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class FP4Weights:
    """float64 weights of the records of one layer, read back from the pool
    bytes.  With a pool that repeats `distinct` records, dequantised records
    are cached by record so each is decoded once."""

    def __init__(self, pool_np, glob, sh, layer, distinct=None, cache=None):
        self.pool, self.glob, self.sh, self.layer = pool_np, glob, sh, layer
        self.distinct = distinct
        self.cache = {} if cache is None else cache

    def __call__(self, e):
        sh, rb = self.sh, self.sh.record_bytes
        fid = self.layer * sh.E + e
        key = fid % self.distinct if self.distinct else fid
        if key not in self.cache:
            rec = self.pool[fid * rb:(fid + 1) * rb]
            if sh.fmt == synth.FMT_MXFP4:
                self.cache[key] = mx.record_weights(rec, sh.H, sh.F)
            elif sh.fmt == synth.FMT_FP8:
                self.cache[key] = f8.record_weights(rec, sh.H, sh.F)
            else:
                self.cache[key] = fp4.record_weights(rec, sh.H, sh.F, float(self.glob[fid]))
        return self.cache[key]


def _repeated_pool(sh, seed, distinct):
    """Pinned pool whose record l*E+e is the encoding of drawn expert
    (l*E+e) mod `distinct` of layer 0 (valid records, generated in a fraction
    of the time).  A prime `distinct` keeps neighbouring experts and the same
    expert of neighbouring layers on different records, so that reading the
    wrong record still changes the output."""
    import torch
    rb = sh.record_bytes
    pool = torch.empty(sh.L * sh.E * rb, dtype=torch.uint8, pin_memory=True)
    pn = pool.numpy()
    enc = {synth.FMT_NVFP4: synth.record_nvfp4, synth.FMT_MXFP4: synth.record_mxfp4,
           synth.FMT_FP8: synth.record_fp8}[sh.fmt]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(min(distinct, os.cpu_count() or 1)) as ex:
        got = list(ex.map(lambda e: enc(seed, 0, e, sh.H, sh.F), range(distinct)))
    recs = [g[0] for g in got] if sh.fmt == synth.FMT_NVFP4 else got
    for fid in range(sh.L * sh.E):
        pn[fid * rb:(fid + 1) * rb] = recs[fid % distinct]
    glob = None
    if sh.fmt == synth.FMT_NVFP4:
        glob = np.array([got[fid % distinct][1] for fid in range(sh.L * sh.E)], dtype=np.float32)
    return pool, glob


def _check_tokens(got, ref, where):
    """rel-L2 over the checked tokens, and over each token on its own, so
    that one wrong token row cannot hide in the norm."""
    rel = nm.rel_l2(got, ref)
    assert rel <= NVFP4_REL_L2, (where, rel)
    per_tok = [nm.rel_l2(got[i], ref[i]) for i in range(len(got))]
    worst = int(np.argmax(per_tok))
    assert per_tok[worst] <= NVFP4_REL_L2, (where, "token row", worst, per_tok[worst])
    return rel


def _replay(ft, sh, S, schedule, B_P, B_H, rho, samples, tok_sample=None, seed=0, distinct=None, repeat=False):
    """schedule: list of (T, steps).  Every call bit-exact; sampled calls
    numerically: on every token when tok_sample is None, else on every token
    of the sampled calls of each phase's first step and on the tok_sample
    tokens of the later ones.  repeat: each sampled forward is run a second
    time on the same inputs (its fills are then already in their slots, and
    the launch's counters must have returned to rest); the two outputs must
    be identical bit for bit."""
    import torch
    pool, glob = _repeated_pool(sh, seed, distinct) if distinct else hz.pinned_pool(sh, seed)
    pool_np = pool.numpy()
    T_max = max(t for t, _ in schedule)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, S, pool, fmt=sh.fmt, T_max=T_max, nvfp4_global=glob)
    st = ctl.CacheState.empty(sh.L, sh.E, S)
    step = 0
    done = []
    cache = {}
    for T, steps in schedule:
        logits = synth.ar1_logits(seed, steps, sh.L, T, sh.E, rho, None) if rho else None
        first = step
        for s in range(steps):
            for layer in range(sh.L):
                lg = logits[s, layer] if rho else synth.iid_logits(seed, (step, layer), T, sh.E)
                ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in lg])
                r = ctl.route_ctl(st, layer, ids, B_P, B_H)
                ctl.check_invariants(st, r)
                ctx.route_ctl(layer, T, logits=_dev(lg), B_P=B_P, B_H=B_H)
                hz.compare_ctl(ctx, st, r, T, f"T={T} step={s} layer={layer}")
                if (step, layer) in samples:
                    if tok_sample is None or step == first:
                        toks = list(range(T))
                    else:
                        toks = sorted(set(min(t, T - 1) for t in tok_sample))
                    w = FP4Weights(pool_np, glob, sh, layer, distinct, cache if distinct else None)
                    xb = synth.tokens_bf16(seed, step, layer, T, sh.H)
                    x = nm.bf16_to_f64(xb)
                    sub_ids = [ids[t] for t in toks]
                    sub_g = [gates[t] for t in toks]
                    sub_sl = [r.slots_topk[t] for t in toks]
                    y_gpu_ref, pc_sub = nm.moe_layer_split(x[toks], sub_ids, sub_g, sub_sl, w)
                    pc = np.zeros((T, sh.H), dtype=np.float32)
                    pc[toks] = pc_sub
                    xd = _dev(xb.view(np.int16)).view(torch.bfloat16)
                    y = torch.empty(T, sh.H, dtype=torch.float32, device="cuda")
                    ctx.moe_forward(xd, _dev(pc), y)
                    torch.cuda.synchronize()
                    got = y.cpu().numpy()[toks]
                    ref = nm.merged_output(y_gpu_ref, pc_sub)
                    assert np.isfinite(y.cpu().numpy()).all()
                    done.append(_check_tokens(got, ref, (T, step, layer)))
                    if repeat:
                        y2 = torch.empty_like(y)
                        ctx.moe_forward(xd, _dev(pc), y2)
                        torch.cuda.synchronize()
                        assert np.array_equal(y2.cpu().numpy(), y.cpu().numpy()), ("repeat", T, step, layer)
                    for f, v in zip(r.F, r.victims):
                        fid = layer * sh.E + f
                        rb = sh.record_bytes
                        assert np.array_equal(ctx.read_slot(v), pool_np[fid * rb:(fid + 1) * rb])
            step += 1
    assert ctx.status() == ft.FT_OK
    ctx.close()
    return done


@pytest.mark.parametrize("H,F,E,k,S,T", [
    (256, 256, 16, 4, 12, 3),       # x fp32 in shared memory
    (1024, 512, 16, 4, 24, 9),      # x bf16 in shared memory
    (1024, 512, 16, 4, 24, 20),     # x from global memory
    (1024, 2048, 8, 4, 8, 40),      # phase-B items of several token groups
])
def test_nvfp4_small(ft, H, F, E, k, S, T):
    sh = synth.Shape(L=2, E=E, k=k, H=H, F=F, fmt=synth.FMT_NVFP4)
    samples = {(s, l) for s in range(4) for l in range(2)}
    done = _replay(ft, sh, S, [(T, 4)], 25.0, 75.0, None, samples, repeat=True)
    assert len(done) == len(samples)


@pytest.mark.slow
def test_large_nvfp4_decode(ft):
    """Large NVFP4 decode: 8 layers, E=256, top-8, H=4096, F=2048, 512 slots,
    64 steps at T=1 then 64 at T=64, AR(1) rho=0.8, B_P=52.7, B_H=150.  The
    pool repeats 13 drawn records; every token of the sampled calls of the
    first T=64 step is checked, and every checked token also on its own."""
    wl = synth.LARGE_NVFP4
    samples = {(s, l) for s in (0, 1, 63) for l in (0, 7)} | {(s, l) for s in (64, 65, 127) for l in (0, 3, 7)}
    done = _replay(ft, wl.shape, wl.S, [(1, 64), (64, 64)], wl.B_P, wl.B_H, wl.rho, samples,
                   tok_sample=[0, 21, 42, 63], distinct=13)
    assert len(done) == len(samples)


def _tile_rows(lg, k, E, M_TILE=128):
    """Tokens whose rows open and close each expert's M tiles in the prefill
    GEMMs.  The rows of expert e are its tokens in ascending order (a stable
    counting sort), cut into tiles of M_TILE rows: per expert, its first
    token, the first token of its last tile and its last token."""
    rows = {}
    for t in range(lg.shape[0]):
        for e in ctl.topk_route(lg[t], k)[0]:
            rows.setdefault(int(e), []).append(t)
    toks = set()
    for e, ts in rows.items():
        toks.update((ts[0], ts[((len(ts) - 1) // M_TILE) * M_TILE], ts[-1]))
    return sorted(toks)


def _run_prefill_fp4(ft, sh, S, T, check_layers, tok_sample=None, seed=0, distinct=None):
    """One prefill chunk of every layer through the double buffer; the
    checked layers against the oracle on every token (tok_sample None), on
    the given tokens, or ("tiles") on each expert's M-tile edge rows."""
    import torch
    pool, glob = _repeated_pool(sh, seed, distinct) if distinct else hz.pinned_pool(sh, seed)
    pool_np = pool.numpy()
    cs, ts = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, S, pool, fmt=sh.fmt, T_max=1, T_prefill_max=T,
                     nvfp4_global=glob, compute_stream=cs.cuda_stream, transfer_stream=ts.cuda_stream)
    xs = [synth.tokens_bf16(seed, 901, l, T, sh.H) for l in range(sh.L)]
    lgs = [synth.iid_logits(seed, (901, l), T, sh.E) for l in range(sh.L)]
    xd = [_dev(x.view(np.int16)).view(torch.bfloat16) for x in xs]
    ld = [_dev(lg) for lg in lgs]
    ys = [torch.empty(T, sh.H, dtype=torch.float32, device="cuda") for _ in range(sh.L)]
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        ctx.prefill_begin(0)
        for l in range(sh.L):
            ctx.prefill_layer(l & 1, l, l + 1 if l + 1 < sh.L else -1, T, xd[l], ld[l], ys[l])
    torch.cuda.synchronize()
    assert ctx.status() == ft.FT_OK
    rels = []
    cache = {}
    for l in check_layers:
        if tok_sample == "tiles":
            toks = _tile_rows(lgs[l], sh.k, sh.E)
        else:
            toks = list(range(T)) if tok_sample is None else tok_sample
        ids, gates = zip(*[ctl.topk_route(lgs[l][t], sh.k) for t in toks])
        ref = nm.gated_sum(nm.bf16_to_f64(xs[l][toks]), ids, gates, lambda t, j: True,
                           FP4Weights(pool_np, glob, sh, l, distinct, cache if distinct else None))
        y = ys[l].cpu().numpy()
        assert np.isfinite(y).all()
        rels.append(_check_tokens(y[toks], ref, ("layer", l, len(toks))))
    ctx.close()
    return rels


def test_nvfp4_prefill_small(ft):
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=256, fmt=synth.FMT_NVFP4)
    _run_prefill_fp4(ft, sh, 16, 300, [0, 1])


@pytest.mark.slow
def test_large_nvfp4_prefill(ft):
    """Large NVFP4 prefill: T=4096 through all 8 layers of E=256, H=4096,
    F=2048 (a pool of 13 drawn records repeated).  Every layer is checked on
    the tokens that open and close each expert's M tiles (about 600 per
    layer), each token also on its own."""
    wl = synth.LARGE_NVFP4
    _run_prefill_fp4(ft, wl.shape, wl.S, 4096, list(range(wl.shape.L)), tok_sample="tiles", distinct=13)


# ------------------------------------------------------------------ MXFP4

@pytest.mark.parametrize("H,F,E,k,S,T", [
    (256, 512, 16, 4, 12, 3),       # x fp32 in shared memory, 8-byte W_gu scale rows
    (1024, 512, 16, 4, 24, 9),      # x bf16 in shared memory
    (1024, 512, 16, 4, 24, 20),     # x from global memory
    (1024, 2048, 8, 4, 8, 40),      # phase-B items of several token groups
])
def test_mxfp4_small(ft, H, F, E, k, S, T):
    sh = synth.Shape(L=2, E=E, k=k, H=H, F=F, fmt=synth.FMT_MXFP4)
    samples = {(s, l) for s in range(4) for l in range(2)}
    done = _replay(ft, sh, S, [(T, 4)], 25.0, 75.0, None, samples, repeat=True)
    assert len(done) == len(samples)


def test_mxfp4_prefill_small(ft):
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=512, fmt=synth.FMT_MXFP4)
    _run_prefill_fp4(ft, sh, 16, 300, [0, 1])


@pytest.mark.slow
def test_large_mxfp4_decode(ft):
    """Large shapes with MXFP4 banks: 8 layers, E=256, top-8, H=4096, F=2048,
    512 slots, 16 steps at T=1 then 8 at T=64, AR(1) rho=0.8.  The pool
    repeats the records of 13 drawn experts (routing does not depend on
    the values; a prime count keeps neighbouring records distinct)."""
    wl = synth.LARGE_MXFP4
    samples = {(s, l) for s in (0, 15) for l in (0, 7)} | {(s, l) for s in (16, 23) for l in (0, 7)}
    done = _replay(ft, wl.shape, wl.S, [(1, 16), (64, 8)], wl.B_P, wl.B_H, wl.rho, samples,
                   tok_sample=[0, 21, 42, 63], distinct=13)
    assert len(done) == len(samples)


# ------------------------------------------------------------ block-FP8

@pytest.mark.parametrize("H,F,E,k,S,T", [
    (256, 256, 16, 4, 12, 3),       # x fp32 in shared memory
    (1024, 512, 16, 4, 24, 9),      # several scale blocks along K and rows
    (1024, 512, 16, 4, 24, 40),     # x read from global memory
])
def test_fp8_small(ft, H, F, E, k, S, T):
    sh = synth.Shape(L=2, E=E, k=k, H=H, F=F, fmt=synth.FMT_FP8)
    samples = {(s, l) for s in range(4) for l in range(2)}
    done = _replay(ft, sh, S, [(T, 4)], 25.0, 75.0, None, samples, repeat=True)
    assert len(done) == len(samples)


def test_fp8_prefill_small(ft):
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=256, fmt=synth.FMT_FP8)
    _run_prefill_fp4(ft, sh, 16, 300, [0, 1])


@pytest.mark.slow
def test_large_fp8_decode(ft):
    """The Large layer shape with block-FP8 banks on 2 layers: E=256, top-8,
    H=4096, F=2048, 512 slots, 8 steps at T=1 then 4 at T=64, AR(1) rho=0.8.
    The pool repeats the records of 13 drawn experts."""
    sh = synth.Shape(L=2, E=256, k=8, H=4096, F=2048, fmt=synth.FMT_FP8)
    samples = {(s, l) for s in (0, 7) for l in (0, 1)} | {(s, l) for s in (8, 11) for l in (0, 1)}
    done = _replay(ft, sh, 512, [(1, 8), (64, 4)], 52.7, 150.0, 0.8, samples,
                   tok_sample=[0, 21, 42, 63], distinct=13)
    assert len(done) == len(samples)


def test_fp4_init_rejects_a_t_max_without_a_kernel_plan(ft):
    """T_max = 256 at the Large layer shape leaves the FP4 decode kernel no
    shared-memory plan (its per-route output rows and worklist no longer fit
    beside two ring slots): init refuses it instead of the first forward
    failing.  T_max = 64 has a plan."""
    import torch
    pool = torch.empty(4096, dtype=torch.uint8, pin_memory=True)
    with pytest.raises(ft.FtError):
        ft.Context(1, 256, 8, 4096, 2048, 16, pool, fmt=ft.FT_FMT_NVFP4, T_max=256,
                   nvfp4_global=np.ones(256, dtype=np.float32))
    with pytest.raises(ft.FtError):
        ft.Context(1, 256, 8, 4096, 2048, 16, pool, fmt=ft.FT_FMT_MXFP4, T_max=256)
    ctx = ft.Context(1, 256, 8, 4096, 2048, 16, pool, fmt=ft.FT_FMT_MXFP4, T_max=64)
    ctx.close()
