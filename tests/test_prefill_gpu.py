"""GPU parity of the prefill path through the C ABI: full-layer double buffer,
tcgen05 grouped GEMMs, SwiGLU and gated combine, against the fp64 oracle's
dense masked MoE; control state after prefill against the oracle's buffer
invalidation; the hostile decode -> prefill -> decode sequence."""
import numpy as np
import pytest

import synth
from oracle import control as ctl
from oracle import numerics as nm
from tests import harness as hz

pytestmark = pytest.mark.gpu


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


def _pool_weights(pool_np, sh, layer):
    rb = sh.record_bytes
    cache = {}

    def w(e):
        if e not in cache:
            fid = layer * sh.E + e
            cache[e] = nm.record_weights_bf16(pool_np[fid * rb:(fid + 1) * rb], sh.H, sh.F)
        return cache[e]
    return w


def _run_prefill(ft, sh, S, T, layers, seed=0, sample=None, streams=True):
    import torch
    pool, _ = hz.pinned_pool(sh, seed)
    cs = torch.cuda.Stream()
    ts = torch.cuda.Stream()
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, S, pool, T_max=4, T_prefill_max=T,
                     compute_stream=cs.cuda_stream, transfer_stream=ts.cuda_stream if streams else 0)
    xs, lgs, ys = [], [], []
    for i, l in enumerate(layers):
        lgs.append(synth.iid_logits(seed, (900, l), T, sh.E))
        xs.append(synth.tokens_bf16(seed, 900, l, T, sh.H))
        ys.append(torch.empty(T, sh.H, dtype=torch.float32, device="cuda"))
    xd = [_dev(x.view(np.int16)).view(torch.bfloat16) for x in xs]
    ld = [_dev(lg) for lg in lgs]
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        ctx.prefill_begin(layers[0])
        for i, l in enumerate(layers):
            nxt = layers[i + 1] if i + 1 < len(layers) else -1
            ctx.prefill_layer(i & 1, l, nxt, T, xd[i], ld[i], ys[i])
    torch.cuda.synchronize()
    assert ctx.status() == ft.FT_OK
    pool_np = pool.numpy()
    results = []
    for i, l in enumerate(layers):
        toks = range(T) if sample is None else sample
        ids, gates = zip(*[ctl.topk_route(lgs[i][t], sh.k) for t in toks])
        x = nm.bf16_to_f64(xs[i][list(toks)])
        ref = nm.gated_sum(x, ids, gates, lambda t, j: True, _pool_weights(pool_np, sh, l))
        y = ys[i].cpu().numpy()[list(toks)]
        assert np.isfinite(ys[i].cpu().numpy()).all()
        rel, mab = nm.rel_l2(y, ref), nm.max_abs(y, ref)
        assert rel <= hz.BF16_REL_L2 and mab <= hz.BF16_MAX_ABS, (l, rel, mab)
        results.append((rel, mab))
    return ctx, results


@pytest.mark.parametrize("shape,S,T", [
    (synth.Shape(L=3, E=8, k=2, H=256, F=128), 16, 600),       # ragged M tiles, one N tile
    (synth.Shape(L=2, E=16, k=4, H=512, F=256), 40, 1000),     # two N tiles in both GEMMs
    (synth.Shape(L=2, E=8, k=2, H=256, F=128), 16, 33),        # one partial M tile per expert
])
def test_prefill_small_parity(ft, shape, S, T):
    layers = list(range(shape.L))
    ctx, res = _run_prefill(ft, shape, S, T, layers)
    # every slot of both buffers is empty after the chunk, like the oracle's invalidation
    st = ctl.CacheState.empty(shape.L, shape.E, S)
    for i, _ in enumerate(layers):
        ctl.prefill_invalidate(st, i & 1)
    sfi, ifs, stp, clk = ctx.ctl_state()
    assert ifs.tolist() == st.id_for_slot and stp.tolist() == st.stamp and sfi.tolist() == st.slot_for_id
    ctx.close()


def test_prefill_single_stream(ft):
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=128)
    ctx, _ = _run_prefill(ft, sh, 16, 300, [1, 0], streams=False)
    ctx.close()


def test_hostile_sequence(ft):
    """deepmox "How residency follows demand...": one request uses layer-0
    experts, a prefill materialises other layers into every slot, the request
    routes back: every route misses and is refilled from layer 0's records."""
    import torch
    sh = synth.Shape(L=4, E=8, k=2, H=256, F=128)
    S = 16
    pool, _ = hz.pinned_pool(sh, 0)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, S, pool, T_max=4, T_prefill_max=64)
    st = ctl.CacheState.empty(sh.L, sh.E, S)
    routes = np.array([[1, 2], [3, 4], [1, 5], [6, 2]], dtype=np.int32)
    w = _dev(np.full(routes.shape, 0.5, np.float32))
    for _ in range(2):
        r = ctl.route_ctl(st, 0, routes.tolist(), 1.0, 1.0)
        ctx.route_ctl(0, 4, topk_ids=_dev(routes), topk_w=w, B_P=1.0, B_H=1.0)
        hz.compare_ctl(ctx, st, r, 4)
    assert r.q == 0 and len(r.hits) == 6
    T = 64
    xs = [_dev(synth.tokens_bf16(0, 1, l, T, sh.H).view(np.int16)).view(torch.bfloat16) for l in range(4)]
    lgs = [_dev(synth.iid_logits(0, (5, l), T, sh.E)) for l in range(4)]
    y = torch.empty(T, sh.H, dtype=torch.float32, device="cuda")
    ctx.prefill_begin(0)
    for i in range(4):
        ctx.prefill_layer(i & 1, i, i + 1 if i < 3 else -1, T, xs[i], lgs[i], y)
        ctl.prefill_invalidate(st, i & 1)
    torch.cuda.synchronize()
    r = ctl.route_ctl(st, 0, routes.tolist(), 1.0, 1.0)
    ctx.route_ctl(0, 4, topk_ids=_dev(routes), topk_w=w, B_P=1.0, B_H=1.0)
    hz.compare_ctl(ctx, st, r, 4)
    assert r.hits == [] and r.q == 6
    for f, v in zip(r.F, r.victims):
        assert np.array_equal(ctx.read_slot(v), synth.record_bf16(0, 0, f, sh.H, sh.F))
    assert ctx.status() == ft.FT_OK
    ctx.close()


def test_prefill_state_errors(ft):
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=128)
    pool, _ = hz.pinned_pool(sh, 0)
    small = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, 15, pool, T_max=4, T_prefill_max=64)  # S < 2E
    with pytest.raises(ft.FtError) as ei:
        small.prefill_begin(0)
    assert ei.value.status == ft.FT_ERR_CAPACITY
    small.close()
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, 16, pool, T_max=4)  # prefill disabled
    with pytest.raises(ft.FtError):
        ctx.prefill_begin(0)
    ctx.close()
    import torch
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, 16, pool, T_max=4, T_prefill_max=64)
    x = torch.zeros(64, sh.H, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(64, sh.E, device="cuda")
    y = torch.empty(64, sh.H, device="cuda")
    with pytest.raises(ft.FtError):
        ctx.prefill_layer(0, 0, -1, 64, x, lg, y)  # no open chunk
    ctx.prefill_begin(0)
    with pytest.raises(ft.FtError):
        ctx.route_ctl(0, 1, logits=lg[:1], B_P=1.0, B_H=1.0)  # decode while a chunk is open
    with pytest.raises(ft.FtError):
        ctx.prefill_layer(1, 0, -1, 64, x, lg, y)  # wrong buffer
    ctx.prefill_layer(0, 0, -1, 64, x, lg, y)
    torch.cuda.synchronize()
    assert ctx.status() == ft.FT_OK
    ctx.close()


@pytest.mark.slow
def test_prefill_full_size(ft):
    """Prefill workload: 4 layers, E=128, top-8, H=2048, F=768, T=8192, 256 slots."""
    wl = synth.PREFILL
    rng = np.random.default_rng(7)
    sample = sorted(rng.choice(wl.T, size=48, replace=False).tolist()) + [wl.T - 1]
    ctx, res = _run_prefill(ft, wl.shape, wl.S, wl.T, list(range(wl.shape.L)), sample=sample)
    ctx.close()
