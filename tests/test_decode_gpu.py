"""GPU parity of the decode path through the C ABI: control state bit-exact
against the oracle on every call, outputs within the BF16 tolerance on every
call of the tiny layer and on sampled calls of the full-size workloads."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import control as ctl
from oracle import numerics as nm
from tests import harness as hz

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_control_hand.json")


@pytest.fixture(scope="module")
def ft():
    import torch
    assert torch.cuda.is_available()
    import moe_expert_cache_gb300 as ft
    ft.load()
    return ft


@pytest.fixture(scope="module")
def tiny_pool():
    return hz.pinned_pool(synth.TINY.shape, seed=0)[0]


def _dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def _tiny_step(ft, ctx, st, wl, step, S_label, weights):
    import torch
    sh = wl.shape
    logits = synth.iid_logits(wl.seed, (step,), wl.T, sh.E)
    xb = synth.tokens_bf16(wl.seed, step, 0, wl.T, sh.H)
    ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits])
    r = ctl.route_ctl(st, 0, ids, wl.B_P, wl.B_H)
    ctl.check_invariants(st, r)
    ctx.route_ctl(0, wl.T, logits=_dev(logits), B_P=wl.B_P, B_H=wl.B_H)
    got = hz.compare_ctl(ctx, st, r, wl.T, f"S={S_label} step={step}")
    assert np.array_equal(got["ids"], np.array(ids, dtype=np.int32))
    assert np.allclose(got["gates"], np.array(gates), rtol=2e-6, atol=1e-7)
    _, pc = nm.moe_layer_split(nm.bf16_to_f64(xb), ids, gates, r.slots_topk, weights)
    x = _dev(xb.view(np.int16)).view(torch.bfloat16)
    y = torch.empty(wl.T, sh.H, dtype=torch.float32, device="cuda")
    ctx.moe_forward(x, _dev(pc), y)
    torch.cuda.synchronize()
    hz.check_output(y, xb, ids, gates, r.slots_topk, weights, pc, f"S={S_label} step={step}")
    # the merged output equals the dense result whatever the split
    y_all = nm.gated_sum(nm.bf16_to_f64(xb), ids, gates, lambda t, j: True, weights)
    assert nm.rel_l2(y.cpu().numpy(), y_all) <= hz.BF16_REL_L2
    return r


@pytest.mark.parametrize("S", [4, 1, 2, 8, 16])
def test_tiny_decode_parity(ft, tiny_pool, S):
    wl = synth.TINY
    sh = wl.shape
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, S, tiny_pool, T_max=wl.T)
    st = ctl.CacheState.empty(sh.L, sh.E, S)
    w = hz.Weights(wl.seed, sh, 0)
    for step in range(wl.steps):
        _tiny_step(ft, ctx, st, wl, step, S, w)
    assert ctx.status() == ft.FT_OK
    # complete-record rule: every occupied slot holds the whole record of its owner
    for s, fid in enumerate(st.id_for_slot):
        if fid >= 0:
            l, e = divmod(fid, sh.E)
            assert np.array_equal(ctx.read_slot(s), synth.record_bf16(wl.seed, l, e, sh.H, sh.F)), s
    c = ctx.counters()
    assert c["calls"] == wl.steps
    ctx.close()


def test_hand_worked_table_through_topk(ft, tiny_pool):
    import torch
    g = json.load(open(GOLDEN))
    ctx = ft.Context(g["L"], g["E"], g["k"], 64, 128, g["S"], tiny_pool, T_max=4)
    for i, step in enumerate(g["steps"]):
        ids = np.array(step["routes"], dtype=np.int32)
        w = np.full(ids.shape, 0.5, dtype=np.float32)
        ctx.route_ctl(0, 4, topk_ids=_dev(ids), topk_w=_dev(w), B_P=g["B_P"], B_H=g["B_H"])
        got = ctx.last_ctl(4)
        assert got["info"].q0 == step["q0"] and got["info"].q == step["q"], i
        assert got["F"] == step["F"] and got["C"] == step["C"] and got["victims"] == step["victims"], i
        assert got["slots_topk"].tolist() == step["slots_topk"], i
        sfi, ifs, stp, clk = ctx.ctl_state()
        assert ifs.tolist() == step["id_for_slot"] and stp.tolist() == step["stamps"], i
    assert sfi.tolist() == g["final_slot_for_id"] and clk == g["final_clock"]
    ctx.close()


def test_invalid_routes_latch_device_error(ft, tiny_pool):
    import torch
    ctx = ft.Context(1, 8, 2, 64, 128, 4, tiny_pool, T_max=4)
    good = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], dtype=np.int32)
    w = np.full(good.shape, 0.5, dtype=np.float32)
    ctx.route_ctl(0, 4, topk_ids=_dev(good), topk_w=_dev(w), B_P=1.0, B_H=1.0)
    assert ctx.status() == ft.FT_OK
    before = ctx.ctl_state()
    for bad in ([[0, 1], [2, 3], [4, 9], [6, 7]], [[0, 1], [2, 2], [4, 5], [6, 7]], [[0, -1], [2, 3], [4, 5], [6, 7]]):
        ctx.route_ctl(0, 4, topk_ids=_dev(np.array(bad, dtype=np.int32)), topk_w=_dev(w), B_P=1.0, B_H=1.0)
        assert ctx.status() == ft.FT_ERR_DEVICE
        after = ctx.ctl_state()
        for a, b in zip(before, after):
            assert np.array_equal(np.asarray(a), np.asarray(b))
        # the forward of an invalid pass returns the CPU partial sum alone
        x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
        pc = torch.randn(4, 64, device="cuda")
        y = torch.empty_like(pc)
        ctx.moe_forward(x, pc, y)
        torch.cuda.synchronize()
        assert torch.equal(y, pc)
    nan_logits = torch.zeros(4, 8, device="cuda")
    nan_logits[2, 3] = float("nan")
    ctx.route_ctl(0, 4, logits=nan_logits, B_P=1.0, B_H=1.0)
    assert ctx.status() == ft.FT_ERR_DEVICE
    assert ctx.status() == ft.FT_OK  # the error word is cleared once read
    with pytest.raises(ft.FtError):
        ctx.route_ctl(0, 5, logits=nan_logits, B_P=1.0, B_H=1.0)  # T > T_max
    with pytest.raises(ft.FtError):
        ctx.route_ctl(0, 4, logits=nan_logits, B_P=0.0, B_H=1.0)
    ctx.close()


# ------------------------------------------------------------ full-size runs

@pytest.fixture(scope="module")
def big_pool():
    """The 48-layer BF16 host pool shared by both decode workloads (58 GB)."""
    return hz.pinned_pool(synth.DECODE_T1.shape, seed=0)[0]


def _replay(ft, pool, wl, samples, resize=()):
    """Run every control call of a decode workload on the GPU and the oracle,
    bit-exact on every call; outputs checked at the sampled (step, layer)."""
    import torch
    sh = wl.shape
    logits = synth.ar1_logits(wl.seed, wl.steps, sh.L, wl.T, sh.E, wl.rho, wl.sigma)
    logits_d = _dev(logits)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, pool, T_max=wl.T)
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    resize = dict(resize)
    checked = []
    for step in range(wl.steps):
        if step in resize:
            ctx.cache_resize(resize[step])
            ctl.resize(st, resize[step])
            sfi, ifs, stp, clk = ctx.ctl_state()
            assert ifs.tolist() == st.id_for_slot and stp.tolist() == st.stamp and sfi.tolist() == st.slot_for_id
        for layer in range(sh.L):
            ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits[step, layer]])
            r = ctl.route_ctl(st, layer, ids, wl.B_P, wl.B_H)
            ctl.check_invariants(st, r)
            ctx.route_ctl(layer, wl.T, logits=logits_d[step, layer], B_P=wl.B_P, B_H=wl.B_H)
            hz.compare_ctl(ctx, st, r, wl.T, f"step={step} layer={layer}")
            if (step, layer) in samples:
                w = hz.Weights(wl.seed, sh, layer)
                xb = synth.tokens_bf16(wl.seed, step, layer, wl.T, sh.H)
                _, pc = nm.moe_layer_split(nm.bf16_to_f64(xb), ids, gates, r.slots_topk, w)
                x = _dev(xb.view(np.int16)).view(torch.bfloat16)
                y = torch.empty(wl.T, sh.H, dtype=torch.float32, device="cuda")
                ctx.moe_forward(x, _dev(pc), y)
                torch.cuda.synchronize()
                checked.append(hz.check_output(y, xb, ids, gates, r.slots_topk, w, pc, f"{step}/{layer}"))
                # complete records: the fills of this call hold their owner's bytes
                for f, v in zip(r.F, r.victims):
                    assert np.array_equal(ctx.read_slot(v), synth.record_bf16(wl.seed, layer, f, sh.H, sh.F))
    assert ctx.status() == ft.FT_OK
    cnt = ctx.counters()
    ctx.close()
    return checked, cnt


@pytest.mark.slow
def test_decode_t1_full_size(ft, big_pool):
    wl = synth.DECODE_T1
    samples = {(s, l) for s in (0, 1, 100, 255) for l in (0, 17, 47)}
    checked, cnt = _replay(ft, big_pool, wl, samples)
    assert len(checked) == len(samples)
    assert cnt["calls"] == wl.steps * wl.shape.L


@pytest.mark.slow
def test_decode_t16_with_resize(ft, big_pool):
    wl = synth.DECODE_T16
    samples = {(s, l) for s in (0, 31, 32, 63, 64, 127) for l in (0, 47)}
    checked, cnt = _replay(ft, big_pool, wl, samples, resize=synth.DECODE_T16_RESIZE)
    assert len(checked) == len(samples)


def test_measure_link_leaves_the_cache_untouched(ft):
    """B_P measured with the fill path (explainer section 5; the txtmix
    write-up's one-off bandwidth measurement): a positive rate, and the cache
    state and statistics are unchanged by the call."""
    import torch
    sh = synth.Shape(L=2, E=8, k=2, H=256, F=128)
    pool, _ = hz.pinned_pool(sh, 0)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, 8, pool, T_max=4)
    routes = np.array([[1, 2], [3, 4], [1, 5], [6, 2]], dtype=np.int32)
    ctx.route_ctl(0, 4, topk_ids=_dev(routes), topk_w=_dev(np.full(routes.shape, 0.5, np.float32)),
                  B_P=1.0, B_H=1.0)
    x = torch.zeros(4, sh.H, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(4, sh.H, device="cuda")
    ctx.moe_forward(x, None, y)
    before, cnt = ctx.ctl_state(), ctx.counters()
    gbps = ctx.measure_link(16, 2)
    assert gbps > 1.0
    after = ctx.ctl_state()
    assert all(np.array_equal(a, b) for a, b in zip(before[:3], after[:3])) and before[3] == after[3]
    assert ctx.counters() == cnt
    with pytest.raises(ft.FtError):
        ctx.measure_link(0, 1)
    with pytest.raises(ft.FtError):
        ctx.measure_link(sh.L * sh.E + 1, 1)
    assert ctx.status() == ft.FT_OK
    ctx.close()


# ------------------------------------------------------- failure handling

def _tiny_oracle_step(ctx, st, wl, step, weights, T=None):
    import torch
    sh = wl.shape
    T = T or wl.T
    logits = synth.iid_logits(wl.seed, (step,), T, sh.E)
    xb = synth.tokens_bf16(wl.seed, step, 0, T, sh.H)
    ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits])
    r = ctl.route_ctl(st, 0, ids, wl.B_P, wl.B_H)
    ctx.route_ctl(0, T, logits=_dev(logits), B_P=wl.B_P, B_H=wl.B_H)
    hz.compare_ctl(ctx, st, r, T, f"step={step}")
    _, pc = nm.moe_layer_split(nm.bf16_to_f64(xb), ids, gates, r.slots_topk, weights)
    x = _dev(xb.view(np.int16)).view(torch.bfloat16)
    y = torch.empty(T, sh.H, dtype=torch.float32, device="cuda")
    ctx.moe_forward(x, _dev(pc), y)
    torch.cuda.synchronize()
    hz.check_output(y, xb, ids, gates, r.slots_topk, weights, pc, f"step={step}")
    return r


def test_wait_that_runs_out_is_reported_and_the_cache_recovers(ft):
    """A bounded wait in the decode kernel gives up: with its progress waits
    limited to 1 microsecond, a forward whose fills stream over the host link
    (the first chunks land after several microseconds) latches the timeout
    and winds down without a fault.  ft_get_status reports FT_ERR_TIMEOUT and
    empties the cache (a fill may be incomplete); the next calls refill from
    the host pool and match the oracle started from an empty cache with the
    same clock."""
    import torch
    wl = synth.Workload("fail", synth.Shape(L=1, E=16, k=4, H=1024, F=512), S=8, steps=6, T=4, rho=None, sigma=None,
                        B_P=1.0, B_H=1.0)
    sh = wl.shape
    pool, _ = hz.pinned_pool(sh, 0)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, pool, T_max=wl.T)
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    w = hz.Weights(wl.seed, sh, 0)
    _tiny_oracle_step(ctx, st, wl, 0, w)
    assert ctx.status() == ft.FT_OK
    with pytest.raises(ft.FtError):
        ctx.set_wait_limit(999)  # below the 1 us floor
    ctx.set_wait_limit(1000)
    logits = synth.iid_logits(wl.seed, (1,), wl.T, sh.E)
    ids, _ = zip(*[ctl.topk_route(r, sh.k) for r in logits])
    r = ctl.route_ctl(st.copy(), 0, ids, wl.B_P, wl.B_H)
    assert r.q >= 2  # real fills stream during the forward
    ctx.route_ctl(0, wl.T, logits=_dev(logits), B_P=wl.B_P, B_H=wl.B_H)
    y = torch.empty(wl.T, sh.H, dtype=torch.float32, device="cuda")
    ctx.moe_forward(_dev(synth.tokens_bf16(wl.seed, 1, 0, wl.T, sh.H).view(np.int16)).view(torch.bfloat16), None, y)
    assert ctx.status() == ft.FT_ERR_TIMEOUT
    sfi, ifs, stp, clk = ctx.ctl_state()
    assert (sfi == -1).all() and (ifs == -1).all() and (stp == 0).all() and clk == st.clock + 1
    ctx.set_wait_limit(0)  # back to the default
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    st.clock = clk
    for step in range(2, wl.steps):
        _tiny_oracle_step(ctx, st, wl, step, w)
    assert ctx.status() == ft.FT_OK
    ctx.close()


def test_resize_that_cannot_allocate_leaves_the_cache_intact(ft):
    """ft_cache_resize "on any failure the old cache is left unchanged": a
    resize to more slots than device memory holds fails in cudaMalloc (a
    genuine out-of-memory answer, no fault); the maps, stamps and slot bytes
    are unchanged and decoding continues against the oracle."""
    wl = synth.Workload("oom", synth.Shape(L=1, E=16, k=4, H=2048, F=2048), S=6, steps=5, T=2, rho=None,
                        sigma=None, B_P=1.0, B_H=2.0)
    sh = wl.shape
    pool, _ = hz.pinned_pool(sh, 0)
    # a BF16 shape whose decode kernel has no shared-memory plan is refused at init
    with pytest.raises(ft.FtError) as ei:
        ft.Context(1, 16, 4, 4096, 2048, 6, pool, T_max=2)
    assert ei.value.status == ft.FT_ERR_ARG
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, pool, T_max=wl.T)
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    w = hz.Weights(wl.seed, sh, 0)
    for step in range(2):
        _tiny_oracle_step(ctx, st, wl, step, w)
    before = ctx.ctl_state()
    slots = [ctx.read_slot(s) for s in range(wl.S)]
    # 13000 records of 25 MB: about 327 GB, more than the GPU's memory
    with pytest.raises(ft.FtError) as ei:
        ctx.cache_resize(13000)
    assert ei.value.status == ft.FT_ERR_OOM
    assert ctx.S == wl.S
    after = ctx.ctl_state()
    assert all(np.array_equal(a, b) for a, b in zip(before[:3], after[:3])) and before[3] == after[3]
    assert all(np.array_equal(ctx.read_slot(s), slots[s]) for s in range(wl.S))
    for step in range(2, wl.steps):
        _tiny_oracle_step(ctx, st, wl, step, w)
    assert ctx.status() == ft.FT_OK
    ctx.close()


def test_set_ctl_state_round_trip(ft, tiny_pool):
    """ft_set_ctl_state: putting back the state just read changes nothing
    (later calls still match the oracle, outputs included); a fresh context
    given an empty cache at clock 1000 follows the oracle from that clock; and
    states that break the map bijection, name an id or slot out of range or
    carry a stamp past the clock are refused with the state unchanged."""
    wl = synth.TINY
    sh = wl.shape
    w = hz.Weights(wl.seed, sh, 0)
    ctx = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, tiny_pool, T_max=wl.T)
    st = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    for step in range(6):
        _tiny_oracle_step(ctx, st, wl, step, w)
    sfi, ifs, stp, clk = ctx.ctl_state()
    ctx.set_ctl_state(sfi, ifs, stp, clk)
    for step in range(6, 10):
        _tiny_oracle_step(ctx, st, wl, step, w)
    good = ctx.ctl_state()
    bad_states = []
    b = [a.copy() for a in good[:3]]
    occ = int(np.flatnonzero(b[1] >= 0)[0])
    b[0][b[1][occ]] = (occ + 1) % wl.S          # slot_for_id disagrees with id_for_slot
    bad_states.append((b, good[3]))
    b = [a.copy() for a in good[:3]]
    b[1][occ] = sh.L * sh.E                     # id out of range
    bad_states.append((b, good[3]))
    b = [a.copy() for a in good[:3]]
    b[2][occ] = good[3] + 1                     # stamp past the clock
    bad_states.append((b, good[3]))
    for (a0, a1, a2), c in bad_states:
        with pytest.raises(ft.FtError) as ei:
            ctx.set_ctl_state(a0, a1, a2, c)
        assert ei.value.status == ft.FT_ERR_ARG
        now = ctx.ctl_state()
        assert all(np.array_equal(x, y) for x, y in zip(good[:3], now[:3])) and good[3] == now[3]
    ctx.close()
    ctx2 = ft.Context(sh.L, sh.E, sh.k, sh.H, sh.F, wl.S, tiny_pool, T_max=wl.T)
    empty = ctl.CacheState.empty(sh.L, sh.E, wl.S)
    ctx2.set_ctl_state(empty.slot_for_id, empty.id_for_slot, empty.stamp, 1000)
    empty.clock = 1000
    for step in range(4):
        _tiny_oracle_step(ctx2, empty, wl, step, w)
    assert ctx2.status() == ft.FT_OK
    ctx2.close()
