"""The allocation-free expert FFN entry point, through the C ABI.

Some callers may not allocate device memory once they run: serving engines
that own all device memory through pools carved at start-up, and
latency-critical paths that cannot afford the synchronisation of cudaMalloc.
ft_expert_ffn_noalloc serves them from a fixed device scratch array.

Two calls in a row (the second with fewer tokens, on the scratch the first
left behind) are compared with ft_moe_forward on the same routes and with the
fp64 oracle, within the BF16 tolerance of the other parity tests.  A call
whose routes all go to the CPU set returns partial_C exactly; an out-of-range
record index is reported by ft_noalloc_status and routes nothing.  The file
is collected last, so that a run stopping at the first failure has run every
other test first.
"""
import numpy as np
import pytest

import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

E, K, H, F = 32, 8, 2048, 768


@pytest.fixture(scope="module")
def setup():
    import torch
    import moe_expert_cache_gb300 as ft
    sh = synth.Shape(L=1, E=E, k=K, H=H, F=F)
    pool = torch.empty(E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
    synth.fill_host_pool(pool.numpy(), sh, 0)
    records = pool.cuda()  # record e of layer 0 at e * record_bytes
    assert ft.noalloc_status(None) == ft.FT_OK  # clears anything an earlier test left
    return ft, sh, pool, records


def _inputs(T, call):
    import torch
    xb = synth.tokens_bf16(0, 70 + call, 0, T, H)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    pc = torch.from_numpy(synth.random_f32(0, (70 + call,), (T, H), 0.1)).cuda()
    return xb, x, pc


def _noalloc(ft, records, rr_np, g_np, x, pc, T):
    import torch
    rr = torch.from_numpy(np.ascontiguousarray(rr_np, dtype=np.int32)).cuda()
    g = torch.from_numpy(np.ascontiguousarray(g_np, dtype=np.float32)).cuda()
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    st = ft.expert_ffn_noalloc(records.data_ptr(), E, rr.data_ptr(), g.data_ptr(), x.data_ptr(),
                               pc.data_ptr() if pc is not None else None, y.data_ptr(), T, K, H, F, None)
    assert st == ft.FT_OK, ft.status_str(st)
    return y


def test_noalloc_matches_context_path_and_oracle_twice(setup):
    import torch
    from oracle import numerics as nm
    ft, sh, pool, records = setup
    weights = hz.Weights(0, sh, 0)
    ctx = ft.Context(1, E, K, H, F, 12, pool, T_max=16)  # 12 slots: some routes go to the CPU set
    for call, T in enumerate((16, 5)):
        logits = torch.from_numpy(synth.iid_logits(0, (70 + call,), T, E)).cuda()
        xb, x, pc = _inputs(T, call)
        ctx.route_ctl(0, T, logits=logits, B_P=1.0, B_H=3.0)
        y_ref = torch.empty(T, H, dtype=torch.float32, device="cuda")
        ctx.moe_forward(x, pc, y_ref)
        got = ctx.last_ctl(T)
        assert got["info"].nC > 0 and got["info"].u_gpu > 0
        route_records = np.where(got["slots_topk"] >= 0, got["ids"], -1).astype(np.int32)
        y = _noalloc(ft, records, route_records, got["gates"], x, pc, T)
        assert ft.noalloc_status(None) == ft.FT_OK
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert nm.rel_l2(a, b) <= hz.BF16_REL_L2 and nm.max_abs(a, b) <= hz.BF16_MAX_ABS, call
        # the oracle: fp64 SwiGLU of the GPU routes, gated, plus the same partial_C
        ids = got["ids"].tolist()
        gates = got["gates"].astype(np.float64).tolist()
        y_gpu = nm.gated_sum(nm.bf16_to_f64(xb), ids, gates, lambda t, j: route_records[t][j] >= 0, weights)
        ref = nm.merged_output(y_gpu, pc.cpu().numpy())
        assert nm.rel_l2(a, ref) <= hz.BF16_REL_L2 and nm.max_abs(a, ref) <= hz.BF16_MAX_ABS, call
    assert ctx.status() == ft.FT_OK
    ctx.close()


def test_noalloc_cpu_only_routes_and_bad_index(setup):
    import torch
    ft, sh, pool, records = setup
    T = 3
    _, x, pc = _inputs(T, 5)
    g = np.full((T, K), 1.0 / K, dtype=np.float32)
    # every route on the CPU set: y is partial_C exactly (and zero without it)
    y = _noalloc(ft, records, np.full((T, K), -1), g, x, pc, T)
    torch.cuda.synchronize()
    assert torch.equal(y, pc)
    y0 = _noalloc(ft, records, np.full((T, K), -1), g, x, None, T)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y0).item() == 0
    assert ft.noalloc_status(None) == ft.FT_OK
    # a record index past the array: reported on the device, nothing routed
    bad = np.tile(np.arange(K, dtype=np.int32), (T, 1))
    bad[1, 3] = E
    y = _noalloc(ft, records, bad, g, x, pc, T)
    assert ft.noalloc_status(None) == ft.FT_ERR_DEVICE
    assert torch.equal(y, pc)
    assert ft.noalloc_status(None) == ft.FT_OK  # read once, then cleared
    # sizes beyond the scratch array are rejected before any launch
    rr = torch.zeros(129, K, dtype=torch.int32, device="cuda")
    yb = torch.empty(129, H, device="cuda")
    xb = torch.zeros(129, H, dtype=torch.bfloat16, device="cuda")
    big = ft.expert_ffn_noalloc(records.data_ptr(), E, rr.data_ptr(), rr.data_ptr(), xb.data_ptr(), None,
                                yb.data_ptr(), 129, K, H, F, None)
    assert big == ft.FT_ERR_ARG
