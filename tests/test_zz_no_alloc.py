"""The allocation-free expert FFN entry point against the context path.

Some callers cannot allocate device memory while they run (inside a CUDA
graph capture, or in engines that own all device memory through their own
pools); ft_expert_ffn_noalloc serves them with a fixed device scratch array.
This test calls it through the C ABI twice in a row and compares each output
with ft_moe_forward on the same routes, within the BF16 tolerance of the
other parity tests.  It is collected last so that a run stopping at the first
failure has run every other test first.
"""
import numpy as np
import pytest

import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu


def test_noalloc_matches_context_path_twice():
    import torch
    import moe_expert_cache_gb300 as ft
    from oracle import numerics as nm

    E, k, H, F = 32, 8, 2048, 768
    sh = synth.Shape(L=1, E=E, k=k, H=H, F=F)
    pool = torch.empty(E * sh.record_bytes, dtype=torch.uint8, pin_memory=True)
    synth.fill_host_pool(pool.numpy(), sh, 0)
    records = pool.cuda()  # record e of layer 0 at e * record_bytes
    ctx = ft.Context(1, E, k, H, F, 12, pool, T_max=16)  # 12 slots: some routes go to the CPU set
    for call, T in enumerate((16, 5)):
        logits = torch.from_numpy(synth.iid_logits(0, (70 + call,), T, E)).cuda()
        xb = synth.tokens_bf16(0, 70 + call, 0, T, H)
        x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
        pc = torch.from_numpy(synth.random_f32(0, (70 + call,), (T, H), 0.1)).cuda()
        ctx.route_ctl(0, T, logits=logits, B_P=1.0, B_H=3.0)
        y_ref = torch.empty(T, H, dtype=torch.float32, device="cuda")
        ctx.moe_forward(x, pc, y_ref)
        got = ctx.last_ctl(T)
        assert got["info"].nC > 0 and got["info"].u_gpu > 0
        route_records = np.where(got["slots_topk"] >= 0, got["ids"], -1).astype(np.int32)
        rr = torch.from_numpy(route_records).cuda()
        g = torch.from_numpy(np.ascontiguousarray(got["gates"])).cuda()
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        st = ft.expert_ffn_noalloc(records.data_ptr(), E, rr.data_ptr(), g.data_ptr(), x.data_ptr(),
                                   pc.data_ptr(), y.data_ptr(), T, k, H, F, None)
        assert st == ft.FT_OK, ft.status_str(st)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert nm.rel_l2(a, b) <= hz.BF16_REL_L2 and nm.max_abs(a, b) <= hz.BF16_MAX_ABS, call
    # sizes beyond the scratch array are rejected before any launch
    big = ft.expert_ffn_noalloc(records.data_ptr(), E, rr.data_ptr(), g.data_ptr(), x.data_ptr(), None,
                                y.data_ptr(), 129, k, H, F, None)
    assert big == ft.FT_ERR_ARG
    assert ctx.status() == ft.FT_OK
    ctx.close()
