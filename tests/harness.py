"""Shared helpers of the GPU parity tests: pinned host pools, a context per
workload, and the comparison of the library's control state with the
oracle's, call by call."""
from __future__ import annotations

import numpy as np

import synth
from oracle import control as ctl
from oracle import numerics as nm

# Tolerances stated for BF16 decode / prefill outputs against the fp64 oracle.
BF16_REL_L2 = 2e-3
BF16_MAX_ABS = 2e-2


def torch_mod():
    import torch
    return torch


def pinned_pool(shape: synth.Shape, seed: int = 0):
    """Page-locked host pool (torch uint8 tensor) holding every record."""
    torch = torch_mod()
    pool = torch.empty(shape.L * shape.E * shape.record_bytes, dtype=torch.uint8, pin_memory=True)
    glob = synth.fill_host_pool(pool.numpy(), shape, seed)
    return pool, glob


class Weights:
    """float64 logical weights of one layer, regenerated from the seed on demand."""

    def __init__(self, seed, shape: synth.Shape, layer: int):
        self.seed, self.shape, self.layer = seed, shape, layer
        self.cache = {}

    def __call__(self, e):
        if e not in self.cache:
            H, F = self.shape.H, self.shape.F
            self.cache[e] = tuple(nm.bf16_to_f64(a) for a in synth.expert_weights_bf16(self.seed, self.layer, e, H, F))
        return self.cache[e]


def compare_ctl(ctx, st: ctl.CacheState, r: ctl.CtlResult, T: int, where: str = ""):
    """Bit-exact comparison of the last control pass and the whole state."""
    got = ctx.last_ctl(T)
    info = got["info"]
    assert info.layer == r.layer, where
    assert info.u == len(r.counts), where
    assert info.h == len(r.hits) and info.m == len(r.misses), where
    assert (info.q0, info.q1, info.q) == (r.fc.q0, r.fc.q1, r.fc.q), where
    assert info.nC == len(r.C), where
    assert got["F"] == r.F, (where, got["F"], r.F)
    assert got["C"] == r.C, (where, got["C"], r.C)
    assert got["victims"] == r.victims, (where, got["victims"], r.victims)
    assert np.array_equal(got["slots_topk"], np.array(r.slots_topk, dtype=np.int32)), where
    assert info.clock == r.clock == st.clock, where
    sfi, ifs, stp, clk = ctx.ctl_state()
    assert clk == st.clock, where
    assert np.array_equal(sfi, np.array(st.slot_for_id, dtype=np.int32)), where
    assert np.array_equal(ifs, np.array(st.id_for_slot, dtype=np.int32)), where
    assert np.array_equal(stp, np.array(st.stamp, dtype=np.uint32)), where
    return got


def check_output(y_gpu_dev, x_bits, ids, gates, slots_topk, weights, partial_C, where=""):
    """y from the library vs the oracle's GPU-part sum + the same partial_C."""
    x = nm.bf16_to_f64(x_bits)
    y_ref_gpu = nm.gated_sum(x, ids, gates, lambda t, j: slots_topk[t][j] >= 0, weights)
    ref = nm.merged_output(y_ref_gpu, partial_C)
    y = y_gpu_dev.float().cpu().numpy().astype(np.float64)
    rel = nm.rel_l2(y, ref)
    mab = nm.max_abs(y, ref)
    assert rel <= BF16_REL_L2 and mab <= BF16_MAX_ABS, (where, rel, mab)
    return rel, mab
