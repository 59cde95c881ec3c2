"""Pins of the oracle's expert arithmetic: dense brute force with plain loops,
capacity independence of the merged output, closed forms of SiLU / SwiGLU,
and the record byte layout."""
import math
import random

import numpy as np
import pytest

import synth
from oracle import control as ctl
from oracle import numerics as nm

TINY = synth.TINY


def _tiny_weights(layer=0):
    sh = TINY.shape
    cache = {}

    def w(e):
        if e not in cache:
            cache[e] = tuple(nm.bf16_to_f64(a) for a in synth.expert_weights_bf16(0, layer, e, sh.H, sh.F))
        return cache[e]
    return w


def test_silu_closed_forms():
    assert nm.silu(np.array([0.0]))[0] == 0.0
    assert abs(nm.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(nm.silu(np.array([50.0]))[0] - 50.0) < 1e-12
    assert abs(nm.silu(np.array([-800.0]))[0]) == 0.0


def test_expert_ffn_hand_example():
    # H=2, F=1: a = 1*x0 + 0*x1, b = 2*x0 + 1*x1, h = silu(a)*b, y = [3h, -h]
    Wg = np.array([[1.0, 0.0]])
    Wu = np.array([[2.0, 1.0]])
    Wd = np.array([[3.0], [-1.0]])
    x = np.array([[1.0, 2.0]])
    h = (1.0 / (1.0 + math.exp(-1.0))) * 4.0
    y = nm.expert_ffn(Wg, Wu, Wd, x)
    assert np.allclose(y, [[3 * h, -h]], rtol=0, atol=1e-15)


def test_dense_bruteforce_matches_gated_sum():
    sh = TINY.shape
    w = _tiny_weights()
    logits = synth.iid_logits(0, (99,), 4, sh.E)
    x = nm.bf16_to_f64(synth.tokens_bf16(0, 0, 0, 4, sh.H))
    ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits])
    y = nm.gated_sum(x, ids, gates, lambda t, j: True, w)
    mask = [[e in ids[t] for e in range(sh.E)] for t in range(4)]
    gm = [[gates[t][list(ids[t]).index(e)] if e in ids[t] else 0.0 for e in range(sh.E)] for t in range(4)]
    wl = [tuple(a.tolist() for a in w(e)) for e in range(sh.E)]
    yb = nm.dense_masked_bruteforce(x.tolist(), mask, gm, wl)
    assert nm.rel_l2(y, yb) < 1e-13


def test_bruteforce_catches_planted_mistakes():
    """A dropped term, a transposed operand or a wrong gate must move the result."""
    sh = TINY.shape
    w = _tiny_weights()
    x = nm.bf16_to_f64(synth.tokens_bf16(0, 1, 0, 2, sh.H))
    ids = [[0, 1], [2, 3]]
    gates = [[0.6, 0.4], [0.3, 0.7]]
    y = nm.gated_sum(x, ids, gates, lambda t, j: True, w)
    y_drop = nm.gated_sum(x, ids, gates, lambda t, j: j == 0, w)
    assert nm.rel_l2(y_drop, y) > 0.1
    y_swapgate = nm.gated_sum(x, ids, [[0.4, 0.6], [0.7, 0.3]], lambda t, j: True, w)
    assert nm.rel_l2(y_swapgate, y) > 0.05

    def w_swapped(e):
        Wg, Wu, Wd = w(e)
        return Wu, Wg, Wd
    assert nm.rel_l2(nm.gated_sum(x, ids, gates, lambda t, j: True, w_swapped), y) > 0.1


@pytest.mark.parametrize("S", [1, 2, 4, 8])
@pytest.mark.parametrize("ratio", [(1.0, 3.0), (1.0, 1.0), (1.0, 10.0)])
def test_capacity_independence(S, ratio):
    """The merged output does not depend on cache size or the q split
    (explainer section 11; deepmox: the cache needs to be truthful, not perfect)."""
    sh = TINY.shape
    w = _tiny_weights()
    st = ctl.CacheState.empty(1, sh.E, S)
    for step in range(6):
        logits = synth.iid_logits(0, (step,), 4, sh.E)
        x = nm.bf16_to_f64(synth.tokens_bf16(0, step, 0, 4, sh.H))
        ids, gates = zip(*[ctl.topk_route(r, sh.k) for r in logits])
        r = ctl.route_ctl(st, 0, ids, *ratio)
        ctl.check_invariants(st, r)
        y_gpu = nm.gated_sum(x, ids, gates, lambda t, j: r.slots_topk[t][j] >= 0, w)
        y_cpu = nm.gated_sum(x, ids, gates, lambda t, j: r.slots_topk[t][j] < 0, w)
        y_all = nm.gated_sum(x, ids, gates, lambda t, j: True, w)
        assert nm.rel_l2(y_gpu + y_cpu, y_all) < 1e-12
        # with the float32 partial sum, the merge stays within float32 rounding
        y_gpu2, pc = nm.moe_layer_split(x, ids, gates, r.slots_topk, w)
        assert nm.rel_l2(nm.merged_output(y_gpu2, pc), y_all) < 1e-6


def test_bf16_record_layout():
    """The record bytes hold W_gu rows as 16 gate rows then the 16 matching up
    rows, repeated, then W_d row-major; read back here by byte offsets."""
    H, F = 64, 128
    Wg, Wu, Wd = synth.expert_weights_bf16(0, 0, 3, H, F)
    rec = synth.record_bf16(0, 0, 3, H, F)
    assert rec.size == 3 * H * F * 2
    r16 = rec.view(np.uint16)
    for f in [0, 5, 15, 16, 31, 100, 127]:
        grp, i = divmod(f, 16)
        gate_row = r16[(grp * 32 + i) * H:(grp * 32 + i + 1) * H]
        up_row = r16[(grp * 32 + 16 + i) * H:(grp * 32 + 16 + i + 1) * H]
        assert np.array_equal(gate_row, Wg[f]) and np.array_equal(up_row, Wu[f])
    assert np.array_equal(r16[2 * F * H:].reshape(H, F), Wd)


def test_bf16_rounding_of_generator():
    # round-to-nearest-even on exact halfway cases and plain values
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.14159], dtype=np.float32)
    b = synth.f32_to_bf16_bits(vals)
    back = nm.bf16_to_f64(b)
    assert back[0] == 1.0
    assert back[1] == 1.0                      # tie -> even mantissa (1.0)
    assert back[2] == 1.0 + 4 * 2 ** -8        # tie -> even (1 + 2^-6)
    assert back[3] == -2.5
    assert abs(back[4] - 3.14159) <= 2 ** -7 * 2


def test_oracle_record_reader_matches_generator():
    H, F = 64, 128
    for e in (0, 5):
        rec = synth.record_bf16(0, 0, e, H, F)
        got = nm.record_weights_bf16(rec, H, F)
        want = [nm.bf16_to_f64(a) for a in synth.expert_weights_bf16(0, 0, e, H, F)]
        for g, w in zip(got, want):
            assert np.array_equal(g, w)
    # a record whose gate/up groups were swapped reads back differently
    rec = synth.record_bf16(0, 0, 1, H, F)
    sw = rec.copy().view(np.uint16)
    blk = 16 * H
    a = sw[:blk].copy()
    sw[:blk] = sw[blk:2 * blk]
    sw[blk:2 * blk] = a
    Wg2, Wu2, _ = nm.record_weights_bf16(sw.view(np.uint8), H, F)
    Wg, Wu, _ = nm.record_weights_bf16(rec, H, F)
    assert not np.array_equal(Wg2, Wg) and np.array_equal(Wg2[:16], Wu[:16])
