"""Pins of the oracle's cache control: the hand-worked table, the Figure-2
split, invariants, and agreement with an independent brute-force LRU model
that keeps an explicit recency list instead of stamps."""
import json
import os
import random
from fractions import Fraction

import pytest

from oracle import control as ctl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_control_hand.json")


def test_hand_worked_tiny_table():
    g = json.load(open(GOLDEN))
    st = ctl.CacheState.empty(g["L"], g["E"], g["S"])
    for i, step in enumerate(g["steps"]):
        r = ctl.route_ctl(st, 0, step["routes"], g["B_P"], g["B_H"])
        ctl.check_invariants(st, r)
        assert r.hits == step["hits"], i
        assert len(r.misses) == step["m"], i
        assert r.fc.q0 == step["q0"] and r.q == step["q"], i
        assert r.F == step["F"] and r.C == step["C"], i
        assert r.victims == step["victims"], i
        assert st.id_for_slot == step["id_for_slot"], i
        assert st.stamp == step["stamps"], i
        assert r.slots_topk == step["slots_topk"], i
    assert st.slot_for_id == g["final_slot_for_id"]
    assert st.clock == g["final_clock"]


def test_figure2_split():
    """METAL MEDIA Figure 2: 12 routed, 8 hits, m=4, one fill, three on the CPU."""
    st = ctl.CacheState.empty(1, 16, 16)
    ctl.route_ctl(st, 0, [list(range(8))], 1.0, 1.0)            # warm 8 experts (q = m)
    r = ctl.route_ctl(st, 0, [list(range(12))], 1.0, 4.0)
    ctl.check_invariants(st, r)
    assert len(r.hits) == 8 and len(r.misses) == 4
    assert r.q == 1 and len(r.F) == 1 and len(r.C) == 3


def test_topk_route_bruteforce():
    rng = random.Random(3)
    import itertools
    import math
    for _ in range(200):
        E = rng.randint(2, 6)
        k = rng.randint(1, E)
        # small integer-valued logits make ties frequent
        logits = [float(rng.randint(-2, 2)) for _ in range(E)]
        ids, gates = ctl.topk_route(logits, k)
        best = None
        for perm in itertools.permutations(range(E), k):
            key = tuple((-logits[e], e) for e in perm)
            if list(key) == sorted(key) and (best is None or key < best[0]):
                best = (key, list(perm))
        assert ids == best[1]
        assert abs(sum(gates) - 1.0) < 1e-15
        ex = [math.exp(logits[e]) for e in ids]
        for g, v in zip(gates, ex):
            assert abs(g - v / sum(ex)) < 1e-15


class ListLRU:
    """Independent model: slots kept in an explicit least-recent-first list.

    Empty slots (never filled, or cleared by a prefill buffer) sit at the
    front in slot order; every slot touched by a call (its hits and its fills)
    moves to the back, the touched ones in slot order among themselves.
    """

    def __init__(self, L, E, S):
        self.L, self.E, self.S = L, E, S
        self.owner = {}          # slot -> flat id
        self.where = {}          # flat id -> slot
        self.empty = set(range(S))
        self.recency = []        # occupied slots, least recent first

    def order(self):
        return sorted(self.empty) + self.recency

    def call(self, layer, routes, BP, BH):
        E = self.E
        counts = {}
        for row in routes:
            for e in row:
                counts[e] = counts.get(e, 0) + 1
        hits = sorted(e for e in counts if layer * E + e in self.where)
        misses = [e for e in counts if layer * E + e not in self.where]
        m = len(misses)
        if m:
            x = Fraction(m) * Fraction(str(BP)) / Fraction(str(BH))
            q = int(x) + (1 if x - int(x) >= Fraction(1, 2) else 0)
            q = min(max(q, 1), m, self.S - len(hits))
        else:
            q = 0
        misses.sort(key=lambda e: (-counts[e], e))
        F = misses[:q]
        hit_slots = {self.where[layer * E + e] for e in hits}
        victims = [s for s in self.order() if s not in hit_slots][:q]
        for f, s in zip(F, victims):
            if s in self.owner:
                del self.where[self.owner[s]]
            self.owner[s] = layer * E + f
            self.where[layer * E + f] = s
            self.empty.discard(s)
        touched = hit_slots | set(victims)
        self.recency = [s for s in self.recency if s not in touched] + sorted(touched)
        return victims

    def clear_buffer(self, b):
        for s in range(b * self.E, (b + 1) * self.E):
            if s in self.owner:
                del self.where[self.owner.pop(s)]
            self.empty.add(s)
        self.recency = [s for s in self.recency if s not in self.empty]

    def resize(self, S_new):
        if S_new >= self.S:
            self.empty |= set(range(self.S, S_new))
            self.S = S_new
            return
        keep = self.recency[-S_new:] if S_new else []
        keep_sorted = sorted(keep)
        rename = {s: i for i, s in enumerate(keep_sorted)}
        new_owner = {rename[s]: self.owner[s] for s in keep}
        self.owner = new_owner
        self.where = {fid: s for s, fid in new_owner.items()}
        self.recency = [rename[s] for s in keep]
        self.empty = set(range(len(keep), S_new))
        self.S = S_new


def _state_matches(st, model):
    assert st.S == model.S
    for s in range(st.S):
        assert st.id_for_slot[s] == model.owner.get(s, ctl.EMPTY)
    # the stamp order equals the list order
    by_stamp = sorted(range(st.S), key=lambda s: (st.stamp[s], s))
    assert by_stamp == model.order()


@pytest.mark.parametrize("seed", range(6))
def test_random_sequences_match_list_model(seed):
    rng = random.Random(seed)
    L, E = 3, 8
    S = rng.choice([1, 2, 3, 5, 16, 20])
    st = ctl.CacheState.empty(L, E, S)
    model = ListLRU(L, E, S)
    for call in range(300):
        op = rng.random()
        if op < 0.05 and st.S >= 2 * E:
            b = rng.randint(0, 1)
            ctl.prefill_invalidate(st, b)
            model.clear_buffer(b)
        elif op < 0.09:
            S_new = rng.randint(1, 24)
            ctl.resize(st, S_new)
            model.resize(S_new)
        else:
            layer = rng.randrange(L)
            T = rng.randint(1, 4)
            k = rng.randint(1, 4)
            routes = [rng.sample(range(E), k) for _ in range(T)]
            BP = rng.choice([1.0, 25.0, 52.7, 90.0])
            BH = rng.choice([90.0, 120.0, 4.0, 52.7])
            if BH < BP:
                BP, BH = BH, BP
            r = ctl.route_ctl(st, layer, routes, BP, BH)
            ctl.check_invariants(st, r)
            v = model.call(layer, routes, BP, BH)
            assert r.victims == v
        ctl.check_invariants(st)
        _state_matches(st, model)


def test_hostile_sequence_control():
    """deepmox "How residency follows demand": a request uses layer-0 experts,
    prefill materialises other layers into every slot, the request returns:
    every route must miss (no stale hit on another layer's bytes)."""
    L, E = 4, 8
    st = ctl.CacheState.empty(L, E, 2 * E)
    routes = [[1, 2], [3, 4]]
    r = ctl.route_ctl(st, 0, routes, 1.0, 1.0)
    assert r.q == 4
    r = ctl.route_ctl(st, 0, routes, 1.0, 1.0)
    assert len(r.hits) == 4 and r.q == 0
    for layer in range(L):
        ctl.prefill_invalidate(st, layer & 1)
    ctl.check_invariants(st)
    assert all(s == ctl.EMPTY for s in st.slot_for_id)
    r = ctl.route_ctl(st, 0, routes, 1.0, 1.0)
    assert r.hits == [] and r.q == 4


def test_resize_keeps_most_recent_and_packs():
    st = ctl.CacheState.empty(1, 16, 8)
    for step in range(8):
        ctl.route_ctl(st, 0, [[step]], 1.0, 1.0)              # expert `step` lands in slot `step`, stamp step+1
    ctl.route_ctl(st, 0, [[0]], 1.0, 1.0)                      # refresh expert 0 -> most recent
    moves = ctl.resize(st, 3)
    ctl.check_invariants(st)
    # kept: expert 0 (stamp 9), 7 (stamp 8), 6 (stamp 7); packed in old-slot order
    assert st.id_for_slot == [0, 6, 7]
    assert moves == [(0, 0), (6, 1), (7, 2)]
    assert st.stamp == [9, 7, 8]
    assert st.slot_for_id[:8] == [0, -1, -1, -1, -1, -1, 1, 2]
    ctl.resize(st, 6)
    assert st.id_for_slot == [0, 6, 7, -1, -1, -1] and st.stamp[3:] == [0, 0, 0]
    assert st.clock == 9
