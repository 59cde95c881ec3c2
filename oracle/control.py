"""Exact-integer control oracle of the expert cache (test infrastructure only).

Sources (FreeToken pages):
  * explainer "FreeToken: Making Large MoE Models Practical on a Single
    Machine", sections 4-7 (the q* split), 8 (global LRU), 10 (device-side
    dedup / classify / q / victims / rewrite), 11 (resize, host pool is the
    source of truth);
  * deepmox chapter "The Expert Cache That Follows the Router", sections
    "One logical expert, two physical levels of memory" (flat id, slot_for_id
    and the reverse map, prefill buffers invalidate owners) and "How residency
    follows demand without leaving the device" (dedup, hits refresh recency,
    victims, in-place rewrite to slots, CPU execution does not warm the cache);
  * txtmix write-up, section "miss 的去向不能拍脑袋" (always at least one fill;
    q -> m as B_H -> B_P) and "CUDA-graph 兼容的 LRU 缓存" (one scan yields the
    K least-recently-used candidates, the miss path takes the first q <= K).

Readings taken where the pages are silent (each is also stated where used):
  R1 top-k order: logit descending, lower expert id first on equal logits.
  R2 q0 = round((m*B_P)/B_H) in float64, in that order, rounding half away
     from zero.
  R3 capacity clamp: q = min(clamp(q0, 1, m), S - h); hits are never evicted.
  R4 fill order: misses by routed-token count descending, lower id first.
  R5 LRU encoding: a clock incremented at the start of every control call;
     hits and fills get stamp = clock; empty slots have stamp 0; victims are
     the q smallest (stamp, slot) among slots that do not hold a hit; the i-th
     fill expert goes to the i-th victim.
  R6 resize: shrinking evicts occupied entries in the victim-scan order
     (smallest (stamp, slot) first) until min(S', occupied) remain, and packs
     the survivors, in ascending old slot order, into slots 0..n-1; growing
     keeps every slot index; stamps and clock are kept.
  R7 prefill: the i-th layer of a prefill chunk is copied into buffer
     b = i & 1 (slots [b*E, (b+1)*E)); before the copy every owner of those
     slots is cleared, and the slots are left empty with stamp 0 after the
     prefill.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from fractions import Fraction

EMPTY = -1


# ------------------------------------------------------------------ routing

def topk_route(logits_row, k: int):
    """Top-k experts of one token and their gates.

    The router picks k of E experts per token (explainer section 1, "token t ->
    router -> Expert 3, 7, 12, 18"); the gate weights are the softmax over the
    k selected logits.  Reading R1: order by logit descending, lower expert id
    first on equal logits; logits compared exactly as the float32 values given.
    Gates are computed in float64.
    Returns (ids: list[int], gates: list[float]).
    """
    vals = [float(v) for v in logits_row]
    order = sorted(range(len(vals)), key=lambda e: (-vals[e], e))[:k]
    top = [vals[e] for e in order]
    mx = max(top)
    ex = [math.exp(v - mx) for v in top]
    s = sum(ex)
    return order, [v / s for v in ex]


# ----------------------------------------------------------------------- q

def round_half_away(x: float) -> int:
    """Round a non-negative float to the nearest integer, halves away from zero."""
    assert x >= 0.0
    f = math.floor(x)
    return int(f) + 1 if x - f >= 0.5 else int(f)


def round_half_away_exact(x: Fraction) -> int:
    assert x >= 0
    f = math.floor(x)
    return f + 1 if x - f >= Fraction(1, 2) else f


@dataclass
class FillCount:
    q0: int          # round(m * B_P / B_H)
    q1: int          # at-least-one-fill clamp to [1, m]
    q: int           # after the capacity clamp (reading R3)
    q0_exact: int    # q0 recomputed in exact rationals from the decimal B_P, B_H


def fill_count(m: int, h: int, S: int, B_P: float, B_H: float) -> FillCount:
    """Number of misses to fill into the GPU cache.

    Explainer section 5 "Deriving q*": equating the fill time q*S/B_P with the
    CPU time (m-q)*S/(B_H-B_P) gives q* = m*B_P/B_H.  txtmix write-up: at least
    one fill is always kept, and q -> m as B_H -> B_P.  Reading R2 (float64
    (m*B_P)/B_H, halves away from zero) and R3 (no more fills than slots not
    holding a hit of this call).
    """
    if m == 0:
        return FillCount(0, 0, 0, 0)
    x = (float(m) * float(B_P)) / float(B_H)
    q0 = round_half_away(x)
    q0e = round_half_away_exact(Fraction(m) * Fraction(str(B_P)) / Fraction(str(B_H)))
    q1 = min(max(q0, 1), m)
    q = min(q1, S - h)
    return FillCount(q0=q0, q1=q1, q=max(q, 0), q0_exact=q0e)


# ------------------------------------------------------------- cache state

@dataclass
class CacheState:
    """Residency maps and recency of the all-layer slot cache.

    deepmox "One logical expert...": flat id = layer*E + expert;
    slot_for_id answers where a flat id lives, id_for_slot (the pages'
    id_of_slot) which flat id owns a slot.  Stamps and clock: reading R5.
    """
    L: int
    E: int
    S: int
    slot_for_id: list = field(default_factory=list)
    id_for_slot: list = field(default_factory=list)
    stamp: list = field(default_factory=list)
    clock: int = 0

    @classmethod
    def empty(cls, L: int, E: int, S: int) -> "CacheState":
        return cls(L, E, S, [EMPTY] * (L * E), [EMPTY] * S, [0] * S, 0)

    def copy(self) -> "CacheState":
        return CacheState(self.L, self.E, self.S, list(self.slot_for_id), list(self.id_for_slot),
                          list(self.stamp), self.clock)


@dataclass
class CtlResult:
    layer: int
    clock: int
    counts: dict            # expert -> routed-token count n_e (unique experts U)
    hits: list              # experts resident before the call, ascending id
    misses: list            # ascending id
    fc: FillCount
    F: list                 # fill experts, fill order (reading R4)
    C: list                 # CPU-set experts, same order
    victims: list           # slots, ascending (stamp, slot)
    evicted: list           # flat id that owned each victim (EMPTY if none)
    slots_topk: list        # [T][k] slot of each route, EMPTY for C

    @property
    def q(self) -> int:
        return self.fc.q


def route_ctl(state: CacheState, layer: int, topk_ids, B_P: float, B_H: float) -> CtlResult:
    """One control pass for one MoE layer, updating ``state`` in place.

    deepmox "How residency follows demand without leaving the device": the
    routed ids are reduced to unique layer-experts; each is looked up in the
    residency row (resident = hit); hits refresh recency; victims are chosen
    for the misses that will be fetched; the route ids are rewritten to slots.
    Explainer section 4 / Figure 2 of the METAL MEDIA page: the misses split
    into the fill set F (copied into slots and run on the GPU) and the CPU set
    C (run from the host pool; deepmox: it does not change GPU residency).
    Readings R3, R4, R5 apply.
    """
    E, S = state.E, state.S
    assert 0 <= layer < state.L
    state.clock += 1
    clk = state.clock
    counts: dict = {}
    for row in topk_ids:
        assert len(set(int(e) for e in row)) == len(row), "duplicate expert within a token"
        for e in row:
            e = int(e)
            assert 0 <= e < E
            counts[e] = counts.get(e, 0) + 1
    U = sorted(counts)
    hits = [e for e in U if state.slot_for_id[layer * E + e] != EMPTY]
    misses = [e for e in U if state.slot_for_id[layer * E + e] == EMPTY]
    fc = fill_count(len(misses), len(hits), S, B_P, B_H)
    order = sorted(misses, key=lambda e: (-counts[e], e))
    F, C = order[:fc.q], order[fc.q:]

    hit_slots = set()
    for e in hits:
        s = state.slot_for_id[layer * E + e]
        hit_slots.add(s)
        state.stamp[s] = clk
    cand = sorted((state.stamp[s], s) for s in range(S) if s not in hit_slots)
    victims = [s for _, s in cand[:fc.q]]
    assert len(victims) == fc.q

    evicted = []
    for f, s in zip(F, victims):
        o = state.id_for_slot[s]
        evicted.append(o)
        if o != EMPTY:
            state.slot_for_id[o] = EMPTY
        fid = layer * E + f
        state.id_for_slot[s] = fid
        state.slot_for_id[fid] = s
        state.stamp[s] = clk

    Cset = set(C)
    slots_topk = [[EMPTY if int(e) in Cset else state.slot_for_id[layer * E + int(e)] for e in row]
                  for row in topk_ids]
    return CtlResult(layer, clk, counts, hits, misses, fc, F, C, victims, evicted, slots_topk)


def check_invariants(state: CacheState, res: CtlResult | None = None) -> None:
    """Invariants that hold after every control call (raises AssertionError)."""
    E, S = state.E, state.S
    for s in range(S):
        o = state.id_for_slot[s]
        if o != EMPTY:
            assert 0 <= o < state.L * E
            assert state.slot_for_id[o] == s, f"slot {s} owner {o} maps to {state.slot_for_id[o]}"
            assert 0 <= state.stamp[s] <= state.clock
    for fid, s in enumerate(state.slot_for_id):
        if s != EMPTY:
            assert 0 <= s < S and state.id_for_slot[s] == fid
    if res is None:
        return
    U = set(res.counts)
    assert set(res.hits) | set(res.F) | set(res.C) == U
    assert len(res.hits) + len(res.F) + len(res.C) == len(U)
    assert len(res.F) == res.q == len(res.victims)
    assert len(set(res.victims)) == len(res.victims)
    l = res.layer
    hit_slots = {state.slot_for_id[l * E + e] for e in res.hits}
    assert not (hit_slots & set(res.victims)), "a victim held a hit"
    for e in list(res.hits) + list(res.F):
        s = state.slot_for_id[l * E + e]
        assert s != EMPTY and state.stamp[s] == res.clock
    for e in res.C:
        assert state.slot_for_id[l * E + e] == EMPTY
    if len(res.misses) >= 1 and state.S - len(res.hits) >= 1:
        assert res.q >= 1, "at least one fill"


# ------------------------------------------------------------------ resize

def resize(state: CacheState, S_new: int):
    """Rebuild the slot cache for a new slot count (reading R6).

    Explainer section 11 and the txtmix section on "ft ctl cache": the cache is
    rebuilt for a new VRAM budget at a safe point; the host pool stays the
    source of truth, so dropped entries only turn into later misses.
    Returns the list of (old_slot, new_slot) moves of the kept records.
    """
    assert S_new >= 1
    moves = []
    if S_new >= state.S:
        grow = S_new - state.S
        state.id_for_slot += [EMPTY] * grow
        state.stamp += [0] * grow
        state.S = S_new
        return moves
    occ = [s for s in range(state.S) if state.id_for_slot[s] != EMPTY]
    lru_first = sorted(occ, key=lambda s: (state.stamp[s], s))
    keep = lru_first[max(0, len(occ) - S_new):]
    keep_set = set(keep)
    for s in occ:
        if s not in keep_set:
            state.slot_for_id[state.id_for_slot[s]] = EMPTY
    new_ids = [EMPTY] * S_new
    new_stamp = [0] * S_new
    for ns, s in enumerate(sorted(keep)):
        fid = state.id_for_slot[s]
        new_ids[ns] = fid
        new_stamp[ns] = state.stamp[s]
        state.slot_for_id[fid] = ns
        moves.append((s, ns))
    state.id_for_slot, state.stamp, state.S = new_ids, new_stamp, S_new
    return moves


# ----------------------------------------------------------------- prefill

def prefill_invalidate(state: CacheState, buffer: int) -> None:
    """Clear the owners of prefill buffer ``buffer`` (reading R7).

    deepmox: the two full-layer buffers are the first two expert-layer regions
    of the slot pool; when a layer is copied into one, the previous owners of
    those slots are invalidated and their slot_for_id entries cleared, and the
    recency is cleared so decode does not treat volatile contents as entries.
    """
    E = state.E
    assert state.S >= 2 * E and buffer in (0, 1)
    for s in range(buffer * E, (buffer + 1) * E):
        o = state.id_for_slot[s]
        if o != EMPTY:
            state.slot_for_id[o] = EMPTY
        state.id_for_slot[s] = EMPTY
        state.stamp[s] = 0


def prefill_routes(logits, k: int):
    """Top-k ids/gates of every token plus the expert-sorted assignment order.

    The assignments (t, j) are ordered by expert, then token (stable counting
    sort); offsets[e] is the first assignment of expert e.
    """
    ids, gates = [], []
    for row in logits:
        i, g = topk_route(row, k)
        ids.append(i)
        gates.append(g)
    E = len(logits[0])
    counts = [0] * E
    for row in ids:
        for e in row:
            counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    return ids, gates, offsets
