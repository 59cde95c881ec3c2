"""float64 expert arithmetic of the MoE layer (test infrastructure only).

What is computed (FreeToken pages):
  * an expert is a gate/up projection plus a down projection (deepmox, "One
    logical expert, two physical levels of memory"); the expert FFN is the
    SwiGLU form FFN(x) = W_d (SiLU(W_g x) * (W_u x)), SiLU(a) = a / (1 + e^-a);
  * the layer output of token t is the gate-weighted sum of the FFNs of its
    top-k experts; the GPU part (hits and fills) and the CPU part (set C) are
    partial sums that merge exactly (METAL MEDIA page, Figure 2 caption;
    explainer section 14, "merge");
  * whether an expert ran on the GPU or the CPU, and how large the cache is,
    does not change the output (explainer section 11; deepmox "the cache does
    not need to be perfect to preserve model semantics").

Inputs arrive as bf16 bit patterns (uint16) and are widened exactly to
float64; all arithmetic is float64.  Readings: the CPU-set partial sum
partial_C is the float32 rounding of its float64 value (it is a float32
buffer handed to the GPU), and y is returned in float64.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def silu(a: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def expert_ffn(Wg, Wu, Wd, x) -> np.ndarray:
    """SwiGLU FFN of one expert for a batch of tokens.

    Wg, Wu: [F, H]; Wd: [H, F]; x: [n, H] (all float64).  Returns [n, H].
    """
    a = x @ Wg.T
    b = x @ Wu.T
    return (silu(a) * b) @ Wd.T


def gated_sum(x, ids, gates, select, weights) -> np.ndarray:
    """sum_{j : select(t, j)} g_tj * FFN_{e_tj}(x_t) for every token t, float64 [T, H].

    ``weights(e)`` returns float64 (Wg, Wu, Wd) of expert e of this layer.
    ``select(t, j)`` picks the routes that belong to this partial sum.
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    y = np.zeros((T, H), dtype=np.float64)
    by_expert: dict = {}
    for t in range(T):
        for j, e in enumerate(ids[t]):
            if select(t, j):
                by_expert.setdefault(int(e), []).append((t, j))
    for e, routes in by_expert.items():
        Wg, Wu, Wd = weights(e)
        toks = [t for t, _ in routes]
        out = expert_ffn(Wg, Wu, Wd, x[toks])
        for (t, j), o in zip(routes, out):
            y[t] += gates[t][j] * o
    return y


def moe_layer_split(x, ids, gates, slots_topk, weights):
    """GPU and CPU partial sums of one decode layer after a control pass.

    A route (t, j) runs on the GPU when the control pass gave it a slot
    (hit or fill) and on the CPU when its expert is in C (slot -1).
    Returns (y_gpu float64 [T,H], partial_C float32 [T,H]).
    """
    y_gpu = gated_sum(x, ids, gates, lambda t, j: slots_topk[t][j] >= 0, weights)
    y_cpu = gated_sum(x, ids, gates, lambda t, j: slots_topk[t][j] < 0, weights)
    return y_gpu, y_cpu.astype(np.float32)


def merged_output(y_gpu, partial_C) -> np.ndarray:
    """Exact merge: y = GPU partial sum + the supplied CPU partial sum (float64)."""
    return np.asarray(y_gpu, dtype=np.float64) + np.asarray(partial_C, dtype=np.float32).astype(np.float64)


def dense_masked_bruteforce(x, mask, gate_matrix, weights_list) -> np.ndarray:
    """y_t = sum_e mask[t][e] * g[t][e] * FFN_e(x_t), with plain Python loops.

    Written with no numpy linear algebra so that it shares nothing with
    ``expert_ffn``; for tiny sizes only.  weights_list[e] = (Wg, Wu, Wd) as
    nested float lists or arrays.
    """
    import math
    T = len(x)
    H = len(x[0])
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        xt = [float(v) for v in x[t]]
        for e, (Wg, Wu, Wd) in enumerate(weights_list):
            if not mask[t][e]:
                continue
            F = len(Wg)
            hvec = []
            for f in range(F):
                a = 0.0
                b = 0.0
                rg = Wg[f]
                ru = Wu[f]
                for i in range(H):
                    a += float(rg[i]) * xt[i]
                    b += float(ru[i]) * xt[i]
                hvec.append(a / (1.0 + math.exp(-a)) * b)
            g = float(gate_matrix[t][e])
            for o in range(H):
                rd = Wd[o]
                acc = 0.0
                for f in range(F):
                    acc += float(rd[f]) * hvec[f]
                y[t][o] += g * acc
    return np.array(y, dtype=np.float64)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def record_weights_bf16(record, H: int, F: int):
    """(Wg [F,H], Wu [F,H], Wd [H,F]) float64 read from one BF16 record's bytes.

    Layout (the library's record definition): bank W_gu [2F, H] row-major with
    gate and up rows interleaved in groups of 16 (16 gate rows, then the 16
    matching up rows), then bank W_d [H, F] row-major.
    """
    r16 = np.asarray(record, dtype=np.uint8).view(np.uint16)
    assert r16.size == 3 * H * F
    gu = bf16_to_f64(r16[:2 * F * H]).reshape(F // 16, 2, 16, H)
    Wg = gu[:, 0].reshape(F, H)
    Wu = gu[:, 1].reshape(F, H)
    Wd = bf16_to_f64(r16[2 * F * H:]).reshape(H, F)
    return Wg, Wu, Wd
