"""Seeded synthetic inputs for the expert-cache MoE layer.

This module is shared by the oracle, the tests and the benchmark.  It holds
no arithmetic of the method itself (no routing, no cache control, no expert
FFN): only random draws, the bf16 / NVFP4 / MXFP4 / block-FP8 encodings of the drawn weights and
the byte layout of one expert record in the host pool.

Random streams: numpy ``PCG64`` seeded by ``SeedSequence([seed, tag, ...])``
so that any tensor (one expert record, the logits of one layer, the tokens of
one step) can be regenerated on its own, without materialising the others.

Workload recipe (FreeToken, "The Expert Cache That Follows the Router", and
the explainer's section 3 "Decode: Exploit Expert Locality"): decode routing
has short-range temporal locality, which an AR(1) process over the router
logits stands in for, one independent chain per (layer, token lane):
``l_0 ~ N(0,1)``, ``l_t = rho*l_{t-1} + sigma*eps_t``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

# Stream tags (first word after the seed in every SeedSequence).
TAG_WEIGHTS = 1
TAG_LOGITS = 2
TAG_X = 3
TAG_PARTIAL_C = 4
TAG_TOPK = 5

FMT_BF16 = 0
FMT_NVFP4 = 1
FMT_MXFP4 = 2
FMT_FP8 = 3

# Record layout: gate and up rows are interleaved in groups of this many rows
# (16 gate rows, then the 16 matching up rows, ...).
GU_INTERLEAVE = 16
# NVFP4: one e4m3 scale per this many consecutive values along K.
NVFP4_BLOCK = 16
# MXFP4: one E8M0 (power-of-two) scale per this many consecutive values along K.
MXFP4_BLOCK = 32
# Block-FP8: one fp32 scale per FP8_BLOCK x FP8_BLOCK block (rows x K) of each matrix.
FP8_BLOCK = 128


@dataclass(frozen=True)
class Shape:
    """Sizes of one MoE layer family (names follow the pages' notation)."""
    L: int   # MoE layers
    E: int   # experts per layer
    k: int   # top-k
    H: int   # hidden size
    F: int   # expert ffn size
    fmt: int = FMT_BF16

    @property
    def record_bytes(self) -> int:
        return record_bytes(self.H, self.F, self.fmt)


def record_bytes(H: int, F: int, fmt: int) -> int:
    """Bytes of one complete layer-expert record (all banks of one expert)."""
    n = 3 * H * F
    if fmt == FMT_BF16:
        return 2 * n
    if fmt == FMT_NVFP4:
        return n // 2 + n // NVFP4_BLOCK
    if fmt == FMT_MXFP4:
        return n // 2 + n // MXFP4_BLOCK
    if fmt == FMT_FP8:
        return n + 4 * 3 * (H // FP8_BLOCK) * (F // FP8_BLOCK)
    raise ValueError(f"unknown format {fmt}")


# ---------------------------------------------------------------- bf16 bits

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(w) for w in words])))


# ------------------------------------------------------------- BF16 experts

def expert_weights_bf16(seed: int, layer: int, expert: int, H: int, F: int):
    """Logical weights of one layer-expert as bf16 bit patterns.

    Returns (Wg [F,H], Wu [F,H], Wd [H,F]) uint16, each element
    bf16(0.02 * N(0,1)) drawn in that order from the record's own stream.
    """
    rng = _rng(seed, TAG_WEIGHTS, layer, expert)
    w = rng.standard_normal(3 * H * F, dtype=np.float32)
    w *= np.float32(0.02)
    b = f32_to_bf16_bits(w)
    n = H * F
    return b[:n].reshape(F, H), b[n:2 * n].reshape(F, H), b[2 * n:].reshape(H, F)


def pack_record_bf16(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Byte image of one BF16 record.

    Layout: bank W_gu [2F, H] row-major (K = H contiguous) whose rows are gate
    and up rows interleaved in groups of GU_INTERLEAVE, then bank W_d [H, F]
    row-major (K = F contiguous).
    """
    F, H = Wg.shape
    g = GU_INTERLEAVE
    assert F % g == 0
    gu = np.empty((F // g, 2, g, H), dtype=np.uint16)
    gu[:, 0] = Wg.reshape(F // g, g, H)
    gu[:, 1] = Wu.reshape(F // g, g, H)
    nb = record_bytes(H, F, FMT_BF16)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    o16 = out.view(np.uint16)
    o16[: 2 * F * H] = gu.reshape(-1)
    o16[2 * F * H:] = Wd.reshape(-1)
    return out


def record_bf16(seed: int, layer: int, expert: int, H: int, F: int, out=None) -> np.ndarray:
    return pack_record_bf16(*expert_weights_bf16(seed, layer, expert, H, F), out=out)


# ------------------------------------------------------------ NVFP4 experts
# Encoding of the drawn weights into NVFP4 (input preparation, done once):
#   per expert global  gs = amax|W| / (6 * 448)   (all three matrices)
#   per block of 16 along K:  s = e4m3(amax_block / (6 * gs))
#   values:  v = e2m1(w / (s_dec * gs))
# e2m1 / e4m3 rounding is round-to-nearest-even with saturation, written
# from the OCP microscaling formats' definitions.

_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _e4m3_table() -> np.ndarray:
    vals = np.zeros(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 7
        if e == 0xF and m == 7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = _e4m3_table()
_E4M3_POS = _E4M3[:127]  # codes 0..126: 0 .. 448 ascending


def _rne_to_grid(x: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to |x| (grid ascending, non-negative);
    ties go to the even index (the even code); saturates at the top."""
    ax = np.minimum(np.abs(x), grid[-1])
    hi = np.searchsorted(grid, ax, side="left")
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    dlo = ax - grid[lo]
    dhi = grid[hi] - ax
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """float -> 4-bit e2m1 code (sign in bit 3)."""
    idx = _rne_to_grid(x, _E2M1_GRID).astype(np.uint8)
    sign = (np.signbit(x) & (idx != 0)).astype(np.uint8) << 3
    return idx | sign


def encode_e4m3_pos(x: np.ndarray) -> np.ndarray:
    """non-negative float -> e4m3 code (0..126), RNE with saturation to 448."""
    return _rne_to_grid(x, _E4M3_POS).astype(np.uint8)


def quantize_nvfp4(W: np.ndarray, gs: float):
    """W [rows, K] float -> (codes uint8 [rows, K], scale codes uint8 [rows, K/16])."""
    rows, K = W.shape
    Wb = W.reshape(rows, K // NVFP4_BLOCK, NVFP4_BLOCK).astype(np.float64)
    amax = np.abs(Wb).max(axis=2)
    sc = encode_e4m3_pos(amax / (6.0 * gs))
    sdec = _E4M3[sc]
    denom = sdec * gs
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(denom[..., None] > 0, Wb / denom[..., None], 0.0)
    codes = encode_e2m1(v).reshape(rows, K)
    return codes, sc


def _pack_nibbles(codes: np.ndarray) -> np.ndarray:
    c = codes.reshape(-1)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def expert_nvfp4(seed: int, layer: int, expert: int, H: int, F: int):
    """NVFP4 encoding of one layer-expert drawn like the BF16 weights.

    Returns dict with e2m1 codes (uint8, one per value), e4m3 scale codes and
    the fp32 global, for gate [F,H], up [F,H] and down [H,F].
    """
    rng = _rng(seed, TAG_WEIGHTS, layer, expert)
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    n = H * F
    Wg, Wu, Wd = w[:n].reshape(F, H), w[n:2 * n].reshape(F, H), w[2 * n:].reshape(H, F)
    gs = float(np.float32(np.abs(w).max() / np.float32(6.0 * 448.0)))
    out = {"global": np.float32(gs)}
    for name, W in (("g", Wg), ("u", Wu), ("d", Wd)):
        codes, sc = quantize_nvfp4(W, gs)
        out[name] = codes
        out[name + "_scale"] = sc
    return out


def pack_record_nvfp4(q: dict, out: np.ndarray | None = None) -> np.ndarray:
    """Byte image of one NVFP4 record.

    Layout: [W_gu values: 2F x H e2m1, two per byte, low nibble first, rows
    interleaved in groups of GU_INTERLEAVE like the BF16 bank]
    [W_d values: H x F, same packing]
    [W_gu scales: 2F x H/16 e4m3, same row order] [W_d scales: H x F/16 e4m3].
    The fp32 global is not part of the record (it stays device-resident).
    """
    F, H = q["g"].shape
    g = GU_INTERLEAVE
    gu = np.empty((F // g, 2, g, H), dtype=np.uint8)
    gu[:, 0] = q["g"].reshape(F // g, g, H)
    gu[:, 1] = q["u"].reshape(F // g, g, H)
    gus = np.empty((F // g, 2, g, H // NVFP4_BLOCK), dtype=np.uint8)
    gus[:, 0] = q["g_scale"].reshape(F // g, g, -1)
    gus[:, 1] = q["u_scale"].reshape(F // g, g, -1)
    parts = [_pack_nibbles(gu), _pack_nibbles(q["d"]), gus.reshape(-1), q["d_scale"].reshape(-1)]
    nb = record_bytes(H, F, FMT_NVFP4)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    off = 0
    for p in parts:
        out[off:off + p.size] = p
        off += p.size
    assert off == nb
    return out


def record_nvfp4(seed: int, layer: int, expert: int, H: int, F: int, out=None):
    """(record bytes, fp32 global) of one NVFP4 layer-expert."""
    q = expert_nvfp4(seed, layer, expert, H, F)
    return pack_record_nvfp4(q, out=out), q["global"]


# ------------------------------------------------------------ MXFP4 experts
# Encoding of the drawn weights into MXFP4 (OCP Microscaling v1.0 conversion):
# per block of 32 along K the shared exponent is floor(log2 amax) - 2 (2 being
# the largest e2m1 exponent), clamped to [-127, 127], stored biased by 127 in
# one E8M0 byte; values are e2m1(w / 2^exponent), round to nearest even with
# saturation.  An all-zero block takes exponent -127.

def quantize_mxfp4(W: np.ndarray):
    """W [rows, K] float -> (codes uint8 [rows, K], E8M0 codes uint8 [rows, K/32])."""
    rows, K = W.shape
    Wb = W.reshape(rows, K // MXFP4_BLOCK, MXFP4_BLOCK).astype(np.float64)
    amax = np.abs(Wb).max(axis=2)
    _, ex = np.frexp(amax)              # amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    se = np.where(amax > 0, ex - 1 - 2, -127)
    se = np.clip(se, -127, 127).astype(np.int64)
    v = Wb / np.ldexp(1.0, se)[..., None]
    codes = encode_e2m1(v).reshape(rows, K)
    return codes, (se + 127).astype(np.uint8)


def expert_mxfp4(seed: int, layer: int, expert: int, H: int, F: int):
    """MXFP4 encoding of one layer-expert drawn like the BF16 weights: e2m1
    codes and E8M0 scale codes of gate [F,H], up [F,H] and down [H,F]."""
    rng = _rng(seed, TAG_WEIGHTS, layer, expert)
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    n = H * F
    out = {}
    for name, W in (("g", w[:n].reshape(F, H)), ("u", w[n:2 * n].reshape(F, H)), ("d", w[2 * n:].reshape(H, F))):
        codes, sc = quantize_mxfp4(W)
        out[name] = codes
        out[name + "_scale"] = sc
    return out


def pack_record_mxfp4(q: dict, out: np.ndarray | None = None) -> np.ndarray:
    """Byte image of one MXFP4 record: the NVFP4 layout with E8M0 block-32
    scales in place of the e4m3 block-16 ones, and no global.

    [W_gu values: 2F x H e2m1, two per byte, low nibble first, rows
    interleaved in groups of GU_INTERLEAVE] [W_d values: H x F]
    [W_gu scales: 2F x H/32, same row order] [W_d scales: H x F/32].
    """
    F, H = q["g"].shape
    g = GU_INTERLEAVE
    gu = np.empty((F // g, 2, g, H), dtype=np.uint8)
    gu[:, 0] = q["g"].reshape(F // g, g, H)
    gu[:, 1] = q["u"].reshape(F // g, g, H)
    gus = np.empty((F // g, 2, g, H // MXFP4_BLOCK), dtype=np.uint8)
    gus[:, 0] = q["g_scale"].reshape(F // g, g, -1)
    gus[:, 1] = q["u_scale"].reshape(F // g, g, -1)
    parts = [_pack_nibbles(gu), _pack_nibbles(q["d"]), gus.reshape(-1), q["d_scale"].reshape(-1)]
    nb = record_bytes(H, F, FMT_MXFP4)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    off = 0
    for p in parts:
        out[off:off + p.size] = p
        off += p.size
    assert off == nb
    return out


def record_mxfp4(seed: int, layer: int, expert: int, H: int, F: int, out=None) -> np.ndarray:
    """Record bytes of one MXFP4 layer-expert."""
    return pack_record_mxfp4(expert_mxfp4(seed, layer, expert, H, F), out=out)


# --------------------------------------------------------- block-FP8 experts
# Encoding of the drawn weights into block-FP8: per 128 x 128 block the fp32
# scale amax / 448 (1 for an all-zero block), values e4m3(w / scale) rounded
# to nearest even with saturation at 448.

def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float -> signed e4m3 code (sign in bit 7), RNE, saturating at 448."""
    idx = encode_e4m3_pos(x)
    sign = (np.signbit(x) & (idx != 0)).astype(np.uint8) << 7
    return idx | sign


def quantize_fp8(W: np.ndarray):
    """W [rows, K] float32 -> (codes uint8 [rows, K], scales float32 [rows/128, K/128])."""
    rows, K = W.shape
    b = FP8_BLOCK
    Wb = np.asarray(W, dtype=np.float32).reshape(rows // b, b, K // b, b)
    amax = np.abs(Wb).max(axis=(1, 3))
    sc = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    v = Wb.astype(np.float64) / sc.astype(np.float64)[:, None, :, None]
    return encode_e4m3(v).reshape(rows, K), sc


def expert_fp8(seed: int, layer: int, expert: int, H: int, F: int):
    """Block-FP8 encoding of one layer-expert drawn like the BF16 weights: e4m3
    codes and fp32 block scales of gate [F,H], up [F,H] and down [H,F]."""
    rng = _rng(seed, TAG_WEIGHTS, layer, expert)
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    n = H * F
    out = {}
    for name, W in (("g", w[:n].reshape(F, H)), ("u", w[n:2 * n].reshape(F, H)), ("d", w[2 * n:].reshape(H, F))):
        codes, sc = quantize_fp8(W)
        out[name] = codes
        out[name + "_scale"] = sc
    return out


def pack_record_fp8(q: dict, out: np.ndarray | None = None) -> np.ndarray:
    """Byte image of one block-FP8 record.

    [W_gu values: 2F x H e4m3, rows interleaved in groups of GU_INTERLEAVE]
    [W_d values: H x F] [W_g scales: F/128 x H/128 fp32] [W_u scales]
    [W_d scales: H/128 x F/128].
    """
    F, H = q["g"].shape
    g = GU_INTERLEAVE
    gu = np.empty((F // g, 2, g, H), dtype=np.uint8)
    gu[:, 0] = q["g"].reshape(F // g, g, H)
    gu[:, 1] = q["u"].reshape(F // g, g, H)
    parts = [gu.reshape(-1), q["d"].reshape(-1)] + [
        np.ascontiguousarray(q[k], dtype=np.float32).reshape(-1).view(np.uint8)
        for k in ("g_scale", "u_scale", "d_scale")]
    nb = record_bytes(H, F, FMT_FP8)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    off = 0
    for p in parts:
        out[off:off + p.size] = p
        off += p.size
    assert off == nb
    return out


def record_fp8(seed: int, layer: int, expert: int, H: int, F: int, out=None) -> np.ndarray:
    """Record bytes of one block-FP8 layer-expert."""
    return pack_record_fp8(expert_fp8(seed, layer, expert, H, F), out=out)


# -------------------------------------------------------------- host pool

def fill_host_pool(pool: np.ndarray, shape: Shape, seed: int, threads: int | None = None) -> np.ndarray | None:
    """Write every record [l*E+e] of the host pool (uint8 [L*E*record_bytes]).

    Returns the per-record fp32 globals [L*E] for NVFP4, else None (BF16,
    MXFP4 and block-FP8 records carry no global).
    """
    rb = shape.record_bytes
    n = shape.L * shape.E
    assert pool.size >= n * rb
    glob = np.zeros(n, dtype=np.float32) if shape.fmt == FMT_NVFP4 else None

    def work(fid: int):
        l, e = divmod(fid, shape.E)
        dst = pool[fid * rb:(fid + 1) * rb]
        if shape.fmt == FMT_BF16:
            record_bf16(seed, l, e, shape.H, shape.F, out=dst)
        elif shape.fmt == FMT_MXFP4:
            record_mxfp4(seed, l, e, shape.H, shape.F, out=dst)
        elif shape.fmt == FMT_FP8:
            record_fp8(seed, l, e, shape.H, shape.F, out=dst)
        else:
            _, gsv = record_nvfp4(seed, l, e, shape.H, shape.F, out=dst)
            glob[fid] = gsv

    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, range(n)))
    return glob


# --------------------------------------------------------- router / tokens

def ar1_logits(seed: int, steps: int, L: int, T: int, E: int, rho: float, sigma: float | None = None) -> np.ndarray:
    """AR(1) router logits, float32 [steps, L, T, E].

    One chain per (layer, token lane); l_0 ~ N(0,1), l_t = rho*l_{t-1} + sigma*eps.
    sigma defaults to sqrt(1 - rho^2) (stationary unit variance).
    """
    if sigma is None:
        sigma = float(np.sqrt(1.0 - rho * rho))
    rng = _rng(seed, TAG_LOGITS, L, T, E)
    out = np.empty((steps, L, T, E), dtype=np.float32)
    cur = rng.standard_normal((L, T, E))
    for s in range(steps):
        if s:
            cur = rho * cur + sigma * rng.standard_normal((L, T, E))
        out[s] = cur
    return out


def iid_logits(seed: int, tag_words: tuple, T: int, E: int) -> np.ndarray:
    """i.i.d. N(0,1) router logits float32 [T, E]."""
    return _rng(seed, TAG_LOGITS, *tag_words).standard_normal((T, E), dtype=np.float32)


def tokens_bf16(seed: int, step: int, layer: int, T: int, H: int) -> np.ndarray:
    """Hidden states x ~ N(0,1) rounded to bf16; uint16 bits [T, H]."""
    return f32_to_bf16_bits(_rng(seed, TAG_X, step, layer, T, H).standard_normal((T, H), dtype=np.float32))


def random_f32(seed: int, tag_words: tuple, shape, scale: float = 1.0) -> np.ndarray:
    """Generic seeded float32 N(0, scale^2) tensor."""
    return (_rng(seed, TAG_PARTIAL_C, *tag_words).standard_normal(shape, dtype=np.float32) * np.float32(scale))


def random_topk(seed: int, tag_words: tuple, T: int, E: int, k: int) -> np.ndarray:
    """Top-k ids int32 [T, k]: k distinct experts per token, uniformly drawn."""
    rng = _rng(seed, TAG_TOPK, *tag_words)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


# --------------------------------------------------------------- configs

@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    S: int
    steps: int
    T: int
    rho: float | None
    sigma: float | None
    B_P: float
    B_H: float
    seed: int = 0


TINY = Workload("tiny", Shape(L=1, E=8, k=2, H=64, F=128), S=4, steps=16, T=4,
                rho=None, sigma=None, B_P=25.0, B_H=75.0)
DECODE_T1 = Workload("decode_t1", Shape(L=48, E=128, k=8, H=2048, F=768), S=1536, steps=256, T=1,
                     rho=0.8, sigma=0.6, B_P=52.7, B_H=120.0)
DECODE_T16 = Workload("decode_t16", Shape(L=48, E=128, k=8, H=2048, F=768), S=768, steps=128, T=16,
                      rho=0.7, sigma=None, B_P=25.0, B_H=90.0)
PREFILL = Workload("prefill", Shape(L=4, E=128, k=8, H=2048, F=768), S=256, steps=1, T=8192,
                   rho=None, sigma=None, B_P=0.0, B_H=0.0)
LARGE_NVFP4 = Workload("large_nvfp4", Shape(L=8, E=256, k=8, H=4096, F=2048, fmt=FMT_NVFP4), S=512,
                       steps=64, T=1, rho=0.8, sigma=None, B_P=52.7, B_H=150.0)
# The Large shapes with MXFP4 banks (a further record format; same routing).
LARGE_MXFP4 = Workload("large_mxfp4", Shape(L=8, E=256, k=8, H=4096, F=2048, fmt=FMT_MXFP4), S=512,
                       steps=64, T=1, rho=0.8, sigma=None, B_P=52.7, B_H=150.0)
# Decode T=16 resizes its cache: shrink to this many slots before step 32,
# grow back before step 64.
DECODE_T16_RESIZE = ((32, 384), (64, 768))
