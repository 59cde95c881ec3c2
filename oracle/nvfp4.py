"""NVFP4 decoding and the block-16 activation quantiser (test infrastructure only).

The pages name NVFP4 banks as packed four-bit values plus block scales, with a
per-expert fp32 global that stays GPU-resident (deepmox, "One logical expert,
two physical levels of memory").  The codes themselves follow the public
format definitions:
  * e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6;
  * e4m3 (OCP FP8 E4M3): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
    infinities, S.1111.111 is NaN, largest finite 448, subnormals 2^-6 * m/8;
  * one e4m3 scale per 16 consecutive values along K; value = e2m1 * scale *
    global.

Record layout read here (written independently of the generator that
produces it): [W_gu values 2F x H, two codes per byte, low nibble first,
gate/up rows interleaved in groups of 16] [W_d values H x F] [W_gu scales
2F x H/16] [W_d scales H x F/16].
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
INTERLEAVE = 16


def e2m1_value(code: int) -> float:
    """Magnitude from the bit fields (not from a table)."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = 0.5 * m              # subnormal: 2^(1-1) * m/2
    else:
        mag = (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return s * mag


def e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3 = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def unpack_codes(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p & 0xF
    out[1::2] = p >> 4
    return out.reshape(rows, cols)


def dequant(codes: np.ndarray, scales: np.ndarray, gs: float) -> np.ndarray:
    """float64 weights from e2m1 codes [rows, K], e4m3 scale codes [rows, K/16]."""
    v = E2M1[codes]
    s = np.repeat(E4M3[scales], BLOCK, axis=1)
    return v * s * float(gs)


def record_weights(record: np.ndarray, H: int, F: int, gs: float):
    """(Wg [F,H], Wu [F,H], Wd [H,F]) float64 of one NVFP4 record."""
    r = np.asarray(record, dtype=np.uint8)
    n_gu = 2 * F * H
    n_d = H * F
    o = 0
    gu_codes = unpack_codes(r[o:o + n_gu // 2], 2 * F, H); o += n_gu // 2
    d_codes = unpack_codes(r[o:o + n_d // 2], H, F); o += n_d // 2
    gu_sc = r[o:o + n_gu // BLOCK].reshape(2 * F, H // BLOCK); o += n_gu // BLOCK
    d_sc = r[o:o + n_d // BLOCK].reshape(H, F // BLOCK); o += n_d // BLOCK
    assert o == r.size
    Wgu = dequant(gu_codes, gu_sc, gs)
    g = INTERLEAVE
    grp = Wgu.reshape(F // g, 2, g, H)
    Wg = grp[:, 0].reshape(F, H)
    Wu = grp[:, 1].reshape(F, H)
    Wd = dequant(d_codes, d_sc, gs)
    return Wg, Wu, Wd


def _nearest_code(x: float, table_pos: list) -> int:
    """Index of the nearest magnitude in an ascending table; ties to the even
    index; saturate at the largest.  Plain loop, one value at a time."""
    ax = min(abs(x), table_pos[-1])
    best = 0
    for i in range(1, len(table_pos)):
        if table_pos[i] <= ax:
            best = i
    if best + 1 < len(table_pos):
        lo, hi = table_pos[best], table_pos[best + 1]
        if ax - lo > hi - ax or (ax - lo == hi - ax and (best + 1) % 2 == 0):
            best += 1
    return best


_E2M1_POS = [e2m1_value(c) for c in range(8)]
_E4M3_POS = [e4m3_value(c) for c in range(127)]


def quantize_block16(x: np.ndarray, gs: float = 1.0):
    """Block-16 NVFP4 quantisation of activations (one row at a time).

    scale = e4m3(amax_block / (6*gs)); value code = e2m1(x / (scale*gs)).
    The divisions are done in float32, correctly rounded, to match a device
    quantiser that divides in float32.  Returns (codes [n, K], scales [n, K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    n, K = x.shape
    codes = np.zeros((n, K), dtype=np.uint8)
    scales = np.zeros((n, K // BLOCK), dtype=np.uint8)
    g32 = np.float32(gs)
    for r in range(n):
        for b in range(K // BLOCK):
            blk = x[r, b * BLOCK:(b + 1) * BLOCK]
            amax = np.float32(np.max(np.abs(blk)))
            s_in = np.float32(amax / np.float32(np.float32(6.0) * g32))
            sc = _nearest_code(float(s_in), _E4M3_POS)
            scales[r, b] = sc
            denom = np.float32(np.float32(E4M3[sc]) * g32)
            for i in range(BLOCK):
                v = float(np.float32(blk[i] / denom)) if denom > 0 else 0.0
                c = _nearest_code(v, _E2M1_POS)
                if v < 0 and c != 0:
                    c |= 0x8
                codes[r, b * BLOCK + i] = c
    return codes, scales
