"""MXFP4 decoding and the block-32 quantiser (test infrastructure only).

The pages list MXFP4 among the quantised bank layouts a slot record may use,
beside NVFP4 and block-FP8, each with its own packed layout and dequantisation
(deepmox, "One logical expert, two physical levels of memory"); they do not
spell the format out.  It is read here as the OCP Microscaling (MX) format,
version 1.0, MXFP4 variant:
  * element type e2m1 (the same four-bit code as NVFP4: magnitudes 0, 0.5, 1,
    1.5, 2, 3, 4, 6; sign in bit 3);
  * one shared scale per block of 32 consecutive values along K, of type
    E8M0: an unsigned biased exponent, value 2^(code - 127), code 0xFF = NaN,
    no sign, no zero, no mantissa;
  * value = e2m1 * 2^(code - 127).  There is no per-expert global.

Record layout read here (written independently of the generator that
produces it): [W_gu values 2F x H, two codes per byte, low nibble first,
gate/up rows interleaved in groups of 16] [W_d values H x F] [W_gu scales
2F x H/32] [W_d scales H x F/32].
"""
from __future__ import annotations

import math

import numpy as np

from oracle.nvfp4 import E2M1, INTERLEAVE, e2m1_value, unpack_codes

BLOCK = 32
E8M0_BIAS = 127
E2M1_EMAX = 2  # exponent of the largest normal e2m1 magnitude, 6 = 1.5 * 2^2


def e8m0_value(code: int) -> float:
    """2^(code - 127) for codes 0..254; code 255 is NaN."""
    if code == 0xFF:
        return float("nan")
    return math.ldexp(1.0, code - E8M0_BIAS)


E8M0 = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 weights from e2m1 codes [rows, K] and E8M0 codes [rows, K/32]."""
    v = E2M1[codes]
    s = np.repeat(E8M0[scales], BLOCK, axis=1)
    return v * s


def record_weights(record: np.ndarray, H: int, F: int):
    """(Wg [F,H], Wu [F,H], Wd [H,F]) float64 of one MXFP4 record."""
    r = np.asarray(record, dtype=np.uint8)
    n_gu = 2 * F * H
    n_d = H * F
    o = 0
    gu_codes = unpack_codes(r[o:o + n_gu // 2], 2 * F, H); o += n_gu // 2
    d_codes = unpack_codes(r[o:o + n_d // 2], H, F); o += n_d // 2
    gu_sc = r[o:o + n_gu // BLOCK].reshape(2 * F, H // BLOCK); o += n_gu // BLOCK
    d_sc = r[o:o + n_d // BLOCK].reshape(H, F // BLOCK); o += n_d // BLOCK
    assert o == r.size
    Wgu = dequant(gu_codes, gu_sc)
    g = INTERLEAVE
    grp = Wgu.reshape(F // g, 2, g, H)
    Wg = grp[:, 0].reshape(F, H)
    Wu = grp[:, 1].reshape(F, H)
    Wd = dequant(d_codes, d_sc)
    return Wg, Wu, Wd


def shared_exponent(amax: float) -> int:
    """The MX conversion's shared exponent of a block whose largest magnitude
    is amax: floor(log2(amax)) minus the element type's largest exponent,
    clamped to what E8M0 holds.  An all-zero block takes the smallest scale
    (reading: the spec's log2(0) = -inf clamps to the lower end)."""
    if amax == 0.0:
        return -E8M0_BIAS
    e = math.frexp(amax)[1] - 1  # floor(log2(amax)), exact for any double
    return max(-E8M0_BIAS, min(E8M0_BIAS, e - E2M1_EMAX))


def _e2m1_code(v: float) -> int:
    """Nearest e2m1 code to v, ties to the even code, saturating at 6.
    Plain scan over the eight magnitudes."""
    mags = [e2m1_value(c) for c in range(8)]
    a = min(abs(v), mags[-1])
    best = 0
    for i in range(8):
        d, db = abs(a - mags[i]), abs(a - mags[best])
        if d < db or (d == db and i % 2 == 0 and best % 2 == 1):
            best = i
    if v < 0 and best != 0:
        best |= 0x8
    return best


def quantize_block32(x: np.ndarray):
    """MX conversion of rows of x, one block of 32 at a time: shared scale
    X = 2^shared_exponent(amax), element = e2m1(x / X) (round to nearest even,
    saturating).  Returns (codes [n, K], E8M0 codes [n, K/32])."""
    x = np.asarray(x, dtype=np.float64)
    n, K = x.shape
    codes = np.zeros((n, K), dtype=np.uint8)
    scales = np.zeros((n, K // BLOCK), dtype=np.uint8)
    for r in range(n):
        for b in range(K // BLOCK):
            blk = x[r, b * BLOCK:(b + 1) * BLOCK]
            se = shared_exponent(float(np.max(np.abs(blk))))
            scales[r, b] = se + E8M0_BIAS
            X = math.ldexp(1.0, se)
            for i in range(BLOCK):
                codes[r, b * BLOCK + i] = _e2m1_code(float(blk[i]) / X)
    return codes, scales
