"""Block-FP8 decoding and its block quantiser (test infrastructure only).

The pages say a block-FP8 bank keeps FP8 weights and block-scale data
(deepmox, "One logical expert, two physical levels of memory") and give no
further detail.  It is read here as the common block-wise FP8 layout:
  * values are OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits, no infinities, S.1111.111 NaN, largest finite 448);
  * each weight matrix is cut into 128 x 128 blocks (rows x K) and every
    block has one fp32 scale: value = e4m3(code) * scale.
Quantisation (used only to pin the generator): scale = amax(block) / 448,
computed in fp32, and codes = e4m3(w / scale) rounded to nearest even with
saturation; an all-zero block takes scale 1.

Record layout read here (written independently of the generator): [W_gu
values 2F x H, one byte each, gate/up rows interleaved in groups of 16]
[W_d values H x F] [W_g scales F/128 x H/128 fp32] [W_u scales F/128 x
H/128] [W_d scales H/128 x F/128], every part row-major.
"""
from __future__ import annotations

import numpy as np

from oracle.nvfp4 import E4M3, INTERLEAVE, e4m3_value

BLOCK = 128
E4M3_MAX = 448.0


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 weights from e4m3 codes [rows, K] and fp32 scales [rows/128, K/128]."""
    v = E4M3[codes]
    s = np.repeat(np.repeat(np.asarray(scales, dtype=np.float64), BLOCK, axis=0), BLOCK, axis=1)
    return v * s


def record_weights(record: np.ndarray, H: int, F: int):
    """(Wg [F,H], Wu [F,H], Wd [H,F]) float64 of one block-FP8 record."""
    r = np.asarray(record, dtype=np.uint8)
    o = 0
    gu = r[o:o + 2 * F * H].reshape(2 * F, H); o += 2 * F * H
    d = r[o:o + H * F].reshape(H, F); o += H * F
    nb = (F // BLOCK) * (H // BLOCK)
    sc = r[o:].view(np.float32)
    assert sc.size == 3 * nb
    sg = sc[:nb].reshape(F // BLOCK, H // BLOCK)
    su = sc[nb:2 * nb].reshape(F // BLOCK, H // BLOCK)
    sd = sc[2 * nb:].reshape(H // BLOCK, F // BLOCK)
    g = INTERLEAVE
    grp = gu.reshape(F // g, 2, g, H)
    Wg = dequant(grp[:, 0].reshape(F, H), sg)
    Wu = dequant(grp[:, 1].reshape(F, H), su)
    Wd = dequant(d, sd)
    return Wg, Wu, Wd


def _e4m3_code(v: float) -> int:
    """Nearest e4m3 code to v, ties to the even code, saturating at 448.
    Plain scan over the 127 non-negative finite magnitudes."""
    a = min(abs(v), E4M3_MAX)
    best = 0
    for c in range(127):
        d, db = abs(a - e4m3_value(c)), abs(a - e4m3_value(best))
        if d < db or (d == db and c % 2 == 0 and best % 2 == 1):
            best = c
    if v < 0 and best != 0:
        best |= 0x80
    return best


def quantize_block128(W: np.ndarray):
    """Block-FP8 quantisation of a matrix [rows, K] (multiples of 128), one
    value at a time.  Returns (codes uint8 [rows, K], scales fp32 [rows/128, K/128])."""
    W = np.asarray(W, dtype=np.float32)
    rows, K = W.shape
    codes = np.zeros((rows, K), dtype=np.uint8)
    scales = np.zeros((rows // BLOCK, K // BLOCK), dtype=np.float32)
    for bi in range(rows // BLOCK):
        for bj in range(K // BLOCK):
            blk = W[bi * BLOCK:(bi + 1) * BLOCK, bj * BLOCK:(bj + 1) * BLOCK]
            amax = np.float32(np.max(np.abs(blk)))
            s = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
            scales[bi, bj] = s
            for i in range(BLOCK):
                for j in range(BLOCK):
                    codes[bi * BLOCK + i, bj * BLOCK + j] = _e4m3_code(float(blk[i, j]) / float(s))
    return codes, scales
