"""Pins of the NVFP4 codecs: exhaustive code tables from the format
definitions, round-to-nearest-even ties at every grid midpoint, agreement of
two independently written quantisers, and the record byte layout."""
import math

import numpy as np
import pytest

import synth
from oracle import nvfp4 as fp4


def test_e2m1_table():
    assert list(fp4.E2M1[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(fp4.E2M1[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e4m3_table():
    assert fp4.e4m3_value(0x38) == 1.0
    assert fp4.e4m3_value(0x7E) == 448.0
    assert fp4.e4m3_value(0x08) == 2.0 ** -6
    assert fp4.e4m3_value(0x01) == 2.0 ** -9
    assert fp4.e4m3_value(0xB8) == -1.0
    assert math.isnan(fp4.e4m3_value(0x7F)) and math.isnan(fp4.e4m3_value(0xFF))
    pos = fp4.E4M3[:127]
    assert np.all(np.diff(pos) > 0)
    # every finite positive value is (1+m/8)*2^(e-7) or m/8*2^-6: check a few by hand
    assert fp4.e4m3_value(0x3F) == 1.875 and fp4.e4m3_value(0x40) == 2.0


def test_e2m1_ties_to_even_and_saturation():
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             6.5: 6.0, 100.0: 6.0, 0.2: 0.0, 0.3: 0.5, -0.75: -1.0, -5.0: -4.0}
    for v, want in cases.items():
        got_o = fp4.E2M1[synth.encode_e2m1(np.array([v]))[0]]
        assert got_o == want, (v, got_o)
        assert fp4.E2M1[fp4._nearest_code(abs(v), fp4._E2M1_POS) | (8 if v < 0 else 0)] == want


def test_e4m3_ties_to_even_all_midpoints():
    pos = fp4.E4M3[:127]
    for i in range(126):
        mid = (pos[i] + pos[i + 1]) / 2
        c_ora = fp4._nearest_code(mid, fp4._E4M3_POS)
        c_gen = int(synth.encode_e4m3_pos(np.array([mid]))[0])
        want = i if i % 2 == 0 else i + 1
        assert c_ora == want and c_gen == want, i
    assert int(synth.encode_e4m3_pos(np.array([1000.0]))[0]) == 126


def test_every_representable_value_round_trips():
    for c in range(16):
        v = fp4.E2M1[c]
        code = int(synth.encode_e2m1(np.array([v]))[0])
        assert fp4.E2M1[code] == v
    for c in range(127):
        assert int(synth.encode_e4m3_pos(np.array([fp4.E4M3[c]]))[0]) == c


def test_two_quantisers_agree():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 64)) * rng.uniform(0.01, 10, size=(6, 1))).astype(np.float32)
    x[2, :16] = 0.0
    for gs in [1.0, 0.37]:
        c1, s1 = fp4.quantize_block16(x, gs)
        c2, s2 = synth.quantize_nvfp4(x, gs)
        assert np.array_equal(s1, s2)
        # the generator divides in float64, the oracle in float32: codes may
        # differ only where the quotient sits within float32 rounding of a midpoint
        diff = c1 != c2
        assert diff.mean() < 0.01


def test_quantiser_error_bound():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 128)).astype(np.float32)
    c, s = fp4.quantize_block16(x, 1.0)
    xd = fp4.dequant(c, s, 1.0)
    # per block: e2m1 spacing near amax is 2 units of (amax/6)/2... bound by half the largest gap
    for r in range(8):
        for b in range(8):
            blk = x[r, b * 16:(b + 1) * 16].astype(np.float64)
            sc = fp4.E4M3[s[r, b]]
            err = np.abs(xd[r, b * 16:(b + 1) * 16] - blk)
            assert np.all(err <= 1.0 * sc + 1e-12)
            assert abs(np.abs(blk).max() / 6.0 - sc) <= sc / 16 + 1e-12


def test_nvfp4_record_layout_round_trip():
    H, F = 64, 128
    q = synth.expert_nvfp4(0, 0, 1, H, F)
    rec, gs = synth.record_nvfp4(0, 0, 1, H, F)
    assert rec.size == synth.record_bytes(H, F, synth.FMT_NVFP4)
    Wg, Wu, Wd = fp4.record_weights(rec, H, F, gs)
    assert np.array_equal(Wg, fp4.dequant(q["g"], q["g_scale"], gs))
    assert np.array_equal(Wu, fp4.dequant(q["u"], q["u_scale"], gs))
    assert np.array_equal(Wd, fp4.dequant(q["d"], q["d_scale"], gs))
    # the quantised weights stay close to the N(0, 0.02) draw they came from
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, synth.TAG_WEIGHTS, 0, 1])))
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    rel = np.linalg.norm(Wg.reshape(-1) - w[:H * F]) / np.linalg.norm(w[:H * F])
    assert rel < 0.15
