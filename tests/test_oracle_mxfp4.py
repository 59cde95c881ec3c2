"""Pins of the MXFP4 codecs: the E8M0 scale against IEEE-754 single bit
patterns, blocks converted by hand (tests/golden/mxfp4_blocks.json), the
properties the MX conversion guarantees (block range, error bound, exact
round trip of representable blocks), agreement of two independently written
quantisers and the record byte layout."""
import json
import math
import os

import numpy as np

import synth
from oracle import mxfp4 as mx
from oracle import nvfp4 as fp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp4_blocks.json")


def test_e8m0_matches_ieee_single_exponent_field():
    # a float32 whose only set bits are the exponent field c is 2^(c-127);
    # code 0 is the subnormal 2^-127 (top mantissa bit only)
    for c in range(1, 255):
        assert np.array([c << 23], dtype=np.uint32).view(np.float32)[0] == mx.E8M0[c], c
    assert np.array([1 << 22], dtype=np.uint32).view(np.float32)[0] == mx.E8M0[0]
    assert mx.E8M0[127] == 1.0 and mx.E8M0[128] == 2.0 and mx.E8M0[126] == 0.5
    assert math.isnan(mx.E8M0[255])


def _block(case):
    x = np.zeros((1, 32))
    for i, v in case["x"].items():
        x[0, int(i)] = v
    return x


def test_hand_worked_blocks():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) == 5
    for case in cases:
        x = _block(case)
        want_codes = np.zeros(32, dtype=np.uint8)
        for i, c in case["codes"].items():
            want_codes[int(i)] = c
        want_deq = np.zeros(32)
        for i, v in case["deq"].items():
            want_deq[int(i)] = v
        for codes, sc in (mx.quantize_block32(x), synth.quantize_mxfp4(x)):
            assert int(sc[0, 0]) == case["scale_code"], case["name"]
            assert np.array_equal(codes[0], want_codes), (case["name"], codes[0])
            assert np.array_equal(mx.dequant(codes, sc)[0], want_deq), case["name"]


def test_nan_scale_poisons_its_block_only():
    codes = np.ones((1, 64), dtype=np.uint8)
    sc = np.array([[255, 127]], dtype=np.uint8)
    d = mx.dequant(codes, sc)
    assert np.isnan(d[0, :32]).all() and (d[0, 32:] == 0.5).all()


def test_block_range_and_error_bound():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((16, 256)) * rng.uniform(1e-4, 1e3, size=(16, 1))
    x[3, :32] = 0.0
    codes, sc = mx.quantize_block32(x)
    d = mx.dequant(codes, sc)
    for r in range(16):
        for b in range(8):
            blk = x[r, b * 32:(b + 1) * 32]
            X = mx.E8M0[sc[r, b]]
            amax = np.abs(blk).max()
            if amax > 0:
                assert 4.0 <= amax / X < 8.0          # the shared exponent's range
            err = np.abs(d[r, b * 32:(b + 1) * 32] - blk)
            # half the widest e2m1 gap (4 -> 6) is 1 unit of X; saturated
            # values (above 6X, below 8X) lose |x| - 6X < 2X
            bound = np.maximum(X, np.abs(blk) - 6 * X)
            assert np.all(err <= bound + 1e-300)
            assert np.all(np.sign(d[r, b * 32:(b + 1) * 32]) * np.sign(blk) >= 0)


def test_representable_blocks_round_trip_exactly():
    rng = np.random.default_rng(12)
    for se in (-20, -3, 0, 5):
        codes = rng.integers(0, 16, size=(4, 64)).astype(np.uint8)
        codes[:, 0] = 7  # amax 6 * 2^se in every block
        codes[:, 32] = 15
        x = fp4.E2M1[codes] * math.ldexp(1.0, se)
        c2, s2 = mx.quantize_block32(x)
        assert (s2 == se + 127).all()
        assert np.array_equal(mx.dequant(c2, s2), x)


def test_unit_scale_equals_the_nvfp4_decode_with_unit_scale():
    # with every scale 1.0 both formats are the bare e2m1 values
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    a = mx.dequant(codes, np.full((3, 2), 127, dtype=np.uint8))
    b = fp4.dequant(codes, np.full((3, 4), 0x38, dtype=np.uint8), 1.0)
    assert np.array_equal(a, b)


def test_two_quantisers_agree():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((8, 128)) * rng.uniform(1e-3, 10, size=(8, 1))
    x[2, 32:64] = 0.0
    c1, s1 = mx.quantize_block32(x)
    c2, s2 = synth.quantize_mxfp4(x)
    assert np.array_equal(s1, s2)
    # both divide by a power of two (exact) and round on the same grid
    assert np.array_equal(c1, c2)


def test_mxfp4_record_layout_round_trip():
    H, F = 64, 128
    q = synth.expert_mxfp4(0, 0, 1, H, F)
    rec = synth.record_mxfp4(0, 0, 1, H, F)
    assert rec.size == synth.record_bytes(H, F, synth.FMT_MXFP4) == 3 * H * F // 2 + 3 * H * F // 32
    Wg, Wu, Wd = mx.record_weights(rec, H, F)
    assert np.array_equal(Wg, mx.dequant(q["g"], q["g_scale"]))
    assert np.array_equal(Wu, mx.dequant(q["u"], q["u_scale"]))
    assert np.array_equal(Wd, mx.dequant(q["d"], q["d_scale"]))
    # the oracle's own quantiser reproduces the generator's codes on the same draw
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, synth.TAG_WEIGHTS, 0, 1])))
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    c, s = mx.quantize_block32(w[:H * F].reshape(F, H).astype(np.float64))
    assert np.array_equal(c, q["g"]) and np.array_equal(s, q["g_scale"])
    rel = np.linalg.norm(Wg.reshape(-1) - w[:H * F]) / np.linalg.norm(w[:H * F])
    assert rel < 0.2
