"""Pins of the block-FP8 codecs: blocks quantised by hand
(tests/golden/fp8_blocks.json), the error bound of round-to-nearest E4M3,
exact round trip of representable blocks, agreement of two independently
written quantisers and the record byte layout."""
import json
import os

import numpy as np

import synth
from oracle import fp8
from oracle import nvfp4 as fp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_blocks.json")


def _block(case):
    x = np.zeros((128, 128), dtype=np.float32)
    for i, j, v in case["x"]:
        x[i, j] = v
    return x


def test_hand_worked_blocks():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) == 3
    for case in cases:
        x = _block(case)
        want = np.zeros((128, 128), dtype=np.uint8)
        for i, j, c in case["codes"]:
            want[i, j] = c
        s_want = np.float32(float.fromhex(case["scale"]))
        for codes, sc in (fp8.quantize_block128(x), synth.quantize_fp8(x)):
            assert sc[0, 0] == s_want, (case["name"], float(sc[0, 0]).hex())
            assert np.array_equal(codes, want), case["name"]
            d = fp8.dequant(codes, sc)
            for i, j, c in case["codes"]:
                assert d[i, j] == fp4.E4M3[c] * float(s_want)


def test_error_bound_and_scale():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((256, 256)) * rng.uniform(1e-4, 10, size=(256, 1))).astype(np.float32)
    x[:128, 128:] = 0.0
    codes, sc = synth.quantize_fp8(x)
    d = fp8.dequant(codes, sc)
    for bi in range(2):
        for bj in range(2):
            blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128].astype(np.float64)
            s = float(sc[bi, bj])
            err = np.abs(d[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128] - blk)
            # half an E4M3 ulp: 2^-4 of the value's binade, 2^-10 in the subnormal range
            bound = s * np.maximum(np.abs(blk) / s * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
            assert np.all(err <= bound)
            amax = np.abs(blk).max()
            if amax > 0:
                assert s == np.float32(np.float32(amax) / np.float32(448.0))
            else:
                assert s == 1.0


def test_representable_blocks_round_trip():
    rng = np.random.default_rng(22)
    for e in (-12, -3, 0, 4):
        codes = rng.integers(0, 255, size=(128, 128)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x7E       # no NaN codes
        codes[0, 0] = 0x7E                         # amax = 448 * 2^e
        x = (fp4.E4M3[codes] * 2.0 ** e).astype(np.float32)
        c2, s2 = synth.quantize_fp8(x)
        assert s2[0, 0] == np.float32(2.0 ** e)
        assert np.array_equal(fp8.dequant(c2, s2), x.astype(np.float64))


def test_two_quantisers_agree_on_a_weight_block():
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, synth.TAG_WEIGHTS, 0, 3])))
    w = (rng.standard_normal((128, 128), dtype=np.float32) * np.float32(0.02))
    c1, s1 = fp8.quantize_block128(w)
    c2, s2 = synth.quantize_fp8(w)
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)


def test_fp8_record_layout_round_trip():
    H, F = 256, 128
    q = synth.expert_fp8(0, 0, 2, H, F)
    rec = synth.record_fp8(0, 0, 2, H, F)
    assert rec.size == synth.record_bytes(H, F, synth.FMT_FP8) == 3 * H * F + 12 * (H // 128) * (F // 128)
    Wg, Wu, Wd = fp8.record_weights(rec, H, F)
    assert np.array_equal(Wg, fp8.dequant(q["g"], q["g_scale"]))
    assert np.array_equal(Wu, fp8.dequant(q["u"], q["u_scale"]))
    assert np.array_equal(Wd, fp8.dequant(q["d"], q["d_scale"]))
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, synth.TAG_WEIGHTS, 0, 2])))
    w = rng.standard_normal(3 * H * F, dtype=np.float32) * np.float32(0.02)
    rel = np.linalg.norm(Wd.reshape(-1) - w[2 * H * F:]) / np.linalg.norm(w[2 * H * F:])
    assert rel < 0.05
