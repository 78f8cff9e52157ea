"""Pins for the oracle's NVFP4 block rule (CPU only).

NVFP4 is the memra-bench card's archived "kf4" KV-cache arm; the rule is the
library's reading of NVIDIA's published format (E2M1 codes, an e4m3 scale byte
per 16 elements, a float32 per-tensor scale), stated in oracle/quant.py.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")

# OCP FP4 E2M1 by definition: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_all_codes():
    vals = quant.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(vals[:8]) == E2M1_TABLE
    assert list(-vals[8:]) == E2M1_TABLE
    assert np.signbit(vals[8])                      # code 8 is -0


def test_e2m1_encode_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(0)
    mids = [(a + b) / 2 for a, b in zip(E2M1_TABLE, E2M1_TABLE[1:])]
    y = np.concatenate([rng.uniform(-8, 8, 20000), mids, [-m for m in mids], E2M1_TABLE, [6.5, 100.0, -7.0]])
    y = y.astype(np.float32)
    got = quant.e2m1_encode_rne_satfinite(y)
    for v, c in zip(y.astype(np.float64), got):
        a = min(abs(Fraction(float(v))), Fraction(6))
        dist = [abs(a - Fraction(t)) for t in E2M1_TABLE]
        best = min(dist)
        cands = [i for i, d in enumerate(dist) if d == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        if np.signbit(v):
            want |= 8
        assert c == want, (v, c, want)


def test_e2m1_round_trip():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(quant.e2m1_encode_rne_satfinite(quant.e2m1_decode(codes).astype(np.float32)), codes)


def _f32(v):
    """Round a float64 value to float32.  For one product or quotient of two
    float32 values, rounding the float64 result again is innocuous (53 >= 2*24 + 2)."""
    return np.float32(v)


@pytest.mark.parametrize("seed", range(4))
def test_nvfp4_steps_follow_the_rule(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((64, 128)) * 10.0 ** rng.uniform(-5, 3, (64, 1))).astype(np.float16)
    s = float(np.float32(np.abs(x.astype(np.float32)).max() / np.float32(2688.0))) * [1.0, 0.5, 3.0, 1e-3][seed]
    c, sb = quant.quantize_nvfp4(x, s)
    s32 = np.float32(s)
    for r in range(0, 64, 7):
        for b in range(8):
            blk = x[r, 16 * b:16 * b + 16].astype(np.float64)
            u = _f32(float(np.max(np.abs(blk))) / float(_f32(6.0 * float(s32))))
            byte = quant.e4m3_encode_rne_satfinite(np.float32(u))
            assert byte == sb[r, b]
            scale_val = float(quant.e4m3_decode(byte))
            eff = float(_f32(scale_val * float(s32)))
            for j in range(16):
                if byte == 0:
                    assert c[r, 16 * b + j] == 0
                    continue
                y = _f32(blk[j] / eff)
                assert c[r, 16 * b + j] == quant.e2m1_encode_rne_satfinite(y)


def test_nvfp4_error_bound():
    """Every code is the nearest E2M1 value of x / (s_b s): within half the local gap, or saturated."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((200, 128)).astype(np.float16)
    s = float(np.float32(np.abs(x.astype(np.float32)).max() / np.float32(2688.0)))
    c, sb = quant.quantize_nvfp4(x, s)
    eff = quant.e4m3_decode(sb) * float(np.float32(s))
    y = x.astype(np.float64).reshape(200, 8, 16) / eff[..., None]
    v = quant.e2m1_decode(c).reshape(200, 8, 16)
    gap = np.where(np.abs(y) <= 2, 0.5, np.where(np.abs(y) <= 4, 1.0, 2.0))
    inside = np.abs(y) <= 6
    assert (np.abs(y - v)[inside] <= gap[inside] / 2 * (1 + 2 ** -20)).all()
    assert (np.abs(v[~inside]) == 6).all()
    # the block maximum lands on the top of the E2M1 range (s_b rounds u to 3 significant bits)
    top = np.abs(v).max(axis=-1)
    assert (top >= 4).all()


def golden_records():
    recs = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        scale, xs, sb, cs = [f.strip() for f in line.split(";")]
        x = np.zeros(16, np.float16)
        vals = [float(t) for t in xs.split()]
        x[:len(vals)] = vals
        codes = np.zeros(16, np.uint8)
        cv = [int(t) for t in cs.split()]
        codes[:len(cv)] = cv
        recs.append((float(scale), x, int(sb, 16), codes))
    return recs


@pytest.mark.parametrize("rec", golden_records(), ids=lambda r: f"s{r[0]}_sb{r[2]:02x}")
def test_golden_blocks(rec):
    scale, x, sb, codes = rec
    c, b = quant.quantize_nvfp4(x[None, :], scale)
    assert b[0, 0] == sb
    assert np.array_equal(c[0], codes)


def test_non_finite_raises():
    with pytest.raises(ValueError):
        quant.quantize_nvfp4(np.array([[np.inf] + [0] * 15], np.float16), 1.0)
