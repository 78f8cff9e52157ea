"""Pins for the oracle's block quantizers (CPU only).

Each rule is re-derived with exact rational arithmetic (``fractions.Fraction``)
and an exact fp16 rounding written from the IEEE binary16 definition, on random
and adversarial blocks; checked against hand-worked blocks; bounded by the
closed-form error |x - x^| <= d/2; and, for fp8, compared with PyTorch's own
float8_e4m3fn conversion (a library routine).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.txt")


# ------------------------------------------------------------ exact helpers --

def rne_int(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def fp16_rne_exact(fr: Fraction) -> Fraction:
    """Round a rational to binary16 (10 stored mantissa bits, emin -14), half to even."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -14) - 10)
    return sign * rne_int(a / quantum) * quantum


def exact_q8_0(x):
    xs = [Fraction(float(v)) for v in x]
    d = fp16_rne_exact(max(abs(v) for v in xs) / 127)
    q = [0 if d == 0 else max(-127, min(127, rne_int(v / d))) for v in xs]
    return d, q


def exact_q4_0(x):
    xs = [Fraction(float(v)) for v in x]
    d = fp16_rne_exact(max(abs(v) for v in xs) / 7)
    q = [0 if d == 0 else max(-8, min(7, rne_int(v / d))) for v in xs]
    return d, q


def exact_q5_1(x):
    xs = [Fraction(float(v)) for v in x]
    mn, mx = min(xs), max(xs)
    d = fp16_rne_exact((mx - mn) / 31)
    q = [0 if d == 0 else max(0, min(31, rne_int((v - mn) / d))) for v in xs]
    return d, mn, q


def adversarial_blocks(rng):
    """Blocks built to sit on rounding ties, subnormals, signed zeros and flat ranges."""
    blocks = []
    blocks.append(np.zeros(32))
    blocks.append(-np.zeros(32))
    blocks.append(np.full(32, 3.0))                                     # max == min
    blocks.append(np.full(32, -2.0 ** -20))                            # flat subnormals
    sub = rng.integers(-1023, 1024, 32) * 2.0 ** -24                    # all fp16 subnormals
    blocks.append(sub)
    blocks.append(np.concatenate([[127.0], np.arange(31) - 15.5]))     # q8_0 ties at d = 1
    blocks.append(np.concatenate([[7.0], (np.arange(31) % 15) - 7.5]))  # q4_0 ties at d = 1
    blocks.append(np.concatenate([[-1.0, 30.0], np.arange(30) - 0.5])) # q5_1 ties at d = 1, m = -1
    blocks.append(np.concatenate([[65504.0, -65504.0], rng.standard_normal(30) * 1000]))  # fp16 extremes
    blocks.append(np.concatenate([[2.0 ** -14], rng.integers(-1024, 1024, 31) * 2.0 ** -24]))
    for scale in (1e-3, 1.0, 300.0):
        blocks.append(rng.standard_normal(32) * scale)
    return [np.asarray(b).astype(np.float16) for b in blocks]


def random_blocks(rng, n):
    out = []
    for i in range(n):
        scale = 10.0 ** rng.uniform(-6, 4)
        out.append((rng.standard_normal(32) * scale).astype(np.float16))
    return out


@pytest.fixture(scope="module")
def blocks():
    rng = np.random.default_rng(1234)
    return adversarial_blocks(rng) + random_blocks(rng, 400)


# --------------------------------------------------------------------- pins --

def test_fp16_cast_is_exact_rne():
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.uniform(-9, 4, 2000),
                           # exact midpoints between neighbouring fp16 values
                           (np.arange(1, 2000) + 0.5) * 2.0 ** -24,
                           (np.arange(1024, 3000) + 0.5) * 2.0 ** -10])
    got = quant.fp16_rne(vals).astype(np.float64)
    for v, g in zip(vals, got):
        assert Fraction(float(g)) == fp16_rne_exact(Fraction(float(v))), v


def test_q8_0_exact(blocks):
    for x in blocks:
        q, d = quant.quantize_q8_0(x)
        de, qe = exact_q8_0(x)
        assert Fraction(float(d[0])) == de
        assert q.tolist() == qe


def test_q4_0_exact(blocks):
    for x in blocks:
        q, d = quant.quantize_q4_0(x)
        de, qe = exact_q4_0(x)
        assert Fraction(float(d[0])) == de
        assert q.tolist() == qe


def test_q5_1_exact(blocks):
    for x in blocks:
        q, d, m = quant.quantize_q5_1(x)
        de, me, qe = exact_q5_1(x)
        assert Fraction(float(d[0])) == de
        assert Fraction(float(m[0])) == me
        assert q.tolist() == qe


def test_error_bounds(blocks):
    """|x - x^| <= d/2 whenever d is a normal fp16 number.

    With a subnormal d the fp16 rounding of d can fall far below max|x|/127
    (resp. /7, /31), so x/d can pass the code range and the clamp decides:
    there the bound is replaced by 'the code sits on the clamp'.
    """
    FP16_MIN_NORMAL = 2.0 ** -14
    for x in blocks:
        xf = x.astype(np.float64)
        q, d = quant.quantize_q8_0(x)
        dv = float(d[0])
        err = np.abs(xf - quant.dequantize_q8_0(q, d))
        if dv >= FP16_MIN_NORMAL:
            assert np.all(err <= dv / 2) and np.abs(q).max() <= 127
        elif dv > 0:
            over = err > dv / 2
            assert np.all(np.abs(q[over]) == 127)
        q, d = quant.quantize_q4_0(x)
        dv = float(d[0])
        err = np.abs(xf - quant.dequantize_q4_0(q, d))
        if dv >= FP16_MIN_NORMAL:
            assert np.all(err <= dv / 2)
            assert q.min() >= -7          # with a normal d the symmetric /7 rule never needs -8
        elif dv > 0:
            over = err > dv / 2
            assert np.all((q[over] == 7) | (q[over] == -8))
        q, d, m = quant.quantize_q5_1(x)
        dv = float(d[0])
        xh = quant.dequantize_q5_1(q, d, m)
        if dv >= FP16_MIN_NORMAL:
            assert np.all(np.abs(xf - xh) <= dv / 2)
            assert xh.min() >= float(m[0]) and xh.max() <= float(m[0]) + 31 * dv
        elif dv > 0:
            over = np.abs(xf - xh) > dv / 2
            assert np.all(q[over] == 31)
        else:
            assert np.all(xh == float(m[0]))


def test_subnormal_scale_reaches_the_clamp():
    """A flat block of -2^-20: d = fp16(2^-20/7) rounds to 2^-23, so x/d = -8 and q4_0 uses -8."""
    x = np.full(32, -2.0 ** -20).astype(np.float16)
    q, d = quant.quantize_q4_0(x)
    assert float(d[0]) == 2.0 ** -23 and np.all(q == -8)
    # q8_0: 2^-20/127 -> fp16 quantum 2^-24: 16/127 = 0.126 -> d = 0 -> all codes 0
    q, d = quant.quantize_q8_0(x)
    assert float(d[0]) == 0 and np.all(q == 0)
    # q8_0 with max|x| = 2^-16: 2^-16/127 * 2^24 = 2.0157 -> d = 2^-23, x/d = 128 -> clamp 127
    x = np.zeros(32, np.float16)
    x[0] = np.float16(2.0 ** -16)
    q, d = quant.quantize_q8_0(x)
    assert float(d[0]) == 2.0 ** -23 and q[0] == 127


def test_rows_split_into_blocks_along_head_dim():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 5, 256)).astype(np.float16)
    q, d = quant.quantize_q8_0(x)
    assert q.shape == x.shape and d.shape == (3, 5, 8)
    for blk in range(8):
        qb, db = quant.quantize_q8_0(x[1, 2, 32 * blk:32 * blk + 32])
        assert np.array_equal(q[1, 2, 32 * blk:32 * blk + 32], qb) and d[1, 2, blk] == db[0]


def test_non_finite_raises():
    x = np.zeros(32, np.float16)
    x[3] = np.inf
    with pytest.raises(ValueError):
        quant.quantize_q8_0(x)
    with pytest.raises(ValueError):
        quant.quantize_fp8(x, 1.0)


def _parse_list(s):
    out = []
    for tok in s.split():
        if "*" in tok:
            v, n = tok.split("*")
            out += [v] * int(n)
        else:
            out.append(tok)
    return out


def golden_records():
    recs = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, xs, d, m, qs = [p.strip() for p in line.split(";")]
            recs.append((fmt, _parse_list(xs), d, m, _parse_list(qs)))
    return recs


@pytest.mark.parametrize("rec", golden_records(), ids=lambda r: r[0])
def test_golden_blocks(rec):
    fmt, xs, d, m, qs = rec
    x = np.zeros(32, np.float16)
    x[:len(xs)] = np.array([float(v) for v in xs], dtype=np.float64).astype(np.float16)
    if fmt == "fp8":
        got = quant.quantize_fp8(x, float(d))
        want = np.zeros(32, np.uint8)
        want[:len(qs)] = [int(v, 16) for v in qs]
        assert got.tolist() == want.tolist()
        return
    want_q = np.zeros(32, np.int64)
    want_q[:len(qs)] = [int(v) for v in qs]
    if fmt == "q8_0":
        q, dd = quant.quantize_q8_0(x)
    elif fmt == "q4_0":
        q, dd = quant.quantize_q4_0(x)
    else:
        q, dd, mm = quant.quantize_q5_1(x)
        assert float(mm[0]) == float(m)
    assert float(dd[0]) == float(d)
    assert q.astype(np.int64).tolist() == want_q.tolist()


# --------------------------------------------------------------------- fp8 ---

def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = quant.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # encode(decode(c)) == c for every finite code (signed zero included)
    finite = codes[~nan]
    assert np.array_equal(quant.e4m3_encode_rne_satfinite(quant.e4m3_decode(finite).astype(np.float32)), finite)


def test_e4m3_encode_matches_torch_inside_range():
    rng = np.random.default_rng(11)
    y = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-4, 2.3, 20000),
                        # exact midpoints between neighbouring e4m3 values
                        (quant.e4m3_decode(np.arange(0, 0x7E)) + quant.e4m3_decode(np.arange(1, 0x7F))) / 2])
    y = np.clip(y, -448, 448).astype(np.float32)
    ours = quant.e4m3_encode_rne_satfinite(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_fp8_saturates_and_divides_in_float32():
    x = np.array([500, -500, 65504, 448, 464], dtype=np.float16)
    assert quant.quantize_fp8(x, 1.0).tolist() == [0x7E, 0xFE, 0x7E, 0x7E, 0x7E]
    # the quotient is one float32 division: pick a scale whose reciprocal is inexact
    rng = np.random.default_rng(5)
    x = rng.standard_normal(4096).astype(np.float16)
    s = np.float32(np.abs(x.astype(np.float32)).max() / np.float32(448))
    y = x.astype(np.float32) / s
    assert np.array_equal(quant.quantize_fp8(x, float(s)), quant.e4m3_encode_rne_satfinite(y))
    # error bound: half an e4m3 spacing, times the scale
    xh = quant.dequantize_fp8(quant.quantize_fp8(x, float(s)), float(s))
    a = np.abs(y.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    half_ulp = 2.0 ** (e - 3) / 2 * float(s)
    assert np.all(np.abs(xh - x.astype(np.float64)) <= half_ulp * (1 + 1e-12) + 1e-300)
