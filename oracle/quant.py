"""Block quantization rules of the KV formats, written out in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The memra-bench card ("drafts/kf4/ - archived experiment") names the KV-cache
format knobs: K = q8_0 | fp8, V = q5_1 | q4_0 | fp8, defaults q8_0 / q5_1.
It prints no rule, so the library states these definitions, applied to each
block of 32 consecutive elements of one fp16 row along head_dim:

q8_0   d = fp16_rne(max|x| / 127)          q = rne(x / d)          x^ = d q
q5_1   m = min x,  d = fp16_rne((max x - min x) / 31)
                                           q = rne((x - m) / d)    x^ = d q + m
q4_0   d = fp16_rne(max|x| / 7)            q = clamp(rne(x / d), -8, 7)
                                                                   x^ = d q
fp8    per-tensor float32 scale s;  byte = e4m3_rne_satfinite(fp32(x) /_rn fp32(s))
                                                                   x^ = s e4m3(byte)
nvfp4  (the card's archived "kf4" arm, an NVFP4 KV cache; reading: NVIDIA's
       published NVFP4 block format) blocks of 16 elements, a float32
       per-tensor scale s, an e4m3 scale byte per block and OCP FP4 E2M1 codes:
           u   = fp32(max|x|) /_rn (6 *_rn s)            (float32 operations)
           s_b = e4m3_rne_satfinite(u)
           c   = e2m1_rne_satfinite(fp32(x) /_rn (e4m3(s_b) *_rn s))   (0 if s_b = 0)
           x^  = s e4m3(s_b) e2m1(c)

"rne" rounds the exact real value half-to-even.  The quotient uses the stored
fp16 d.  With a normal fp16 d the clamps never act (|x/d| < 127.5, 7.5, 31.5);
with a subnormal d the fp16 rounding of d can fall well below max|x|/127 and
the clamp decides the code.  When the stored d is 0 (all-zero block, a block whose max|x|/127
rounds to fp16 zero, or max == min for q5_1) every q is 0.  Non-finite inputs
are outside the contract: these functions raise.

Exactness of the float64 evaluation: x, d and m are fp16 values, so x - m is
exact in float64 and the float64 quotient can never land on a rounding tie it
was not already on (a tie of x/d is a short binary fraction, and a non-tie is
at least 2^-12 relative away from one, far above float64's 2^-53).  The
float64 -> fp16 cast of numpy rounds to nearest even; one float64 rounding
before it is harmless at these precisions.  Both facts are pinned by exact
rational arithmetic in tests/test_oracle_quant.py.

Pins: exact ``fractions.Fraction`` re-derivation on random and adversarial
blocks (ties, subnormals, max == min, signed zeros); the closed-form error
bound |x - x^| <= d/2; hand-worked blocks in tests/golden/; fp8 decode of all
256 codes and encode inside +-448 against torch.float8_e4m3fn (a library
conversion).
"""
from __future__ import annotations

import numpy as np

QBLOCK = 32
E4M3_MAX = 448.0


def _blocks(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("quantizers take fp16 rows")
    if x.shape[-1] % QBLOCK:
        raise ValueError("head_dim must be a multiple of 32")
    xb = x.astype(np.float64).reshape(x.shape[:-1] + (x.shape[-1] // QBLOCK, QBLOCK))
    if not np.isfinite(xb).all():
        raise ValueError("non-finite input is outside the contract")
    return xb


def fp16_rne(v) -> np.ndarray:
    """Round float64 values to fp16, half-to-even (numpy's cast)."""
    return np.asarray(v, dtype=np.float64).astype(np.float16)


def quantize_q8_0(x: np.ndarray):
    """fp16 [..., D] -> (codes int8 [..., D], d fp16 [..., D/32])."""
    xb = _blocks(x)
    amax = np.abs(xb).max(axis=-1)
    d = fp16_rne(amax / 127.0)
    dd = d.astype(np.float64)[..., None]
    safe = np.where(dd > 0, dd, 1.0)
    q = np.where(dd > 0, np.rint(xb / safe), 0.0)
    q = np.clip(q, -127, 127).astype(np.int8)
    return q.reshape(x.shape), d


def quantize_q5_1(x: np.ndarray):
    """fp16 [..., D] -> (codes uint8 0..31 [..., D], d fp16 [..., D/32], m fp16 [..., D/32])."""
    xb = _blocks(x)
    mn = xb.min(axis=-1)
    mx = xb.max(axis=-1)
    d = fp16_rne((mx - mn) / 31.0)
    m = mn.astype(np.float16)          # exact: the minimum is one of the fp16 inputs
    dd = d.astype(np.float64)[..., None]
    safe = np.where(dd > 0, dd, 1.0)
    q = np.where(dd > 0, np.rint((xb - mn[..., None]) / safe), 0.0)
    q = np.clip(q, 0, 31).astype(np.uint8)
    return q.reshape(x.shape), d, m


def quantize_q4_0(x: np.ndarray):
    """fp16 [..., D] -> (codes int8 -8..7 [..., D], d fp16 [..., D/32])."""
    xb = _blocks(x)
    amax = np.abs(xb).max(axis=-1)
    d = fp16_rne(amax / 7.0)
    dd = d.astype(np.float64)[..., None]
    safe = np.where(dd > 0, dd, 1.0)
    q = np.where(dd > 0, np.rint(xb / safe), 0.0)
    q = np.clip(q, -8, 7).astype(np.int8)
    return q.reshape(x.shape), d


def dequantize_q8_0(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    qb = q.astype(np.float64).reshape(q.shape[:-1] + (q.shape[-1] // QBLOCK, QBLOCK))
    return (qb * d.astype(np.float64)[..., None]).reshape(q.shape)


def dequantize_q5_1(q: np.ndarray, d: np.ndarray, m: np.ndarray) -> np.ndarray:
    qb = q.astype(np.float64).reshape(q.shape[:-1] + (q.shape[-1] // QBLOCK, QBLOCK))
    return (qb * d.astype(np.float64)[..., None] + m.astype(np.float64)[..., None]).reshape(q.shape)


dequantize_q4_0 = dequantize_q8_0


# ---------------------------------------------------------------- fp8 e4m3 ---
# OCP 8-bit floating point, E4M3 variant ("fn"): sign bit 7, exponent bits 6..3
# with bias 7, mantissa bits 2..0; exponent 0 encodes subnormals m * 2^-9;
# S.1111.111 is NaN; there is no infinity; the largest finite value is 448.

def e4m3_decode(byte) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    b = np.asarray(byte, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    mant = b & 0x7
    val = np.where(e == 0, mant * 2.0 ** -9, (1.0 + mant / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & (mant == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0x7F, dtype=np.uint8)          # 0x00..0x7E: every non-negative finite code
_POS_VALS = e4m3_decode(_POS_CODES)                    # strictly increasing


def e4m3_encode_rne_satfinite(y) -> np.ndarray:
    """float32 values -> e4m3 bytes, nearest value, ties to the even code, |y| > 448 -> 448."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    if not np.isfinite(y).all():
        raise ValueError("non-finite input is outside the contract")
    a = np.minimum(np.abs(y), E4M3_MAX)
    hi = np.searchsorted(_POS_VALS, a, side="left")      # first code with value >= a
    hi = np.minimum(hi, _POS_VALS.size - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _POS_VALS[lo]
    dhi = _POS_VALS[hi] - a
    exact = dhi == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(exact | pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    return np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)


def quantize_fp8(x: np.ndarray, scale: float) -> np.ndarray:
    """fp16 [...] with float32 per-tensor scale -> e4m3 bytes [...]."""
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("quantizers take fp16 rows")
    y = x.astype(np.float32) / np.float32(scale)     # one IEEE float32 division, round to nearest even
    return e4m3_encode_rne_satfinite(y)


def dequantize_fp8(b: np.ndarray, scale: float) -> np.ndarray:
    return e4m3_decode(b) * float(np.float32(scale))


# ------------------------------------------------------- nvfp4 (e2m1) -------
# OCP 4-bit floating point E2M1: sign bit 3, exponent bits 2..1 with bias 1,
# mantissa bit 0; exponent 0 encodes 0 and the subnormal 0.5; no NaN or
# infinity; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.

NVFP4_BLOCK = 16
E2M1_MAX = 6.0


def e2m1_decode(code) -> np.ndarray:
    """4-bit codes (uint8 0..15) -> float64 values."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    mant = c & 0x1
    val = np.where(e == 0, mant * 0.5, (1.0 + mant / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return sign * val


_E2M1_CODES = np.arange(8, dtype=np.uint8)             # non-negative codes, values strictly increasing
_E2M1_VALS = e2m1_decode(_E2M1_CODES)


def e2m1_encode_rne_satfinite(y) -> np.ndarray:
    """float32 values -> E2M1 codes, nearest value, ties to the even code, |y| > 6 -> 6."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    if not np.isfinite(y).all():
        raise ValueError("non-finite input is outside the contract")
    a = np.minimum(np.abs(y), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_E2M1_VALS, a, side="left"), _E2M1_VALS.size - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E2M1_VALS[lo]
    dhi = _E2M1_VALS[hi] - a
    pick_hi = (dhi == 0) | (dhi < dlo) | ((dhi == dlo) & (_E2M1_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _E2M1_CODES[hi], _E2M1_CODES[lo]).astype(np.uint8)
    return np.where(np.signbit(y), code | 0x8, code).astype(np.uint8)


def quantize_nvfp4(x: np.ndarray, scale: float):
    """fp16 [..., D] with float32 per-tensor scale -> (codes uint8 0..15 [..., D], scale bytes uint8 [..., D/16])."""
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("quantizers take fp16 rows")
    if x.shape[-1] % NVFP4_BLOCK:
        raise ValueError("head_dim must be a multiple of 16")
    xb = x.astype(np.float32).reshape(x.shape[:-1] + (x.shape[-1] // NVFP4_BLOCK, NVFP4_BLOCK))
    if not np.isfinite(xb).all():
        raise ValueError("non-finite input is outside the contract")
    s = np.float32(scale)
    amax = np.abs(xb).max(axis=-1)                                  # exact: an fp16 value
    u = amax / (np.float32(6.0) * s)                                # float32 multiply, then float32 divide
    sb = e4m3_encode_rne_satfinite(u.astype(np.float32))
    eff = (e4m3_decode(sb).astype(np.float32) * s).astype(np.float32)   # float32 product
    safe = np.where(eff > 0, eff, np.float32(1.0)).astype(np.float32)
    y = (xb / safe[..., None]).astype(np.float32)                   # one float32 division per element
    c = e2m1_encode_rne_satfinite(y)
    c = np.where((sb == 0)[..., None], np.uint8(0), c).astype(np.uint8)
    return c.reshape(x.shape), sb


def dequantize_nvfp4(c: np.ndarray, sb: np.ndarray, scale: float) -> np.ndarray:
    cb = e2m1_decode(c).reshape(c.shape[:-1] + (c.shape[-1] // NVFP4_BLOCK, NVFP4_BLOCK))
    return (cb * e4m3_decode(sb)[..., None] * float(np.float32(scale))).reshape(c.shape)


# ------------------------------------------------------ format dispatchers ---

def quantize_rows(x: np.ndarray, fmt: str, scale: float = 1.0) -> dict:
    """Quantize fp16 rows [..., D]; returns the canonical block fields of the format."""
    if fmt == "q8_0":
        q, d = quantize_q8_0(x)
        return {"fmt": fmt, "q": q, "d": d}
    if fmt == "q5_1":
        q, d, m = quantize_q5_1(x)
        return {"fmt": fmt, "q": q, "d": d, "m": m}
    if fmt == "q4_0":
        q, d = quantize_q4_0(x)
        return {"fmt": fmt, "q": q, "d": d}
    if fmt == "fp8":
        return {"fmt": fmt, "q": quantize_fp8(x, scale), "scale": float(np.float32(scale))}
    if fmt == "nvfp4":
        c, sb = quantize_nvfp4(x, scale)
        return {"fmt": fmt, "q": c, "sb": sb, "scale": float(np.float32(scale))}
    raise ValueError(fmt)


def dequantize_rows(blk: dict) -> np.ndarray:
    fmt = blk["fmt"]
    if fmt in ("q8_0", "q4_0"):
        return dequantize_q8_0(blk["q"], blk["d"])
    if fmt == "q5_1":
        return dequantize_q5_1(blk["q"], blk["d"], blk["m"])
    if fmt == "fp8":
        return dequantize_fp8(blk["q"], blk["scale"])
    if fmt == "nvfp4":
        return dequantize_nvfp4(blk["q"], blk["sb"], blk["scale"])
    raise ValueError(fmt)


def select_rows(blk: dict, idx) -> dict:
    """Sub-select rows (first axis) of a quantized field set."""
    out = {"fmt": blk["fmt"]}
    for k, v in blk.items():
        if isinstance(v, np.ndarray):
            out[k] = v[idx]
        elif k != "fmt":
            out[k] = v
    return out
