"""Byte layout of the paged, block-quantized KV pools, written out per element.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The memra pages define no layout (the README says the engine "repacks" model
data into its own internal layout and stops there), so the layout is this
library's ABI, stated in include/memra.h.  This module restates those formulas
element by element, independently of the CUDA code, so that the bytes the
quantize-append kernel writes can be compared bit for bit.

Pool = [num_pages][n_kv_heads][segment]; a segment holds one page (16 tokens)
of one KV head.  For token t (0..15) and element j (0..D-1) of its row, with
nb = D/32, b = j // 32 and r = j % 32:

K side (q8_0 codes, stored as the byte q + 128, and fp8 codes)
    kc = r // 8, e = r % 8, tg = t % 8, tp = t // 8, lane = 4 tg + kc
    code byte   ((tp (nb/2) + b//2) 32 + lane) 16 + (b%2) 8 + e
    q8_0 d      16 D + (t nb + b) 2                       (fp16, little endian)

V side
    vg = r // 4, h = (r % 4) // 2, s = r % 2
    c = (t % 8) // 2, f = t % 2, p = t // 8, lane = 4 vg + c, k = 2 f + p
    nibble      byte ((b//2) 32 + lane) 16 + (b%2) 8 + 4 h + k, bits 4s..4s+3
                (q5_1: the low 4 bits of q; q4_0: q + 8)
    q5_1 bit 4  byte 8 D + (lane (nb/2) + b//2) 4 + k, bit 4 s + 2 (b%2) + h
    q5_1 d, m   10 D (d) / 11 D (m) + ((c nb + b) 4 + 2 p + f) 2
    q4_0 d      8 D + ((c nb + b) 4 + 2 p + f) 2
    fp8 byte    (b 32 + lane) 16 + 8 h + 2 (2 p + s) + f

NVFP4 (K or V; scales per 16-element block b16 = j // 16; each 32-bit word of a
lane holds the 8 codes of one m16n8k16 A fragment, 4 bits each, and every byte
two codes of one token)
    K codes     b = j // 32, r = j % 32, c = r // 8, e = r % 8, lane = 4 (t % 8) + c,
                w = 2 b + e // 4
                byte ((w // 4) 32 + lane) 16 + (w % 4) 4 + (t // 8) + 2 ((e % 4) // 2),
                bits 4 (e % 2) ..                          (elements e, e + 1 share a byte)
    K scales    8 D + t (D/16) + b16                       (e4m3 bytes)
    V codes     r = j % 16, c = (t % 8) // 2, lane = 4 (r % 8) + c
                byte ((b16 // 4) 32 + lane) 16 + (b16 % 4) 4 + (t % 2) + 2 (t // 8),
                bits 4 (r // 8) ..                         (elements r, r + 8 share a byte)
    V scales    8 D + (c (D/16) + b16) 4 + (t % 2) + 2 (t // 8)

Segment sizes: K q8_0 17 D, K fp8 16 D, K nvfp4 9 D, V q5_1 12 D, V q4_0 9 D,
V fp8 16 D, V nvfp4 9 D.  Every byte of a segment belongs to exactly one token.

Pin: this module has no source outside the library's own header, so its
parity is pinned only by (a) the round trip unpack(pack(x)) == x, (b) the
check that the offsets of each format tile the segment exactly once, and
(c) hand-worked offsets in tests/golden/layout_offsets.txt.
"""
from __future__ import annotations

import numpy as np

PAGE = 16


def k_segment_bytes(fmt: str, D: int) -> int:
    return {"q8_0": 17 * D, "fp8": 16 * D, "nvfp4": 9 * D}[fmt]


def v_segment_bytes(fmt: str, D: int) -> int:
    return {"q5_1": 12 * D, "q4_0": 9 * D, "fp8": 16 * D, "nvfp4": 9 * D}[fmt]


def segment_bytes(side: str, fmt: str, D: int) -> int:
    return k_segment_bytes(fmt, D) if side == "k" else v_segment_bytes(fmt, D)


# --------------------------------------------------------------- K side -----

def k_code_offset(t, j, D):
    nb = D // 32
    b, r = j // 32, j % 32
    kc, e = r // 8, r % 8
    tg, tp = t % 8, t // 8
    lane = 4 * tg + kc
    return ((tp * (nb // 2) + b // 2) * 32 + lane) * 16 + (b % 2) * 8 + e


def k_d_offset(t, b, D):
    nb = D // 32
    return 16 * D + (t * nb + b) * 2


# --------------------------------------------------------------- V side -----

def _v_coords(t, j):
    b, r = j // 32, j % 32
    vg, h, s = r // 4, (r % 4) // 2, r % 2
    c, f, p = (t % 8) // 2, t % 2, t // 8
    lane = 4 * vg + c
    k = 2 * f + p
    return b, vg, h, s, c, f, p, lane, k


def v_nibble_offset(t, j, D):
    """(byte, shift) of the low nibble of element j of token t."""
    b, vg, h, s, c, f, p, lane, k = _v_coords(t, j)
    return ((b // 2) * 32 + lane) * 16 + (b % 2) * 8 + 4 * h + k, 4 * s


def v_hibit_offset(t, j, D):
    """(byte, bit) of bit 4 of a q5_1 code."""
    nb = D // 32
    b, vg, h, s, c, f, p, lane, k = _v_coords(t, j)
    return 8 * D + (lane * (nb // 2) + b // 2) * 4 + k, 4 * s + 2 * (b % 2) + h


def v_param_offset(t, b, D, base):
    nb = D // 32
    c, f, p = (t % 8) // 2, t % 2, t // 8
    return base + ((c * nb + b) * 4 + 2 * p + f) * 2


def v_fp8_offset(t, j, D):
    b, vg, h, s, c, f, p, lane, k = _v_coords(t, j)
    return (b * 32 + lane) * 16 + 8 * h + 2 * (2 * p + s) + f


# ------------------------------------------------------------ NVFP4 side ---

def nvfp4_code_offset(side: str, t, j, D):
    """(byte, shift) of the E2M1 code of element j of token t."""
    b16, r = j // 16, j % 16
    if side == "k":
        r32 = j % 32
        e = r32 % 8
        lane = 4 * (t % 8) + r32 // 8
        w = 2 * (j // 32) + e // 4
        return ((w // 4) * 32 + lane) * 16 + (w % 4) * 4 + t // 8 + 2 * ((e % 4) // 2), 4 * (e % 2)
    else:
        lane = 4 * (r % 8) + (t % 8) // 2
        byte_in_word = t % 2 + 2 * (t // 8)
        shift = 4 * (r // 8)
    return ((b16 // 4) * 32 + lane) * 16 + (b16 % 4) * 4 + byte_in_word, shift


def nvfp4_scale_offset(side: str, t, b16, D):
    if side == "k":
        return 8 * D + t * (D // 16) + b16
    c = (t % 8) // 2
    return 8 * D + (c * (D // 16) + b16) * 4 + t % 2 + 2 * (t // 8)


# ------------------------------------------------- one token row -> bytes ---

def _fp16_bytes(x: np.ndarray) -> np.ndarray:
    """fp16 [..., n] -> uint8 [..., n, 2] little endian."""
    u = np.ascontiguousarray(x, dtype=np.float16).view(np.uint16).astype(np.uint32)
    return np.stack([u & 0xFF, u >> 8], axis=-1).astype(np.uint8)


def row_bytes(side: str, fields: dict, t: np.ndarray, D: int):
    """Bytes owned by each row.

    fields: canonical fields of N rows (``q`` [N, D], ``d``/``m`` [N, nb]).
    t: int array [N] of the row's token position in its page.
    Returns (offsets int64 [N, n], values uint8 [N, n]).
    """
    fmt = fields["fmt"]
    q = np.asarray(fields["q"])
    N = q.shape[0]
    t = np.asarray(t, dtype=np.int64).reshape(N, 1)
    nb = D // 32
    j = np.arange(D, dtype=np.int64).reshape(1, D)
    offs, vals = [], []
    if fmt == "nvfp4":
        # two codes of the row per byte: elements (j, j + 1) for K, (j, j + 8) for V
        if side == "k":
            lo_j = j[:, 0::2]
            hi_q = q[:, 1::2]
        else:
            lo_j = j[:, (j[0] % 16) < 8]
            hi_q = q[:, (j[0] % 16) >= 8]
        off, sh = nvfp4_code_offset(side, t, lo_j, D)
        assert (np.asarray(sh) == 0).all()
        offs.append(np.broadcast_to(off, (N, D // 2)))
        vals.append((q[:, lo_j[0]] | (hi_q << 4)).astype(np.uint8))
        nb16 = D // 16
        bb = np.arange(nb16, dtype=np.int64).reshape(1, nb16)
        offs.append(np.broadcast_to(nvfp4_scale_offset(side, t, bb, D), (N, nb16)))
        vals.append(np.asarray(fields["sb"]).astype(np.uint8))
        return np.concatenate(offs, axis=1).astype(np.int64), np.concatenate(vals, axis=1).astype(np.uint8)
    if side == "k":
        if fmt not in ("q8_0", "fp8"):
            raise ValueError(f"K format {fmt} is not a K knob")
        offs.append(np.broadcast_to(k_code_offset(t, j, D), (N, D)))
        vals.append((q.astype(np.int64) + 128).astype(np.uint8) if fmt == "q8_0" else q.astype(np.uint8))
        if fmt == "q8_0":
            bb = np.arange(nb, dtype=np.int64).reshape(1, nb)
            o = k_d_offset(t, bb, D)                                   # [N, nb]
            offs.append(np.stack([o, o + 1], axis=-1).reshape(N, 2 * nb))
            vals.append(_fp16_bytes(fields["d"]).reshape(N, 2 * nb))
    else:
        if fmt in ("q5_1", "q4_0"):
            code = q.astype(np.int64) + (8 if fmt == "q4_0" else 0)     # q4_0 stores q + 8
            lo4 = code & 0xF
            je = j[:, 0::2]                                            # elements with s == 0
            byte_off, _ = v_nibble_offset(t, je, D)
            offs.append(np.broadcast_to(byte_off, (N, D // 2)))
            vals.append((lo4[:, 0::2] | (lo4[:, 1::2] << 4)).astype(np.uint8))
            if fmt == "q5_1":
                hb = (code >> 4) & 1
                # Elements sharing a bit-4 byte: same (vg, b // 2); order j so that the 8
                # elements of each byte are adjacent, then OR their bits together.
                jj = np.arange(D, dtype=np.int64)
                group = (jj % 32) // 4 * (nb // 2) + (jj // 32) // 2
                perm = np.argsort(group, kind="stable")
                _, bit = v_hibit_offset(np.zeros(1, np.int64), jj, D)
                bits = (hb[:, perm] << bit[perm]).reshape(N, D // 8, 8).sum(axis=-1)
                first = perm.reshape(D // 8, 8)[:, 0].reshape(1, D // 8)
                hoff, _ = v_hibit_offset(t, first, D)
                offs.append(np.broadcast_to(hoff, (N, D // 8)))
                vals.append(bits.astype(np.uint8))
            bb = np.arange(nb, dtype=np.int64).reshape(1, nb)
            dbase = 10 * D if fmt == "q5_1" else 8 * D
            o = v_param_offset(t, bb, D, dbase)
            offs.append(np.stack([o, o + 1], axis=-1).reshape(N, 2 * nb))
            vals.append(_fp16_bytes(fields["d"]).reshape(N, 2 * nb))
            if fmt == "q5_1":
                o = v_param_offset(t, bb, D, 11 * D)
                offs.append(np.stack([o, o + 1], axis=-1).reshape(N, 2 * nb))
                vals.append(_fp16_bytes(fields["m"]).reshape(N, 2 * nb))
        elif fmt == "fp8":
            offs.append(np.broadcast_to(v_fp8_offset(t, j, D), (N, D)))
            vals.append(q.astype(np.uint8))
        else:
            raise ValueError(f"V format {fmt} is not a V knob")
    return np.concatenate(offs, axis=1).astype(np.int64), np.concatenate(vals, axis=1).astype(np.uint8)


def write_rows(pool: np.ndarray, side: str, fields: dict, slots: np.ndarray, head: int, D: int,
               chunk: int = 65536) -> None:
    """Scatter quantized rows of one KV head into a pool [num_pages, Hkv, seg] (in place)."""
    slots = np.asarray(slots, dtype=np.int64)
    flat = pool.reshape(pool.shape[0], pool.shape[1], -1)
    for s0 in range(0, slots.size, chunk):
        sl = slots[s0:s0 + chunk]
        sub = {k: (v[s0:s0 + chunk] if isinstance(v, np.ndarray) else v) for k, v in fields.items()}
        offs, vals = row_bytes(side, sub, sl % PAGE, D)
        pages = (sl // PAGE).reshape(-1, 1)
        flat[np.broadcast_to(pages, offs.shape), head, offs] = vals


def read_rows(pool: np.ndarray, side: str, fmt: str, slots: np.ndarray, head: int, D: int,
              scale: float = 1.0) -> dict:
    """Decode rows of one KV head from pool bytes back into canonical fields."""
    slots = np.asarray(slots, dtype=np.int64)
    N = slots.size
    nb = D // 32
    t = (slots % PAGE).reshape(N, 1)
    page = (slots // PAGE).reshape(N, 1)
    seg = pool.reshape(pool.shape[0], pool.shape[1], -1)[:, head, :]
    j = np.arange(D, dtype=np.int64).reshape(1, D)
    bb = np.arange(nb, dtype=np.int64).reshape(1, nb)

    def f16_at(o):
        lo = seg[page, o].astype(np.uint16)
        hi = seg[page, o + 1].astype(np.uint16)
        return (lo | (hi << 8)).view(np.float16)

    if fmt == "nvfp4":
        off, sh = nvfp4_code_offset(side, t, j, D)
        code = (seg[page, off].astype(np.int64) >> sh) & 0xF
        b16 = np.arange(D // 16, dtype=np.int64).reshape(1, D // 16)
        return {"fmt": fmt, "q": code.astype(np.uint8), "sb": seg[page, nvfp4_scale_offset(side, t, b16, D)],
                "scale": float(np.float32(scale))}
    if side == "k":
        code = seg[page, k_code_offset(t, j, D)]
        if fmt == "q8_0":
            return {"fmt": fmt, "q": (code.astype(np.int64) - 128).astype(np.int8), "d": f16_at(k_d_offset(t, bb, D))}
        return {"fmt": fmt, "q": code, "scale": float(np.float32(scale))}
    if fmt in ("q5_1", "q4_0"):
        off, sh = v_nibble_offset(t, j, D)
        code = (seg[page, off].astype(np.int64) >> sh) & 0xF
        if fmt == "q5_1":
            hoff, hbit = v_hibit_offset(t, j, D)
            code |= ((seg[page, hoff].astype(np.int64) >> hbit) & 1) << 4
            return {"fmt": fmt, "q": code.astype(np.uint8), "d": f16_at(v_param_offset(t, bb, D, 10 * D)),
                    "m": f16_at(v_param_offset(t, bb, D, 11 * D))}
        return {"fmt": fmt, "q": (code - 8).astype(np.int8), "d": f16_at(v_param_offset(t, bb, D, 8 * D))}
    if fmt == "fp8":
        return {"fmt": fmt, "q": seg[page, v_fp8_offset(t, j, D)], "scale": float(np.float32(scale))}
    raise ValueError(fmt)
