"""Pins for the oracle's restatement of the pool byte layout (CPU only)."""
import os

import numpy as np
import pytest

from oracle import layout, quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_offsets.txt")

COMBOS = [("k", "q8_0"), ("k", "fp8"), ("k", "nvfp4"), ("v", "q5_1"), ("v", "q4_0"), ("v", "fp8"), ("v", "nvfp4")]


def _rows(fmt, n, D, rng):
    x = rng.standard_normal((n, D)).astype(np.float16)
    return quant.quantize_rows(x, fmt, 0.0123)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("side,fmt", COMBOS)
def test_offsets_tile_the_segment_once(side, fmt, D):
    rng = np.random.default_rng(0)
    f = _rows(fmt, 16, D, rng)
    offs, _ = layout.row_bytes(side, f, np.arange(16), D)
    seg = layout.segment_bytes(side, fmt, D)
    flat = np.sort(offs.reshape(-1))
    assert flat.size == seg and np.array_equal(flat, np.arange(seg))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("side,fmt", COMBOS)
def test_pack_unpack_round_trip(side, fmt, D):
    rng = np.random.default_rng(1)
    num_pages, hkv = 5, 3
    n = 57
    slots = rng.choice(num_pages * 16, size=n, replace=False)
    pool = rng.integers(0, 256, (num_pages, hkv, layout.segment_bytes(side, fmt, D)), dtype=np.uint8)
    before = pool.copy()
    fields = _rows(fmt, n, D, rng)
    layout.write_rows(pool, side, fields, slots, 1, D)
    back = layout.read_rows(pool, side, fmt, slots, 1, D, scale=0.0123)
    for key in ("q", "d", "m", "sb"):
        if key in fields:
            assert np.array_equal(back[key].view(np.uint8) if back[key].dtype == np.float16 else back[key],
                                  fields[key].view(np.uint8) if fields[key].dtype == np.float16 else fields[key])
    # other heads untouched, and untouched slots keep their bytes
    assert np.array_equal(pool[:, 0], before[:, 0]) and np.array_equal(pool[:, 2], before[:, 2])
    free = np.setdiff1d(np.arange(num_pages * 16), slots)
    zeros = _rows(fmt, free.size, D, rng)
    offs, _ = layout.row_bytes(side, zeros, free % 16, D)
    pg = (free // 16)[:, None]
    assert np.array_equal(pool[np.broadcast_to(pg, offs.shape), 1, offs],
                          before[np.broadcast_to(pg, offs.shape), 1, offs])


def test_q5_1_high_bit_and_nibble_split():
    """Codes 16..31 put their bit 4 in the bit-4 region, the rest in the nibble region."""
    D = 128
    q = np.zeros((1, D), np.uint8)
    q[0, 77] = 0x1B                    # bit 4 set, low nibble 0xB
    f = {"fmt": "q5_1", "q": q, "d": np.ones((1, 4), np.float16), "m": np.zeros((1, 4), np.float16)}
    pool = np.zeros((1, 1, layout.v_segment_bytes("q5_1", D)), np.uint8)
    layout.write_rows(pool, "v", f, np.array([11]), 0, D)
    seg = pool[0, 0]
    assert seg[723] == 0xB0            # t=11, j=77: nibble byte 723, upper nibble
    assert seg[1135] == 0x10           # bit-4 byte 1135, bit 4
    assert seg[:1024].sum() == 0xB0 and seg[1024:1280].sum() == 0x10


def golden_rows():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                what, t, jb, byte, extra = [p.strip() for p in line.split(";")]
                out.append((what, int(t), int(jb), int(byte), extra))
    return out


@pytest.mark.parametrize("row", golden_rows(), ids=lambda r: f"{r[0]}-t{r[1]}-{r[2]}")
def test_golden_offsets(row):
    what, t, jb, byte, extra = row
    D = 128
    if what == "kcode":
        assert layout.k_code_offset(t, jb, D) == byte
    elif what == "kd":
        assert layout.k_d_offset(t, jb, D) == byte
    elif what == "vnib":
        assert layout.v_nibble_offset(t, jb, D) == (byte, int(extra))
    elif what == "vhi":
        assert layout.v_hibit_offset(t, jb, D) == (byte, int(extra))
    elif what == "vd51":
        assert layout.v_param_offset(t, jb, D, 10 * D) == byte
    elif what == "vm51":
        assert layout.v_param_offset(t, jb, D, 11 * D) == byte
    elif what == "vd40":
        assert layout.v_param_offset(t, jb, D, 8 * D) == byte
    elif what == "vfp8":
        assert layout.v_fp8_offset(t, jb, D) == byte
    elif what in ("k4code", "v4code"):
        assert layout.nvfp4_code_offset(what[0], t, jb, D) == (byte, int(extra))
    elif what in ("k4scale", "v4scale"):
        assert layout.nvfp4_scale_offset(what[0], t, jb, D) == byte
    else:
        raise AssertionError(what)
