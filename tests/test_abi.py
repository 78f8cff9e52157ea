"""The C ABI library loads, exports every declared symbol, and validates on the host (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "memra.h")


@pytest.fixture(scope="module")
def memra():
    from decode_attention_block_memra_gb300 import _build
    try:
        _build.build()
    except RuntimeError as e:          # no nvcc on this machine
        pytest.skip(str(e))
    import decode_attention_block_memra_gb300 as m
    m.lib()
    return m


def declared_functions():
    """Every function declared in include/*.h."""
    names = set()
    inc = os.path.dirname(HEADER)
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(memra_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(memra):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(memra.library_path())
    for n in names:
        assert hasattr(lib, n), n


def test_segment_and_pool_sizes(memra):
    D = 128
    assert memra.kv_segment_bytes("q8_0", False, D) == 17 * D
    assert memra.kv_segment_bytes("fp8", False, D) == 16 * D
    assert memra.kv_segment_bytes("q5_1", True, D) == 12 * D
    assert memra.kv_segment_bytes("q4_0", True, 256) == 9 * 256
    assert memra.kv_segment_bytes("fp8", True, 256) == 16 * 256
    assert memra.kv_segment_bytes("nvfp4", False, D) == 9 * D
    assert memra.kv_segment_bytes("nvfp4", True, 256) == 9 * 256
    # K knobs are q8_0 | fp8 and V knobs q5_1 | q4_0 | fp8 only
    assert memra.kv_segment_bytes("q5_1", False, D) == 0
    assert memra.kv_segment_bytes("q8_0", True, D) == 0
    assert memra.kv_segment_bytes("q8_0", False, 64) == 0
    assert memra.kv_pool_bytes("q8_0", False, 16384, 4, 128) == 16384 * 4 * 2176
    assert memra.kv_pool_bytes("q8_0", False, 10, 4, 128, page_size=32) == 0
    from oracle import layout
    for side, fmt in (("k", "q8_0"), ("k", "fp8"), ("k", "nvfp4"), ("v", "q5_1"), ("v", "q4_0"), ("v", "fp8"),
                      ("v", "nvfp4")):
        for D in (128, 256):
            assert memra.kv_segment_bytes(fmt, side == "v", D) == layout.segment_bytes(side, fmt, D)


def test_split_plan_and_workspace(memra):
    assert memra.num_splits(0) == 0
    assert memra.num_splits(1) == 1
    C = memra.SPLIT_TOKENS
    assert C == 1280
    assert memra.num_splits(C) == 1
    assert memra.num_splits(C + 1) == 2
    assert memra.num_splits(262144) == 205
    rows, ns, D = 1 * 1 * 32, 205, 128
    o = rows * ns * D * 4
    assert memra.decode_attn_workspace_bytes(1, 1, 32, 128, 262144) == ((o + 255) // 256) * 256 + rows * ns * 4
    assert memra.decode_attn_workspace_bytes(4, 1, 8, 128, 0) == 0
    assert memra.decode_attn_workspace_bytes(1, 0, 8, 128, 10) == 0


def _cache(memra, **kw):
    c = memra.KVCacheStruct(0, 1, 16, 2, 128, 4, 4096, 8192, 1.0, 1.0, 0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _decode(memra, c, **kw):
    a = dict(q=4096, pt=4096, maxp=4, sl=4096, maxlen=64, B=1, Q=1, Hq=8, Hkv=2, D=128, scale=0.1, ws=4096,
             wsb=1 << 20, out=4096)
    a.update(kw)
    return memra.lib().memra_decode_attn(ctypes.byref(c), a["q"], a["pt"], a["maxp"], a["sl"], a["maxlen"], a["B"],
                                         a["Q"], a["Hq"], a["Hkv"], a["D"], a["scale"], a["ws"], a["wsb"], a["out"],
                                         None)


def test_host_validation_without_gpu(memra):
    """Every argument error is caught on the host before any CUDA call."""
    L = memra.lib()
    assert L.memra_kv_append(None, 16, 16, 16, 1, None) == 1
    assert L.memra_kv_append(ctypes.byref(_cache(memra, k_fmt=1)), 16, 16, 16, 1, None) == 2    # q5_1 is not a K knob
    assert L.memra_kv_append(ctypes.byref(_cache(memra, v_fmt=0)), 16, 16, 16, 1, None) == 2    # q8_0 is not a V knob
    assert L.memra_kv_append(ctypes.byref(_cache(memra, page_size=32)), 16, 16, 16, 1, None) == 2
    assert L.memra_kv_append(ctypes.byref(_cache(memra, head_dim=64)), 16, 16, 16, 1, None) == 2
    assert L.memra_kv_append(ctypes.byref(_cache(memra, k_pool=4100)), 16, 16, 16, 1, None) == 1  # misaligned
    assert L.memra_kv_append(ctypes.byref(_cache(memra, k_fmt=3, k_scale=0.0)), 16, 16, 16, 1, None) == 1
    assert L.memra_kv_append(ctypes.byref(_cache(memra, v_fmt=4, v_scale=float("inf"))), 16, 16, 16, 1, None) == 1
    assert L.memra_kv_append(ctypes.byref(_cache(memra, k_fmt=5)), 16, 16, 16, 1, None) == 2      # no format 5
    assert L.memra_kv_append(ctypes.byref(_cache(memra)), 16, 16, 16, -1, None) == 1
    assert L.memra_kv_append(ctypes.byref(_cache(memra)), 0, 16, 16, 1, None) == 1
    assert L.memra_kv_append(ctypes.byref(_cache(memra)), 16, 16, 16, 0, None) == 0               # no-op
    c = _cache(memra)
    assert _decode(memra, c, B=0) == 0                                  # empty batch: no-op
    assert _decode(memra, c, Hq=7) == 1                                 # 7 query heads over 2 KV heads
    assert _decode(memra, c, Hkv=4) == 1                                # disagrees with the cache
    assert _decode(memra, c, D=256) == 1
    assert _decode(memra, c, wsb=10) == 3                               # workspace too small
    assert _decode(memra, c, q=4097) == 1
    assert _decode(memra, c, scale=float("nan")) == 1
    assert _decode(memra, c, Q=0) == 1
    assert _decode(memra, c, Q=9, Hq=16, wsb=10) == 3                   # 72 rows per KV head pass the limits
    assert _decode(memra, c, Q=17, Hq=16) == 2                          # q_len above MEMRA_MAX_Q_LEN
    assert _decode(memra, c, Hq=258) == 2                               # group 129 > MEMRA_MAX_GROUP
    assert _decode(memra, c, B=65536) == 2                              # grid z limit
    assert L.memra_read_status(None, None, None) == 1
    # the test hook of the bounded waits checks its limit before anything else
    for bad_ns in (0, 10 ** 9 + 1):
        assert L.memra_testing_decode_attn_short_page(ctypes.byref(c), 4096, 4096, 4, 4096, 64, 1, 1, 8, 2, 128,
                                                      0.1, 4096, 1 << 20, 4096, bad_ns, None) == 1
    assert L.memra_testing_scale_division_mismatches(None, 1, 4096, None) == 1
    assert L.memra_testing_scale_division_mismatches(4096, 0, 4096, None) == 1
    assert L.memra_testing_scale_division_mismatches(4096, 65536, 4096, None) == 1
    assert memra.status_string(3) == "workspace too small"
    assert memra.status_string(99) == "unknown status"


def _cascade(memra, c, prefix, **kw):
    a = dict(q=4096, pt=4096, maxp=4, sl=4096, maxlen=64, B=1, Q=1, Hq=8, Hkv=2, D=128, scale=0.1, ws=4096,
             wsb=1 << 20, out=4096)
    a.update(kw)
    return memra.lib().memra_decode_attn_cascade(ctypes.byref(c), a["q"], a["pt"], a["maxp"], a["sl"], a["maxlen"],
                                                 prefix, a["B"], a["Q"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                                                 a["ws"], a["wsb"], a["out"], None)


def test_cascade_workspace_and_host_validation(memra):
    # 16 sequences of 4,860 tokens over a 4,096-token prefix, 32 query heads
    for D, chunk in ((128, 64), (256, 64)):
        # own keys (764 of them) split no finer than 512 tokens: 2 partials per row
        rows, chunks, ns = 16 * 32, 4096 // chunk, 2
        suf = ((rows * ns * D * 4 + 255) // 256) * 256 + rows * ns * 4
        pre_o = rows * chunks * D * 4
        want = ((suf + 255) // 256) * 256 + ((pre_o + 255) // 256) * 256 + rows * chunks * 4
        assert memra.decode_attn_cascade_workspace_bytes(16, 1, 32, D, 4860, 4096) == want
    assert memra.decode_attn_cascade_workspace_bytes(16, 1, 32, 128, 4860, 4004) == 0     # not whole pages
    assert memra.decode_attn_cascade_workspace_bytes(16, 1, 32, 128, 4860, 4880) == 0     # beyond the context
    assert memra.decode_attn_cascade_workspace_bytes(16, 1, 32, 128, 4860, 0) >= \
        memra.decode_attn_workspace_bytes(16, 1, 32, 128, 4860)
    c = _cache(memra)
    assert _cascade(memra, c, 8) == 1                       # not a multiple of 16
    assert _cascade(memra, c, -16) == 1
    assert _cascade(memra, c, 64) == 1                      # no key left for the new token
    assert _cascade(memra, c, 48, wsb=10) == 3              # workspace too small
    assert _cascade(memra, c, 80, maxlen=100) == 1          # five prefix pages, four table columns
    assert _cascade(memra, c, 16, B=0) == 0                 # empty batch: no-op


def _header_defines():
    text = open(HEADER).read()
    out = {}
    for name, val in re.findall(r"^#define\s+(MEMRA_[A-Z0-9_]+)\s+(.+?)\s*(?:/\*.*)?$", text, flags=re.M):
        out[name] = val
    return out


def test_binding_constants_match_the_header():
    """The Python binding's copies of the header's constants agree with include/memra.h."""
    import decode_attention_block_memra_gb300 as m
    d = _header_defines()

    def value(name):
        return int(eval(d[name].replace("u", ""), {}))           # e.g. "(16u << 20)"

    assert value("MEMRA_NOALLOC_SCRATCH_BYTES") == m.NOALLOC_SCRATCH_BYTES
    assert value("MEMRA_PAGE_SIZE") == m.PAGE_SIZE
    assert value("MEMRA_SPLIT_TOKENS") == m.SPLIT_TOKENS
    for bit in ("BAD_PAGE", "BAD_SLOT", "BAD_SEQ_LEN", "TIMEOUT", "PREFIX"):
        assert value("MEMRA_DEVERR_" + bit) == getattr(m, "DEVERR_" + bit)
