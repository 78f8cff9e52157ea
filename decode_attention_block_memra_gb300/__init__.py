"""Python binding of the memra decode-attention C ABI (include/memra.h).

Argument marshalling only: every step of the hot path (quantize-append,
split-K decode, log-sum-exp combine) runs in the CUDA kernels of
``libmemra.so``.  PyTorch supplies device memory and the current stream; the
functions take torch tensors (or raw integers for pointers) and raise
``MemraError`` on any non-zero status.  There is no CPU fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

FORMATS = {"q8_0": 0, "q5_1": 1, "q4_0": 2, "fp8": 3, "nvfp4": 4}
PAGE_SIZE = 16
SPLIT_TOKENS = 1280

DEVERR_BAD_PAGE = 1
DEVERR_BAD_SLOT = 2
DEVERR_BAD_SEQ_LEN = 4
DEVERR_TIMEOUT = 8
DEVERR_PREFIX = 16


class MemraError(RuntimeError):
    def __init__(self, status: int, where: str, flags: int = 0):
        self.status = status
        self.flags = flags
        msg = f"{where}: {status_string(status)} (status {status})"
        if flags:
            msg += f", device flags 0x{flags:x}"
        super().__init__(msg)


class KVCacheStruct(ctypes.Structure):
    """Mirror of memra_kv_cache."""
    _fields_ = [
        ("k_fmt", ctypes.c_int32),
        ("v_fmt", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("status", ctypes.c_void_p),
    ]


_LIB = None

_SIGS = {
    "memra_kv_segment_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 3),
    "memra_kv_pool_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 6),
    "memra_kv_append": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "memra_decode_attn_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 5),
    "memra_decode_attn": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_void_p] + [ctypes.c_int32] * 6 +
                          [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "memra_decode_attn_partials": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_int32, ctypes.c_void_p] + [ctypes.c_int32] * 6 +
                                   [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                    ctypes.c_void_p]),
    "memra_decode_attn_combine": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p] +
                                  [ctypes.c_int32] * 6 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                          ctypes.c_void_p]),
    "memra_decode_step": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] +
                          [ctypes.c_int32] * 6 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                  ctypes.c_void_p]),
    "memra_decode_attn_window": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_void_p] + [ctypes.c_int32] * 6 +
                                 [ctypes.c_float, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                  ctypes.c_void_p]),
    "memra_decode_step_window": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] +
                                 [ctypes.c_int32] * 6 + [ctypes.c_float, ctypes.c_int32, ctypes.c_void_p,
                                                         ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "memra_decode_attn_cascade_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 6),
    "memra_decode_attn_cascade": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int32, ctypes.c_void_p] + [ctypes.c_int32] * 7 +
                                  [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                   ctypes.c_void_p]),
    "memra_decode_step_cascade": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] +
                                  [ctypes.c_int32] * 7 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                                          ctypes.c_void_p, ctypes.c_void_p]),
    "memra_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int32, ctypes.c_void_p] + [ctypes.c_int32] * 6 +
                                  [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]),
    "memra_testing_decode_attn_short_page": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.c_void_p,
                                                            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] +
                                             [ctypes.c_int32] * 6 + [ctypes.c_float, ctypes.c_void_p,
                                                                     ctypes.c_size_t, ctypes.c_void_p,
                                                                     ctypes.c_uint64, ctypes.c_void_p]),
    "memra_testing_scale_division_mismatches": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                                ctypes.c_void_p]),
    "memra_read_status": (ctypes.c_int, [ctypes.POINTER(KVCacheStruct), ctypes.POINTER(ctypes.c_int32),
                                         ctypes.c_void_p]),
    "memra_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "memra_num_splits": (ctypes.c_int32, [ctypes.c_int32]),
}


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libmemra.so (built in-tree by ``_build.build()``); raises if absent."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libmemra.so is not built ({path}); run __graft_entry__.build() first")
        h = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = h
    return _LIB


def status_string(status: int) -> str:
    return lib().memra_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise MemraError(rc, where)


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fmt_id(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def kv_segment_bytes(fmt, is_v: bool, head_dim: int) -> int:
    return int(lib().memra_kv_segment_bytes(fmt_id(fmt), int(bool(is_v)), head_dim))


def kv_pool_bytes(fmt, is_v: bool, num_pages: int, n_kv_heads: int, head_dim: int, page_size: int = PAGE_SIZE) -> int:
    return int(lib().memra_kv_pool_bytes(fmt_id(fmt), int(bool(is_v)), num_pages, page_size, n_kv_heads, head_dim))


def num_splits(seq_len: int) -> int:
    return int(lib().memra_num_splits(int(seq_len)))


def decode_attn_workspace_bytes(batch: int, q_len: int, n_heads: int, head_dim: int, max_seq_len: int) -> int:
    return int(lib().memra_decode_attn_workspace_bytes(batch, q_len, n_heads, head_dim, max_seq_len))


class KVCache:
    """A paged KV cache: the two pools and the status word as torch device tensors."""

    def __init__(self, k_fmt, v_fmt, num_pages: int, n_kv_heads: int, head_dim: int, k_scale: float = 1.0,
                 v_scale: float = 1.0, device="cuda", k_pool=None, v_pool=None):
        import torch
        self.k_fmt, self.v_fmt = k_fmt, v_fmt
        self.num_pages, self.n_kv_heads, self.head_dim = num_pages, n_kv_heads, head_dim
        kb = kv_pool_bytes(k_fmt, False, num_pages, n_kv_heads, head_dim)
        vb = kv_pool_bytes(v_fmt, True, num_pages, n_kv_heads, head_dim)
        if kb == 0 or vb == 0:
            raise MemraError(2, "KVCache")
        self.k_pool = k_pool if k_pool is not None else torch.zeros(kb, dtype=torch.uint8, device=device)
        self.v_pool = v_pool if v_pool is not None else torch.zeros(vb, dtype=torch.uint8, device=device)
        assert self.k_pool.numel() == kb and self.v_pool.numel() == vb
        self.status = torch.zeros(4, dtype=torch.int32, device=device)
        self.struct = KVCacheStruct(fmt_id(k_fmt), fmt_id(v_fmt), PAGE_SIZE, n_kv_heads, head_dim, num_pages,
                                    self.k_pool.data_ptr(), self.v_pool.data_ptr(), float(k_scale), float(v_scale),
                                    self.status.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self.struct)


def kv_append(cache: KVCache, k, v, slot_mapping, n_tok: int | None = None, stream=None) -> None:
    """memra_kv_append: k, v fp16 [n_tok, Hkv, D]; slot_mapping int32 [n_tok]."""
    n = int(slot_mapping.shape[0]) if n_tok is None else n_tok
    _check(lib().memra_kv_append(cache.ref, _ptr(k), _ptr(v), _ptr(slot_mapping), n, _stream(stream)),
           "memra_kv_append")


def _decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace, sm_scale):
    B, Q, Hq, D = q.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return (cache.ref, _ptr(q), _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens), int(max_seq_len), B, Q,
            Hq, cache.n_kv_heads, D, float(sm_scale if sm_scale is not None else D ** -0.5), _ptr(workspace),
            ws_bytes, _ptr(out))


def decode_attn(cache: KVCache, q, page_table, seq_lens, max_seq_len: int, out, workspace, sm_scale=None,
                stream=None, window: int = 0) -> None:
    """memra_decode_attn: q fp16 [B, Q, Hq, D] -> out fp16 [B, Q, Hq, D].

    window > 0: memra_decode_attn_window (sliding window; page_table rows are rings).
    """
    a = _decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace, sm_scale)
    if window:
        _check(lib().memra_decode_attn_window(*a[:12], int(window), *a[12:], _stream(stream)),
               "memra_decode_attn_window")
        return
    _check(lib().memra_decode_attn(*a, _stream(stream)), "memra_decode_attn")


def decode_attn_partials(cache: KVCache, q, page_table, seq_lens, max_seq_len: int, out, workspace, sm_scale=None,
                         stream=None) -> None:
    _check(lib().memra_decode_attn_partials(*_decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace,
                                                          sm_scale), _stream(stream)), "memra_decode_attn_partials")


def decode_attn_combine(cache: KVCache, seq_lens, max_seq_len: int, max_pages_per_seq: int, batch: int, q_len: int,
                        n_heads: int, out, workspace, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().memra_decode_attn_combine(cache.ref, _ptr(seq_lens), int(max_seq_len), int(max_pages_per_seq), batch,
                                           q_len, n_heads, cache.head_dim, _ptr(workspace), ws_bytes, _ptr(out),
                                           _stream(stream)), "memra_decode_attn_combine")


def decode_step(cache: KVCache, k_new, v_new, q, page_table, seq_lens, max_seq_len: int, out, workspace,
                sm_scale=None, stream=None, window: int = 0) -> None:
    """memra_decode_step: store the step's rows (k_new, v_new fp16 [B, Q, Hkv, D]) and attend, in one pass.

    seq_lens include the Q new tokens; their rows go to the positions
    seq_lens[b] - Q .. seq_lens[b] - 1 of each sequence's pages.  window > 0:
    memra_decode_step_window (sliding window; page_table rows are rings).
    """
    a = _decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace, sm_scale)
    if window:
        _check(lib().memra_decode_step_window(a[0], _ptr(k_new), _ptr(v_new), *a[1:12], int(window), *a[12:],
                                              _stream(stream)), "memra_decode_step_window")
        return
    _check(lib().memra_decode_step(a[0], _ptr(k_new), _ptr(v_new), *a[1:], _stream(stream)), "memra_decode_step")


def decode_attn_cascade_workspace_bytes(batch: int, q_len: int, n_heads: int, head_dim: int, max_seq_len: int,
                                        prefix_len: int) -> int:
    return int(lib().memra_decode_attn_cascade_workspace_bytes(batch, q_len, n_heads, head_dim, max_seq_len,
                                                               prefix_len))


def decode_attn_cascade(cache: KVCache, q, page_table, seq_lens, max_seq_len: int, prefix_len: int, out, workspace,
                        sm_scale=None, stream=None, k_new=None, v_new=None) -> None:
    """memra_decode_attn_cascade (or memra_decode_step_cascade when k_new / v_new are given).

    Keys 0 .. prefix_len - 1 of every sequence are the pages of page_table row
    0's first prefix_len / 16 columns, attended once per KV head for all rows
    on the tcgen05 tensor cores; each sequence's own keys go through the split
    kernel; the workspace is decode_attn_cascade_workspace_bytes(...).
    """
    a = _decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace, sm_scale)
    if k_new is not None or v_new is not None:
        _check(lib().memra_decode_step_cascade(a[0], _ptr(k_new), _ptr(v_new), *a[1:6], int(prefix_len), *a[6:],
                                               _stream(stream)), "memra_decode_step_cascade")
        return
    _check(lib().memra_decode_attn_cascade(*a[:6], int(prefix_len), *a[6:], _stream(stream)),
           "memra_decode_attn_cascade")


NOALLOC_SCRATCH_BYTES = 16 << 20


def decode_attn_noalloc(cache: KVCache, q, page_table, seq_lens, max_seq_len: int, out, sm_scale=None,
                        stream=None) -> None:
    """memra_decode_attn_noalloc: decode attention without a workspace, for callers that cannot allocate.

    The split-K partials go to a fixed library-owned device array of
    NOALLOC_SCRATCH_BYTES; calls that may overlap on the GPU race on it.
    """
    B, Q, Hq, D = q.shape
    _check(lib().memra_decode_attn_noalloc(cache.ref, _ptr(q), _ptr(page_table), int(page_table.shape[1]),
                                           _ptr(seq_lens), int(max_seq_len), B, Q, Hq, cache.n_kv_heads, D,
                                           float(sm_scale if sm_scale is not None else D ** -0.5), _ptr(out),
                                           _stream(stream)), "memra_decode_attn_noalloc")


def testing_decode_attn_short_page(cache: KVCache, q, page_table, seq_lens, max_seq_len: int, out, workspace,
                                   page_wait_ns: int, sm_scale=None, stream=None) -> None:
    """memra_testing_decode_attn_short_page (memra_testing.h): decode attention whose first CTA's first
    page wait cannot complete and runs out after page_wait_ns; the call then flags DEVERR_TIMEOUT."""
    a = _decode_args(cache, q, page_table, seq_lens, max_seq_len, out, workspace, sm_scale)
    _check(lib().memra_testing_decode_attn_short_page(*a, int(page_wait_ns), _stream(stream)),
           "memra_testing_decode_attn_short_page")


def testing_scale_division_mismatches(scales, mismatches, stream=None) -> None:
    """memra_testing_scale_division_mismatches (memra_testing.h): adds to mismatches (one int64 on the device)
    the (fp16 x, scale) pairs whose division-free quotient differs from the IEEE one."""
    _check(lib().memra_testing_scale_division_mismatches(_ptr(scales), int(scales.numel()), _ptr(mismatches),
                                                         _stream(stream)), "memra_testing_scale_division_mismatches")


def read_status(cache: KVCache, stream=None) -> int:
    """memra_read_status: synchronizes, returns and clears the device error bits."""
    flags = ctypes.c_int32(0)
    rc = lib().memra_read_status(cache.ref, ctypes.byref(flags), _stream(stream))
    if rc not in (0, 5):
        raise MemraError(rc, "memra_read_status")
    return int(flags.value)
