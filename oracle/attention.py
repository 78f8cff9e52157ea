"""Decode attention on the dequantized paged cache, written as its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

For sequence b with context T_b (the cache after the step's append) and
q_len Q, query row i sits at absolute position T_b - Q + i and sees keys
0 .. T_b - Q + i (for Q = 1 this is plain decode over the whole context; for
Q = K + 1 it is the causal verify of K speculative drafts, the memra README's
"Speculative decoding" item of the serving surface and the MTP rows of its
performance table).  Query head h reads KV head floor(h / G), G = Hq / Hkv.
With K^ and V^ the dequantized rows,

    s_t = (sum_j q_j K^[t, j]) / sqrt(D)
    p   = softmax(s)            (max subtracted first)
    o   = sum_t p_t V^[t, :]

all in float64.  Rows with no visible key return zeros.  The shared-prefix
workload needs nothing special here: page tables that point at the same pages
read the same rows.

Sliding window (the README's SWA ring, "Recent fixes" list): with a window of
W tokens the row at position p sees only keys max(0, p - W + 1) .. p.  Ring
page tables map position p to column (p // 16) % R of the sequence's row, so
only the last R pages of a sequence hold rows.

Pins: explicit triple loops on tiny inputs; a context of one token returns
that V^ row; q = 0 returns the mean of the visible V^ rows; float64
``torch.nn.functional.scaled_dot_product_attention`` (a library routine) on
the dequantized, GQA-expanded tensors with a causal mask; invariance under a
permutation of the page pool; for the window: explicit loops, a window of
one returns the row's own V^, q = 0 returns the mean of the window, a window
wider than the context is full attention, and float64 SDPA with a band mask
(tests/test_oracle_attention.py).
"""
from __future__ import annotations

import numpy as np

from . import quant

PAGE = 16


def attention_rows(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, sm_scale: float, window: int = 0,
                   start: int = 0) -> np.ndarray:
    """q [Q, Hq, D], k_hat / v_hat [T', Hkv, D] -> out [Q, Hq, D] float64 (causal over the last Q keys).

    The rows hold positions start .. start + T' - 1 of the sequence.  window > 0
    hides keys more than window - 1 positions before the query row.
    """
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    v_hat = np.asarray(v_hat, dtype=np.float64)
    Q, Hq, D = q.shape
    T, Hkv, _ = k_hat.shape
    G = Hq // Hkv
    out = np.zeros((Q, Hq, D), dtype=np.float64)
    for h in range(Hq):
        kh = h // G
        s_all = k_hat[:, kh, :] @ q[:, h, :].T * sm_scale          # [T, Q]
        for i in range(Q):
            last = T - Q + i                                       # last visible key (row index)
            if last < 0:
                continue
            first = 0
            if window > 0:
                first_pos = max(0, start + last - window + 1)
                if first_pos < start:
                    raise ValueError("the window reaches keys before the first row given")
                first = first_pos - start
            s = s_all[first: last + 1, i]
            p = np.exp(s - s.max())
            out[i, h] = (p @ v_hat[first: last + 1, kh, :]) / p.sum()
    return out


def quantize_cache(w) -> dict:
    """Quantize every unique cached row of a workload, per KV head: {'k': [fields per head], 'v': [...]}."""
    out = {"k": [], "v": []}
    for h in range(w.n_kv_heads):
        out["k"].append(quant.quantize_rows(w.k_rows[:, h, :], w.k_fmt, w.k_scale))
        out["v"].append(quant.quantize_rows(w.v_rows[:, h, :], w.v_fmt, w.v_scale))
    return out


def first_position(w, b: int) -> int:
    """First position of sequence b that holds a row (0 unless the page table is a ring)."""
    return int(w.first_pos[b]) if getattr(w, "ring", False) else 0


def sequence_rows(w, b: int) -> np.ndarray:
    """Indices (into the unique rows) of sequence b's tokens first_position .. T_b - 1, through its page table."""
    T = int(w.seq_lens[b])
    tok = np.arange(first_position(w, b), T, dtype=np.int64)
    col = tok // PAGE
    if getattr(w, "ring", False):
        col = col % w.page_table.shape[1]
    slots = w.page_table[b, col].astype(np.int64) * PAGE + tok % PAGE
    order = np.argsort(w.slots, kind="stable")
    pos = np.searchsorted(w.slots[order], slots)
    rows = order[pos]
    if not np.array_equal(w.slots[rows], slots):
        raise ValueError("page table points at a slot no row was written to")
    return rows


def reference(w, cache=None, rows=None) -> np.ndarray:
    """Oracle output [B, Q, Hq, D] float64.

    rows: optional iterable of (b, i, h) to compute; other entries stay NaN.
    """
    if cache is None:
        cache = quantize_cache(w)
    B, Q, Hq, D = w.q.shape
    G = Hq // w.n_kv_heads
    out = np.full((B, Q, Hq, D), np.nan)
    want = None
    if rows is not None:
        want = {}
        for (b, i, h) in rows:
            want.setdefault(b, set()).add(h // G)
    for b in range(B):
        if want is not None and b not in want:
            continue
        r = sequence_rows(w, b)
        for kh in range(w.n_kv_heads):
            if want is not None and kh not in want[b]:
                continue
            k_hat = quant.dequantize_rows(quant.select_rows(cache["k"][kh], r))[:, None, :]
            v_hat = quant.dequantize_rows(quant.select_rows(cache["v"][kh], r))[:, None, :]
            heads = slice(kh * G, (kh + 1) * G)
            out[b, :, heads, :] = attention_rows(w.q[b, :, heads, :], k_hat, v_hat, w.sm_scale,
                                                 window=getattr(w, "window", 0), start=first_position(w, b))
    if rows is not None:
        mask = np.zeros(out.shape[:3], dtype=bool)
        for (b, i, h) in rows:
            mask[b, i, h] = True
        out[~mask] = np.nan
    return out


def build_pools(w, cache=None, fill=None, rows=None):
    """Pool bytes [num_pages, Hkv, seg] for K and V holding the given rows (default: all unique rows).

    fill: (k_pool, v_pool) arrays to start from (the bytes of unwritten slots), else zeros.
    """
    from . import layout
    if cache is None:
        cache = quantize_cache(w)
    D = w.head_dim
    kseg = layout.k_segment_bytes(w.k_fmt, D)
    vseg = layout.v_segment_bytes(w.v_fmt, D)
    if fill is None:
        kp = np.zeros((w.num_pages, w.n_kv_heads, kseg), np.uint8)
        vp = np.zeros((w.num_pages, w.n_kv_heads, vseg), np.uint8)
    else:
        kp, vp = (np.array(f, dtype=np.uint8, copy=True).reshape(w.num_pages, w.n_kv_heads, -1) for f in fill)
    idx = np.arange(w.slots.size) if rows is None else np.asarray(rows)
    for h in range(w.n_kv_heads):
        layout.write_rows(kp, "k", quant.select_rows(cache["k"][h], idx), w.slots[idx], h, D)
        layout.write_rows(vp, "v", quant.select_rows(cache["v"][h], idx), w.slots[idx], h, D)
    return kp, vp
