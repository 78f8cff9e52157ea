"""Complete parity of a workload: every pool byte and every output row against the oracle.

Test infrastructure (imports ``oracle/``).  At the full sizes the oracle is
too slow for one core (the head_dim 256 sweep quantizes 2.4 G values per
side), so the work is cut into independent pieces and spread over the host's
cores with a ``spawn`` process pool (a forked child of a process that has
used CUDA can hang):

* pool pieces: (side, KV head, range of pages).  The oracle quantizes every
  unique row whose slot lies in the range, writes it into a copy of the bytes
  the pool started from, and compares the whole range with the GPU's bytes,
  so untouched slots must also be unchanged;
* attention pieces: (sequence, KV head).  The oracle quantizes and
  dequantizes that sequence's rows through its page table, runs the float64
  definition for the query rows of that KV head, and compares them all with
  the GPU output.

Every piece calls the oracle's own functions unchanged; nothing is sampled.
The arrays reach the workers as ``.npy`` files in a temporary directory
(memory-mapped there), on ``/dev/shm`` when it has room.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile
from concurrent.futures import ProcessPoolExecutor
from types import SimpleNamespace

import numpy as np

PAGE = 16

_OPEN = {}


def _load(spec, name):
    key = (spec["dir"], name)
    if key not in _OPEN:
        _OPEN[key] = np.load(os.path.join(spec["dir"], name + ".npy"), mmap_mode="r")
    return _OPEN[key]


def _view(spec):
    """The page-table fields the oracle's sequence_rows reads, from the shared files."""
    return SimpleNamespace(seq_lens=_load(spec, "seq_lens"), page_table=_load(spec, "page_table"),
                           slots=_load(spec, "slots"), ring=spec["ring"],
                           first_pos=_load(spec, "first_pos") if spec["ring"] else None)


def _pool_piece(spec, side, head, p0, p1):
    """Expected bytes of pages [p0, p1) of one KV head against the GPU's; returns (bad bytes, first bad)."""
    from oracle import layout, quant
    fmt = spec[side + "_fmt"]
    order = _load(spec, "slot_order")
    sorted_slots = _load(spec, "sorted_slots")
    lo = np.searchsorted(sorted_slots, p0 * PAGE)
    hi = np.searchsorted(sorted_slots, p1 * PAGE)
    rows = np.sort(np.asarray(order[lo:hi]))
    fill = _load(spec, side + "_fill")
    want = np.array(fill[p0:p1, head:head + 1, :], copy=True)
    if rows.size:
        src = _load(spec, side + "_rows")
        fields = quant.quantize_rows(np.asarray(src[rows, head, :]), fmt, spec[side + "_scale"])
        slots = np.asarray(_load(spec, "slots")[rows]).astype(np.int64) - p0 * PAGE
        layout.write_rows(want, side, fields, slots, 0, spec["head_dim"])
    got = np.asarray(_load(spec, side + "_gpu")[p0:p1, head:head + 1, :])
    bad = np.argwhere(want != got)
    if bad.size == 0:
        return 0, None
    first = bad[0]
    return int(len(bad)), (int(first[0]) + p0, head, int(first[2]))


def _attention_piece(spec, b, kh):
    """Oracle rows of sequence b, KV head kh against the GPU's; returns (max |err|, all finite, rows)."""
    from oracle import attention, quant
    w = _view(spec)
    rows = attention.sequence_rows(w, b)
    k = quant.quantize_rows(np.asarray(_load(spec, "k_rows")[rows, kh, :]), spec["k_fmt"], spec["k_scale"])
    v = quant.quantize_rows(np.asarray(_load(spec, "v_rows")[rows, kh, :]), spec["v_fmt"], spec["v_scale"])
    k_hat = quant.dequantize_rows(k)[:, None, :]
    v_hat = quant.dequantize_rows(v)[:, None, :]
    G = spec["group"]
    heads = slice(kh * G, (kh + 1) * G)
    q = np.asarray(_load(spec, "q")[b, :, heads, :])
    ref = attention.attention_rows(q, k_hat, v_hat, spec["sm_scale"], window=spec["window"],
                                   start=attention.first_position(w, b))
    got = np.asarray(_load(spec, "out")[b, :, heads, :]).astype(np.float64)
    finite = bool(np.isfinite(got).all())
    err = float(np.abs(got - ref).max()) if finite else float("inf")
    return err, finite, ref.shape[0] * ref.shape[1]


def _workdir(nbytes):
    shm = "/dev/shm"
    try:
        if os.path.isdir(shm) and shutil.disk_usage(shm).free > 2 * nbytes + (1 << 30):
            return tempfile.mkdtemp(prefix="memra_parity_", dir=shm)
    except OSError:
        pass
    return tempfile.mkdtemp(prefix="memra_parity_")


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def check(w, out, k_pool=None, v_pool=None, k_fill=None, v_fill=None, tol=2e-3, pages_per_piece=2048):
    """Compare every output row (and, given the GPU pools, every pool byte) of w with the oracle.

    out: GPU fp16 [B, Q, Hq, D].  k_pool / v_pool: GPU pool bytes; k_fill / v_fill:
    the bytes the pools started from (zeros if None).  Returns a summary dict and
    raises AssertionError on the first mismatch class found.
    """
    B, Q, Hq, D = w.q.shape
    arrays = {"q": w.q, "out": np.asarray(out), "k_rows": w.k_rows, "v_rows": w.v_rows,
              "slots": w.slots, "seq_lens": w.seq_lens, "page_table": w.page_table}
    if getattr(w, "ring", False):
        arrays["first_pos"] = w.first_pos
    check_pools = k_pool is not None
    if check_pools:
        order = np.argsort(w.slots, kind="stable")
        arrays["slot_order"] = order
        arrays["sorted_slots"] = w.slots[order]
        for side, pool, fill in (("k", k_pool, k_fill), ("v", v_pool, v_fill)):
            pool = np.asarray(pool).reshape(w.num_pages, w.n_kv_heads, -1)
            arrays[side + "_gpu"] = pool
            arrays[side + "_fill"] = np.zeros_like(pool) if fill is None else \
                np.asarray(fill).reshape(pool.shape)
    total = sum(a.nbytes for a in arrays.values())
    d = _workdir(total)
    try:
        for name, a in arrays.items():
            np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(a))
        spec = {"dir": d, "k_fmt": w.k_fmt, "v_fmt": w.v_fmt, "k_scale": float(w.k_scale),
                "v_scale": float(w.v_scale), "head_dim": D, "group": Hq // w.n_kv_heads, "sm_scale": w.sm_scale,
                "window": int(getattr(w, "window", 0)), "ring": bool(getattr(w, "ring", False))}
        ctx = mp.get_context("spawn")
        with ProcessPoolExecutor(max_workers=workers(), mp_context=ctx) as ex:
            attn = [ex.submit(_attention_piece, spec, b, kh) for b in range(B) for kh in range(w.n_kv_heads)]
            pools = []
            if check_pools:
                for side in ("k", "v"):
                    for h in range(w.n_kv_heads):
                        for p0 in range(0, w.num_pages, pages_per_piece):
                            pools.append((side, ex.submit(_pool_piece, spec, side, h, p0,
                                                          min(w.num_pages, p0 + pages_per_piece))))
            errs = [f.result() for f in attn]
            pool_res = [(side, f.result()) for side, f in pools]
    finally:
        shutil.rmtree(d, ignore_errors=True)
    summary = {"rows": sum(n for _, _, n in errs), "max_err": max((e for e, _, _ in errs), default=0.0)}
    assert all(fin for _, fin, _ in errs), "non-finite output"
    for side in ("k", "v"):
        bad = [r for s, r in pool_res if s == side and r[0]]
        if bad:
            n = sum(r[0] for r in bad)
            raise AssertionError(f"{side.upper()} pool differs at {n} bytes, first (page, head, byte) {bad[0][1]}")
    if check_pools:
        summary["pool_bytes"] = int(arrays["k_gpu"].size + arrays["v_gpu"].size)
    assert summary["rows"] == B * Q * Hq, "not every output row was compared"
    assert summary["max_err"] <= tol, f"max |gpu - oracle| = {summary['max_err']:.3e} > {tol}"
    return summary
