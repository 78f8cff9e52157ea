"""Seeded synthetic inputs for decode attention over a block-quantized paged KV cache.

This module only draws random numbers and lays tokens out in pages.  It holds
none of the method's arithmetic (no quantization, no attention); the CUDA
library and the CPU oracle both receive exactly the arrays built here.

Source of the shapes: the memra project pages (GitHub README mirror, "Long
context and larger models" and the shared-prefix serving measurement of the
introduction; Hugging Face card "memra-bench", kf4 archive section for the KV
format names).  The pages name no random generator, so the recipe is:

* ``numpy.random.default_rng(seed)``; every draw is ``standard_normal`` in
  float64, rounded to float16 (round-to-nearest-even by numpy's cast).
* Draw order: (ragged sweep only: the context lengths) -> q -> k -> v
  (long context: k is multiplied by 0.5 before the fp16 rounding)
  -> (long context only: a permutation of the page pool).
* k and v are drawn once for every *unique* cached row, in slot order: the
  shared prefix first (once), then each sequence's own tokens.
* Pages are handed out sequentially unless the workload says otherwise; each
  sequence starts on a fresh page.
* fp8 per-tensor scales are ``float32(amax / 448)`` over the whole K (resp. V)
  tensor of the workload, nvfp4 ones ``float32(amax / 2688)`` (6 x 448), passed
  to both sides as an input.
* The last ``q_len`` rows of every sequence are the rows the step appends
  (quantize-append runs inside the timed step); all other rows are written
  into the cache before timing.
* Sliding-window workloads (the README's SWA ring, "Recent fixes"): every
  sequence owns a ring of R pages and position p lives in ring page
  (p // 16) % R, so only the rows of the last R pages exist; they are drawn
  sequence-major in position order (q -> k -> v -> page permutation).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 16
FP8_E4M3_MAX = 448.0

K_FORMATS = ("q8_0", "fp8", "nvfp4")
V_FORMATS = ("q5_1", "q4_0", "fp8", "nvfp4")
NVFP4_RANGE = 6.0 * 448.0          # largest E2M1 magnitude x largest e4m3 block scale


@dataclass
class Workload:
    name: str
    batch: int
    q_len: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    k_fmt: str
    v_fmt: str
    seq_lens: np.ndarray          # int32 [B], context after the step's append
    page_table: np.ndarray        # int32 [B, max_pages_per_seq]
    num_pages: int
    q: np.ndarray                 # fp16 [B, Q, Hq, D]
    slots: np.ndarray             # int32 [N] slot (= page*16 + offset) of each unique row
    k_rows: np.ndarray            # fp16 [N, Hkv, D]
    v_rows: np.ndarray            # fp16 [N, Hkv, D]
    step_rows: np.ndarray         # int64 [B*Q] indices into the unique rows appended by the step
    k_scale: float = 1.0          # fp8 only: float32 per-tensor scale of K
    v_scale: float = 1.0          # fp8 only: float32 per-tensor scale of V
    shared_prefix: int = 0
    window: int = 0               # sliding window in tokens (0: every earlier key is visible)
    ring: bool = False            # page_table rows are rings: position p -> column (p // 16) % columns
    first_pos: np.ndarray | None = None   # int64 [B] first position with a row (ring workloads)
    notes: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def sm_scale(self) -> float:
        return float(1.0 / np.sqrt(self.head_dim))

    @property
    def prefill_rows(self) -> np.ndarray:
        """Indices of the unique rows that are in the cache before the step."""
        mask = np.ones(self.slots.shape[0], dtype=bool)
        mask[self.step_rows] = False
        return np.nonzero(mask)[0]

    def with_formats(self, k_fmt: str, v_fmt: str) -> "Workload":
        """Same tensors, other KV formats (fp8 scales are recomputed from the data)."""
        w = Workload(**{**self.__dict__})
        w.k_fmt, w.v_fmt = k_fmt, v_fmt
        w.name = f"{self.name.split('[')[0]}[{k_fmt}/{v_fmt}]"
        w.k_scale, w.v_scale = _fp8_scales(w)
        return w


def _normal_f16(rng: np.random.Generator, shape, mult: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """float64 standard normal draws rounded to fp16, drawn in chunks (same stream as one draw)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        x = rng.standard_normal(stop - start)
        if mult != 1.0:
            x *= mult
        out[start:stop] = x.astype(np.float16)
    return out.reshape(shape)


def _amax_f16(x: np.ndarray, chunk: int = 1 << 24) -> float:
    flat = x.reshape(-1)
    m = 0.0
    for s in range(0, flat.size, chunk):
        m = max(m, float(np.abs(flat[s:s + chunk].astype(np.float32)).max()))
    return m


def _tensor_scale(fmt: str, rows: np.ndarray) -> float:
    """float32 per-tensor scale of the formats that take one (fp8, nvfp4); 1 for the others."""
    div = {"fp8": FP8_E4M3_MAX, "nvfp4": NVFP4_RANGE}.get(fmt)
    if div is None:
        return 1.0
    s = float(np.float32(_amax_f16(rows)) / np.float32(div))
    return float(np.float32(s)) if s > 0.0 else 1.0


def _fp8_scales(w: Workload) -> tuple[float, float]:
    return _tensor_scale(w.k_fmt, w.k_rows), _tensor_scale(w.v_fmt, w.v_rows)


def _layout(seq_lens, shared_prefix: int, page_perm_rng=None, extra_pages: int = 0):
    """Assign pages: shared prefix pages first, then each sequence's own pages.

    Returns page_table [B, maxp], num_pages, slots [N] for the unique rows
    (prefix rows first, then sequence 0's own rows, sequence 1's ...), and the
    per-sequence row index map (list of int64 arrays, one per sequence).
    """
    B = len(seq_lens)
    assert shared_prefix % PAGE_SIZE == 0
    n_prefix_pages = shared_prefix // PAGE_SIZE
    own_pages = [-(-(int(t) - shared_prefix) // PAGE_SIZE) for t in seq_lens]
    num_pages = n_prefix_pages + sum(own_pages) + extra_pages
    maxp = max([n_prefix_pages + p for p in own_pages] + [1])
    logical = np.arange(num_pages, dtype=np.int64)
    if page_perm_rng is not None:
        phys = page_perm_rng.permutation(num_pages).astype(np.int64)
    else:
        phys = logical
    page_table = np.zeros((B, maxp), dtype=np.int32)
    slots = []
    seq_rows = []
    # prefix rows
    prefix_slots = np.array([phys[t // PAGE_SIZE] * PAGE_SIZE + t % PAGE_SIZE for t in range(shared_prefix)],
                            dtype=np.int64)
    slots.append(prefix_slots)
    next_page = n_prefix_pages
    row_base = shared_prefix
    for b, t_b in enumerate(seq_lens):
        t_b = int(t_b)
        pages = list(range(n_prefix_pages)) + list(range(next_page, next_page + own_pages[b]))
        next_page += own_pages[b]
        page_table[b, :len(pages)] = phys[pages]
        own = t_b - shared_prefix
        tok = np.arange(shared_prefix, t_b, dtype=np.int64)
        pg = np.asarray(pages, dtype=np.int64)[tok // PAGE_SIZE]
        slots.append(phys[pg] * PAGE_SIZE + tok % PAGE_SIZE)
        seq_rows.append(np.concatenate([np.arange(shared_prefix, dtype=np.int64),
                                        np.arange(row_base, row_base + own, dtype=np.int64)]))
        row_base += own
    slots = np.concatenate(slots).astype(np.int32)
    return page_table, num_pages, slots, seq_rows


def make_workload(name: str, *, batch: int, q_len: int, n_heads: int, n_kv_heads: int, head_dim: int,
                  k_fmt: str, v_fmt: str, seed: int, seq_lens=None, ctx_range=None, shared_prefix: int = 0,
                  k_mult: float = 1.0, permute_pages: bool = False, extra_pages: int = 0) -> Workload:
    """Build one workload with the documented draw order."""
    assert k_fmt in K_FORMATS and v_fmt in V_FORMATS
    rng = np.random.default_rng(seed)
    if ctx_range is not None:
        lo, hi = ctx_range
        seq_lens = rng.integers(lo, hi, size=batch, endpoint=True)
    seq_lens = np.asarray(seq_lens, dtype=np.int64).reshape(batch)
    assert (seq_lens >= max(q_len, 1)).all() and (seq_lens >= shared_prefix + q_len).all()
    n_unique = shared_prefix + int((seq_lens - shared_prefix).sum())
    q = _normal_f16(rng, (batch, q_len, n_heads, head_dim))
    k_rows = _normal_f16(rng, (n_unique, n_kv_heads, head_dim), mult=k_mult)
    v_rows = _normal_f16(rng, (n_unique, n_kv_heads, head_dim))
    perm_rng = rng if permute_pages else None
    page_table, num_pages, slots, seq_rows = _layout(seq_lens, shared_prefix, perm_rng, extra_pages)
    step_rows = np.concatenate([r[-q_len:] for r in seq_rows]) if batch else np.zeros(0, np.int64)
    w = Workload(name=name, batch=batch, q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                 head_dim=head_dim, k_fmt=k_fmt, v_fmt=v_fmt, seq_lens=seq_lens.astype(np.int32),
                 page_table=page_table, num_pages=num_pages, q=q, slots=slots, k_rows=k_rows, v_rows=v_rows,
                 step_rows=step_rows.astype(np.int64), shared_prefix=shared_prefix)
    w.k_scale, w.v_scale = _fp8_scales(w)
    return w


def min_ring_pages(window: int, q_len: int) -> int:
    """Fewest ring pages that hold every key a window of `window` tokens shows to q_len query rows."""
    return (window + q_len - 2) // PAGE_SIZE + 2


def make_window_workload(name: str, *, batch: int, q_len: int, n_heads: int, n_kv_heads: int, head_dim: int,
                         k_fmt: str, v_fmt: str, seed: int, seq_lens, window: int, ring_pages: int | None = None,
                         permute_pages: bool = False, extra_pages: int = 0) -> Workload:
    """Sliding-window attention over a ring of pages per sequence."""
    assert k_fmt in K_FORMATS and v_fmt in V_FORMATS and window >= 1
    R = min_ring_pages(window, q_len) if ring_pages is None else int(ring_pages)
    assert R >= min_ring_pages(window, q_len)
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64).reshape(batch)
    assert (seq_lens >= max(q_len, 1)).all()
    first = np.maximum(0, ((seq_lens - 1) // PAGE_SIZE - R + 1) * PAGE_SIZE)
    counts = seq_lens - first
    n_unique = int(counts.sum())
    q = _normal_f16(rng, (batch, q_len, n_heads, head_dim))
    k_rows = _normal_f16(rng, (n_unique, n_kv_heads, head_dim))
    v_rows = _normal_f16(rng, (n_unique, n_kv_heads, head_dim))
    num_pages = batch * R + extra_pages
    phys = rng.permutation(num_pages).astype(np.int64) if permute_pages else np.arange(num_pages, dtype=np.int64)
    page_table = phys[:batch * R].reshape(batch, R).astype(np.int32)
    slots, step = [], []
    base = 0
    for b in range(batch):
        pos = np.arange(first[b], seq_lens[b], dtype=np.int64)
        slots.append(page_table[b, (pos // PAGE_SIZE) % R].astype(np.int64) * PAGE_SIZE + pos % PAGE_SIZE)
        step.append(np.arange(base + counts[b] - q_len, base + counts[b], dtype=np.int64))
        base += int(counts[b])
    w = Workload(name=name, batch=batch, q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                 head_dim=head_dim, k_fmt=k_fmt, v_fmt=v_fmt, seq_lens=seq_lens.astype(np.int32),
                 page_table=page_table, num_pages=num_pages, q=q,
                 slots=np.concatenate(slots).astype(np.int32) if batch else np.zeros(0, np.int32),
                 k_rows=k_rows, v_rows=v_rows,
                 step_rows=np.concatenate(step) if batch else np.zeros(0, np.int64),
                 window=int(window), ring=True, first_pos=first.astype(np.int64))
    w.k_scale, w.v_scale = _fp8_scales(w)
    return w


# The five workloads of the hot path, by what they are.
def tiny() -> Workload:
    """batch 1, q_len 1, 8/2 heads, D 128, 256-token context, seed 0."""
    return make_workload("tiny_b1_ctx256_h8kv2_d128", batch=1, q_len=1, n_heads=8, n_kv_heads=2, head_dim=128,
                         k_fmt="q8_0", v_fmt="q5_1", seed=0, seq_lens=[256])


def shared_prefix() -> Workload:
    """16 sequences of 4,860 tokens sharing a 4,096-token prefix, 32/4 heads, D 128, seed 1."""
    return make_workload("shared_prefix_b16_ctx4860_prefix4096_h32kv4_d128", batch=16, q_len=1, n_heads=32,
                         n_kv_heads=4, head_dim=128, k_fmt="q8_0", v_fmt="q5_1", seed=1,
                         seq_lens=[4860] * 16, shared_prefix=4096)


def shared_prefix_long() -> Workload:
    """16 sequences of 33,532 tokens sharing a 32,768-token prefix (a long shared document or system
    prompt before each request's own 764 tokens), 32/4 heads, D 128, seed 6."""
    return make_workload("shared_prefix_long_b16_ctx33532_prefix32768_h32kv4_d128", batch=16, q_len=1,
                         n_heads=32, n_kv_heads=4, head_dim=128, k_fmt="q8_0", v_fmt="q5_1", seed=6,
                         seq_lens=[33532] * 16, shared_prefix=32768)


def long_context() -> Workload:
    """batch 1, 262,144-token context, 32/4 heads, D 128, pages in a random permutation, k x0.5, seed 2."""
    return make_workload("long_context_b1_ctx262144_h32kv4_d128", batch=1, q_len=1, n_heads=32, n_kv_heads=4,
                         head_dim=128, k_fmt="q8_0", v_fmt="q5_1", seed=2, seq_lens=[262144], k_mult=0.5,
                         permute_pages=True)


def mtp_verify() -> Workload:
    """8 sequences, q_len 4 (3 drafts + 1) causal, prior context 6,300, 32/4 heads, D 128, seed 3."""
    return make_workload("mtp_verify_b8_q4_ctx6300_h32kv4_d128", batch=8, q_len=4, n_heads=32, n_kv_heads=4,
                         head_dim=128, k_fmt="q8_0", v_fmt="q5_1", seed=3, seq_lens=[6304] * 8)


SWEEP_FORMATS = {"a": ("q8_0", "q4_0"), "b": ("fp8", "fp8"), "c": ("q8_0", "q5_1")}


def format_sweep(variant: str = "c") -> Workload:
    """64 ragged sequences (512..32,768 tokens, seed 4), 16/2 heads, D 256, in one of three KV formats."""
    k_fmt, v_fmt = SWEEP_FORMATS[variant]
    return make_workload(f"format_sweep_b64_ragged512-32768_h16kv2_d256[{k_fmt}/{v_fmt}]", batch=64, q_len=1,
                         n_heads=16, n_kv_heads=2, head_dim=256, k_fmt=k_fmt, v_fmt=v_fmt, seed=4,
                         ctx_range=(512, 32768))


WORKLOADS = {
    "tiny": tiny,
    "shared_prefix": shared_prefix,
    "shared_prefix_long": shared_prefix_long,
    "long_context": long_context,
    "mtp_verify": mtp_verify,
    "sweep_a": lambda: format_sweep("a"),
    "sweep_b": lambda: format_sweep("b"),
    "sweep_c": lambda: format_sweep("c"),
}


def random_case(seed: int, *, batch: int = 2, q_len: int = 1, n_heads: int = 8, n_kv_heads: int = 2,
                head_dim: int = 128, k_fmt: str = "q8_0", v_fmt: str = "q5_1", ctx=(1, 300),
                shared_prefix: int = 0, permute_pages: bool = True, extra_pages: int = 3) -> Workload:
    """Small randomized case for parity tests (ragged contexts, shuffled pages, spare pages)."""
    lo, hi = ctx
    lo = max(lo, q_len + shared_prefix)
    hi = max(hi, lo)
    return make_workload(f"random_{seed}", batch=batch, q_len=q_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                         head_dim=head_dim, k_fmt=k_fmt, v_fmt=v_fmt, seed=seed, ctx_range=(lo, hi),
                         shared_prefix=shared_prefix, permute_pages=permute_pages, extra_pages=extra_pages)
