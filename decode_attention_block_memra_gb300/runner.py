"""Runs one workload through the C ABI on the current CUDA device.

Plumbing only: uploads a ``workloads.Workload`` (fp16 rows, page tables,
query), fills the paged cache with quantize-append for the rows that exist
before the step, then runs the step itself (quantize-append of the step's
new rows, split-K decode, combine).  All arithmetic runs in libmemra.so.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import (KVCache, decode_attn, decode_attn_cascade, decode_attn_cascade_workspace_bytes,
               decode_attn_workspace_bytes, decode_step, kv_append, read_status)


@dataclass
class DeviceWorkload:
    w: object
    cache: KVCache
    q: object
    page_table: object
    seq_lens: object
    out: object
    workspace: object
    step_k: object
    step_v: object
    step_slots: object
    cascade_workspace: object = None

    def step(self, stream=None, fused: bool = False, cascade: bool = False) -> None:
        """One pass of the hot path: append the step's rows, then attend.

        fused: one memra_decode_step (the split kernel stores the rows) instead
        of memra_kv_append followed by memra_decode_attn.  cascade: the
        workload's shared prefix through the cascade calls
        (memra_decode_step_cascade when fused, else memra_kv_append +
        memra_decode_attn_cascade).
        """
        w = self.w
        window = getattr(w, "window", 0)
        if cascade:
            import torch
            if self.cascade_workspace is None:
                n = decode_attn_cascade_workspace_bytes(w.batch, w.q_len, w.n_heads, w.head_dim, w.max_seq_len,
                                                        w.shared_prefix)
                self.cascade_workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=self.q.device)
            B, Q = w.batch, w.q_len
            kn = vn = None
            if fused:
                kn = self.step_k.view(B, Q, w.n_kv_heads, w.head_dim)
                vn = self.step_v.view(B, Q, w.n_kv_heads, w.head_dim)
            else:
                kv_append(self.cache, self.step_k, self.step_v, self.step_slots, stream=stream)
            decode_attn_cascade(self.cache, self.q, self.page_table, self.seq_lens, w.max_seq_len, w.shared_prefix,
                                self.out, self.cascade_workspace, w.sm_scale, stream=stream, k_new=kn, v_new=vn)
            return
        if fused:
            B, Q = w.batch, w.q_len
            decode_step(self.cache, self.step_k.view(B, Q, w.n_kv_heads, w.head_dim),
                        self.step_v.view(B, Q, w.n_kv_heads, w.head_dim), self.q, self.page_table, self.seq_lens,
                        w.max_seq_len, self.out, self.workspace, w.sm_scale, stream=stream, window=window)
            return
        kv_append(self.cache, self.step_k, self.step_v, self.step_slots, stream=stream)
        decode_attn(self.cache, self.q, self.page_table, self.seq_lens, w.max_seq_len, self.out, self.workspace,
                    w.sm_scale, stream=stream, window=window)


def upload(w, fill_seed: int | None = None, device="cuda", prefill_chunk: int = 1 << 20) -> DeviceWorkload:
    """Allocate and fill the cache for the rows that precede the step.

    fill_seed: if given, the pools start as seeded random bytes (so tokens
    never written are garbage, which the kernels must ignore); else zeros.
    """
    import torch
    cache = KVCache(w.k_fmt, w.v_fmt, w.num_pages, w.n_kv_heads, w.head_dim, w.k_scale, w.v_scale, device=device)
    if fill_seed is not None:
        g = torch.Generator(device="cpu").manual_seed(fill_seed)
        cache.k_pool.copy_(torch.randint(0, 256, cache.k_pool.shape, dtype=torch.uint8, generator=g))
        cache.v_pool.copy_(torch.randint(0, 256, cache.v_pool.shape, dtype=torch.uint8, generator=g))
    pre = w.prefill_rows
    for s in range(0, pre.size, prefill_chunk):
        idx = pre[s:s + prefill_chunk]
        k = torch.from_numpy(np.ascontiguousarray(w.k_rows[idx])).to(device)
        v = torch.from_numpy(np.ascontiguousarray(w.v_rows[idx])).to(device)
        sl = torch.from_numpy(np.ascontiguousarray(w.slots[idx])).to(device)
        kv_append(cache, k, v, sl)
    step = w.step_rows
    dw = DeviceWorkload(
        w=w, cache=cache,
        q=torch.from_numpy(np.ascontiguousarray(w.q)).to(device),
        page_table=torch.from_numpy(np.ascontiguousarray(w.page_table)).to(device),
        seq_lens=torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device),
        out=torch.empty(w.q.shape, dtype=torch.float16, device=device),
        workspace=torch.empty(max(1, decode_attn_workspace_bytes(w.batch, w.q_len, w.n_heads, w.head_dim,
                                                                 w.max_seq_len)), dtype=torch.uint8, device=device),
        step_k=torch.from_numpy(np.ascontiguousarray(w.k_rows[step])).to(device),
        step_v=torch.from_numpy(np.ascontiguousarray(w.v_rows[step])).to(device),
        step_slots=torch.from_numpy(np.ascontiguousarray(w.slots[step])).to(device),
    )
    return dw


@dataclass
class StepResult:
    out: np.ndarray          # fp16 [B, Q, Hq, D]
    k_pool: np.ndarray       # uint8 [num_pages, Hkv, seg]
    v_pool: np.ndarray
    flags: int
    initial_k_pool: np.ndarray | None = None
    initial_v_pool: np.ndarray | None = None


def run_workload(w, fill_seed: int | None = None, want_pools: bool = False, fused: bool = False,
                 cascade: bool = False) -> StepResult:
    """Upload, fill, run one step (fused: through memra_decode_step; cascade: the
    shared-prefix cascade calls), copy everything back."""
    import torch
    init_k = init_v = None
    dw = upload(w, fill_seed=fill_seed)
    if want_pools and fill_seed is not None:
        # the bytes the pools started from (regenerated with the same seed)
        g = torch.Generator(device="cpu").manual_seed(fill_seed)
        init_k = torch.randint(0, 256, dw.cache.k_pool.shape, dtype=torch.uint8, generator=g).numpy()
        init_v = torch.randint(0, 256, dw.cache.v_pool.shape, dtype=torch.uint8, generator=g).numpy()
    dw.step(fused=fused, cascade=cascade)
    flags = read_status(dw.cache)
    torch.cuda.synchronize()
    out = dw.out.cpu().numpy()
    kp = vp = None
    if want_pools:
        kp = dw.cache.k_pool.cpu().numpy().reshape(w.num_pages, w.n_kv_heads, -1)
        vp = dw.cache.v_pool.cpu().numpy().reshape(w.num_pages, w.n_kv_heads, -1)
    return StepResult(out=out, k_pool=kp, v_pool=vp, flags=flags, initial_k_pool=init_k, initial_v_pool=init_v)
