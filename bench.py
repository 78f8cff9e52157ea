#!/usr/bin/env python3
"""Benchmark of one decode step over a block-quantized paged KV cache.

A step is one pass of the whole hot path on one batch: quantize-append of the
step's new K/V rows, the split-K decode kernel, the log-sum-exp combine.  The
default workload is the 262,144-token long-context decode (batch 1, 32 query
heads / 4 KV heads, head_dim 128, K q8_0 / V q5_1, pages in a random
permutation of the pool).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  value = query tokens per second of the whole
job (decode-attention throughput); kv_gbs = unique quantized-KV bytes per
second.  Timing: CUDA events on the launching stream around every step, an
L2 flush (256 MiB write, then read back so no dirty line is left) between
steps outside the events, max over ranks.  The line also carries
``per_workload``: the same step and its split kernel timed on the other
workloads (tiny, shared prefix plain and cascade, MTP verify, the head_dim
256 format sweep in three formats).
With --gpus N (under torchrun) every rank runs an independent replica of the
workload (the path shards into independent sequences; there is no exchange).

The oracle's leg (``cpu_baseline``, and ``--impl reference``) runs the CPU
oracle as it stands on whole steps of the same workload: the step's new rows
quantized, then attention for every query row of every KV head, spread over
the host's cores as independent (sequence, KV head) pieces in a spawn
process pool, one BLAS thread per process.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn tokens/s (quantized-KV GB/s, % of HBM peak)"
# quantized-KV algorithmic bytes per element of a row: codes + block parameters
K_BYTES_PER_ELEM = {"q8_0": 34 / 32, "fp8": 1.0, "nvfp4": 9 / 16}
V_BYTES_PER_ELEM = {"q5_1": 24 / 32, "q4_0": 18 / 32, "fp8": 1.0, "nvfp4": 9 / 16}
BYTES_PER_TOKEN_HEAD = {  # per token per KV head, K + V, by head_dim
    (k, v): K_BYTES_PER_ELEM[k] + V_BYTES_PER_ELEM[v] for k in K_BYTES_PER_ELEM for v in V_BYTES_PER_ELEM
}
KERNEL_SOURCES = ["decode_attention_block_memra_gb300/csrc/decode_kernel.cuh",
                  "decode_attention_block_memra_gb300/csrc/memra_device.cuh",
                  "decode_attention_block_memra_gb300/csrc/kv_quant.cuh",
                  "decode_attention_block_memra_gb300/csrc/api.cu", "include/memra.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def unique_kv_bytes(w) -> int:
    """Algorithmic quantized-KV bytes of one decode launch: every unique (token, KV head) once."""
    per = BYTES_PER_TOKEN_HEAD[(w.k_fmt, w.v_fmt)] * w.head_dim
    return int(round(w.slots.size * w.n_kv_heads * per))


def logical_kv_bytes(w) -> int:
    per = BYTES_PER_TOKEN_HEAD[(w.k_fmt, w.v_fmt)] * w.head_dim
    return int(round(int(w.seq_lens.sum()) * w.n_kv_heads * per))


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def stored_traffic(workload: str):
    """ncu DRAM bytes per launch of the decode kernel, if taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == "decode_split_kernel" \
                        and parts[1] == workload and parts[2] == kernel_hash():
                    return int(parts[3])
    except FileNotFoundError:
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"memra_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax = float(p[2])
                except ValueError:
                    continue
                for name, val in zip(names[1:], p[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(seconds: float, world: int, device=None) -> float:
    """The job's time: the slowest rank's (replicas run independently; no data exchange)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank processes its own replica of the workload."""
    return world * tokens_per_step * steps / seconds


def make_workload(name: str, formats: str | None = None):
    import workloads as W
    w = W.WORKLOADS[name]()
    if formats:
        w = w.with_formats(*formats.split("/"))
    return w


def workload_config(w) -> dict:
    """The workload a line measures (the same dict in the native and the oracle arm)."""
    return {"workload": w.name, "batch": w.batch, "q_len": w.q_len, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "context_tokens": int(w.seq_lens.sum()), "unique_tokens": int(w.slots.size),
            "kv_format": f"{w.k_fmt}/{w.v_fmt}", "page_size": 16, "split_tokens": "max(1280, T / (SMs x CTAs per SM / KV heads))",
            "l2": "flushed between steps (256 MiB write, then read back, outside the timed events)"}


# ------------------------------------------------------------ the oracle leg --
# The step on the CPU: quantize the step's new rows, then attention for every
# query row over the dequantized cache.  The rows in the cache before the step
# are quantized beforehand (untimed, as the GPU cache is filled before its
# timed steps).  Pieces: one per (sequence, KV head), independent, in a spawn
# pool; the arrays reach the workers as memory-mapped .npy files.

_ORACLE_FILES = {}


def _oracle_load(d, name):
    import numpy as np
    key = (d, name)
    if key not in _ORACLE_FILES:
        _ORACLE_FILES[key] = np.load(os.path.join(d, name + ".npy"), mmap_mode="r+" if name.startswith("pre_")
                                     else "r")
    return _ORACLE_FILES[key]


def _oracle_prep_piece(spec, side, kh, r0, r1):
    """Quantize cached rows [r0, r1) (of the rows present before the step) of one side and KV head."""
    import numpy as np
    from oracle import quant
    d = spec["dir"]
    pre = _oracle_load(d, "prefill_rows")[r0:r1]
    src = _oracle_load(d, side + "_rows")
    fields = quant.quantize_rows(np.asarray(src[np.asarray(pre), kh, :]), spec[side + "_fmt"], spec[side + "_scale"])
    for key in spec[side + "_keys"]:
        _oracle_load(d, f"pre_{side}_{key}")[kh, r0:r1] = fields[key]
    for key in spec[side + "_keys"]:
        _oracle_load(d, f"pre_{side}_{key}").flush()


def _oracle_step_piece(spec, b, kh):
    """One (sequence, KV head) piece of the step: quantize its new rows, attend for its query rows."""
    import numpy as np
    from oracle import attention, quant
    d = spec["dir"]
    w = SimpleNamespace(seq_lens=_oracle_load(d, "seq_lens"), page_table=_oracle_load(d, "page_table"),
                        slots=_oracle_load(d, "slots"), ring=spec["ring"],
                        first_pos=_oracle_load(d, "first_pos") if spec["ring"] else None)
    rows = attention.sequence_rows(w, b)
    pre_idx = np.asarray(_oracle_load(d, "pre_index"))[rows]
    step_idx = np.asarray(_oracle_load(d, "step_index"))[rows]
    new_at = step_idx >= 0
    hats = []
    for side in ("k", "v"):
        new = quant.quantize_rows(np.asarray(_oracle_load(d, side + "_step"))[step_idx[new_at], kh, :],
                                  spec[side + "_fmt"], spec[side + "_scale"])
        fields = dict(new)
        for key in spec[side + "_keys"]:
            cached = _oracle_load(d, f"pre_{side}_{key}")[kh]
            arr = np.empty((rows.size,) + cached.shape[1:], dtype=cached.dtype)
            arr[~new_at] = cached[pre_idx[~new_at]]
            arr[new_at] = new[key]
            fields[key] = arr
        hats.append(quant.dequantize_rows(fields)[:, None, :])
    G = spec["group"]
    heads = slice(kh * G, (kh + 1) * G)
    q = np.asarray(_oracle_load(d, "q")[b, :, heads, :])
    out = attention.attention_rows(q, hats[0], hats[1], spec["sm_scale"], window=spec["window"],
                                   start=attention.first_position(w, b))
    return float(out.sum())


class OracleStep:
    """The CPU oracle on whole steps of a workload, over the host's cores."""

    def __init__(self, workload: str, formats: str | None = None, workers: int | None = None):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor

        import numpy as np
        from oracle import quant
        for var in BLAS_ENV:              # one BLAS thread per worker process (inherited at spawn)
            os.environ[var] = "1"
        self.w = w = make_workload(workload, formats)
        self.host_cpus = os.cpu_count() or 1
        self.workers = workers or max(1, min(self.host_cpus, 16))
        self.dir = tempfile.mkdtemp(prefix="memra_oracle_")
        pre = w.prefill_rows
        pre_index = np.full(w.slots.size, -1, np.int64)
        pre_index[pre] = np.arange(pre.size)
        step_index = np.full(w.slots.size, -1, np.int64)
        step_index[w.step_rows] = np.arange(w.step_rows.size)
        arrays = {"q": w.q, "slots": w.slots, "seq_lens": w.seq_lens, "page_table": w.page_table,
                  "prefill_rows": pre, "pre_index": pre_index, "step_index": step_index,
                  "k_rows": w.k_rows, "v_rows": w.v_rows,
                  "k_step": w.k_rows[w.step_rows], "v_step": w.v_rows[w.step_rows]}
        if getattr(w, "ring", False):
            arrays["first_pos"] = w.first_pos
        for name, a in arrays.items():
            np.save(os.path.join(self.dir, name + ".npy"), np.ascontiguousarray(a))
        self.spec = {"dir": self.dir, "k_fmt": w.k_fmt, "v_fmt": w.v_fmt, "k_scale": float(w.k_scale),
                     "v_scale": float(w.v_scale), "group": w.n_heads // w.n_kv_heads, "sm_scale": w.sm_scale,
                     "window": int(getattr(w, "window", 0)), "ring": bool(getattr(w, "ring", False))}
        # the fields of each format, from one quantized row; one file per field: [Hkv, rows before the step, ...]
        for side, fmt, sc in (("k", w.k_fmt, w.k_scale), ("v", w.v_fmt, w.v_scale)):
            one = quant.quantize_rows(w.k_rows[:1, 0, :] if side == "k" else w.v_rows[:1, 0, :], fmt, sc)
            keys = [k for k, v in one.items() if isinstance(v, np.ndarray)]
            self.spec[side + "_keys"] = keys
            for key in keys:
                np.lib.format.open_memmap(os.path.join(self.dir, f"pre_{side}_{key}.npy"), mode="w+",
                                          dtype=one[key].dtype, shape=(w.n_kv_heads, pre.size) + one[key].shape[1:])
        self.pool = ProcessPoolExecutor(max_workers=self.workers, mp_context=mp.get_context("spawn"))
        chunk = 1 << 16
        jobs = [self.pool.submit(_oracle_prep_piece, self.spec, side, kh, r0, min(pre.size, r0 + chunk))
                for side in ("k", "v") for kh in range(w.n_kv_heads) for r0 in range(0, pre.size, chunk)]
        for j in jobs:
            j.result()
        # the source rows are not needed by the steps
        self.pieces = [(b, kh) for b in range(w.batch) for kh in range(w.n_kv_heads)]

    def run(self) -> float:
        """Wall seconds of one whole step."""
        t0 = time.perf_counter()
        futs = [self.pool.submit(_oracle_step_piece, self.spec, b, kh) for b, kh in self.pieces]
        for f in futs:
            f.result()
        return time.perf_counter() - t0

    def close(self):
        self.pool.shutdown()
        shutil.rmtree(self.dir, ignore_errors=True)

    def describe(self, how: str) -> dict:
        w = self.w
        busy = min(self.workers, len(self.pieces))       # pieces of one step that can run at once
        return {"kind": "oracle", "cores": busy, "host_cpus": self.host_cpus, "blas_threads_per_core": 1,
                "workers": self.workers,
                "sample": (f"whole steps of {w.name} ({w.k_fmt}/{w.v_fmt}): the step's {w.step_rows.size} new rows "
                           f"quantized, then attention for all {w.batch * w.q_len * w.n_heads} query rows over "
                           f"{int(w.seq_lens.sum())} keys per query head in float64, as {len(self.pieces)} "
                           f"(sequence, KV head) pieces on {self.workers} worker processes; {how}")}


def oracle_sample(workload: str, formats: str | None, reps: int) -> dict:
    st = OracleStep(workload, formats)
    try:
        st.run()                                         # warm the workers (imports, page cache)
        times = [st.run() for _ in range(reps)]
    finally:
        st.close()
    per_step = statistics.median(times)
    w = st.w
    return {"value": w.batch * w.q_len / per_step, "unit": "tokens/s", **st.describe(f"median of {reps} steps"),
            "seconds_per_step": per_step}


def cpu_baseline(workload: str, formats: str | None, reps: int) -> dict:
    """The oracle, as it stands, on whole steps over the host's cores (in a subprocess, before any CUDA work)."""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload, "--steps", str(reps)]
    if formats:
        cmd += ["--formats", formats]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        tail = r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"
        return {"value": None, "unit": "tokens/s", "cores": None, "kind": "oracle", "sample": "failed: " + tail}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference_arm(args) -> None:
    world, rank, _ = dist_env()
    if rank != 0:
        return
    t_start = time.perf_counter()
    st = OracleStep(args.workload, args.formats)
    try:
        for _ in range(args.warmup):
            st.run()
        t0 = time.perf_counter()
        times = [st.run() for _ in range(args.steps)]
        wall = time.perf_counter() - t0
    finally:
        st.close()
    w = st.w
    per_step = statistics.mean(times)
    value = w.batch * w.q_len / per_step
    cb = {"value": value, "unit": "tokens/s", **st.describe(f"mean of {args.steps} steps")}
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": workload_config(w), "parallelism": "host processes",
            "cpu_baseline": cb, "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0},
            "timed_wall_s": wall, "total_wall_s": time.perf_counter() - t_start}
    print(json.dumps(line), flush=True)


def percentile(xs, pct):
    """Linear-interpolated percentile of a non-empty list (numpy's default rule)."""
    ys = sorted(xs)
    pos = (len(ys) - 1) * pct / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


# ------------------------------------------------------------ the GPU leg --

class Bench:
    """Times the hot path of one workload through the public entry points."""

    def __init__(self, w, two_call=False, cascade=False, pack_inputs=False):
        import torch
        import decode_attention_block_memra_gb300 as memra
        from decode_attention_block_memra_gb300.runner import upload
        self.torch, self.memra = torch, memra
        self.w, self.two_call, self.cascade = w, two_call, cascade
        self.dw = dw = upload(w)
        self.stream = torch.cuda.current_stream()
        if pack_inputs:
            # The step's inputs (q, the new rows, the lengths, the page table) live in one device buffer at
            # 256-byte offsets, so that the end-to-end step uploads them from one pinned buffer in one copy.
            step_inputs = [("q", dw.q), ("step_k", dw.step_k), ("step_v", dw.step_v), ("seq_lens", dw.seq_lens),
                           ("page_table", dw.page_table)] + ([("step_slots", dw.step_slots)] if two_call else [])
            offsets, total = [], 0
            for _, t in step_inputs:
                offsets.append(total)
                total += -(-t.numel() * t.element_size() // 256) * 256
            self.dev_pack = torch.empty(total, dtype=torch.uint8, device="cuda")
            self.host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
            for (name, t), off in zip(step_inputs, offsets):
                nbytes = t.numel() * t.element_size()
                view = self.dev_pack[off:off + nbytes].view(t.dtype).view(t.shape)
                view.copy_(t)
                self.host_pack[off:off + nbytes].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
                setattr(dw, name, view)
        B, Q = w.batch, w.q_len
        self.k_new = dw.step_k.view(B, Q, w.n_kv_heads, w.head_dim)
        self.v_new = dw.step_v.view(B, Q, w.n_kv_heads, w.head_dim)
        self.cws = None
        if cascade:
            if not w.shared_prefix:
                raise SystemExit("--cascade needs a workload with a shared prefix")
            self.cws = torch.empty(memra.decode_attn_cascade_workspace_bytes(B, Q, w.n_heads, w.head_dim,
                                                                             w.max_seq_len, w.shared_prefix),
                                   dtype=torch.uint8, device="cuda")
        # the split kernel, the combine (left out when every row fits one split), the separate append of the
        # two-call form, the cascade's prefix pass
        combine = 1 if (cascade or w.max_seq_len > memra.SPLIT_TOKENS) else 0
        self.launches_per_step = 1 + combine + (1 if two_call else 0) + (1 if cascade else 0)

    def hot_path(self):
        """Store the step's rows and attend: one memra_decode_step (split-K with the rows stored inside, then
        the combine), or the two-call form, or the cascade calls."""
        memra, dw, w, s = self.memra, self.dw, self.w, self.stream
        if self.cascade:
            if self.two_call:
                memra.kv_append(dw.cache, dw.step_k, dw.step_v, dw.step_slots, stream=s)
                memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                                          w.shared_prefix, dw.out, self.cws, w.sm_scale, stream=s)
            else:
                memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                                          w.shared_prefix, dw.out, self.cws, w.sm_scale, stream=s, k_new=self.k_new,
                                          v_new=self.v_new)
        elif self.two_call:
            memra.kv_append(dw.cache, dw.step_k, dw.step_v, dw.step_slots, stream=s)
            memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace,
                              w.sm_scale, stream=s)
        else:
            memra.decode_step(dw.cache, self.k_new, self.v_new, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                              dw.out, dw.workspace, w.sm_scale, stream=s)

    def split_pass(self):
        """The split-K kernel alone (its partials pass), for its roofline; for the cascade the whole cascade
        attention (prefix pass, split-K, merge)."""
        memra, dw, w, s = self.memra, self.dw, self.w, self.stream
        if self.cascade:
            memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, w.shared_prefix,
                                      dw.out, self.cws, w.sm_scale, stream=s)
        else:
            memra.decode_attn_partials(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out,
                                       dw.workspace, w.sm_scale, stream=s)

    def timed(self, fn, n, flush_l2):
        """Event-timed ms of n calls of fn on the launching stream, L2 flushed before each (outside the events)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush_l2()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def flags(self) -> int:
        return self.memra.read_status(self.dw.cache)


def summarize(w, step_ms, split_ms, peak, cascade=False) -> dict:
    kv = unique_kv_bytes(w)
    step_s = statistics.mean(step_ms) / 1e3
    split_s = statistics.mean(split_ms) / 1e3
    return {"workload": w.name, "step_form": "cascade (memra_decode_step_cascade)" if cascade
            else "fused (memra_decode_step)",
            "config": workload_config(w), "tokens_per_s": w.batch * w.q_len / step_s,
            "step_us": {"median": statistics.median(step_ms) * 1e3, "mean": step_s * 1e6},
            "kv_bytes_unique": kv, "kv_bytes_logical": logical_kv_bytes(w),
            "kv_gbs_step": kv / step_s / 1e9,
            "split_kernel": "cascade attention (prefix pass + split-K + merge)" if cascade else "decode_split_kernel",
            "split_us": split_s * 1e6, "split_kv_gbs": kv / split_s / 1e9, "split_hbm_frac": kv / split_s / 1e9 / peak,
            # ncu DRAM bytes of one split-kernel launch, when profiles/traffic.txt holds a capture of the
            # current kernel source for this workload (else None)
            "split_traffic": None if cascade else stored_traffic(w.name)}


def per_workload_lines(args, flush_l2, peak) -> list:
    """Every other workload's step and split kernel, timed like the main one (fewer steps)."""
    import workloads as W
    torch = __import__("torch")
    out = []
    n, warm = args.per_workload_steps, 3

    def one(w, cascade=False):
        b = Bench(w, cascade=cascade)
        for _ in range(warm):
            flush_l2()
            b.hot_path()
        torch.cuda.synchronize()
        if b.flags():
            raise RuntimeError(f"device status flagged on {w.name}")
        step_ms = b.timed(b.hot_path, n, flush_l2)
        b.timed(b.split_pass, warm, flush_l2)
        split_ms = b.timed(b.split_pass, n, flush_l2)
        flags = b.flags()
        r = summarize(w, step_ms, split_ms, peak, cascade)
        r["device_flags"] = flags
        out.append(r)
        del b
        torch.cuda.empty_cache()

    for name in ("tiny", "shared_prefix", "mtp_verify"):
        w = W.WORKLOADS[name]()
        one(w)
        if name == "shared_prefix":
            one(w, cascade=True)
    base = W.format_sweep("c")
    for v in ("a", "b", "c"):
        one(base.with_formats(*W.SWEEP_FORMATS[v]))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--formats", default=None, help="K/V formats overriding the workload's, e.g. q8_0/q4_0")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true", help="leave out the per_workload block")
    ap.add_argument("--per-workload-steps", type=int, default=20)
    ap.add_argument("--two-call", action="store_true",
                    help="time memra_kv_append + memra_decode_attn instead of the fused memra_decode_step")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix workloads: the cascade calls (the prefix once per KV head on tcgen05)")
    ap.add_argument("--cpu-reps", type=int, default=3)
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        print(json.dumps(oracle_sample(args.workload, args.formats, args.steps)))
        return
    if args.impl == "reference":
        run_reference_arm(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    world, rank, local = dist_env()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.formats, args.cpu_reps)      # before any CUDA work in this process

    import torch
    import torch.distributed as dist
    import decode_attention_block_memra_gb300 as memra
    from decode_attention_block_memra_gb300 import _build

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    memra.lib()
    w = make_workload(args.workload, args.formats)
    b = Bench(w, two_call=args.two_call, cascade=args.cascade, pack_inputs=True)
    dw, stream = b.dw, b.stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def flush_l2():
        # write a buffer larger than L2, then read it back: the KV lines are gone
        # and no dirty lines are left to be written back during the timed step
        flush.fill_(1)
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=flush_sink)

    b.timed(b.hot_path, args.warmup, flush_l2)
    if b.flags():
        raise RuntimeError("device status flagged during warm-up")

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    step_ms = b.timed(b.hot_path, args.steps, flush_l2)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    flags = b.flags()
    # the split kernel timed alone over as many launches (same inputs, L2 flushed)
    b.timed(b.split_pass, 3, flush_l2)
    k2_ms = b.timed(b.split_pass, args.steps, flush_l2)
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, "cuda")
    tokens_per_step = w.batch * w.q_len
    value = job_throughput(tokens_per_step, args.steps, world, total_s)
    kv_bytes = unique_kv_bytes(w)
    peak, peak_kind = measured_peaks()
    k2_avg_s = statistics.mean(k2_ms) / 1e3
    achieved = kv_bytes / k2_avg_s / 1e9

    # end to end through the public API: the step's inputs from pinned host memory to the device (one
    # copy of the packed buffer), the step, the output back to pinned host memory
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    h2d = b.host_pack.numel()
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        b.dev_pack.copy_(b.host_pack, non_blocking=True)
        b.hot_path()
        out_host.copy_(dw.out, non_blocking=True)

    for _ in range(args.warmup):
        flush_l2()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush_l2()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        z.record(stream)
        z.synchronize()
        e2e_ms.append(a.elapsed_time(z))
    e2e_total = max_over_ranks(sum(e2e_ms) / 1e3, world, "cuda")
    e2e_value = job_throughput(tokens_per_step, args.steps, world, e2e_total)

    launches_per_step = b.launches_per_step
    per_workload = None
    if rank == 0 and not args.no_per_workload:
        del b, dw
        torch.cuda.empty_cache()
        per_workload = per_workload_lines(args, flush_l2, peak)

    if rank == 0:
        traffic = None if args.cascade else stored_traffic(w.name)
        line = {
            "metric": METRIC,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 MMA operands, f32 accumulate (KV q8_0/q5_1 codes)",
            "data": "synthetic (seeded N(0,1) fp16 q/k/v, random page permutation)",
            "config": workload_config(w), "parallelism": f"replicas x{world}",
            "kv_gbs": world * kv_bytes * args.steps / total_s / 1e9,
            "kv_hbm_frac": world * kv_bytes * args.steps / total_s / 1e9 / peak / world,
            "kv_bytes_per_step": kv_bytes, "kv_bytes_logical_per_step": logical_kv_bytes(w),
            "step_ms": {"median": statistics.median(step_ms), "p10": percentile(step_ms, 10),
                        "p90": percentile(step_ms, 90), "min": min(step_ms), "max": max(step_ms)},
            "roofline": {"kernel": "cascade attention (prefix pass + split-K + merge)" if args.cascade
                         else "decode_split_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs", "launch_ms": statistics.mean(k2_ms),
                         "algorithmic_bytes_per_launch": kv_bytes},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_total / args.steps * 1e3},
            # per timed step: split-K (rows stored inside) + combine, or append + split-K + combine
            "gpu_launches": launches_per_step * args.steps,
            "step_form": ("cascade " if args.cascade else "") + (
                "two-call (memra_kv_append + memra_decode_attn)" if args.two_call else "fused (memra_decode_step)"),
            "clocks": clocks,
            "device_flags": flags,
            "library_sources": _build.built_hash(),
            "per_workload": per_workload,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
