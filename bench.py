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
steps outside the events, max over ranks.
With --gpus N (under torchrun) every rank runs an independent replica of the
workload (the path shards into independent sequences; there is no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

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


def cpu_baseline(workload: str, reps: int) -> dict:
    """The oracle, as it stands, timed on host cores in a single-threaded subprocess."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload, "--steps", str(reps)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if r.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": "failed: " +
                r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    return json.loads(r.stdout.strip().splitlines()[-1])


class OracleStep:
    """The CPU oracle on one KV head of one step (its query group over the whole context).

    Preparation (the cache as it stands before the step, i.e. the quantized
    prefill rows) is untimed, like the GPU prefill.  run() times the step:
    quantize the step's new rows, then attention over the dequantized cache.
    """

    def __init__(self, workload: str):
        import workloads as W
        from oracle import quant
        self.w = w = W.WORKLOADS[workload]()
        self.kh = 0
        self.pre = w.prefill_rows
        self.fields = {}
        for s, src, fmt, sc in (("k", w.k_rows, w.k_fmt, w.k_scale), ("v", w.v_rows, w.v_fmt, w.v_scale)):
            self.fields[s] = quant.quantize_rows(src[self.pre, self.kh, :], fmt, sc)
        G = w.n_heads // w.n_kv_heads
        self.G = G
        self.rows = [(b, i, self.kh * G + h) for b in range(w.batch) for i in range(w.q_len) for h in range(G)]

    def run(self) -> float:
        import numpy as np
        from oracle import attention, quant
        w, kh = self.w, self.kh
        t0 = time.perf_counter()
        cache = {"k": [None] * w.n_kv_heads, "v": [None] * w.n_kv_heads}
        for s, src, fmt, sc in (("k", w.k_rows, w.k_fmt, w.k_scale), ("v", w.v_rows, w.v_fmt, w.v_scale)):
            new = quant.quantize_rows(src[w.step_rows, kh, :], fmt, sc)
            full = {"fmt": fmt}
            for key, val in self.fields[s].items():
                if isinstance(val, np.ndarray):
                    arr = np.empty((w.slots.size,) + val.shape[1:], dtype=val.dtype)
                    arr[self.pre] = val
                    arr[w.step_rows] = new[key]
                    full[key] = arr
                elif key != "fmt":
                    full[key] = val
            cache[s][kh] = full
        attention.reference(w, cache=cache, rows=self.rows)
        return (time.perf_counter() - t0) * w.n_kv_heads          # scaled to all KV heads of the step

    def describe(self, how: str) -> str:
        return (f"KV head 0 of one step of {self.w.name} (its {self.G} query heads over the whole context), "
                f"{how}, x{self.w.n_kv_heads} KV heads; single thread")


def oracle_sample(workload: str, reps: int) -> dict:
    st = OracleStep(workload)
    times = [st.run() for _ in range(reps)]
    per_step = statistics.median(times)
    w = st.w
    return {"value": w.batch * w.q_len / per_step, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": st.describe(f"median of {reps} reps"), "seconds_per_step": per_step}


def run_reference_arm(args) -> None:
    world, rank, _ = dist_env()
    if rank != 0:
        return
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(var, "1")
    st = OracleStep(args.workload)
    w = st.w
    for _ in range(args.warmup):
        st.run()
    t0 = time.perf_counter()
    times = [st.run() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    per_step = statistics.mean(times)
    value = w.batch * w.q_len / per_step
    cb = {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
          "sample": st.describe(f"mean of {args.steps} steps")}
    line = {"impl": "reference", "metric": "decode-attn tokens/s (quantized-KV GB/s, % of HBM peak)",
            "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": cb, "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


def workload_config(w) -> dict:
    return {"workload": w.name, "batch": w.batch, "q_len": w.q_len, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "context_tokens": int(w.seq_lens.sum()), "unique_tokens": int(w.slots.size),
            "kv_format": f"{w.k_fmt}/{w.v_fmt}", "page_size": 16, "split_tokens": "max(1024, T / (SMs x CTAs per SM / KV heads))",
            "l2": "flushed between steps (256 MiB write, then read back, outside the timed events)"}


def percentile(xs, pct):
    """Linear-interpolated percentile of a non-empty list (numpy's default rule)."""
    ys = sorted(xs)
    pos = (len(ys) - 1) * pct / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--formats", default=None, help="K/V formats overriding the workload's, e.g. q8_0/q4_0")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--two-call", action="store_true",
                    help="time memra_kv_append + memra_decode_attn instead of the fused memra_decode_step")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix workloads: the cascade calls (the prefix once per KV head on tcgen05)")
    ap.add_argument("--cpu-reps", type=int, default=5)
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        print(json.dumps(oracle_sample(args.workload, args.steps)))
        return
    if args.impl == "reference":
        run_reference_arm(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    world, rank, local = dist_env()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.cpu_reps)      # before any CUDA work in this process

    import torch
    import torch.distributed as dist
    import workloads as W
    import decode_attention_block_memra_gb300 as memra
    from decode_attention_block_memra_gb300 import _build
    from decode_attention_block_memra_gb300.runner import upload

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    memra.lib()
    w = W.WORKLOADS[args.workload]()
    if args.formats:
        w = w.with_formats(*args.formats.split("/"))
    dw = upload(w)
    # The step's inputs (q, the new rows, the lengths, the page table) live in one device buffer at
    # 256-byte offsets, so that the end-to-end step uploads them from one pinned buffer in one copy.
    step_inputs = [("q", dw.q), ("step_k", dw.step_k), ("step_v", dw.step_v), ("seq_lens", dw.seq_lens),
                   ("page_table", dw.page_table)] + ([("step_slots", dw.step_slots)] if args.two_call else [])
    offsets, total = [], 0
    for _, t in step_inputs:
        offsets.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    dev_pack = torch.empty(total, dtype=torch.uint8, device="cuda")
    host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    for (name, t), off in zip(step_inputs, offsets):
        nbytes = t.numel() * t.element_size()
        view = dev_pack[off:off + nbytes].view(t.dtype).view(t.shape)
        view.copy_(t)
        host_pack[off:off + nbytes].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        setattr(dw, name, view)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def flush_l2():
        # write a buffer larger than L2, then read it back: the KV lines are gone
        # and no dirty lines are left to be written back during the timed step
        flush.fill_(1)
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=flush_sink)

    B, Q = w.batch, w.q_len
    k_new = dw.step_k.view(B, Q, w.n_kv_heads, w.head_dim)
    v_new = dw.step_v.view(B, Q, w.n_kv_heads, w.head_dim)
    if args.cascade:
        if not w.shared_prefix:
            raise SystemExit("--cascade needs a workload with a shared prefix")
        cws = torch.empty(memra.decode_attn_cascade_workspace_bytes(B, Q, w.n_heads, w.head_dim, w.max_seq_len,
                                                                    w.shared_prefix), dtype=torch.uint8,
                          device="cuda")

    def hot_path():
        # store the step's rows and attend: one memra_decode_step (split-K with
        # the rows stored inside, then the combine), or the two-call form
        if args.cascade:
            if args.two_call:
                memra.kv_append(dw.cache, dw.step_k, dw.step_v, dw.step_slots, stream=stream)
                memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                                          w.shared_prefix, dw.out, cws, w.sm_scale, stream=stream)
            else:
                memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len,
                                          w.shared_prefix, dw.out, cws, w.sm_scale, stream=stream, k_new=k_new,
                                          v_new=v_new)
        elif args.two_call:
            memra.kv_append(dw.cache, dw.step_k, dw.step_v, dw.step_slots, stream=stream)
            memra.decode_attn(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out, dw.workspace,
                              w.sm_scale, stream=stream)
        else:
            memra.decode_step(dw.cache, k_new, v_new, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out,
                              dw.workspace, w.sm_scale, stream=stream)

    # the split kernel, the combine (left out when every row fits one split), the separate append of the
    # two-call form, the cascade's prefix pass
    combine = 1 if (args.cascade or w.max_seq_len > memra.SPLIT_TOKENS) else 0
    launches_per_step = 1 + combine + (1 if args.two_call else 0) + (1 if args.cascade else 0)

    def step(ev0, ev1):
        # one pass of the hot path through the public entry points, events only
        # at its two ends so the launches chain as they do in use
        ev0.record(stream)
        hot_path()
        ev1.record(stream)

    def split_pass(ev0, ev1):
        # the split-K kernel alone (its partials pass), for its roofline; with
        # --cascade the whole cascade attention (prefix pass, split-K, merge)
        ev0.record(stream)
        if args.cascade:
            memra.decode_attn_cascade(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, w.shared_prefix,
                                      dw.out, cws, w.sm_scale, stream=stream)
        else:
            memra.decode_attn_partials(dw.cache, dw.q, dw.page_table, dw.seq_lens, w.max_seq_len, dw.out,
                                       dw.workspace, w.sm_scale, stream=stream)
        ev1.record(stream)

    def new_events(n):
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]

    for e in new_events(args.warmup):
        flush_l2()
        step(*e)
    torch.cuda.synchronize()
    if memra.read_status(dw.cache):
        raise RuntimeError("device status flagged during warm-up")

    sampler = ClockSampler(local)
    evs = new_events(args.steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for e in evs:
        flush_l2()
        step(*e)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    flags = memra.read_status(dw.cache)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    # the split kernel timed alone over as many launches (same inputs, L2 flushed)
    kev = new_events(args.steps)
    for e in new_events(3):
        flush_l2()
        split_pass(*e)
    for e in kev:
        flush_l2()
        split_pass(*e)
    torch.cuda.synchronize()
    k2_ms = [a.elapsed_time(b) for a, b in kev]
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
    h2d = host_pack.numel()
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        dev_pack.copy_(host_pack, non_blocking=True)
        hot_path()
        out_host.copy_(dw.out, non_blocking=True)

    for _ in range(args.warmup):
        flush_l2()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_total = max_over_ranks(sum(e2e_ms) / 1e3, world, "cuda")
    e2e_value = job_throughput(tokens_per_step, args.steps, world, e2e_total)

    if rank == 0:
        traffic = None if args.cascade else stored_traffic(w.name)
        line = {
            "metric": "decode-attn tokens/s (quantized-KV GB/s, % of HBM peak)",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 MMA operands, f32 accumulate (KV q8_0/q5_1 codes)",
            "data": "synthetic (seeded N(0,1) fp16 q/k/v, random page permutation)",
            "config": {**workload_config(w), "parallelism": f"replicas x{world}"},
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
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
