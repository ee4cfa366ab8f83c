#!/usr/bin/env python
"""Benchmark of one forward pass's hot path: per layer kv_append + ragged paged GQA attention.

Default workload: the Qwen2.5-1.5B-shaped decode batch (28 layers, 12 q / 2 KV heads, head_dim 128,
256 rows with contexts uniform in [256, 768] plus one new token, blocks of 16 scattered over a pool 1.25x
the need, fp16 values from the seeded generator).  A step = one attention plan + 28 x (append + attention).

The timed region replays the step as one CUDA graph (captured from the same library calls), so the
number is the GPU's, not the host's launch rate; `--eager` times the calls issued one by one instead.

Prints one JSON line (rank 0).  `value` is algorithmic HBM bytes per second of the whole step (K/V read
once per row and layer, q read, output written, block tables, append traffic); `ctx_tokens_per_s` is the
number of context tokens attended per second.  `--kv-cache e4m3` runs the same step on the 8-bit cache (E4M3
codes and a power-of-two scale per cached row; its bytes counted as stored).  `--impl reference` times the
CPU oracle instead; `--config sched_trace` runs the scheduler policies' trace.
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")   # the oracle legs are single-threaded by design

import argparse
import ctypes
import hashlib
import json
import math
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload  # noqa: E402

CONFIGS = {
    "qwen_decode": lambda: synth.qwen_decode(0),
    "mixed_step": lambda: synth.mixed_step(0),
    "prefill_8k": lambda: synth.prefill_chunk(0),
    "long_gqa": lambda: synth.long_gqa(0),
    "tiny_decode": lambda: synth.tiny_decode(0),
}

# DRAM bytes per pkv_attention call measured with ncu (dram__bytes_read.sum + dram__bytes_write.sum,
# summed over the call's kernels) on the qwen_decode workload, keyed by the sha256 prefix of the kernel
# source they were taken on and the cache format; reported as null once the source changes.
TRAFFIC = {"68f5e3fd9c44/fp16/qwen_decode": 142.34e6,   # profiles/decode_kernel_qwen_decode.md
           "68f5e3fd9c44/e4m3/qwen_decode": 71.68e6}    # profiles/decode_kernel_qwen_decode_e4m3.md

FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(batch: synth.StepBatch, kv8: bool = False):
    """Per layer: (attention bytes, append bytes) -- each cached K/V row of a row read once (GQA grouping):
    head_dim fp16 values, or head_dim E4M3 codes and one scale byte on the 8-bit cache; q read and output
    written once (fp16), 4 bytes per block-table entry; append reads the fp16 k/v and writes them in the
    cache's format, plus the 8-byte slot of each token."""
    s = batch.shape
    ctx = batch.context_lens.astype(np.int64)
    T = int(batch.q_lens.sum())
    row = s.head_dim + 1 if kv8 else s.head_dim * 2   # bytes of one cached (token, KV head) row of K or V
    attn = (2 * int(ctx.sum()) * s.num_kv_heads * row + T * s.num_q_heads * s.head_dim * 2 * 2
            + 4 * int(((ctx + 15) // 16).sum()))
    append = T * s.num_kv_heads * (s.head_dim * 2 * 2 + row * 2) + 8 * T
    return attn, append


FALLBACK_TENSOR_TFLOPS = 1900.0
PREFILL_MIN_QLEN = 16  # rows with this many new tokens run on the tensor-core tile kernel


def measured_peak(key: str = "hbm_gbs", fallback: float = FALLBACK_HBM_GBS):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback, "fallback"


def long_merge(batch: synth.StepBatch, pool) -> bool:
    """Whether some token of the pass has more than 32 splits (then a merge launch follows each decode)."""
    split = pool.cfg.split_blocks or pkv.DEFAULT_SPLIT_BLOCKS
    nblk = (batch.context_lens.astype(np.int64) + 15) // 16
    return bool((((nblk + split - 1) // split) > 32).any())


def prefill_flops(batch: synth.StepBatch) -> int:
    """Per layer: 4 d Hq (causal query-key pairs) over the rows that take the tile kernel."""
    s = batch.shape
    pairs = 0
    for c, q in zip(batch.context_lens.astype(np.int64), batch.q_lens.astype(np.int64)):
        if q >= PREFILL_MIN_QLEN:
            pairs += int(q * (c - q) + q * (q + 1) // 2)
    return 4 * s.head_dim * s.num_q_heads * pairs


def time_prefill_rows(batch: synth.StepBatch, reps: int = 20, kv_dtype: int = pkv.PKV_KV_F16):
    """Mean CUDA-event time of one attention call over only the batch's prefill rows (the tile kernel,
    plus an empty decode launch; on the 8-bit cache also the dequantizing launch), rotating over the layers;
    None if the batch has no such rows."""
    rows = [b for b in range(batch.num_seqs) if batch.q_lens[b] >= PREFILL_MIN_QLEN]
    if not rows:
        return None
    s = batch.shape
    sub = synth.custom_batch(s, batch.cached_lens[rows], batch.q_lens[rows], seed=batch.seed,
                             req_ids=batch.req_ids[rows])
    layers = list(range(s.num_layers))
    pool = workload.make_pool(sub, kv_dtype=kv_dtype)
    workload.prefill_cache(pool, sub, layers)
    ds = workload.upload(sub, pool)
    qs, _, _ = workload.step_inputs(ds, layers)
    outs = [torch.empty_like(q) for q in qs]
    attn = workload.Attention(pool, ds)
    attn.plan()
    for i, layer in enumerate(layers):
        attn.run(layer, qs[i], outs[i])
    torch.cuda.synchronize()
    ev = []
    for _ in range(reps):
        for i, layer in enumerate(layers):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            attn.run(layer, qs[i], outs[i])
            b.record()
            ev.append((a, b))
    torch.cuda.synchronize()
    assert pool.check() == 0
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def source_hash() -> str:
    """sha256 prefix of the kernel sources with comments and blank lines removed: a measurement stays keyed
    to the code it was taken on, whatever happens to the comments."""
    h = hashlib.sha256()
    for f in ("attention.cu", "decode.cuh", "decode_e4m3.cu", "pkv_internal.cuh"):
        with open(os.path.join(ROOT, "continuous_batching_paged_ragged_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:12]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        loaded = [s for s in sms if s > 0.5 * max(sms)] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: replicas run independently, the job ends with the last one."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------------------
# CPU oracle legs (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------------------------------

def oracle_inputs(batch: synth.StepBatch, layer: int, rows, max_queries: int = 0):
    """Per row: (q, k, v) for the oracle; with max_queries > 0 a longer chunk keeps only its last max_queries
    queries (each still over its whole causal context)."""
    s = batch.shape
    items = []
    for b in rows:
        req, ctx = int(batch.req_ids[b]), int(batch.context_lens[b])
        ql = int(batch.q_lens[b])
        if max_queries > 0:
            ql = min(ql, max_queries)
        k, v = synth.sequence_kv(batch.seed, layer, req, ctx, s.num_kv_heads, s.head_dim)
        q = synth.token_values(synth.KIND_Q, batch.seed, layer, np.full(ql, req), np.arange(ctx - ql, ctx),
                               s.num_q_heads, s.head_dim)
        items.append((q, k, v))
    return items


def oracle_bytes(batch, rows, max_queries: int = 0):
    s = batch.shape
    ctx = batch.context_lens[rows].astype(np.int64)
    ql = batch.q_lens[rows].astype(np.int64)
    if max_queries > 0:
        ql = np.minimum(ql, max_queries)
    return (2 * int(ctx.sum()) * s.num_kv_heads * s.head_dim * 2 + int(ql.sum()) * s.num_q_heads * s.head_dim * 4
            + 4 * int(((ctx + 15) // 16).sum())), int(ctx.sum())


def cpu_baseline(batch, budget_s: float = 12.0, kv8: bool = False, max_queries: int = 0):
    import oracle
    rows = list(range(batch.num_seqs))
    items = oracle_inputs(batch, 0, rows, max_queries)
    nbytes, nctx = oracle_bytes(batch, rows, max_queries)
    if kv8:   # attention over the dequantized 8-bit cache (quantized once, outside the timing)
        from oracle import fp8
        items = [(q, fp8.dequantize_rows(*fp8.quantize_rows(k)), fp8.dequantize_rows(*fp8.quantize_rows(v)))
                 for q, k, v in items]
        s = batch.shape
        nbytes -= int(batch.context_lens.astype(np.int64).sum()) * 2 * s.num_kv_heads * (s.head_dim - 1)
    reps, t0 = 0, time.perf_counter()
    while True:
        for q, k, v in items:
            oracle.attention_row(q, k, v)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    return {"value": nbytes * reps / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "ctx_tokens_per_s": nctx * reps / el,
            "sample": f"layer 0 of {batch.shape.num_layers}, all {batch.num_seqs} rows"
                      + (f" (a chunk's last {max_queries} queries at most)" if max_queries else "")
                      + f", repeated {reps}x ({el:.1f} s, fp64 NumPy, 1 thread of {os.cpu_count()} host cores)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    batch = CONFIGS[args.config]()
    rows_all = list(range(batch.num_seqs))
    probe = oracle_inputs(batch, 0, rows_all[:8])
    t0 = time.perf_counter()
    for q, k, v in probe:
        oracle.attention_row(q, k, v)
    per_row = (time.perf_counter() - t0) / len(probe)
    budget = 150.0 / (args.steps + args.warmup)
    n = int(max(1, min(batch.num_seqs, budget / max(per_row, 1e-6))))
    rows = rows_all[:n]
    items = oracle_inputs(batch, 0, rows)
    nbytes, nctx = oracle_bytes(batch, rows)
    if args.kv_cache == "e4m3":   # attention over the dequantized 8-bit cache (quantized once, untimed)
        from oracle import fp8
        items = [(q, fp8.dequantize_rows(*fp8.quantize_rows(k)), fp8.dequantize_rows(*fp8.quantize_rows(v)))
                 for q, k, v in items]
        s = batch.shape
        nbytes -= nctx * 2 * s.num_kv_heads * (s.head_dim - 1)
    for _ in range(args.warmup):
        for q, k, v in items:
            oracle.attention_row(q, k, v)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for q, k, v in items:
            oracle.attention_row(q, k, v)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": "paged ragged attention: achieved HBM GB/s (% of GB300 peak), ctx tokens/s",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": batch.name, "rows_per_step": n, "layers_per_step": 1, "kv_cache": args.kv_cache},
        "ctx_tokens_per_s": nctx * args.steps / el,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} of {batch.num_seqs} rows of layer 0 per step, fp64 NumPy, 1 thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------------
# GPU path
# ----------------------------------------------------------------------------------------------------

def measure(args, batch, rank, world, local, steps, warmup, cpu_budget_s=12.0, with_e2e=True, cpu_max_queries=0):
    """One workload's timed step (plan + every layer's append and attention, as one CUDA graph unless
    --eager); returns the JSON fields (rank 0) or None."""
    dev = torch.device("cuda", local)
    s = batch.shape
    layers = list(range(s.num_layers))
    kv8 = args.kv_cache == "e4m3"
    fused = not args.unfused
    pool = workload.make_pool(batch, split_blocks=args.split_blocks,
                              kv_dtype=pkv.PKV_KV_E4M3 if kv8 else pkv.PKV_KV_F16)
    split_blocks = pool.cfg.split_blocks or pkv.DEFAULT_SPLIT_BLOCKS
    merge_launch = long_merge(batch, pool)
    workload.prefill_cache(pool, batch, layers)
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, layers)
    outs = [torch.empty_like(q) for q in qs]
    attn = workload.Attention(pool, ds)
    stream = torch.cuda.current_stream(dev)
    step = workload.RawStep(pool, ds, attn, qs, ks, vs, outs, stream.cuda_stream, fused=fused)
    torch.cuda.synchronize()
    assert pool.check() == 0

    # the step as one CUDA graph: the same calls, captured on a side stream, replayed on `stream`
    graph = None
    if not args.eager:
        graph, launches_per_step = workload.capture_step_graph(pool, ds, attn, qs, ks, vs, outs, layers, fused=fused,
                                                               device=dev)
    graphed = graph is not None

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step(layers)

    attn_bytes, append_bytes = algorithmic_bytes(batch, kv8)
    step_bytes = (attn_bytes + append_bytes) * len(layers)
    ctx_tokens = int(batch.context_lens.astype(np.int64).sum()) * len(layers)

    # ---- device-resident timed region ----
    for _ in range(warmup):
        run_step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    step.launches = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    launches = step.launches if graph is None else launches_per_step * steps
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    assert pool.check() == 0

    # ---- per-kernel timing of the dominant call (pkv_attention), events on its stream ----
    kev = []
    n_kernel_steps = max(3, min(steps, 200))
    for _ in range(n_kernel_steps):
        step.plan()
        for i, layer in enumerate(layers):
            if not fused:
                step.append(i, layer)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if fused:
                step.attention_append(i, layer)  # the decode kernel does the append too
            else:
                step.attention(i, layer)
            b.record(stream)
            kev.append((a, b))
    torch.cuda.synchronize()
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)

    # ---- end to end through the public calls with host buffers ----
    e2e = run_e2e(args, batch, pool, ds, attn, qs, ks, vs, outs, stream, layers, step_bytes, steps) if with_e2e else None
    del graph, step, attn, qs, ks, vs, outs, ds
    pool.close()
    del pool
    torch.cuda.empty_cache()
    pf_ms = time_prefill_rows(batch, kv_dtype=pkv.PKV_KV_E4M3 if kv8 else pkv.PKV_KV_F16) if rank == 0 else None
    torch.cuda.empty_cache()

    if rank != 0:
        return None
    peak, peak_src = measured_peak()
    kernel_bytes = attn_bytes + (append_bytes if fused else 0)
    # The dominant kernel's average launch duration over the timed region: with the fused call a step is
    # one plan launch plus one attention launch per layer (plus the long-context merge launch where a
    # token has more than 32 splits), so the step time over the layer count is an upper bound on it (the
    # plan's share is charged to the attention).  Layers are pipelined through programmatic dependent
    # launch inside the timed region; `isolated_call_ms` is the same call issued alone, between events.
    per_call_ms = ms / len(layers) if (fused and graphed) else attn_ms
    achieved = kernel_bytes / (per_call_ms * 1e-3) / 1e9
    sh = source_hash()
    value = step_bytes * world / (ms * 1e-3) / 1e9
    line = {
        "metric": "paged ragged attention: achieved HBM GB/s (% of GB300 peak), ctx tokens/s",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded Philox4x32-10, Irwin-Hall approx N(0,1) fp16)",
        "config": {"workload": batch.name, "layers": s.num_layers, "num_q_heads": s.num_q_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
                   "rows": batch.num_seqs, "new_tokens": batch.num_tokens,
                   "context_tokens_per_layer": int(batch.context_lens.sum()), "pool_blocks": batch.num_blocks,
                   "kv_cache": "e4m3 codes + power-of-two scale per cached row" if kv8 else "fp16",
                   "split_blocks": split_blocks,
                   "l2": f"inputs larger than L2: {step_bytes / 1e9:.2f} GB of K/V per step rotating over "
                         f"{s.num_layers} layer pools", "parallelism": f"replicas x{world}",
                   "launch": "eager" if not graphed else "cuda_graph",
                   "layer_call": "pkv_append + pkv_attention" if args.unfused else "pkv_attention_append"},
        "pct_of_peak": 100.0 * value / world / peak,
        "ctx_tokens_per_s": ctx_tokens * world / (ms * 1e-3),
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": TRAFFIC.get(f"{sh}/{args.kv_cache}/{batch.name}"),
                     "kernel": "decode_kernel (split-K decode, fused merge" + (", fused append)" if fused else ")")
                               + (" + merge_kernel (tokens with > 32 splits)" if merge_launch else ""),
                     "per_launch_bytes": kernel_bytes, "avg_launch_ms": per_call_ms,
                     "avg_launch_over": "timed region (CUDA graph, step time / layers)"
                                        if per_call_ms is not attn_ms else "per-call CUDA events",
                     "isolated_call_ms": attn_ms,
                     "isolated_frac": kernel_bytes / (attn_ms * 1e-3) / 1e9 / peak, "peak_source": peak_src,
                     "source": sh},
        "e2e": e2e,
        "clocks": clocks,
    }
    if pf_ms is not None:
        # a mixed pass: the prefill rows are tensor-bound, the decode rows HBM-bound (report both)
        tpeak, tsrc = measured_peak("bf16_tflops", FALLBACK_TENSOR_TFLOPS)
        flops = prefill_flops(batch)
        decode = line["roofline"]
        decode["kernel"] = "decode_kernel + prefill_kernel (whole attention call)"
        line["roofline"] = {"bound": "tensor", "achieved": flops / (pf_ms * 1e-3) / 1e12, "peak": tpeak,
                            "unit": "TFLOP/s", "frac": flops / (pf_ms * 1e-3) / 1e12 / tpeak, "traffic": None,
                            "kernel": "prefill_kernel (tcgen05, prefill rows alone)", "flops_per_launch": flops,
                            "avg_launch_ms": pf_ms, "peak_source": f"{tsrc} bf16 dense (fp16 runs at the same rate)"}
        line["attention_call_roofline"] = decode
        hbm_ms = step_bytes / (peak * 1e9) * 1e3
        tensor_ms = flops * len(layers) / (tpeak * 1e12) * 1e3
        line["lower_bounds_ms_per_step"] = {"hbm": hbm_ms, "tensor": tensor_ms, "sum": hbm_ms + tensor_ms,
                                            "max": max(hbm_ms, tensor_ms), "measured": ms}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(batch, budget_s=cpu_budget_s, kv8=kv8, max_queries=cpu_max_queries)
    return line


def run_pkv(args, rank, world, local):
    torch.cuda.set_device(local)
    batch = CONFIGS[args.config]()
    if args.layers:
        batch.shape = synth.Shape(args.layers, batch.shape.num_q_heads, batch.shape.num_kv_heads,
                                  batch.shape.head_dim, batch.shape.block_size)
    line = measure(args, batch, rank, world, local, args.steps, args.warmup)
    if args.config == "qwen_decode" and not args.layers and not args.no_configs and world == 1:
        # the other workloads of the pages, each as its own timed region with its clocks and oracle baseline
        extra = {}
        for name, steps, cpu_q in (("mixed_step", min(args.steps, 100), 0), ("prefill_8k", min(args.steps, 20), 256),
                                   ("long_gqa", min(args.steps, 20), 0)):
            t0 = time.perf_counter()
            sub = measure(args, CONFIGS[name](), rank, world, local, max(steps, 3), args.warmup, cpu_budget_s=4.0,
                          cpu_max_queries=cpu_q)
            if sub is not None:
                sub["wall_s"] = time.perf_counter() - t0
                extra[name] = sub
        for cap in (256, 64):
            t0 = time.perf_counter()
            res = run_trace_policies(args, local, [t for t in TRACE_POLICIES if t[0] in
                                                   ("on_demand/pass", "on_demand/pass cap 64") and t[4] == cap],
                                     cpu_baseline_s=4.0 if not args.no_cpu_baseline else 0.0)
            if rank == 0 and res:
                res[0]["wall_s"] = time.perf_counter() - t0
                extra[f"sched_trace_cap{cap}"] = res[0]
        if rank == 0:
            line["configs"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------------
# Scheduler-driven trace under each allocation policy and unit of scheduling
# ----------------------------------------------------------------------------------------------------

# (name, allocation, unit, declared output / real output, max_num_seqs, blocks, prefix caching, cache format).
# The last row spends the bytes of the 5,000-block fp16 pool on the 8-bit cache: 2 d / (d + 1) times the blocks.
TRACE_POLICIES = [
    ("on_demand/pass", pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_PASS, 1.0, 256, 20000, False, "fp16"),
    ("reserve 1x/pass", pkv.PKV_ALLOC_RESERVE, pkv.PKV_UNIT_PASS, 1.0, 256, 20000, False, "fp16"),
    ("reserve 4x/pass", pkv.PKV_ALLOC_RESERVE, pkv.PKV_UNIT_PASS, 4.0, 256, 20000, False, "fp16"),
    ("on_demand/pass cap 64", pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_PASS, 1.0, 64, 20000, False, "fp16"),
    ("on_demand/request cap 64", pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_REQUEST, 1.0, 64, 20000, False, "fp16"),
    ("on_demand/pass 5000 blocks", pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_PASS, 1.0, 256, 5000, False, "fp16"),
    ("on_demand/pass 5000 blocks prefix-cached", pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_PASS, 1.0, 256, 5000, True,
     "fp16"),
    ("on_demand/pass 8-bit cache, 9922 blocks (the bytes of 5000 fp16 blocks)", pkv.PKV_ALLOC_ON_DEMAND,
     pkv.PKV_UNIT_PASS, 1.0, 256, 5000 * 2 * 128 // 129, False, "e4m3"),
]
TRACE_SHAPE = (28, 12, 2, 128)  # layers, q heads, KV heads, head_dim (the Qwen2.5-1.5B cache shape)
TRACE_BUDGET = 8192             # new tokens per pass


def trace_cpu_baseline(passes, reqs, budget_s: float):
    """The oracle on a bounded sample of the trace: one layer of the pass with the most decode rows (each row's
    seeded q/k/v), extrapolated to every pass's context tokens and 28 layers; output tokens per second."""
    import oracle
    L, Hq, Hkv, d = TRACE_SHAPE
    best = max(range(len(passes)), key=lambda i: (passes[i]["decode_rows"], -i))
    p = passes[best]
    t0 = time.perf_counter()
    done_ctx = 0
    for req, ql, ctx in zip(p["req_ids"], p["q_lens"], p["context_lens"]):
        ql = min(int(ql), 16)   # a long chunk contributes its last 16 queries (the sample stays bounded)
        k, v = synth.sequence_kv(0, 0, int(req), int(ctx), Hkv, d)
        q = synth.token_values(synth.KIND_Q, 0, 0, np.full(ql, int(req)), np.arange(int(ctx) - ql, int(ctx)), Hq, d)
        oracle.attention_row(q, k, v)
        done_ctx += int(ctx)
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    total_ctx = sum(int(x["ctx_tokens"]) for x in passes) * L
    est_s = el / max(done_ctx, 1) * total_ctx
    outputs = sum(r.max_output for r in reqs)
    return {"value": outputs / est_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done_ctx} context tokens of pass {best} (layer 0, chunks capped at 16 queries), "
                      f"{el:.1f} s of fp64 NumPy on 1 of {os.cpu_count()} host cores, extrapolated to "
                      f"{total_ctx} context tokens (all passes, {L} layers)"}


def run_trace_policies(args, local, policies, cpu_baseline_s: float = 0.0):
    """256 trace requests (lognormal prompts, U[50, 781] outputs, token budget 8,192, max_num_seqs and pool as
    the policy says) run to exhaustion; every pass is the plan + 28 x fused append and attention on the GPU,
    over the seeded q/k/v of the pass's tokens (generated on the device for every layer before the pass).
    Only the GPU work of a pass is timed (CUDA events around it); the host scheduler, the metadata upload and
    the value generation run between passes, outside the timed work."""
    dev = torch.device("cuda", local)
    L, Hq, Hkv, d = TRACE_SHAPE
    budget = TRACE_BUDGET
    reqs = synth.trace_requests(0)
    max_w = max((r.prompt_len + r.max_output + 15) // 16 for r in reqs)
    cap_all = max(t[4] for t in policies)
    nblk = max(t[5] for t in policies)
    pools = {kv: pkv.Pool(L, Hq, Hkv, d, nblk, kv_dtype=pkv.PKV_KV_E4M3 if kv == "e4m3" else pkv.PKV_KV_F16)
             for kv in sorted({t[7] for t in policies})}
    q = torch.empty(L, budget, Hq, d, dtype=torch.float16, device=dev)
    k = torch.empty(L, budget, Hkv, d, dtype=torch.float16, device=dev)
    v = torch.empty_like(k)
    out = torch.empty(budget, Hq, d, dtype=torch.float16, device=dev)
    bt = torch.empty(cap_all * max_w, dtype=torch.int32, device=dev)
    ctx = torch.empty(cap_all, dtype=torch.int32, device=dev)
    qsl = torch.empty(cap_all + 1, dtype=torch.int32, device=dev)
    slots = torch.empty(budget, dtype=torch.int64, device=dev)
    treq = torch.empty(budget, dtype=torch.int64, device=dev)
    tpos = torch.empty(budget, dtype=torch.int64, device=dev)
    ws_bytes = max(pkv.pkv_attention_workspace_bytes(pl.handle, cap_all, budget, max_w) for pl in pools.values())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    lib = pkv.load()
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    results = []
    for name, alloc, unit, declared, max_seqs, blocks, prefix, kv in policies:
        pool = pools[kv]
        sched = pkv.Scheduler(max_seqs, budget, 16, blocks, synth.block_permutation(blocks, 0), alloc=alloc, unit=unit,
                              prefix_caching=prefix)
        for r in reqs:
            sched.add(r.req_id, r.prompt_len, r.max_output, int(round(declared * r.max_output)))
        events, steps, launches, passes = [], 0, 0, []
        sampler = ClockSampler(local)
        sampler.start()
        while not sched.done():
            st = sched.step()
            B, T, W = len(st["req_ids"]), int(st["query_start_loc"][-1]), st["max_blocks_per_seq"]
            qls = np.diff(st["query_start_loc"]).astype(np.int64)
            cl = st["context_lens"].astype(np.int64)
            tok_req = np.repeat(st["req_ids"].astype(np.int64), qls)
            tok_pos = np.concatenate([np.arange(c - n, c) for c, n in zip(cl, qls)]) if B else np.zeros(0, np.int64)
            bt[:B * W].copy_(torch.from_numpy(st["block_tables"].reshape(-1)))
            ctx[:B].copy_(torch.from_numpy(st["context_lens"]))
            qsl[:B + 1].copy_(torch.from_numpy(st["query_start_loc"]))
            slots[:T].copy_(torch.from_numpy(st["slot_mapping"]))
            treq[:T].copy_(torch.from_numpy(tok_req))
            tpos[:T].copy_(torch.from_numpy(tok_pos))
            for layer in range(L):   # the pass's seeded values, outside the timed work
                synth.device_fill(synth.KIND_Q, 0, layer, treq[:T], tpos[:T], Hq, d, q[layer, :T])
                synth.device_fill(synth.KIND_K, 0, layer, treq[:T], tpos[:T], Hkv, d, k[layer, :T])
                synth.device_fill(synth.KIND_V, 0, layer, treq[:T], tpos[:T], Hkv, d, v[layer, :T])
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pkv._check(lib.pkv_attention_plan(pool.handle, ctx.data_ptr(), qsl.data_ptr(), B, T, W, ws.data_ptr(),
                                              ws_bytes, sp), "pkv_attention_plan")
            launches += lib.pkv_last_launch_count(pool.handle)
            for layer in range(L):
                pkv._check(lib.pkv_attention_append(pool.handle, layer, q[layer].data_ptr(), k[layer].data_ptr(),
                                                    v[layer].data_ptr(), slots.data_ptr(), bt.data_ptr(), W,
                                                    ctx.data_ptr(), qsl.data_ptr(), B, T, out.data_ptr(),
                                                    ws.data_ptr(), ws_bytes, sp), "pkv_attention_append")
                launches += lib.pkv_last_launch_count(pool.handle)
            b.record(stream)
            events.append((a, b))
            steps += 1
            passes.append({"req_ids": st["req_ids"].copy(), "q_lens": qls, "context_lens": cl,
                           "decode_rows": int((qls == 1).sum()), "ctx_tokens": int(cl.sum())})
            if len(events) % 128 == 0:  # keep the host from running far ahead of the device
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        clocks = sampler.stop()
        assert pool.check() == 0
        gpu_s = sum(x.elapsed_time(y) for x, y in events) / 1e3
        stt = sched.stats()
        sched.close()
        outputs = sum(r.max_output for r in reqs)
        res = {"policy": name, "max_num_seqs": max_seqs, "output_tokens_per_s": outputs / gpu_s,
               "gpu_s": gpu_s, "steps": steps, "ms_per_step": gpu_s * 1e3 / steps,
               "preemptions": stt["preemptions"], "recomputed_tokens": stt["recomputed_tokens"],
               "max_batch": stt["max_batch"], "mean_batch": stt["batch_sum"] / max(1, stt["steps"]),
               "live_cache": stt["live_tokens"] / max(1, stt["held_slots"]), "pool_blocks": blocks,
               "prefix_hit_tokens": stt["prefix_hit_tokens"], "kv_cache": kv,
               "tokens_scheduled": stt["tokens_scheduled"], "gpu_launches": launches, "clocks": clocks,
               "values": "seeded q/k/v of every pass's tokens (device generator, all layers)"}
        if cpu_baseline_s > 0:
            res["cpu_baseline"] = trace_cpu_baseline(passes, reqs, cpu_baseline_s)
        results.append(res)
    for pl in pools.values():
        pl.close()
    del q, k, v, ws
    torch.cuda.empty_cache()
    return results


def run_sched_trace(args, rank, world, local):
    torch.cuda.set_device(local)
    policies = [t for t in TRACE_POLICIES if re.search(args.trace_filter, t[0])]
    results = run_trace_policies(args, local, policies)
    if rank != 0:
        return
    head = results[0]
    L, Hq, Hkv, d = TRACE_SHAPE
    line = {"metric": "scheduler-driven trace: output tokens/s over the GPU time of its passes", "value":
            head["output_tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": head["steps"], "warmup": 0,
            "ms_per_step": head["gpu_s"] * 1e3 / head["steps"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded trace: 256 requests, lognormal prompts "
            "median 300 clipped [16, 4096], outputs U[50, 781]; seeded q/k/v)",
            "config": {"workload": "sched_trace", "layers": L, "num_q_heads": Hq, "num_kv_heads": Hkv,
                       "head_dim": d, "pool_blocks": head["pool_blocks"], "max_num_seqs": head["max_num_seqs"],
                       "token_budget": TRACE_BUDGET, "split_blocks": pkv.DEFAULT_SPLIT_BLOCKS,
                       "launch": "eager (per-pass events)"},
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "policies": results}
    print(json.dumps(line), flush=True)


def e2e_chunks(L: int):
    """The end-to-end step's copy chunks over L layers: `ups`, the first layer of each upload chunk after layer 0
    (chunk c is layers [ups[c], ups[c + 1]), the last one up to L), and `cuts`, the layer before which each
    download chunk goes down (chunk c is layers [cuts[c - 1], cuts[c]), the first from 0; the layers from the
    last cut on go down after the step).  Uploads double in size, downloads halve toward the end."""
    ups = [b for b in (1 << k for k in range(32)) if b < L]
    cuts = sorted({L - (1 << k) for k in range(32) if 0 < L - (1 << k) < L})
    return ups, cuts


def run_e2e(args, batch, pool, ds, attn, qs, ks, vs, outs, stream, layers, step_bytes, steps):
    """The same metric end to end through the public calls: every step copies the pass's metadata and every
    layer's q/k/v from pinned host memory and reads every layer's output back.  The copies run beside the
    attention on two copy streams in chunks that double in size, so that only a layer's worth is exposed at
    each end: layer 0's inputs go up before the plan, layers [1, 2), [2, 4), [4, 8), ... on the upload stream
    (the compute stream waits for each chunk before its first layer, by then long landed: a layer's inputs
    take a fraction of its attention time); the outputs come down in chunks that halve toward the end, each
    as soon as its last layer is done, the last layer's after it.  The step (copies, events and library calls)
    is captured as one CUDA graph, as the device-resident timing is (--eager: issued call by call)."""
    dev = stream.device
    L = len(layers)
    h_q = torch.stack([q.cpu() for q in qs]).pin_memory()
    h_k = torch.stack([k.cpu() for k in ks]).pin_memory()
    h_v = torch.stack([v.cpu() for v in vs]).pin_memory()
    h_out = torch.empty((L,) + tuple(outs[0].shape), dtype=torch.float16).pin_memory()
    h_bt = ds.block_tables.cpu().pin_memory()
    h_ctx = ds.context_lens.cpu().pin_memory()
    h_qsl = ds.query_start_loc.cpu().pin_memory()
    h_slots = ds.slot_mapping.cpu().pin_memory()
    d_q = torch.stack(qs)
    d_k = torch.stack(ks)
    d_v = torch.stack(vs)
    d_out = torch.stack(outs)
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_bt, h_ctx, h_qsl, h_slots))
    d2h = h_out.numel() * h_out.element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ups, cuts = e2e_chunks(L)
    ev_up = [torch.cuda.Event() for _ in ups]
    ev_cut = [torch.cuda.Event() for _ in cuts]

    def one(main, step):
        with torch.cuda.stream(main):
            ds.block_tables.copy_(h_bt, non_blocking=True)
            ds.context_lens.copy_(h_ctx, non_blocking=True)
            ds.query_start_loc.copy_(h_qsl, non_blocking=True)
            ds.slot_mapping.copy_(h_slots, non_blocking=True)
            d_q[:1].copy_(h_q[:1], non_blocking=True)
            d_k[:1].copy_(h_k[:1], non_blocking=True)
            d_v[:1].copy_(h_v[:1], non_blocking=True)
        up.wait_stream(main)      # the previous step has read its inputs
        down.wait_stream(main)
        with torch.cuda.stream(up):
            for c, lo in enumerate(ups):
                hi = ups[c + 1] if c + 1 < len(ups) else L
                d_q[lo:hi].copy_(h_q[lo:hi], non_blocking=True)
                d_k[lo:hi].copy_(h_k[lo:hi], non_blocking=True)
                d_v[lo:hi].copy_(h_v[lo:hi], non_blocking=True)
                ev_up[c].record(up)
        step.plan()
        for i, layer in enumerate(layers):
            if i in ups:
                main.wait_event(ev_up[ups.index(i)])
            if i in cuts:
                c = cuts.index(i)
                lo = cuts[c - 1] if c else 0
                ev_cut[c].record(main)
                down.wait_event(ev_cut[c])
                with torch.cuda.stream(down):
                    h_out[lo:i].copy_(d_out[lo:i], non_blocking=True)
            if step.fused:
                step.attention_append(i, layer)
            else:
                step.append(i, layer)
                step.attention(i, layer)
        tail = cuts[-1] if cuts else 0
        with torch.cuda.stream(main):
            h_out[tail:].copy_(d_out[tail:], non_blocking=True)
        main.wait_stream(up)
        main.wait_stream(down)

    n = max(3, min(steps, 200))
    if args.eager:
        step = workload.RawStep(pool, ds, attn, list(d_q), list(d_k), list(d_v), list(d_out), stream.cuda_stream,
                                fused=not args.unfused)
        run = lambda: one(stream, step)  # noqa: E731
    else:
        cap = torch.cuda.Stream(dev)
        step = workload.RawStep(pool, ds, attn, list(d_q), list(d_k), list(d_v), list(d_out), cap.cuda_stream,
                                fused=not args.unfused)
        cap.wait_stream(stream)
        for _ in range(2):
            one(cap, step)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            one(cap, step)
        torch.cuda.synchronize()
        run = graph.replay
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"value": step_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "copies": "layer 0's inputs before the step, the rest on a copy stream in chunks starting at layers "
                      f"{ups}; outputs on a second copy stream in chunks ending at layers {cuts}, the last layer's "
                      "after it" + ("" if args.eager else "; the step captured as one CUDA graph")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--config", default="qwen_decode", choices=sorted(CONFIGS) + ["sched_trace"])
    ap.add_argument("--split-blocks", type=int, default=0)
    ap.add_argument("--trace-filter", default="", help="sched_trace: run the policies whose name matches this "
                    "regular expression")
    ap.add_argument("--kv-cache", default="fp16", choices=["fp16", "e4m3"],
                    help="cache format: fp16 values, or E4M3 codes with a power-of-two scale per cached row")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="the default workload alone (no configs object)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--eager", action="store_true", help="time the calls issued one by one, not a CUDA graph")
    ap.add_argument("--unfused", action="store_true", help="pkv_append then pkv_attention per layer, not the "
                    "fused pkv_attention_append")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        if args.config == "sched_trace":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the attention workloads; "
                                  "the scheduler trace's policies are compared on the GPU path only"}), flush=True)
            return
        return run_reference(args, rank, world)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        if args.config == "sched_trace":
            return run_sched_trace(args, rank, world, local)
        run_pkv(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
