"""Shared pieces of the GPU parity tests: run a pass through libpkv and compare rows with the oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from oracle import fp8
from continuous_batching_paged_ragged_gb300 import pkv, synth, workload

MAX_ABS = 4e-3    # tolerance on fp16 attention outputs vs the fp64 oracle
MEAN_ABS = 5e-4


def oracle_row(batch: synth.StepBatch, layer: int, b: int, kv_heads=None) -> np.ndarray:
    """fp64 [q_len, Hq, d] (or the q heads of KV heads kv_heads=(lo, hi)) for row b of the pass."""
    s = batch.shape
    G = s.num_q_heads // s.num_kv_heads
    req, ctx, ql = int(batch.req_ids[b]), int(batch.context_lens[b]), int(batch.q_lens[b])
    k, v = synth.sequence_kv(batch.seed, layer, req, ctx, s.num_kv_heads, s.head_dim, kv_heads)
    qh = None if kv_heads is None else (kv_heads[0] * G, kv_heads[1] * G)
    q = synth.token_values(synth.KIND_Q, batch.seed, layer, np.full(ql, req), np.arange(ctx - ql, ctx),
                           s.num_q_heads, s.head_dim, qh)
    return oracle.attention_row(q, k, v)


def oracle_row_8bit(batch: synth.StepBatch, layer: int, b: int) -> np.ndarray:
    """The same over an 8-bit cache: every cached row of K and V quantized (oracle.fp8), attention over the
    dequantized values."""
    s = batch.shape
    req, ctx, ql = int(batch.req_ids[b]), int(batch.context_lens[b]), int(batch.q_lens[b])
    k, v = synth.sequence_kv(batch.seed, layer, req, ctx, s.num_kv_heads, s.head_dim)
    kq = fp8.dequantize_rows(*fp8.quantize_rows(k))
    vq = fp8.dequantize_rows(*fp8.quantize_rows(v))
    q = synth.token_values(synth.KIND_Q, batch.seed, layer, np.full(ql, req), np.arange(ctx - ql, ctx),
                           s.num_q_heads, s.head_dim)
    return oracle.attention_row(q, kq, vq)


def assert_close(gpu_fp16: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    g = gpu_fp16.astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    assert stats["max_abs"] <= MAX_ABS, f"{what}: {stats}"
    assert stats["mean_abs"] <= MEAN_ABS, f"{what}: {stats}"
    return stats


def poison(pool) -> None:
    """NaN everywhere not written: fp16 NaN values, or E4M3 NaN codes and scale bytes of 255 (2^128)."""
    if pool.is_8bit:
        pool.cache_view().fill_(0x7F)
        pool.scales_view().fill_(0xFF)
    else:
        pool.cache_view().view(torch.int16).fill_(0x7E00)


def run_batch(batch: synth.StepBatch, layers, num_layers=None, split_blocks=0, poison=True, pool=None,
              kv_dtype=pkv.PKV_KV_F16, fused=False):
    """Allocate a pool (NaN-poisoned), pre-fill the cached tokens, run the pass; returns (pool, ds, outs)."""
    if pool is None:
        pool = workload.make_pool(batch, num_layers, split_blocks, kv_dtype=kv_dtype)
        if poison:
            globals()["poison"](pool)
    workload.prefill_cache(pool, batch, layers)
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, layers)
    outs = [torch.empty_like(q) for q in qs]
    workload.run_pass(pool, ds, layers, qs, ks, vs, outs, fused=fused)
    torch.cuda.synchronize()
    bits = pool.check()
    assert bits == 0, f"device error word set: {bits:#x}"
    return pool, ds, outs


def row_slice(batch: synth.StepBatch, out: torch.Tensor, b: int) -> np.ndarray:
    qsl = batch.query_start_loc
    return out[int(qsl[b]):int(qsl[b + 1])].cpu().numpy()


# --- passes over edited values -------------------------------------------------------------------------
# Some cases need values the seeded generator never produces (a dominant key, queries aligned with a key,
# scores spanning tens of log2 units).  The test builds them on the host from the generator's values, the
# pool receives them through pkv_slot_mapping + pkv_append, and the oracle reads the same host arrays.

def host_rows(batch: synth.StepBatch, layer: int):
    """Per row b: [q (q_len, Hq, d), k (ctx, Hkv, d), v] fp16 host copies of the generator's values."""
    s = batch.shape
    rows = []
    for b in range(batch.num_seqs):
        req, ctx, ql = int(batch.req_ids[b]), int(batch.context_lens[b]), int(batch.q_lens[b])
        k, v = synth.sequence_kv(batch.seed, layer, req, ctx, s.num_kv_heads, s.head_dim)
        q = synth.token_values(synth.KIND_Q, batch.seed, layer, np.full(ql, req), np.arange(ctx - ql, ctx),
                               s.num_q_heads, s.head_dim)
        rows.append([q.copy(), k.copy(), v.copy()])
    return rows


def oracle_host_row(row, kv_dtype=pkv.PKV_KV_F16) -> np.ndarray:
    """fp64 oracle of one row of host values (over the dequantized values on an 8-bit cache)."""
    q, k, v = row
    if kv_dtype == pkv.PKV_KV_E4M3:
        k = fp8.dequantize_rows(*fp8.quantize_rows(k))
        v = fp8.dequantize_rows(*fp8.quantize_rows(v))
    return oracle.attention_row(q, k, v)


def run_host_values(batch: synth.StepBatch, layers, rows_by_layer, kv_dtype=pkv.PKV_KV_F16, fused=False,
                    split_blocks=0, num_layers=None, device="cuda"):
    """Run one pass over host values: every row's cached positions written through pkv_slot_mapping +
    pkv_append, then the pass's append + attention (or the fused call) on its new tokens.  The pool starts
    NaN-poisoned.  Returns (pool, ds, outs)."""
    pool = workload.make_pool(batch, num_layers or (max(layers) + 1), split_blocks, kv_dtype=kv_dtype)
    poison(pool)
    cached = batch.cached_lens
    have = np.nonzero(cached > 0)[0]
    if have.size:
        bt = torch.from_numpy(np.ascontiguousarray(batch.block_tables[have])).to(device)
        ctx = torch.from_numpy(cached[have].astype(np.int32)).to(device)
        qsl_np = np.zeros(have.size + 1, dtype=np.int32)
        np.cumsum(cached[have], out=qsl_np[1:])
        total = int(qsl_np[-1])
        slots = torch.empty(total, dtype=torch.int64, device=device)
        pkv.pkv_slot_mapping(pool.handle, bt, bt.shape[1], ctx, torch.from_numpy(qsl_np).to(device), int(have.size),
                             total, slots)
        for layer in layers:
            rows = rows_by_layer[layer]
            k = torch.from_numpy(np.concatenate([rows[b][1][:cached[b]] for b in have])).to(device)
            v = torch.from_numpy(np.concatenate([rows[b][2][:cached[b]] for b in have])).to(device)
            pkv.pkv_append(pool.handle, layer, k, v, slots, total)
    ds = workload.upload(batch, pool)
    qs, ks, vs = [], [], []
    for layer in layers:
        rows = rows_by_layer[layer]
        qs.append(torch.from_numpy(np.concatenate([r[0] for r in rows])).to(device))
        ks.append(torch.from_numpy(np.concatenate([r[1][cached[b]:] for b, r in enumerate(rows)])).to(device))
        vs.append(torch.from_numpy(np.concatenate([r[2][cached[b]:] for b, r in enumerate(rows)])).to(device))
    outs = [torch.full_like(q, float("nan")) for q in qs]
    workload.run_pass(pool, ds, layers, qs, ks, vs, outs, fused=fused)
    torch.cuda.synchronize()
    bits = pool.check()
    assert bits == 0, f"device error word set: {bits:#x}"
    return pool, ds, outs


def score_span_log2(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Per (query, head): the spread (max - min) of the scaled scores over the visible keys, in log2 units."""
    ql, hq, d = q.shape
    g = hq // k.shape[1]
    ctx = k.shape[0]
    span = np.zeros((ql, hq))
    for i in range(ql):
        last = ctx - ql + i
        for h in range(hq):
            s = k[:last + 1, h // g, :].astype(np.float64) @ q[i, h].astype(np.float64) / math.sqrt(d)
            span[i, h] = (s.max() - s.min()) / math.log(2.0)
    return span
