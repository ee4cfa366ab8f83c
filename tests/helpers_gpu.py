"""Shared pieces of the GPU parity tests: run a pass through libpkv and compare rows with the oracle."""
from __future__ import annotations

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
