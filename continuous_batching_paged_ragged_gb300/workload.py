"""Device-side set-up of a synthetic pass: metadata upload, cache pre-fill and per-layer q/k/v.

Used by the GPU tests and the benchmark.  Everything on the device runs through libpkv's own calls
(pkv_slot_mapping, pkv_append) and the device input generator; nothing here computes attention.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from . import pkv, synth


@dataclasses.dataclass
class DeviceStep:
    batch: synth.StepBatch
    block_tables: torch.Tensor     # int32 [B, max_blocks]
    context_lens: torch.Tensor     # int32 [B]
    query_start_loc: torch.Tensor  # int32 [B + 1]
    slot_mapping: torch.Tensor     # int64 [T]
    tok_req: torch.Tensor          # int64 [T]
    tok_pos: torch.Tensor          # int64 [T]

    @property
    def num_seqs(self) -> int:
        return self.batch.num_seqs

    @property
    def num_tokens(self) -> int:
        return self.batch.num_tokens

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def make_pool(batch: synth.StepBatch, num_layers: Optional[int] = None, split_blocks: int = 0,
              kv_dtype: int = pkv.PKV_KV_F16) -> pkv.Pool:
    s = batch.shape
    return pkv.Pool(num_layers or s.num_layers, s.num_q_heads, s.num_kv_heads, s.head_dim, batch.num_blocks,
                    s.block_size, split_blocks, kv_dtype=kv_dtype)


def upload(batch: synth.StepBatch, pool: pkv.Pool, device="cuda") -> DeviceStep:
    """Metadata to the device; the slot mapping of this pass's tokens is computed by pkv_slot_mapping."""
    bt = torch.from_numpy(np.ascontiguousarray(batch.block_tables)).to(device)
    ctx = torch.from_numpy(batch.context_lens.astype(np.int32)).to(device)
    qsl = torch.from_numpy(batch.query_start_loc).to(device)
    req, pos = batch.token_req_pos()
    slots = torch.empty(batch.num_tokens, dtype=torch.int64, device=device)
    pkv.pkv_slot_mapping(pool.handle, bt, bt.shape[1], ctx, qsl, batch.num_seqs, batch.num_tokens, slots)
    return DeviceStep(batch, bt, ctx, qsl, slots, torch.from_numpy(req).to(device), torch.from_numpy(pos).to(device))


def prefill_cache(pool: pkv.Pool, batch: synth.StepBatch, layers: List[int], chunk_tokens: int = 1 << 17,
                  device="cuda") -> None:
    """Write every row's already-cached tokens (positions 0 .. cached-1) into the pool, layer by layer,
    through pkv_slot_mapping + pkv_append on device-generated K/V."""
    cached = batch.cached_lens
    rows = np.nonzero(cached > 0)[0]
    if rows.size == 0:
        return
    s = batch.shape
    bt = torch.from_numpy(np.ascontiguousarray(batch.block_tables[rows])).to(device)
    ctx = torch.from_numpy(cached[rows].astype(np.int32)).to(device)
    qsl_np = np.zeros(rows.size + 1, dtype=np.int32)
    np.cumsum(cached[rows], out=qsl_np[1:])
    qsl = torch.from_numpy(qsl_np).to(device)
    total = int(qsl_np[-1])
    slots = torch.empty(total, dtype=torch.int64, device=device)
    pkv.pkv_slot_mapping(pool.handle, bt, bt.shape[1], ctx, qsl, int(rows.size), total, slots)
    req = torch.from_numpy(np.repeat(batch.req_ids[rows], cached[rows])).to(device)
    pos = torch.from_numpy(np.concatenate([np.arange(int(c), dtype=np.int64) for c in cached[rows]])).to(device)
    n = min(chunk_tokens, total)
    kbuf = torch.empty(n, s.num_kv_heads, s.head_dim, dtype=torch.float16, device=device)
    vbuf = torch.empty_like(kbuf)
    for layer in layers:
        for lo in range(0, total, chunk_tokens):
            hi = min(lo + chunk_tokens, total)
            m = hi - lo
            synth.device_fill(synth.KIND_K, batch.seed, layer, req[lo:hi], pos[lo:hi], s.num_kv_heads, s.head_dim,
                              kbuf[:m])
            synth.device_fill(synth.KIND_V, batch.seed, layer, req[lo:hi], pos[lo:hi], s.num_kv_heads, s.head_dim,
                              vbuf[:m])
            pkv.pkv_append(pool.handle, layer, kbuf, vbuf, slots[lo:hi], m)


def step_inputs(ds: DeviceStep, layers: List[int], device="cuda"):
    """Per layer: q [T, Hq, d], k and v [T, Hkv, d] of this pass's tokens, generated on the device."""
    b = ds.batch
    s = b.shape
    T = b.num_tokens
    qs, ks, vs = [], [], []
    for layer in layers:
        q = torch.empty(T, s.num_q_heads, s.head_dim, dtype=torch.float16, device=device)
        k = torch.empty(T, s.num_kv_heads, s.head_dim, dtype=torch.float16, device=device)
        v = torch.empty_like(k)
        synth.device_fill(synth.KIND_Q, b.seed, layer, ds.tok_req, ds.tok_pos, s.num_q_heads, s.head_dim, q)
        synth.device_fill(synth.KIND_K, b.seed, layer, ds.tok_req, ds.tok_pos, s.num_kv_heads, s.head_dim, k)
        synth.device_fill(synth.KIND_V, b.seed, layer, ds.tok_req, ds.tok_pos, s.num_kv_heads, s.head_dim, v)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return qs, ks, vs


class Attention:
    """Workspace + plan for one pass's metadata; run(layer, q, out) = pkv_attention."""

    def __init__(self, pool: pkv.Pool, ds: DeviceStep, device="cuda"):
        self.pool = pool
        self.ds = ds
        self.ws_bytes = pkv.pkv_attention_workspace_bytes(pool.handle, ds.num_seqs, ds.num_tokens, ds.max_blocks)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)

    def plan(self, stream=None):
        d = self.ds
        pkv.pkv_attention_plan(self.pool.handle, d.context_lens, d.query_start_loc, d.num_seqs, d.num_tokens,
                               d.max_blocks, self.workspace, self.ws_bytes, stream)

    def run(self, layer: int, q: torch.Tensor, out: torch.Tensor, stream=None):
        d = self.ds
        pkv.pkv_attention(self.pool.handle, layer, q, d.block_tables, d.max_blocks, d.context_lens,
                          d.query_start_loc, d.num_seqs, d.num_tokens, out, self.workspace, self.ws_bytes, stream)

    def run_append(self, layer: int, q, k, v, out, stream=None):
        d = self.ds
        pkv.pkv_attention_append(self.pool.handle, layer, q, k, v, d.slot_mapping, d.block_tables, d.max_blocks,
                                 d.context_lens, d.query_start_loc, d.num_seqs, d.num_tokens, out, self.workspace,
                                 self.ws_bytes, stream)


def run_pass(pool: pkv.Pool, ds: DeviceStep, layers: List[int], qs, ks, vs, outs, attn: Optional[Attention] = None,
             fused: bool = False):
    """One forward pass's hot path: per layer, append this pass's K/V, then attention (fused: one
    pkv_attention_append call per layer)."""
    if attn is None:
        attn = Attention(pool, ds)
    attn.plan()
    for i, layer in enumerate(layers):
        if fused:
            attn.run_append(layer, qs[i], ks[i], vs[i], outs[i])
        else:
            pkv.pkv_append(pool.handle, layer, ks[i], vs[i], ds.slot_mapping, ds.num_tokens)
            attn.run(layer, qs[i], outs[i])
    return attn


class RawStep:
    """One forward pass's hot path with every pointer resolved up front (as a benchmark or a CUDA-graph
    capture wants it): plan + per layer append and attention, as one pkv_attention_append call (fused=True)
    or pkv_append then pkv_attention.  `launches` counts the kernels the calls enqueued."""

    def __init__(self, pool, ds, attn, qs, ks, vs, outs, stream, fused=True):
        self.fused = fused
        self.lib = pkv.load()
        self.pool = pool.handle
        self.ds = ds
        self.ws = attn.workspace.data_ptr()
        self.ws_bytes = attn.ws_bytes
        self.q = [x.data_ptr() for x in qs]
        self.k = [x.data_ptr() for x in ks]
        self.v = [x.data_ptr() for x in vs]
        self.o = [x.data_ptr() for x in outs]
        self.stream = stream
        self.bt = ds.block_tables.data_ptr()
        self.ctx = ds.context_lens.data_ptr()
        self.qsl = ds.query_start_loc.data_ptr()
        self.slots = ds.slot_mapping.data_ptr()
        self.launches = 0

    def plan(self):
        d = self.ds
        st = self.lib.pkv_attention_plan(self.pool, self.ctx, self.qsl, d.num_seqs, d.num_tokens, d.max_blocks,
                                         self.ws, self.ws_bytes, self.stream)
        if st:
            raise pkv.PkvError(st, "pkv_attention_plan", pkv.pkv_last_error())
        self.launches += self.lib.pkv_last_launch_count(self.pool)

    def append(self, i, layer):
        st = self.lib.pkv_append(self.pool, layer, self.k[i], self.v[i], self.slots, self.ds.num_tokens, self.stream)
        if st:
            raise pkv.PkvError(st, "pkv_append", pkv.pkv_last_error())
        self.launches += self.lib.pkv_last_launch_count(self.pool)

    def attention(self, i, layer):
        d = self.ds
        st = self.lib.pkv_attention(self.pool, layer, self.q[i], self.bt, d.max_blocks, self.ctx, self.qsl,
                                    d.num_seqs, d.num_tokens, self.o[i], self.ws, self.ws_bytes, self.stream)
        if st:
            raise pkv.PkvError(st, "pkv_attention", pkv.pkv_last_error())
        self.launches += self.lib.pkv_last_launch_count(self.pool)

    def attention_append(self, i, layer):
        d = self.ds
        st = self.lib.pkv_attention_append(self.pool, layer, self.q[i], self.k[i], self.v[i], self.slots, self.bt,
                                           d.max_blocks, self.ctx, self.qsl, d.num_seqs, d.num_tokens, self.o[i],
                                           self.ws, self.ws_bytes, self.stream)
        if st:
            raise pkv.PkvError(st, "pkv_attention_append", pkv.pkv_last_error())
        self.launches += self.lib.pkv_last_launch_count(self.pool)

    def __call__(self, layers):
        self.plan()
        for i, layer in enumerate(layers):
            if self.fused:
                self.attention_append(i, layer)
            else:
                self.append(i, layer)
                self.attention(i, layer)


def capture_step_graph(pool: pkv.Pool, ds: DeviceStep, attn: Attention, qs, ks, vs, outs, layers: List[int],
                       fused: bool = True, device="cuda", warm: int = 3):
    """The pass as one CUDA graph: the same library calls (RawStep), run `warm` times on a side stream, then
    captured there.  Returns (graph, kernel launches per replay).  Replaying it re-runs the plan, the
    append of this pass's tokens (the same bits to the same slots) and the attention of every layer."""
    stream = torch.cuda.current_stream(device)
    cap = torch.cuda.Stream(device)
    step = RawStep(pool, ds, attn, qs, ks, vs, outs, cap.cuda_stream, fused=fused)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for _ in range(warm):
            step(layers)
    torch.cuda.synchronize()
    step.launches = 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        step(layers)
    torch.cuda.synchronize()
    return graph, step.launches
