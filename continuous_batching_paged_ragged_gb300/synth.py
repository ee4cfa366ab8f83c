"""Seeded synthetic inputs: the one module that both the CUDA path's callers and the oracle's callers use.

It holds random numbers and workload recipes only -- none of the attention, append, slot-mapping or
scheduling arithmetic.  Everything the pages' workloads need is produced here from a seed:

* Tensor values (q, k, v) come from a counter-based generator, Philox4x32-10 as published by Salmon,
  Moraes, Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC 2011).  A value is a pure
  function of (seed, kind, layer, request, position, head, dim), so a re-prefilled token after
  preemption rewrites identical bits, and the oracle can regenerate any sequence's keys and values in
  logical order without reading the device's paged pool.  The device-side twin of this generator
  (``csrc/synth.cu``, loaded through :func:`device_fill`) implements the same published definition
  independently; a GPU test checks the two agree bit for bit.
* Each value approximates N(0, 1) by an Irwin-Hall sum of four 16-bit uniforms, centred and scaled by
  sqrt(3)/65536 in one float32 multiply, then rounded to fp16 (round-to-nearest-even).  All steps are
  exact integer work plus two IEEE roundings, so host and device agree exactly.
* Workload recipes (context lengths, scattered block tables, request traces) use numpy's PCG64.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import List, Optional, Sequence

import numpy as np

# --- Philox4x32-10 (Salmon et al. 2011, section 3, the Philox round and key schedule) -----------------
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

KIND_Q = 1
KIND_K = 2
KIND_V = 3

# float32(sqrt(3) / 65536): the Irwin-Hall(4) sum of 16-bit uniforms has standard deviation 65536/sqrt(3).
NORMAL_SCALE = np.float32(math.sqrt(3.0) / 65536.0)
IRWIN_HALL_CENTER = 131070  # 4 * 32767.5


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox4x32 rounds over arrays of 32-bit counters (broadcast together), key (k0, k1)."""
    c0 = np.asarray(c0, dtype=np.uint64)
    c1 = np.asarray(c1, dtype=np.uint64)
    c2 = np.asarray(c2, dtype=np.uint64)
    c3 = np.asarray(c3, dtype=np.uint64)
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    ka = np.uint64(k0 & 0xFFFFFFFF)
    kb = np.uint64(k1 & 0xFFFFFFFF)
    for _ in range(10):
        p0 = m0 * c0
        p1 = m1 * c2
        n0 = (p1 >> np.uint64(32)) ^ c1 ^ ka
        n1 = p1 & _MASK32
        n2 = (p0 >> np.uint64(32)) ^ c3 ^ kb
        n3 = p0 & _MASK32
        c0, c1, c2, c3 = n0, n1, n2, n3
        ka = (ka + np.uint64(PHILOX_W0)) & _MASK32
        kb = (kb + np.uint64(PHILOX_W1)) & _MASK32
    return (c0.astype(np.uint32), c1.astype(np.uint32), c2.astype(np.uint32), c3.astype(np.uint32))


def _irwin_hall_fp16(wa, wb):
    wa = wa.astype(np.int64)
    wb = wb.astype(np.int64)
    s = (wa & 0xFFFF) + (wa >> 16) + (wb & 0xFFFF) + (wb >> 16) - IRWIN_HALL_CENTER
    x = s.astype(np.float32) * NORMAL_SCALE  # exact int -> f32, one IEEE f32 multiply
    return x.astype(np.float16)              # IEEE round-to-nearest-even


def token_values(kind: int, seed: int, layer: int, req_ids, positions, heads: int, head_dim: int,
                 head_range: Optional[tuple] = None) -> np.ndarray:
    """fp16 [T, heads, head_dim] values of one tensor kind for tokens (req_ids[t], positions[t]).

    Counter layout: key = (seed low word, kind << 24 | layer); counter = (pair index of the flattened
    (head, dim) element, position, request id, seed high word).  An even element takes output words
    0-1 of its pair's Philox call, an odd element words 2-3.  ``head_range=(lo, hi)`` returns only heads
    lo .. hi-1 (same values as the full tensor's slice).
    """
    req = np.asarray(req_ids, dtype=np.int64).reshape(-1)
    pos = np.asarray(positions, dtype=np.int64).reshape(-1)
    assert req.shape == pos.shape
    lo_h, hi_h = head_range if head_range is not None else (0, heads)
    assert 0 <= lo_h < hi_h <= heads and head_dim % 2 == 0
    n_el = (hi_h - lo_h) * head_dim
    pairs = np.arange(lo_h * head_dim // 2, hi_h * head_dim // 2, dtype=np.uint64)
    k0 = seed & 0xFFFFFFFF
    k1 = ((kind & 0xFF) << 24) | (layer & 0xFFFFFF)
    c3 = (seed >> 32) & 0xFFFFFFFF
    out = np.empty((req.shape[0], n_el), dtype=np.float16)
    step = max(1, (1 << 17) // pairs.shape[0])   # bounded temporaries keep numpy in cache
    for lo in range(0, req.shape[0], step):
        hi = min(lo + step, req.shape[0])
        w0, w1, w2, w3 = philox4x32_10(pairs[None, :], pos[lo:hi, None].astype(np.uint64) & _MASK32,
                                       req[lo:hi, None].astype(np.uint64) & _MASK32, np.uint64(c3), k0, k1)
        out[lo:hi, 0::2] = _irwin_hall_fp16(w0, w1)
        out[lo:hi, 1::2] = _irwin_hall_fp16(w2, w3)
    return out.reshape(req.shape[0], hi_h - lo_h, head_dim)


def sequence_kv(seed: int, layer: int, req_id: int, ctx: int, num_kv_heads: int, head_dim: int,
                head_range: Optional[tuple] = None):
    """Contiguous logical-order K and V ([ctx, Hkv, d] fp16) of one sequence at one layer."""
    pos = np.arange(ctx, dtype=np.int64)
    req = np.full(ctx, req_id, dtype=np.int64)
    k = token_values(KIND_K, seed, layer, req, pos, num_kv_heads, head_dim, head_range)
    v = token_values(KIND_V, seed, layer, req, pos, num_kv_heads, head_dim, head_range)
    return k, v


# --- workload recipes --------------------------------------------------------------------------------

@dataclasses.dataclass
class Shape:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int = 16


@dataclasses.dataclass
class StepBatch:
    """One forward pass's ragged batch: rows in batch order, new tokens packed row by row."""
    shape: Shape
    num_blocks: int
    req_ids: np.ndarray          # int64 [B]
    q_lens: np.ndarray           # int32 [B]  new tokens this pass
    context_lens: np.ndarray     # int32 [B]  cached + new tokens (keys each row's last query sees)
    block_tables: np.ndarray     # int32 [B, max_blocks], -1 past each row's used blocks
    block_perm: np.ndarray       # int32 [num_blocks]: the random physical order blocks were handed out in
    seed: int
    name: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def query_start_loc(self) -> np.ndarray:
        qsl = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.q_lens, out=qsl[1:])
        return qsl

    @property
    def cached_lens(self) -> np.ndarray:
        return (self.context_lens - self.q_lens).astype(np.int32)

    def token_req_pos(self):
        """Per new token: (request id, absolute position)."""
        reqs, poss = [], []
        for b in range(self.num_seqs):
            c0 = int(self.cached_lens[b])
            n = int(self.q_lens[b])
            reqs.append(np.full(n, self.req_ids[b], dtype=np.int64))
            poss.append(np.arange(c0, c0 + n, dtype=np.int64))
        return np.concatenate(reqs), np.concatenate(poss)

    def cached_req_pos(self):
        """Per already-cached token (the pool's prior content): (row, request id, absolute position)."""
        rows, reqs, poss = [], [], []
        for b in range(self.num_seqs):
            c0 = int(self.cached_lens[b])
            rows.append(np.full(c0, b, dtype=np.int64))
            reqs.append(np.full(c0, self.req_ids[b], dtype=np.int64))
            poss.append(np.arange(c0, dtype=np.int64))
        return np.concatenate(rows), np.concatenate(reqs), np.concatenate(poss)


def block_permutation(num_blocks: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED_B10C))
    return rng.permutation(num_blocks).astype(np.int32)


def scatter_block_tables(context_lens: Sequence[int], block_size: int, num_blocks: int, seed: int):
    """Hand each row ceil(ctx/bs) physical blocks taken in order from a seeded random permutation."""
    perm = block_permutation(num_blocks, seed)
    need = [(int(c) + block_size - 1) // block_size for c in context_lens]
    assert sum(need) <= num_blocks, "pool too small for the batch"
    max_blocks = max(1, max(need) if need else 1)
    bt = np.full((len(need), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, perm


def _make_batch(name, shape, cached, q_lens, seed, pool_factor=1.25, num_blocks=None, req_base=1000,
                block_seed=None, req_ids=None):
    cached = np.asarray(cached, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx = (cached + q_lens).astype(np.int32)
    need = int(sum((int(c) + shape.block_size - 1) // shape.block_size for c in ctx))
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * need))
    bt, perm = scatter_block_tables(ctx, shape.block_size, num_blocks, seed if block_seed is None else block_seed)
    if req_ids is None:
        req_ids = np.arange(req_base, req_base + len(ctx), dtype=np.int64)
    return StepBatch(shape, num_blocks, np.asarray(req_ids, dtype=np.int64), q_lens, ctx, bt, perm, seed, name)


def custom_batch(shape: Shape, cached, q_lens, seed: int = 0, num_blocks: Optional[int] = None,
                 block_seed: Optional[int] = None, req_ids=None, pool_factor: float = 1.25) -> StepBatch:
    """A pass with the given per-row cached lengths and new-token counts; blocks scattered by block_seed.

    Values depend on (seed, request id, position) only, so two batches that place the same rows in
    different physical blocks (block_seed) or in a different order hold identical logical K/V/Q."""
    return _make_batch("custom", shape, cached, q_lens, seed, pool_factor, num_blocks, block_seed=block_seed,
                       req_ids=req_ids)


def tiny_decode(seed: int = 0) -> StepBatch:
    """1 layer, 4 q / 2 KV heads, d=64, 64-block pool; cached {7,16,33,50}, one new token each."""
    return _make_batch("tiny_decode", Shape(1, 4, 2, 64), [7, 16, 33, 50], [1, 1, 1, 1], seed, num_blocks=64)


def qwen_decode(seed: int = 0, num_seqs: int = 256) -> StepBatch:
    """Qwen2.5-1.5B shape (28 layers, 12/2 heads, d=128); cached ~ U[256, 768]; pool 1.25x the need."""
    rng = np.random.Generator(np.random.PCG64(seed + 2))
    cached = rng.integers(256, 768, size=num_seqs, endpoint=True)
    return _make_batch("qwen_decode", Shape(28, 12, 2, 128), cached, np.ones(num_seqs), seed)


def mixed_step(seed: int = 0) -> StepBatch:
    """83 decode rows (cached ~ U[64, 1100]) then chunked-prefill rows 2048-on-0 and 1024-on-3072."""
    rng = np.random.Generator(np.random.PCG64(seed + 3))
    cached = list(rng.integers(64, 1100, size=83, endpoint=True)) + [0, 3072]
    q_lens = [1] * 83 + [2048, 1024]
    return _make_batch("mixed_step", Shape(28, 12, 2, 128), cached, q_lens, seed)


def prefill_chunk(seed: int = 0, q_len: int = 8192, cached: int = 0) -> StepBatch:
    """Qwen2.5-1.5B shape, one row whose pass is a single chunk of q_len new tokens (the whole per-pass token
    budget of 8,192 by default) on top of `cached` tokens."""
    return _make_batch("prefill_8k" if (q_len, cached) == (8192, 0) else "prefill_chunk", Shape(28, 12, 2, 128),
                       [cached], [q_len], seed)


def long_gqa(seed: int = 0, cached_len: int = 262144, num_seqs: int = 4, num_layers: int = 16) -> StepBatch:
    """16 KV layers, 16 q / 4 KV heads, d=256; 4 rows of 262,144 cached tokens, one query each."""
    return _make_batch("long_gqa", Shape(num_layers, 16, 4, 256), [cached_len] * num_seqs,
                       [1] * num_seqs, seed, pool_factor=1.0)


@dataclasses.dataclass
class TraceRequest:
    req_id: int
    prompt_len: int
    max_output: int


def trace_requests(seed: int = 0, n: int = 256, median: float = 300.0, sigma: float = 1.0,
                   lo: int = 16, hi: int = 4096, out_lo: int = 50, out_hi: int = 781) -> List[TraceRequest]:
    """Prompt = clip(round(median * exp(N(0, sigma))), lo, hi); output budget ~ U[out_lo, out_hi]."""
    rng = np.random.Generator(np.random.PCG64(seed + 5))
    z = rng.standard_normal(n)
    prompts = np.clip(np.rint(median * np.exp(sigma * z)), lo, hi).astype(np.int64)
    outs = rng.integers(out_lo, out_hi, size=n, endpoint=True)
    return [TraceRequest(i, int(p), int(o)) for i, (p, o) in enumerate(zip(prompts, outs))]


# --- device twin of the value generator ---------------------------------------------------------------

_synth_lib = None


def _load_synth():
    global _synth_lib
    if _synth_lib is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.pkv_synth_fill.restype = ctypes.c_int
        lib.pkv_synth_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p]
        _synth_lib = lib
    return _synth_lib


def device_fill(kind: int, seed: int, layer: int, req_ids_dev, positions_dev, heads: int, head_dim: int, out,
                stream: Optional[int] = None) -> None:
    """Fill ``out`` (device fp16 [T, heads, d]) with :func:`token_values` computed on the GPU.

    ``req_ids_dev`` / ``positions_dev`` are int64 device tensors of length T.
    """
    import torch
    lib = _load_synth()
    T = int(req_ids_dev.numel())
    assert positions_dev.numel() == T and out.numel() == T * heads * head_dim
    assert req_ids_dev.dtype == torch.int64 and positions_dev.dtype == torch.int64
    assert out.dtype == torch.float16 and out.is_contiguous()
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    rc = lib.pkv_synth_fill(kind, seed, layer, req_ids_dev.data_ptr(), positions_dev.data_ptr(), T, heads,
                            head_dim, out.data_ptr(), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"pkv_synth_fill failed with CUDA error {rc}")
