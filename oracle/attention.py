"""Attention oracle: the plain definition, float64, from contiguous per-sequence K/V.

Test infrastructure only (see the package docstring).

The pages never print an attention formula; they name the pieces.  A forward pass reads every cached
key/value pair of a sequence instead of recomputing them ("Continuous Batching Is Not a Bigger Batch",
opening section: one K/V pair per token per layer); several query heads share one KV head under
grouped-query attention (same page, "Where the batch size actually comes from"); a prompt may be
consumed in chunks inside one pass with no separate prefill phase (same page, "What the scheduler does
on one step"); the paged layout stores only real tokens ("Static batching", "Ragged batches").

Readings taken where the pages are silent (each listed in the design notes):
  * softmax scale 1/sqrt(head_dim);
  * contiguous GQA groups: query head h reads KV head h // (Hq / Hkv);
  * a chunk of q_len new tokens sits at the END of the row's context (ctx includes this pass's tokens),
    so query i (0-based) is at absolute position ctx - q_len + i and sees keys 0 .. ctx - q_len + i.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np


def round_fp16(x: np.ndarray) -> np.ndarray:
    """float64 -> fp16, IEEE round-to-nearest-even (numpy's conversion), one rounding."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def attention_row(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Causal GQA attention of one row's new queries over its whole context.

    q: fp16 [q_len, Hq, d] -- this pass's query tokens of the row, in position order.
    k, v: [ctx, Hkv, d] -- the row's keys/values in logical (position) order, this pass's included: fp16, or
    the float64 values an 8-bit cache dequantizes to (oracle.fp8).
    Returns float64 [q_len, Hq, d].
    """
    q_len, num_q_heads, d = q.shape
    ctx, num_kv_heads, d2 = k.shape
    assert d == d2 and v.shape == k.shape
    assert num_q_heads % num_kv_heads == 0
    assert 1 <= q_len <= ctx
    group = num_q_heads // num_kv_heads
    scale = 1.0 / math.sqrt(d)
    qf = q.astype(np.float64)
    kf = k.astype(np.float64)
    vf = v.astype(np.float64)
    out = np.zeros((q_len, num_q_heads, d), dtype=np.float64)
    for i in range(q_len):
        last = ctx - q_len + i          # absolute position of query i; keys 0..last are visible
        for h in range(num_q_heads):
            g = h // group
            scores = (kf[: last + 1, g, :] @ qf[i, h, :]) * scale
            weights = np.exp(scores - scores.max())
            weights /= weights.sum()
            out[i, h, :] = weights @ vf[: last + 1, g, :]
    return out


def attention_batch(q: np.ndarray, ks: Sequence[np.ndarray], vs: Sequence[np.ndarray],
                    query_start_loc: Sequence[int]) -> np.ndarray:
    """Ragged batch: row b owns packed query tokens query_start_loc[b] .. query_start_loc[b+1]-1.

    q: fp16 [T, Hq, d]; ks[b], vs[b]: fp16 [ctx_b, Hkv, d] in logical order.  Returns float64 [T, Hq, d].
    Rows are independent: each is attention_row on its own slice.
    """
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(len(ks)):
        lo, hi = int(query_start_loc[b]), int(query_start_loc[b + 1])
        out[lo:hi] = attention_row(q[lo:hi], ks[b], vs[b])
    return out
