"""Oracle jobs for a process pool (started with the 'spawn' method): each regenerates one sequence's inputs
with the seeded generator and returns the fp64 oracle for it.  Imports nothing from the CUDA path."""
from __future__ import annotations

import numpy as np

import oracle
from continuous_batching_paged_ragged_gb300 import synth


def long_row_one_kv_head(args):
    """(seed, layer, req, ctx, kv head g, Hq, Hkv, d) -> fp64 [1, G, d]: the row's last query (position
    ctx - 1) for the G query heads of KV head g, over its whole context."""
    seed, layer, req, ctx, g, hq, hkv, d = args
    G = hq // hkv
    k, v = synth.sequence_kv(seed, layer, req, ctx, hkv, d, (g, g + 1))
    q = synth.token_values(synth.KIND_Q, seed, layer, np.array([req]), np.array([ctx - 1]), hq, d,
                           (g * G, g * G + G))
    return oracle.attention_row(q, k, v)
