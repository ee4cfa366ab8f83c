"""Paged-cache arithmetic oracle: KV sizing, block counts, slot mapping and the append scatter.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """Cache bytes one token of context costs: 2 (K and V) x layers x kv_heads x head_dim x bytes.

    "Continuous Batching Is Not a Bigger Batch", section "Where the batch size actually comes from".
    """
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


def kv_bytes_for_window(window_tokens: int, num_layers: int, num_kv_heads: int, head_dim: int,
                        bytes_per_elem: float) -> float:
    """Raw KV bytes of one window ("An advertised batch limit proves nothing until sampled",
    section "Context math sets the ceiling the fields ignore")."""
    return window_tokens * kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_elem)


def pool_blocks_for_bytes(pool_bytes: int, bytes_per_token: int, block_size: int = 16) -> int:
    """Whole blocks of block_size tokens that fit in a pool ("Continuous Batching Is Not a Bigger Batch",
    section "Where the batch size actually comes from": a pool is counted in 16-token blocks)."""
    return pool_bytes // (bytes_per_token * block_size)


def blocks_for_tokens(num_tokens: int, block_size: int = 16) -> int:
    """Blocks a sequence of num_tokens holds under on-demand allocation: the last block may be partial
    ("Continuous Batching Is Not a Bigger Batch", section "The allocator is the other half")."""
    return -(-num_tokens // block_size)


def max_resident_sequences(pool_blocks: int, blocks_per_sequence: int) -> int:
    """floor(pool / per-sequence footprint) (same page, "Where the batch size actually comes from")."""
    return pool_blocks // blocks_per_sequence


def cache_bytes(num_layers: int, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
                bytes_per_elem: int = 2) -> int:
    """Bytes of a pool holding K and V for every layer: 2 x L x blocks x Hkv x bs x d x bytes."""
    return 2 * num_layers * num_blocks * num_kv_heads * block_size * head_dim * bytes_per_elem


def slot_of(block_table_row: Sequence[int], position: int, block_size: int) -> int:
    """Physical slot of a token at absolute position p: the row's block p // bs, offset p % bs.

    The pages never print this formula; it is the plain reading of "blocks allocated as tokens are
    computed" with a per-sequence block table (reading recorded in the design notes).
    """
    return int(block_table_row[position // block_size]) * block_size + position % block_size


def slot_mapping_for_batch(block_tables: np.ndarray, context_lens: Sequence[int], q_lens: Sequence[int],
                           block_size: int) -> np.ndarray:
    """int64 [T]: slot of every new token, rows in batch order, tokens in position order."""
    out = []
    for b in range(len(q_lens)):
        start = int(context_lens[b]) - int(q_lens[b])
        for p in range(start, start + int(q_lens[b])):
            out.append(slot_of(block_tables[b], p, block_size))
    return np.asarray(out, dtype=np.int64)


def append_reference(pool_k: np.ndarray, pool_v: np.ndarray, k: np.ndarray, v: np.ndarray,
                     slot_mapping: Sequence[int]) -> None:
    """In place: pool[slot // bs, :, slot % bs, :] = new token's [Hkv, d] for K and V; slot -1 is skipped.

    pool_k, pool_v: fp16 [num_blocks, Hkv, bs, d] (one layer); k, v: fp16 [T, Hkv, d].
    A pure copy of fp16 bits: no arithmetic touches the values.
    """
    block_size = pool_k.shape[2]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        pool_k[slot // block_size, :, slot % block_size, :] = k[t]
        pool_v[slot // block_size, :, slot % block_size, :] = v[t]
