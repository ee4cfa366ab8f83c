"""Pins for the paging oracle: the sizing figures the pages print, and brute force on the append scatter."""
import json
import os

import numpy as np
import pytest

import oracle
from continuous_batching_paged_ragged_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kv_sizing.json")))
GIB = 1 << 30


def test_qwen3_8b_bytes_per_token():
    g = GOLDEN["qwen3_8b_bytes_per_token"]
    b = oracle.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["bytes"])
    assert b == g["expected_bytes"]
    assert b / 1024 == g["expected_kib"]


def test_qwen3_8b_pool_blocks():
    g = GOLDEN["qwen3_8b_16gib_pool"]
    blocks = oracle.pool_blocks_for_bytes(g["pool_bytes"], g["bytes_per_token"], g["block_size"])
    assert blocks == g["expected_blocks"]
    assert blocks * g["block_size"] == g["expected_tokens"]


def test_request_block_count_and_concurrency():
    g = GOLDEN["request_blocks"]
    nb = oracle.blocks_for_tokens(g["prompt"] + g["generated"], g["block_size"])
    assert nb == g["expected_blocks"]
    assert oracle.max_resident_sequences(g["pool_blocks"], nb) == g["expected_sequences"]


def test_qwen25_bytes_per_token_and_positions():
    g = GOLDEN["qwen25_1p5b_bytes_per_token"]
    b = oracle.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["bytes"])
    assert b == g["expected_kib"] * 1024
    positions = g["cache_gb"] * 1e9 / b
    assert positions == pytest.approx(g["expected_positions_approx"], rel=0.005)
    assert g["expected_positions_approx"] / g["seq_len"] == pytest.approx(g["expected_batch_approx"], rel=0.005)


def test_long_context_window_bytes():
    g = GOLDEN["long_context_window"]
    for bits, gib in g["expected_gib"].items():
        b = oracle.kv_bytes_for_window(g["window"], g["layers"], g["kv_heads"], g["head_dim"], int(bits) / 8)
        assert b == gib * GIB
    four = 4 * oracle.kv_bytes_for_window(g["window"], g["layers"], g["kv_heads"], g["head_dim"], 0.5)
    assert four == g["four_windows_4bit_gib"] * GIB


def test_max_concurrency_line():
    g = GOLDEN["vllm_max_concurrency"]
    assert round(g["pool_tokens"] / g["max_model_len"], 2) == g["expected"]


def test_cache_bytes_matches_per_token_cost():
    """Pool bytes for L layers = blocks x bs tokens x the per-token cost of the pages' formula."""
    for L, hkv, d, nb in [(28, 2, 128, 1000), (16, 4, 256, 7), (1, 2, 64, 64)]:
        assert oracle.cache_bytes(L, nb, hkv, 16, d) == nb * 16 * oracle.kv_bytes_per_token(L, hkv, d, 2)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 31, 32, 33, 1624])
def test_last_block_waste_below_block_size(n):
    nb = oracle.blocks_for_tokens(n, 16)
    assert 0 <= nb * 16 - n < 16 and nb >= 1


def test_slot_mapping_bruteforce():
    """Every (row, position) lands in a distinct slot of the row's own blocks at offset p % bs."""
    batch = synth.qwen_decode(seed=3, num_seqs=12)
    bt = batch.block_tables
    slots = oracle.slot_mapping_for_batch(bt, batch.context_lens, batch.q_lens, 16)
    assert slots.shape == (batch.num_tokens,)
    assert len(set(slots.tolist())) == len(slots)
    # brute force: enumerate every slot of the row's blocks and find the position that owns it
    t = 0
    for b in range(batch.num_seqs):
        owned = {}
        for i, blk in enumerate(bt[b]):
            if blk < 0:
                break
            for off in range(16):
                owned[int(blk) * 16 + off] = i * 16 + off
        for p in range(int(batch.cached_lens[b]), int(batch.context_lens[b])):
            assert owned[int(slots[t])] == p
            t += 1


def test_append_reference_scatter_and_skip():
    rng = np.random.default_rng(0)
    nb, hkv, bs, d = 6, 2, 4, 8
    pk = np.zeros((nb, hkv, bs, d), np.float16)
    pv = np.zeros((nb, hkv, bs, d), np.float16)
    k = rng.standard_normal((3, hkv, d)).astype(np.float16)
    v = rng.standard_normal((3, hkv, d)).astype(np.float16)
    oracle.append_reference(pk, pv, k, v, [13, -1, 2])
    assert np.array_equal(pk[3, :, 1], k[0]) and np.array_equal(pv[3, :, 1], v[0])
    assert np.array_equal(pk[0, :, 2], k[2]) and np.array_equal(pv[0, :, 2], v[2])
    # exactly 2 tokens' worth of bytes changed (slot -1 skipped)
    assert np.count_nonzero(np.any(pk != 0, axis=-1)) == 2 * hkv


def test_bench_byte_counts_match_the_sizing_formula():
    """The benchmark's algorithmic bytes: K and V once per row and layer at the pages' per-token cost
    (2 x Hkv x d x bytes, per layer), and on the 8-bit cache d code bytes plus one scale byte per row."""
    import bench
    batch = synth.custom_batch(synth.Shape(1, 12, 2, 128), [300, 17], [1, 1], seed=0)
    ctx = int(batch.context_lens.sum())
    a16, _ = bench.algorithmic_bytes(batch)
    a8, _ = bench.algorithmic_bytes(batch, kv8=True)
    other = 2 * 12 * 128 * 2 * 2 + 4 * int(((batch.context_lens + 15) // 16).sum())   # q in, out, tables
    assert a16 - other == ctx * oracle.kv_bytes_per_token(1, 2, 128, 2)
    assert a8 - other == ctx * 2 * 2 * (128 + 1)
