"""GPU parity of the chunked-prefill tile path (rows with >= 16 new tokens, head_dim 64, 128 or 256) against the
fp64 oracle: chunks over zero, short and long cached prefixes, chunk lengths around the tile sizes
(positions per tile = 128 / G, 128 keys per K/V tile, 16-token blocks), every supported head grouping,
and the same rows mixed with decode rows in one pass."""
import numpy as np
import pytest
import torch

import oracle
from continuous_batching_paged_ragged_gb300 import synth
from helpers_gpu import assert_close, oracle_row, row_slice, run_batch

pytestmark = pytest.mark.gpu

# (cached, q_len): chunk boundaries against P = 128 / G positions per tile and 128-key K/V tiles
PREFILL_ROWS = [(0, 16), (0, 21), (0, 22), (0, 127), (0, 128), (0, 129), (0, 300), (5, 43), (127, 16),
                (128, 17), (1000, 64), (2047, 200), (16, 250)]
SHAPES = [(12, 2, 128), (8, 8, 64), (8, 1, 128), (16, 4, 128), (4, 2, 64), (8, 8, 128), (16, 16, 64),
          (16, 4, 256), (12, 2, 256), (8, 8, 256), (16, 2, 256)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
def test_prefill_rows_all_shapes(cuda, built, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached, qls = zip(*PREFILL_ROWS)
    batch = synth.custom_batch(shape, cached, qls, seed=21)
    pool, ds, outs = run_batch(batch, [0])
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row(batch, 0, b), f"{(hq, hkv, d)} row {b} {PREFILL_ROWS[b]}")


def test_prefill_mixed_with_decode_rows(cuda, built):
    """Decode rows, short chunks (decode path) and long chunks (tile path) in one pass, two layers."""
    shape = synth.Shape(2, 12, 2, 128)
    rows = [(300, 1), (0, 40), (17, 1), (700, 15), (64, 16), (3000, 1), (250, 333), (1, 1)]
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=8)
    pool, ds, outs = run_batch(batch, [0, 1])
    for layer in (0, 1):
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, outs[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")


def test_prefill_row_alone_equals_batched(cuda, built):
    """A prefill row's output is bit-identical alone and inside a batch."""
    shape = synth.Shape(1, 12, 2, 128)
    rows = [(100, 1), (0, 180), (900, 1), (40, 77)]
    cached, qls = zip(*rows)
    full = synth.custom_batch(shape, cached, qls, seed=12)
    _, _, of = run_batch(full, [0])
    for b in (1, 3):
        alone = synth.custom_batch(shape, [cached[b]], [qls[b]], seed=12, req_ids=[full.req_ids[b]])
        _, _, oa = run_batch(alone, [0])
        assert np.array_equal(oa[0].cpu().numpy().view(np.uint16), row_slice(full, of[0], b).view(np.uint16))


def test_prefill_output_rows_untouched_outside_the_pass(cuda, built):
    """The tile path writes exactly the pass's tokens: a sentinel past the last token survives."""
    shape = synth.Shape(1, 8, 2, 128)
    batch = synth.custom_batch(shape, [0, 33], [50, 20], seed=3)
    from continuous_batching_paged_ragged_gb300 import workload
    pool = workload.make_pool(batch)
    workload.prefill_cache(pool, batch, [0])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0])
    T = batch.num_tokens
    big = torch.full((T + 4, 8, 128), 7.0, dtype=torch.float16, device=cuda)
    out = big[:T]
    workload.run_pass(pool, ds, [0], qs, ks, vs, [out])
    torch.cuda.synchronize()
    assert pool.check() == 0
    assert torch.all(big[T:] == 7.0)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, out, b), oracle_row(batch, 0, b), f"row {b}")


def test_prefill_split_items_many_entries_per_cta(cuda, built):
    """Chunks on long cached prefixes (more than 24 K/V tiles: split in two key ranges and merged) with more
    work entries than SMs, so CTAs run several entries back to back; two layers reuse the merge slots."""
    shape = synth.Shape(2, 12, 2, 128)
    rows = [(3000, 512), (2500, 300), (4000, 256), (2200, 700), (17, 1), (5000, 40)]
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=31)
    pool, ds, outs = run_batch(batch, [0, 1])
    for layer in (0, 1):
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, outs[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")


def test_prefill_8k_chunk_sampled_positions(cuda, built):
    """One row whose pass is a whole 8,192-token chunk (the per-pass token budget) on an empty cache: 392 work
    entries, ~2.6 per CTA.  Every output row is written (a NaN sentinel everywhere before the pass), and the
    oracle runs query by query at sampled positions (tile and item boundaries, the last position), each over
    its own causal prefix."""
    from continuous_batching_paged_ragged_gb300 import workload
    batch = synth.prefill_chunk(0)
    batch.shape = synth.Shape(1, batch.shape.num_q_heads, batch.shape.num_kv_heads, batch.shape.head_dim)
    s = batch.shape
    pool = workload.make_pool(batch)
    workload.prefill_cache(pool, batch, [0])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0])
    outs = [torch.full_like(qs[0], float("nan"))]
    workload.run_pass(pool, ds, [0], qs, ks, vs, outs)
    torch.cuda.synchronize()
    assert pool.check() == 0
    assert bool(torch.isfinite(outs[0]).all()), "some output rows were never written"
    out = row_slice(batch, outs[0], 0)
    req, ctx = int(batch.req_ids[0]), int(batch.context_lens[0])
    k, v = synth.sequence_kv(batch.seed, 0, req, ctx, s.num_kv_heads, s.head_dim)
    rng = np.random.Generator(np.random.PCG64(88))
    picks = {0, 1, 20, 21, 41, 42, 127, 128, 129, 1023, 1024, 4095, 4096, 6000, 8150, 8190, 8191}
    picks |= set(int(x) for x in rng.integers(0, ctx, size=12))
    for i in sorted(picks):
        q = synth.token_values(synth.KIND_Q, batch.seed, 0, np.array([req]), np.array([i]), s.num_q_heads,
                               s.head_dim)
        ref = oracle.attention_row(q, k[: i + 1], v[: i + 1])
        assert_close(out[i : i + 1], ref, f"position {i}")


def test_prefill_d256_long_prefix_split(cuda, built):
    """head_dim 256 (one Q tile per item, 64-key tiles): chunks on long cached prefixes, so items span more than
    24 tiles and run as two key chunks, mixed with decode rows; two layers reuse the merge slots."""
    shape = synth.Shape(2, 16, 4, 256)
    rows = [(3000, 100), (17, 1), (1500, 64), (5000, 33), (9, 40)]
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=41)
    pool, ds, outs = run_batch(batch, [0, 1])
    for layer in (0, 1):
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, outs[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")
