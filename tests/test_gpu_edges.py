"""GPU edge cases: ragged and boundary lengths, every supported head shape, degenerate inputs,
invariances (physical placement, batch composition, row order) and the device-side error reporting."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, row_slice, run_batch

pytestmark = pytest.mark.gpu

# (cached, q_len) rows around block (16 tokens) and split boundaries (the default split of 32 blocks is 512
# tokens; 16-block splits, 256 tokens, are covered too), plus chunks
ROWS = [(0, 1), (1, 1), (14, 1), (15, 1), (16, 1), (255, 1), (256, 1), (257, 1), (511, 1), (512, 1), (700, 1),
        (1023, 1), (1024, 1), (16, 3), (0, 33), (240, 17), (500, 12), (1020, 6), (0, 2)]
SHAPES = [(4, 2, 64), (12, 2, 128), (16, 4, 256), (8, 8, 128), (8, 1, 128), (16, 2, 64), (4, 1, 256)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
def test_ragged_boundaries_all_shapes(cuda, built, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached, qls = zip(*ROWS)
    batch = synth.custom_batch(shape, cached, qls, seed=11)
    pool, ds, outs = run_batch(batch, [0])
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row(batch, 0, b), f"{(hq, hkv, d)} row {b} {ROWS[b]}")


def test_context_of_one_returns_v_exactly(cuda, built):
    shape = synth.Shape(1, 12, 2, 128)
    batch = synth.custom_batch(shape, [0, 0, 0], [1, 1, 1], seed=5)
    pool, ds, outs = run_batch(batch, [0])
    out = outs[0].cpu().numpy()
    for b in range(3):
        v = synth.token_values(synth.KIND_V, 5, 0, [batch.req_ids[b]], [0], 2, 128)[0]
        for h in range(12):
            assert np.array_equal(out[b, h].view(np.uint16), v[h // 6].view(np.uint16))


@pytest.mark.parametrize("split_blocks", [1, 3, 16, 32])
def test_split_size_does_not_change_the_answer(cuda, built, split_blocks):
    shape = synth.Shape(1, 12, 2, 128)
    batch = synth.custom_batch(shape, [1000, 37, 400, 0], [1, 1, 5, 64], seed=2)
    pool, ds, outs = run_batch(batch, [0], split_blocks=split_blocks)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row(batch, 0, b), f"split {split_blocks} row {b}")


def test_split_size_above_limit_is_refused(cuda, built):
    batch = synth.tiny_decode(0)
    pool = workload.make_pool(batch, split_blocks=64)
    ds = workload.upload(batch, pool)
    attn = workload.Attention(pool, ds)
    with pytest.raises(pkv.PkvError) as e:
        attn.plan()
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


def test_invariant_to_physical_block_placement(cuda, built):
    shape = synth.Shape(1, 12, 2, 128)
    cached, qls = [300, 17, 650, 1, 0], [1, 1, 1, 1, 20]
    a = synth.custom_batch(shape, cached, qls, seed=3, block_seed=100)
    b = synth.custom_batch(shape, cached, qls, seed=3, block_seed=200)
    assert not np.array_equal(a.block_tables, b.block_tables)
    _, _, oa = run_batch(a, [0])
    _, _, ob = run_batch(b, [0])
    assert torch.equal(oa[0].view(torch.int16), ob[0].view(torch.int16))


def test_batched_equals_each_row_alone(cuda, built):
    """The pages' parity method: each row in a ragged batch gives exactly what it gives at batch 1."""
    shape = synth.Shape(1, 12, 2, 128)
    cached, qls = [300, 17, 650, 1, 0, 255], [1, 1, 1, 1, 20, 1]
    full = synth.custom_batch(shape, cached, qls, seed=4)
    _, _, of = run_batch(full, [0])
    for b in range(len(cached)):
        alone = synth.custom_batch(shape, [cached[b]], [qls[b]], seed=4, req_ids=[full.req_ids[b]])
        _, _, oa = run_batch(alone, [0])
        assert torch.equal(oa[0].view(torch.int16), torch.from_numpy(row_slice(full, of[0], b)).to(cuda).view(torch.int16))


def test_row_order_does_not_matter(cuda, built):
    shape = synth.Shape(1, 16, 4, 256)
    cached, qls = [300, 17, 650, 1, 0], [1, 1, 1, 3, 20]
    a = synth.custom_batch(shape, cached, qls, seed=6)
    perm = [3, 0, 4, 2, 1]
    b = synth.custom_batch(shape, [cached[i] for i in perm], [qls[i] for i in perm], seed=6,
                           req_ids=[a.req_ids[i] for i in perm])
    _, _, oa = run_batch(a, [0])
    _, _, ob = run_batch(b, [0])
    for j, i in enumerate(perm):
        assert np.array_equal(row_slice(a, oa[0], i).view(np.uint16), row_slice(b, ob[0], j).view(np.uint16))


def test_empty_pass_launches_nothing(cuda, built):
    batch = synth.tiny_decode(0)
    pool = workload.make_pool(batch)
    ws = torch.empty(256, dtype=torch.uint8, device=cuda)
    z = torch.zeros(1, dtype=torch.int32, device=cuda)
    pkv.pkv_attention_plan(pool.handle, z, z, 0, 0, 1, ws, 256)
    pkv.pkv_attention(pool.handle, 0, ws, z, 1, z, z, 0, 0, ws, ws, 256)
    assert pkv.pkv_last_launch_count(pool.handle) == 0
    pkv.pkv_append(pool.handle, 0, ws, ws, z, 0)
    assert pkv.pkv_last_launch_count(pool.handle) == 0


def test_attention_without_matching_plan_is_refused(cuda, built):
    batch = synth.tiny_decode(0)
    pool, ds, outs = run_batch(batch, [0])
    attn = workload.Attention(pool, ds)
    other = torch.empty_like(attn.workspace)
    q = torch.zeros_like(outs[0])
    with pytest.raises(pkv.PkvError):
        pkv.pkv_attention(pool.handle, 0, q, ds.block_tables, ds.max_blocks, ds.context_lens, ds.query_start_loc,
                          ds.num_seqs, ds.num_tokens, outs[0], other, attn.ws_bytes)


def test_out_of_range_metadata_is_reported_not_dereferenced(cuda, built):
    """Bad block ids and slots are caught by the kernels' own bounds checks and reported."""
    batch = synth.tiny_decode(0)
    pool, ds, outs = run_batch(batch, [0])
    bad_bt = ds.block_tables.clone()
    bad_bt[1, 0] = batch.num_blocks + 5
    bad_bt[2, 1] = -7
    attn = workload.Attention(pool, ds)
    attn.plan()
    q = torch.zeros_like(outs[0])
    pkv.pkv_attention(pool.handle, 0, q, bad_bt, ds.max_blocks, ds.context_lens, ds.query_start_loc, ds.num_seqs,
                      ds.num_tokens, outs[0], attn.workspace, attn.ws_bytes)
    torch.cuda.synchronize()
    assert pool.check() & pkv.PKV_DEVERR_BLOCK_RANGE
    k = torch.zeros(2, 2, 64, dtype=torch.float16, device=cuda)
    slots = torch.tensor([batch.num_blocks * 16, -3], dtype=torch.int64, device=cuda)
    pkv.pkv_append(pool.handle, 0, k, k, slots, 2)
    torch.cuda.synchronize()
    assert pool.check() & pkv.PKV_DEVERR_SLOT_RANGE
    bad_ctx = ds.context_lens.clone()
    bad_ctx[0] = 10 ** 6                                       # longer than the block table allows
    attn2 = workload.Attention(pool, ds)
    pkv.pkv_attention_plan(pool.handle, bad_ctx, ds.query_start_loc, ds.num_seqs, ds.num_tokens, ds.max_blocks,
                           attn2.workspace, attn2.ws_bytes)
    torch.cuda.synchronize()
    assert pool.check() & pkv.PKV_DEVERR_ROW_META
