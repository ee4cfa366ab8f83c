"""Repeated launches on one plan: large batches of small tasks, the case where the decode kernel's warps hand
tasks, queue slots and q buffers to each other most often.  Every launch must leave the device error word
clear (no on-chip wait may give up) and the last outputs of both layers must match the oracle row by row."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import synth, workload
from helpers_gpu import assert_close, oracle_row, row_slice

pytestmark = pytest.mark.gpu

LAUNCHES = 40


@pytest.mark.parametrize("rows,split_blocks", [(512, 0), (512, 4), (1024, 8)])
def test_many_launches_on_one_plan(cuda, built, rows, split_blocks):
    rng = np.random.default_rng(rows + split_blocks)
    ctx = rng.integers(2, 770, size=rows)
    shape = synth.Shape(2, 12, 2, 128)
    batch = synth.custom_batch(shape, ctx - 1, np.ones(rows, dtype=np.int64), seed=13)
    pool = workload.make_pool(batch, split_blocks=split_blocks)
    workload.prefill_cache(pool, batch, [0, 1])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0, 1])
    outs = [torch.full_like(q, float("nan")) for q in qs]
    attn = workload.Attention(pool, ds)
    attn.plan()
    for i in range(LAUNCHES):
        attn.run_append(i % 2, qs[i % 2], ks[i % 2], vs[i % 2], outs[i % 2])
        if i % 8 == 7:
            torch.cuda.synchronize()
            assert pool.check() == 0, f"device error word set after launch {i}"
    torch.cuda.synchronize()
    assert pool.check() == 0
    for layer in (0, 1):
        for b in range(0, rows, 7):
            assert_close(row_slice(batch, outs[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")
