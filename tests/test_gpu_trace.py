"""Scheduler-driven passes on the GPU: the C++ scheduler's batches (256 lognormal-prompt requests, token
budget 8,192) run through slot mapping, kv_append and attention on a persistent paged pool, as the pages'
engine does one pass after another ("Continuous Batching Is Not a Bigger Batch", sections "What the
scheduler does on one step" and "The allocator is the other half").  The 5,000-block pool preempts and
recomputes; a re-prefilled request rewrites identical key/value bits, so its later rows still match the
oracle.  Checked every pass: the device slot mapping against the scheduler's, the device error word, and
sampled rows (decode rows and one bounded prefill row) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, oracle_row_8bit, poison, row_slice

pytestmark = pytest.mark.gpu

SEED = 0
LAYERS = [0, 1]


def _step_batch(shape, num_blocks, st):
    return synth.StepBatch(shape, num_blocks, st["req_ids"], st["q_lens"], st["context_lens"],
                           np.ascontiguousarray(st["block_tables"]), np.zeros(0, dtype=np.int32), SEED, "trace")


@pytest.mark.parametrize("num_blocks,cap,steps,alloc,unit,declared,prefix,kv", [
    (20000, 256, 24, 0, 0, 1.0, False, 0), (5000, 256, 84, 0, 0, 1.0, False, 0), (20000, 64, 16, 0, 0, 1.0, False, 0),
    (5000, 256, 40, pkv.PKV_ALLOC_RESERVE, pkv.PKV_UNIT_PASS, 4.0, False, 0),
    (20000, 64, 40, pkv.PKV_ALLOC_ON_DEMAND, pkv.PKV_UNIT_REQUEST, 1.0, False, 0),
    (5000, 256, 110, 0, 0, 1.0, True, 0),
    (9922, 256, 60, 0, 0, 1.0, False, pkv.PKV_KV_E4M3)])
def test_scheduler_trace_passes(cuda, built, num_blocks, cap, steps, alloc, unit, declared, prefix, kv):
    """The default policy, and the Orca reservation ("The allocator is the other half"), request-level
    batching ("The boundary: when this is worth nothing") and prefix-cached recompute variants of the same
    page.  With prefix caching a readmitted request reads the blocks it wrote before its preemption.  The last
    case is the 8-bit cache ("Checking it on a real system": quantize the cache) at the bytes of 5,000 fp16
    blocks; its rows are checked against the oracle over the dequantized cache."""
    shape = synth.Shape(len(LAYERS), 12, 2, 128)
    sched = pkv.Scheduler(cap, 8192, 16, num_blocks, free_order=synth.block_permutation(num_blocks, SEED),
                          alloc=alloc, unit=unit, prefix_caching=prefix)
    for r in synth.trace_requests(SEED):
        sched.add(r.req_id, r.prompt_len, r.max_output, int(round(declared * r.max_output)))
    probe = synth.custom_batch(shape, [1], [1], seed=SEED, num_blocks=num_blocks)
    pool = workload.make_pool(probe, kv_dtype=kv)
    poison(pool)  # NaN wherever nothing was appended
    reference = oracle_row_8bit if kv == pkv.PKV_KV_E4M3 else oracle_row
    rng = np.random.default_rng(7)
    preempted, rechecked, reused = set(), 0, 0
    for step in range(steps):
        st = sched.step()
        preempted.update(st["preempted"])
        if len(st["req_ids"]) == 0:
            break
        batch = _step_batch(shape, num_blocks, st)
        ds = workload.upload(batch, pool)
        assert np.array_equal(ds.slot_mapping.cpu().numpy(), st["slot_mapping"]), f"step {step}: slot mapping"
        qs, ks, vs = workload.step_inputs(ds, LAYERS)
        outs = [torch.empty_like(q) for q in qs]
        workload.run_pass(pool, ds, LAYERS, qs, ks, vs, outs)
        torch.cuda.synchronize()
        assert pool.check() == 0, f"step {step}: device error word"
        ql, ctx = batch.q_lens, batch.context_lens
        decode = np.nonzero(ql == 1)[0]
        sample = list(rng.choice(decode, size=min(2, decode.size), replace=False)) if decode.size else []
        chunk = [b for b in np.nonzero(ql > 1)[0] if int(ql[b]) * int(ctx[b]) <= 600_000]
        if chunk:
            sample.append(chunk[0])
        back = [b for b in range(batch.num_seqs) if int(batch.req_ids[b]) in preempted]
        if back:
            # a request readmitted after preemption (its cache recomputed, or reused from its own blocks);
            # prefer one whose first row this is, starting past reused blocks
            fresh = [b for b in back if int(batch.req_ids[b]) in st["admitted"] and ctx[b] > ql[b]
                     and int(ql[b]) * int(ctx[b]) <= 2_000_000]
            sample.append(fresh[0] if fresh else back[0])
            rechecked += 1
            reused += len(fresh)
        for b in sample:
            assert_close(row_slice(batch, outs[1], b), reference(batch, 1, int(b)),
                         f"step {step} row {b} (req {batch.req_ids[b]}, q_len {ql[b]}, ctx {ctx[b]})")
    stats = sched.stats()
    if num_blocks == 5000 and alloc == pkv.PKV_ALLOC_ON_DEMAND:
        assert stats["preemptions"] > 0 and rechecked > 0, stats
    if alloc == pkv.PKV_ALLOC_RESERVE:
        assert stats["preemptions"] == 0
    if prefix:
        assert stats["prefix_hit_tokens"] > 0 and reused > 0, stats
    sched.close()


@pytest.mark.parametrize("num_blocks,cap", [(20000, 256), (20000, 64), (5000, 256)])
def test_scheduler_trace_to_exhaustion(cuda, built, num_blocks, cap):
    """Every pass of the trace until the scheduler is done, one layer: slot mapping and device error word
    checked every pass, one row against the oracle every 25th pass and on the last."""
    shape = synth.Shape(1, 12, 2, 128)
    sched = pkv.Scheduler(cap, 8192, 16, num_blocks, free_order=synth.block_permutation(num_blocks, SEED))
    for r in synth.trace_requests(SEED):
        sched.add(r.req_id, r.prompt_len, r.max_output)
    probe = synth.custom_batch(shape, [1], [1], seed=SEED, num_blocks=num_blocks)
    pool = workload.make_pool(probe)
    pool.cache_view().view(torch.int16).fill_(0x7E00)
    step, tokens = 0, 0
    while not sched.done():
        st = sched.step()
        assert len(st["req_ids"]) > 0, f"step {step}: the scheduler made no progress"
        batch = _step_batch(shape, num_blocks, st)
        ds = workload.upload(batch, pool)
        assert np.array_equal(ds.slot_mapping.cpu().numpy(), st["slot_mapping"]), f"step {step}: slot mapping"
        qs, ks, vs = workload.step_inputs(ds, [0])
        outs = [torch.empty_like(qs[0])]
        workload.run_pass(pool, ds, [0], qs, ks, vs, outs, fused=True)
        tokens += batch.num_tokens
        if step % 25 == 0 or sched.done():
            torch.cuda.synchronize()
            assert pool.check() == 0, f"step {step}: device error word"
            b = int(np.argmin(batch.q_lens.astype(np.int64) * batch.context_lens))  # the cheapest row to check
            assert_close(row_slice(batch, outs[0], b), oracle_row(batch, 0, b), f"step {step} row {b}")
        step += 1
    torch.cuda.synchronize()
    assert pool.check() == 0
    stats = sched.stats()
    assert stats["steps"] == step and stats["running"] == 0 and stats["waiting"] == 0
    assert tokens == stats["tokens_scheduled"]
    sched.close()
