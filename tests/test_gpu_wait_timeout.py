"""GPU: an on-chip wait that runs out ([ABL] "Counting jobs while they run": a job must not be left holding the
device).  Every barrier wait in the kernels is bounded; when one gives up the kernel records
PKV_DEVERR_WAIT_TIMEOUT, lets its copies land and returns, and later attention launches on the pool do no
work until the bit is cleared and the pass is planned again.

The expiry is made with the library's test hook (pkv_debug_expire_wait, enabled by PKV_TEST_HOOKS=1): one
thread waits, through the kernels' own bounded wait, on a barrier nobody arrives at, with the limit shortened
to 1 ms.  Nothing traps and nothing waits without a limit."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, row_slice

pytestmark = pytest.mark.gpu


def _pass():
    batch = synth.custom_batch(synth.Shape(1, 12, 2, 128), [300, 40, 0, 700], [1, 3, 20, 1], seed=29)
    pool = workload.make_pool(batch)
    workload.prefill_cache(pool, batch, [0])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0])
    for_layer = (qs[0], ks[0], vs[0])
    pkv.pkv_append(pool.handle, 0, ks[0], vs[0], ds.slot_mapping, ds.num_tokens)
    torch.cuda.synchronize()
    return batch, pool, ds, for_layer


def test_hook_is_off_by_default(cuda, built, monkeypatch):
    monkeypatch.delenv("PKV_TEST_HOOKS", raising=False)
    batch, pool, ds, _ = _pass()
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_debug_expire_wait(pool.handle, 1_000_000)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    assert pkv.pkv_last_launch_count(pool.handle) == 0
    assert pool.check() == 0


def test_expired_wait_poisons_the_pool_until_cleared(cuda, built, monkeypatch):
    monkeypatch.setenv("PKV_TEST_HOOKS", "1")
    batch, pool, ds, (q, k, v) = _pass()
    attn = workload.Attention(pool, ds)
    attn.plan()
    good = torch.empty_like(q)
    attn.run(0, q, good)
    torch.cuda.synchronize()
    assert pool.check(clear=False) == 0

    with pytest.raises(pkv.PkvError) as e:   # limits outside 1 ns .. 100 ms are refused
        pkv.pkv_debug_expire_wait(pool.handle, 0)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_RANGE
    pkv.pkv_debug_expire_wait(pool.handle, 1_000_000)
    assert pkv.pkv_last_launch_count(pool.handle) == 1
    torch.cuda.synchronize()
    assert pool.check(clear=False) == pkv.PKV_DEVERR_WAIT_TIMEOUT

    # while the bit is set, an attention launch does no work: the output keeps its sentinel
    sentinel = torch.full_like(q, 7.0)
    attn.plan()
    attn.run(0, q, sentinel)
    torch.cuda.synchronize()
    assert torch.all(sentinel == 7.0)
    assert pool.check(clear=False) == pkv.PKV_DEVERR_WAIT_TIMEOUT

    # cleared and planned again, the pass is right again (and the same bits as before the expiry)
    assert pool.check(clear=True) == pkv.PKV_DEVERR_WAIT_TIMEOUT
    assert pool.check(clear=False) == 0
    attn.plan()
    out = torch.empty_like(q)
    attn.run(0, q, out)
    torch.cuda.synchronize()
    assert pool.check() == 0
    assert torch.equal(out.view(torch.int16), good.view(torch.int16))
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, out, b), oracle_row(batch, 0, b), f"row {b}")
