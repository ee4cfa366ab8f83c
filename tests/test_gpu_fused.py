"""GPU: pkv_attention_append (kv_append fused into the decode launch) gives bit for bit the cache contents and
the outputs of pkv_append followed by pkv_attention -- decode rows, short chunks, skipped slots -- and falls
back to the two calls when a prefill row is possible."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, row_slice

pytestmark = pytest.mark.gpu


def _pass(batch, layers, fused, skip=()):
    pool = workload.make_pool(batch)
    pool.cache_view().view(torch.int16).fill_(0x7E00)
    workload.prefill_cache(pool, batch, layers)
    ds = workload.upload(batch, pool)
    for t in skip:
        ds.slot_mapping[t] = -1
    qs, ks, vs = workload.step_inputs(ds, layers)
    outs = [torch.empty_like(q) for q in qs]
    workload.run_pass(pool, ds, layers, qs, ks, vs, outs, fused=fused)
    torch.cuda.synchronize()
    assert pool.check() == 0
    return pool, outs


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("rows", [
    [(300, 1), (17, 1), (0, 1), (255, 1), (256, 1), (700, 1), (15, 1)],          # decode rows
    [(300, 1), (40, 3), (0, 7), (255, 2), (16, 1), (900, 4)],                    # short chunks (decode path)
])
def test_fused_equals_append_then_attention(cuda, built, rows):
    shape = synth.Shape(2, 12, 2, 128)
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=14)
    pa, oa = _pass(batch, [0, 1], fused=False)
    pb, ob = _pass(batch, [0, 1], fused=True)
    assert pkv.pkv_last_launch_count(pb.handle) == 1  # one decode launch: no separate append
    assert _same(pa.cache_view(), pb.cache_view())
    for layer in (0, 1):
        assert _same(oa[layer], ob[layer])
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, ob[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")


def test_fused_skips_slot_minus_one(cuda, built):
    shape = synth.Shape(1, 8, 2, 64)
    batch = synth.custom_batch(shape, [100, 30, 0], [1, 1, 1], seed=2)
    pa, _ = _pass(batch, [0], fused=False, skip=[1])
    pb, _ = _pass(batch, [0], fused=True, skip=[1])
    assert _same(pa.cache_view(), pb.cache_view())


@pytest.mark.parametrize("hq,hkv,d", [(12, 2, 128), (16, 4, 256)])
def test_fused_falls_back_when_a_prefill_row_is_possible(cuda, built, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    batch = synth.custom_batch(shape, [200, 0, 50], [1, 40, 1], seed=5)
    pa, oa = _pass(batch, [0], fused=False)
    pb, ob = _pass(batch, [0], fused=True)
    assert _same(pa.cache_view(), pb.cache_view())
    assert _same(oa[0], ob[0])


def test_qwen_decode_fused_full_size_sampled(cuda, built):
    """The benchmark's workload through the fused call: 256 rows, three layers, sampled rows."""
    batch = synth.qwen_decode(0)
    batch.shape = synth.Shape(3, 12, 2, 128)
    pb, ob = _pass(batch, [0, 1, 2], fused=True)
    for layer in (0, 2):
        for b in (0, 77, 255):
            assert_close(row_slice(batch, ob[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")
