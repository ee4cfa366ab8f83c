"""GPU parity: libpkv through its C ABI against the CPU oracle on the seeded synthetic workloads.

Bit-exact: the device input generator, slot mapping, kv_append.  Within max abs 4e-3 / mean abs 5e-4:
attention outputs (fp16) against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, row_slice, run_batch

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host(cuda, built):
    rng = np.random.default_rng(0)
    for kind, heads, d in [(synth.KIND_Q, 12, 128), (synth.KIND_K, 4, 256), (synth.KIND_V, 2, 64)]:
        req = rng.integers(0, 1 << 31, 300)
        pos = rng.integers(0, 300000, 300)
        host = synth.token_values(kind, 123456789012, 7, req, pos, heads, d)
        dev = torch.empty(300, heads, d, dtype=torch.float16, device=cuda)
        synth.device_fill(kind, 123456789012, 7, torch.from_numpy(req).to(cuda), torch.from_numpy(pos).to(cuda),
                          heads, d, dev)
        assert np.array_equal(dev.cpu().numpy().view(np.uint16), host.view(np.uint16))


@pytest.mark.parametrize("make", [synth.tiny_decode, synth.qwen_decode, synth.mixed_step])
def test_slot_mapping_bit_exact(cuda, built, make):
    batch = make(0)
    pool = workload.make_pool(batch, num_layers=1)
    ds = workload.upload(batch, pool)
    ref = oracle.slot_mapping_for_batch(batch.block_tables, batch.context_lens, batch.q_lens, 16)
    assert np.array_equal(ds.slot_mapping.cpu().numpy(), ref)
    assert pool.check() == 0


@pytest.mark.parametrize("make", [synth.tiny_decode, synth.mixed_step])
def test_append_bit_exact(cuda, built, make):
    batch = make(1)
    pool = workload.make_pool(batch, num_layers=2)
    view = pool.cache_view().view(torch.int16)
    view.copy_(torch.randint(-32768, 32767, view.shape, dtype=torch.int16, device=cuda))
    before_k = pool.layer(1, 0).cpu().numpy().copy()
    before_v = pool.layer(1, 1).cpu().numpy().copy()
    other = pool.layer(0, 0).cpu().numpy().copy()
    ds = workload.upload(batch, pool)
    _, ks, vs = workload.step_inputs(ds, [1])
    slots = ds.slot_mapping.clone()
    slots[::7] = -1                                          # padding slots are skipped
    pkv.pkv_append(pool.handle, 1, ks[0], vs[0], slots, batch.num_tokens)
    torch.cuda.synchronize()
    oracle.append_reference(before_k, before_v, ks[0].cpu().numpy(), vs[0].cpu().numpy(), slots.cpu().numpy())
    assert np.array_equal(pool.layer(1, 0).cpu().numpy().view(np.uint16), before_k.view(np.uint16))
    assert np.array_equal(pool.layer(1, 1).cpu().numpy().view(np.uint16), before_v.view(np.uint16))
    assert np.array_equal(pool.layer(0, 0).cpu().numpy().view(np.uint16), other.view(np.uint16))
    assert pool.check() == 0


def test_tiny_decode_parity(cuda, built):
    batch = synth.tiny_decode(0)
    pool, ds, outs = run_batch(batch, [0])
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row(batch, 0, b), f"row {b}")


def test_qwen_decode_full_size_sampled(cuda, built):
    """All 28 layers, 256 rows, in the benchmark's launch configuration: every row on the first and the last
    layer, and on every other layer the shortest and longest contexts and three fixed rows."""
    batch = synth.qwen_decode(0)
    layers = list(range(28))
    pool, ds, outs = run_batch(batch, layers, poison=False)
    order = np.argsort(batch.context_lens)
    sample = sorted(set(order[:3].tolist() + order[-3:].tolist() + [17, 100, 201]))
    for layer in layers:
        rows = range(batch.num_seqs) if layer in (0, 27) else sample
        for b in rows:
            assert_close(row_slice(batch, outs[layer], b), oracle_row(batch, layer, b), f"layer {layer} row {b}")


def test_mixed_step_parity(cuda, built):
    """83 decode rows + chunked-prefill rows of 2048 (on 0) and 1024 (on 3072) new tokens, every row."""
    batch = synth.mixed_step(0)
    pool, ds, outs = run_batch(batch, [0, 1], num_layers=2)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[1], b), oracle_row(batch, 1, b), f"row {b}")


def test_long_context_gqa_every_row_and_head(cuda, built):
    """The long-context workload's rows (four of 262,144 cached tokens, d=256, 16 q / 4 KV heads) in a 16-layer
    pool: all 16 (row, KV head) pairs on the last layer and one KV head of every row on the first, each
    against the oracle element by element.  The oracle runs in a process pool (spawn) on the host cores."""
    import multiprocessing as mp
    import os

    import oracle_workers

    batch = synth.long_gqa(0)
    s = batch.shape
    assert s.num_layers == 16
    pool, ds, outs = run_batch(batch, [0, 15], num_layers=16, poison=False)
    jobs = [(15, b, g) for b in range(4) for g in range(4)] + [(0, b, (b + 1) % 4) for b in range(4)]
    args = [(batch.seed, layer, int(batch.req_ids[b]), int(batch.context_lens[b]), g, s.num_q_heads,
             s.num_kv_heads, s.head_dim) for layer, b, g in jobs]
    with mp.get_context("spawn").Pool(max(1, min(len(jobs), os.cpu_count() or 1))) as workers:
        refs = workers.map(oracle_workers.long_row_one_kv_head, args, chunksize=1)
    G = s.num_q_heads // s.num_kv_heads
    for (layer, b, g), ref in zip(jobs, refs):
        out = outs[0 if layer == 0 else 1]
        assert_close(row_slice(batch, out, b)[:, G * g:G * g + G], ref, f"layer {layer} row {b} kv {g}")
