"""GPU parity of the pass as the benchmark times it: plan + per layer pkv_attention_append, captured as one
CUDA graph (workload.capture_step_graph, the function bench.py uses) and replayed.  Each replay plans again,
re-appends this pass's tokens (the same bits to the same slots) and recomputes every layer; the outputs must
match the oracle after every replay and be bit-identical between replays ("Static batching", "What changed":
the step is launched without the host in the loop)."""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row, oracle_row_8bit, poison, row_slice

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make,num_layers,kv", [
    pytest.param(synth.qwen_decode, 28, pkv.PKV_KV_F16, id="qwen_decode-28-fp16"),
    pytest.param(synth.qwen_decode, 4, pkv.PKV_KV_E4M3, id="qwen_decode-4-e4m3"),
    pytest.param(synth.mixed_step, 3, pkv.PKV_KV_F16, id="mixed_step-3-fp16"),
    pytest.param(synth.mixed_step, 3, pkv.PKV_KV_E4M3, id="mixed_step-3-e4m3"),
])
def test_graph_replayed_step_matches_oracle(cuda, built, make, num_layers, kv):
    batch = make(0)
    s = batch.shape
    batch.shape = synth.Shape(num_layers, s.num_q_heads, s.num_kv_heads, s.head_dim, s.block_size)
    layers = list(range(num_layers))
    pool = workload.make_pool(batch, kv_dtype=kv)
    poison(pool)
    workload.prefill_cache(pool, batch, layers)
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, layers)
    outs = [torch.full_like(q, float("nan")) for q in qs]
    attn = workload.Attention(pool, ds)
    graph, launches = workload.capture_step_graph(pool, ds, attn, qs, ks, vs, outs, layers, fused=True)
    assert launches >= 1 + num_layers
    first = None
    for rep in range(3):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pool.check() == 0
        now = [o.clone() for o in outs]
        if first is None:
            first = now
        else:
            for a, b in zip(first, now):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    order = np.argsort(batch.context_lens)
    rows = sorted(set(order[:2].tolist() + order[-2:].tolist() + [5, batch.num_seqs // 2]))
    rows += [b for b in range(batch.num_seqs) if batch.q_lens[b] > 1]          # every chunked-prefill row
    ref_of = oracle_row_8bit if kv == pkv.PKV_KV_E4M3 else oracle_row
    for layer in sorted({0, num_layers // 2, num_layers - 1}):
        for b in sorted(set(rows)):
            assert_close(row_slice(batch, first[layer], b), ref_of(batch, layer, b), f"layer {layer} row {b}")
