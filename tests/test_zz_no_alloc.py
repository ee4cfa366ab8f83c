"""pkv_attention_noalloc: the attention call for callers that cannot provide a workspace.

Such a caller (an engine whose device memory already belongs to its own allocator, or code that must not
call cudaMalloc in the middle of a pass) gets the split-K scratch from a fixed array inside libpkv.  The
test checks, through the C ABI, that two calls in a row give what the workspace-based pkv_attention gives
on the same inputs, and that a pass too large for the array is refused before anything runs.
This file is collected last on purpose; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


def _with_workspace(pool, ds, layer, q):
    out = torch.empty_like(q)
    attn = workload.Attention(pool, ds)
    attn.plan()
    attn.run(layer, q, out)
    return out


def _noalloc(pool, ds, layer, q):
    out = torch.full_like(q, float("nan"))
    pkv.pkv_attention_noalloc(pool.handle, layer, q, ds.block_tables, ds.max_blocks, ds.context_lens,
                              ds.query_start_loc, ds.num_seqs, ds.num_tokens, out)
    return out


def _close(a, b):
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (err.max().item(), err.mean().item())


def test_noalloc_matches_workspace_call_twice_in_a_row(cuda, built):
    # a Qwen-shaped ragged pass with decode rows spanning several splits and a chunked-prefill row
    shape = synth.Shape(2, 12, 2, 128)
    batch = synth.custom_batch(shape, [700, 17, 300, 0, 511, 1000], [1, 1, 1, 40, 1, 3], seed=21)
    pool = workload.make_pool(batch)
    workload.prefill_cache(pool, batch, [0, 1])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0, 1])
    for layer in (0, 1):
        pkv.pkv_append(pool.handle, layer, ks[layer], vs[layer], ds.slot_mapping, ds.num_tokens)
    need = pkv.pkv_attention_workspace_bytes(pool.handle, ds.num_seqs, ds.num_tokens, ds.max_blocks)
    assert 0 < need <= pkv.PKV_NOALLOC_SCRATCH_BYTES
    for layer in (0, 1):                       # two calls in a row share (and overwrite) the array
        ref = _with_workspace(pool, ds, layer, qs[layer])
        got = _noalloc(pool, ds, layer, qs[layer])
        torch.cuda.synchronize()
        _close(got, ref)
    # a second round on the same layer still agrees (the array keeps the previous call's contents)
    again = _noalloc(pool, ds, 0, qs[0])
    torch.cuda.synchronize()
    _close(again, _with_workspace(pool, ds, 0, qs[0]))
    assert pool.check() == 0


def test_noalloc_refuses_a_pass_beyond_its_scratch(cuda, built):
    shape = synth.Shape(1, 16, 4, 256)
    batch = synth.custom_batch(shape, [2000] * 64, [1] * 64, seed=22)
    pool = workload.make_pool(batch, split_blocks=1)          # one split per block: ~130 MB of partials
    ds = workload.upload(batch, pool)
    need = pkv.pkv_attention_workspace_bytes(pool.handle, ds.num_seqs, ds.num_tokens, ds.max_blocks)
    assert need > pkv.PKV_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(ds.num_tokens, 16, 256, dtype=torch.float16, device=cuda)
    out = torch.zeros_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_attention_noalloc(pool.handle, 0, q, ds.block_tables, ds.max_blocks, ds.context_lens,
                                  ds.query_start_loc, ds.num_seqs, ds.num_tokens, out)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_RANGE
    assert pkv.pkv_last_launch_count(pool.handle) == 0
