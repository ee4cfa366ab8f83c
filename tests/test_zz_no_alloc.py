"""pkv_attention_noalloc: the attention call for callers that cannot provide a workspace.

Such a caller (an engine whose device memory already belongs to its own allocator, or code that must not
call cudaMalloc in the middle of a pass) gets the split-K scratch from a fixed array inside libpkv.  The
tests check, through the C ABI, that two calls in a row give what the workspace-based pkv_attention gives
on the same inputs -- bit for bit, since both run the same kernels on the same plan -- and what the oracle
gives; that the 8-bit cache's prefill rows (whose fp16 shadow then lives in the array) agree too, also when
calls alternate with the workspace call; that a pass too large for the array is refused before anything
runs; and, in a fresh process, that a first call made during a stream capture is refused.
This file is collected last on purpose; it also passes alone in a fresh process.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import MAX_ABS, MEAN_ABS, assert_close, oracle_row, oracle_row_8bit, poison, row_slice

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


def _same_bits(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _against_oracle(batch, out, layer, kv8=False):
    for b in range(batch.num_seqs):
        ref = oracle_row_8bit(batch, layer, b) if kv8 else oracle_row(batch, layer, b)
        assert_close(row_slice(batch, out, b), ref, f"layer {layer} row {b}")


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
        _same_bits(got, ref)
        _against_oracle(batch, got, layer)
    # a second round on the same layer still agrees (the array keeps the previous call's contents)
    again = _noalloc(pool, ds, 0, qs[0])
    torch.cuda.synchronize()
    _same_bits(again, _with_workspace(pool, ds, 0, qs[0]))
    assert pool.check() == 0


def test_noalloc_8bit_cache_with_a_prefill_row(cuda, built):
    """On the 8-bit cache a chunked-prefill row reads an fp16 shadow of its blocks, which for this call lives in
    the built-in array; the shadow's tensor map is re-encoded whenever the call alternates with a workspace."""
    shape = synth.Shape(1, 12, 2, 128)
    batch = synth.custom_batch(shape, [300, 0, 40, 700], [1, 48, 20, 1], seed=23)
    pool = workload.make_pool(batch, kv_dtype=pkv.PKV_KV_E4M3)
    poison(pool)
    workload.prefill_cache(pool, batch, [0])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0])
    pkv.pkv_append(pool.handle, 0, ks[0], vs[0], ds.slot_mapping, ds.num_tokens)
    need = pkv.pkv_attention_workspace_bytes(pool.handle, ds.num_seqs, ds.num_tokens, ds.max_blocks)
    assert 0 < need <= pkv.PKV_NOALLOC_SCRATCH_BYTES
    ref = _with_workspace(pool, ds, 0, qs[0])
    first = _noalloc(pool, ds, 0, qs[0])
    second = _noalloc(pool, ds, 0, qs[0])
    torch.cuda.synchronize()
    _same_bits(first, ref)
    _same_bits(second, ref)
    _against_oracle(batch, first, 0, kv8=True)
    again_ws = _with_workspace(pool, ds, 0, qs[0])   # the shadow map moves back to the workspace ...
    again = _noalloc(pool, ds, 0, qs[0])              # ... and into the array again
    torch.cuda.synchronize()
    _same_bits(again_ws, ref)
    _same_bits(again, ref)
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


_CAPTURE_PROBE = r"""
import sys
sys.path.insert(0, sys.argv[1])
import torch
from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
batch = synth.custom_batch(synth.Shape(1, 12, 2, 128), [100, 30], [1, 1], seed=3)
pool = workload.make_pool(batch)
ds = workload.upload(batch, pool)
q = torch.zeros(ds.num_tokens, 12, 128, dtype=torch.float16, device="cuda")
out = torch.zeros_like(q)
torch.cuda.synchronize()
side = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
status, message = None, ""
with torch.cuda.graph(graph, stream=side):
    try:
        pkv.pkv_attention_noalloc(pool.handle, 0, q, ds.block_tables, ds.max_blocks, ds.context_lens,
                                  ds.query_start_loc, ds.num_seqs, ds.num_tokens, out, side)
    except pkv.PkvError as e:
        status = e.status
        message = str(e)
print("STATUS", status, pkv.pkv_last_launch_count(pool.handle), "capture" in message)
"""


def test_first_noalloc_call_during_capture_is_refused(cuda, built):
    """In a fresh process (no earlier call has looked up the array's address) a first call made while the stream
    is being captured is refused with PKV_ERR_INVALID_ARG, before anything is launched."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_PROBE, root], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("STATUS")][-1]
    assert line == f"STATUS {pkv.PKV_ERR_INVALID_ARG} 0 True", line
