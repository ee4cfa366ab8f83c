"""GPU: PKV_VALIDATE=1 checks a call's device metadata on the host and refuses a bad pass before anything is
launched (no launch counted, the device error word untouched); a good pass gives the same bits either way."""
import pytest
import torch

from continuous_batching_paged_ragged_gb300 import pkv, synth, workload

pytestmark = pytest.mark.gpu


def _setup():
    batch = synth.custom_batch(synth.Shape(1, 12, 2, 128), [300, 40, 0, 700], [1, 3, 20, 1], seed=19)
    pool = workload.make_pool(batch)
    workload.prefill_cache(pool, batch, [0])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0])
    torch.cuda.synchronize()
    return batch, pool, ds, qs[0], ks[0], vs[0]


def _refused(fn, status):
    with pytest.raises(pkv.PkvError) as e:
        fn()
    assert e.value.status == status and "PKV_VALIDATE" in str(e.value)


def test_good_pass_same_bits_with_and_without_validation(cuda, built, monkeypatch):
    batch, pool, ds, q, k, v = _setup()
    outs = []
    for flag in ("0", "1"):
        monkeypatch.setenv("PKV_VALIDATE", flag)
        out = torch.empty_like(q)
        attn = workload.Attention(pool, ds)
        attn.plan()
        attn.run_append(0, q, k, v, out)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert pool.check() == 0


def test_bad_metadata_refused_before_launch(cuda, built, monkeypatch):
    batch, pool, ds, q, k, v = _setup()
    monkeypatch.setenv("PKV_VALIDATE", "1")
    out = torch.empty_like(q)
    attn = workload.Attention(pool, ds)
    attn.plan()
    d = ds
    # a block id past the pool, inside a row's context
    bad_bt = d.block_tables.clone()
    bad_bt[3, 5] = batch.num_blocks + 7
    _refused(lambda: pkv.pkv_attention(pool.handle, 0, q, bad_bt, d.max_blocks, d.context_lens, d.query_start_loc,
                                       d.num_seqs, d.num_tokens, out, attn.workspace, attn.ws_bytes),
             pkv.PKV_ERR_OUT_OF_RANGE)
    assert pkv.pkv_last_launch_count(pool.handle) == 0
    # a slot past the pool
    bad_slots = d.slot_mapping.clone()
    bad_slots[2] = batch.num_blocks * 16
    _refused(lambda: pkv.pkv_append(pool.handle, 0, k, v, bad_slots, d.num_tokens), pkv.PKV_ERR_OUT_OF_RANGE)
    _refused(lambda: pkv.pkv_attention_append(pool.handle, 0, q, k, v, bad_slots, d.block_tables, d.max_blocks,
                                              d.context_lens, d.query_start_loc, d.num_seqs, d.num_tokens, out,
                                              attn.workspace, attn.ws_bytes), pkv.PKV_ERR_OUT_OF_RANGE)
    # query_start_loc decreasing, and a context longer than the block table allows
    bad_qsl = d.query_start_loc.clone()
    bad_qsl[2] = 0
    _refused(lambda: pkv.pkv_attention_plan(pool.handle, d.context_lens, bad_qsl, d.num_seqs, d.num_tokens,
                                            d.max_blocks, attn.workspace, attn.ws_bytes), pkv.PKV_ERR_INVALID_ARG)
    bad_ctx = d.context_lens.clone()
    bad_ctx[0] = d.max_blocks * 16 + 1
    _refused(lambda: pkv.pkv_attention_plan(pool.handle, bad_ctx, d.query_start_loc, d.num_seqs, d.num_tokens,
                                            d.max_blocks, attn.workspace, attn.ws_bytes), pkv.PKV_ERR_INVALID_ARG)
    _refused(lambda: pkv.pkv_slot_mapping(pool.handle, bad_bt, d.max_blocks, d.context_lens, d.query_start_loc,
                                          d.num_seqs, d.num_tokens, torch.empty_like(d.slot_mapping)),
             pkv.PKV_ERR_OUT_OF_RANGE)
    _refused(lambda: pkv.pkv_attention_noalloc(pool.handle, 0, q, bad_bt, d.max_blocks, d.context_lens,
                                               d.query_start_loc, d.num_seqs, d.num_tokens, out),
             pkv.PKV_ERR_OUT_OF_RANGE)
    torch.cuda.synchronize()
    assert pool.check() == 0   # nothing ran: the kernels' own range checks never saw the bad values


def test_two_workspaces_planned_on_one_pool_both_run(cuda, built):
    """Plans live per workspace: planning a second workspace leaves the first one's plan valid."""
    batch, pool, ds, q, k, v = _setup()
    pkv.pkv_append(pool.handle, 0, k, v, ds.slot_mapping, ds.num_tokens)
    a, b = workload.Attention(pool, ds), workload.Attention(pool, ds)
    a.plan()
    b.plan()
    out_a, out_b = torch.empty_like(q), torch.empty_like(q)
    a.run(0, q, out_a)                       # planned before b: still valid
    b.run(0, q, out_b)
    a.run(0, q, out_a)
    torch.cuda.synchronize()
    assert pool.check() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_stale_plan_refused_when_contents_change(cuda, built, monkeypatch):
    """Under PKV_VALIDATE=1 a pass whose context_lens / query_start_loc were rewritten in place after the plan
    (same pointers, same sizes) is refused before anything is launched; a new plan makes it run again."""
    batch, pool, ds, q, k, v = _setup()
    monkeypatch.setenv("PKV_VALIDATE", "1")
    attn = workload.Attention(pool, ds)
    attn.plan()
    out = torch.empty_like(q)
    attn.run_append(0, q, k, v, out)
    torch.cuda.synchronize()
    saved = ds.context_lens.clone()
    ds.context_lens[0] -= 1                  # still a valid row, but not the pass the plan was built for
    torch.cuda.synchronize()
    with pytest.raises(pkv.PkvError) as e:
        attn.run(0, q, out)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG and "changed since" in str(e.value)
    assert pkv.pkv_last_launch_count(pool.handle) == 0
    with pytest.raises(pkv.PkvError) as e:
        attn.run_append(0, q, k, v, out)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    ds.context_lens.copy_(saved)
    attn.run(0, q, out)                      # the contents match the plan again
    attn.plan()
    attn.run(0, q, out)
    torch.cuda.synchronize()
    assert pool.check() == 0
