"""Pins for the scheduler oracle: hand-worked traces and the behaviour rules the pages state."""
import json
import os

import numpy as np
import pytest

import oracle
from continuous_batching_paged_ragged_gb300 import synth

TRACES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sched_traces.json")))["traces"]


def _run(trace):
    s = oracle.Scheduler(trace["max_num_seqs"], trace["token_budget"], trace["block_size"], trace["free_blocks"],
                         trace.get("alloc", oracle.ON_DEMAND), trace.get("unit", oracle.PASS),
                         trace.get("prefix_caching", False))
    for req in trace["requests"]:
        s.add(*req)
    steps = []
    while not s.done():
        steps.append(s.step())
        assert len(steps) < 1000
    return s, steps


@pytest.mark.parametrize("trace", TRACES, ids=[t["name"] for t in TRACES])
def test_hand_worked_trace(trace):
    s, steps = _run(trace)
    assert len(steps) == len(trace["steps"])
    for got, want in zip(steps, trace["steps"]):
        rows = [[int(got.req_ids[b]), int(got.q_lens[b]), int(got.context_lens[b]),
                 [int(x) for x in got.block_tables[b] if x >= 0]] for b in range(len(got.req_ids))]
        assert rows == [r[:4] for r in want["rows"]]
        assert got.slot_mapping.tolist() == [x for r in want["rows"] for x in r[4]]
        assert got.preempted == want["preempted"]
        assert sorted(got.finished) == sorted(want["finished"])
    assert list(s.free) == trace["final_free"]
    assert s.num_preemptions == trace["preemptions"]
    assert s.recomputed_tokens == trace["recomputed"]
    if "live_tokens" in trace:
        assert (s.live_tokens, s.held_slots) == (trace["live_tokens"], trace["held_slots"])
    if "prefix_hit_tokens" in trace:
        assert s.prefix_hit_tokens == trace["prefix_hit_tokens"]


def _trace_sched(num_blocks, cap, seed=0, n=64):
    reqs = synth.trace_requests(seed, n=n)
    s = oracle.Scheduler(cap, 8192, 16, synth.block_permutation(num_blocks, seed))
    for r in reqs:
        s.add(r.req_id, r.prompt_len, r.max_output)
    return s, reqs


def test_invariants_along_a_pressured_trace():
    """Block conservation, budget, per-row block counts, exactly one output per finished token stream."""
    s, reqs = _trace_sched(num_blocks=600, cap=64)
    seen_preempt = 0
    while not s.done():
        running_before = list(s.running)
        rows = s.step()
        assert int(rows.q_lens.sum()) <= s.token_budget
        held = [b for r in s.running for b in r.blocks] + [b for r in s.waiting for b in r.blocks]
        assert len(held) == len(set(held))
        assert len(held) + len(s.free) == s.num_blocks
        assert not set(held) & set(s.free)
        for r in s.running:
            assert len(r.blocks) == -(-r.num_computed // 16)
        for r in s.waiting:
            assert r.blocks == [] and r.num_computed == 0
        if rows.preempted:
            seen_preempt += 1
            assert rows.admitted == []                      # a preempting pass admits nobody
            # victims are the newest running requests, taken from the back
            tail = [r.req_id for r in running_before][-len(rows.preempted):][::-1]
            assert rows.preempted == tail
        assert s.steps < 100000
    assert seen_preempt > 0
    assert all(r.num_output == r.max_output for r in s.by_id.values())


def test_preempted_request_restarts_from_zero():
    s, _ = _trace_sched(num_blocks=600, cap=64)
    while not s.done():
        before = {r.req_id: r.num_output for r in s.running}
        rows = s.step()
        for rid in rows.preempted:
            r = s.by_id[rid]
            assert r.num_computed == 0 and r.status == "PREEMPTED"
            assert r.num_output == before[rid]                # generated outputs are kept, K/V recomputed
        # a readmitted request's first row re-prefills prompt + outputs from position 0
        for b, rid in enumerate(rows.req_ids.tolist()):
            if rid in rows.admitted:
                assert rows.context_lens[b] == rows.q_lens[b]


def test_cap_gates_admission_only_and_lowering_drains():
    s, _ = _trace_sched(num_blocks=20000, cap=32)
    for _ in range(5):
        s.step()
    assert len(s.running) == 32
    s.set_max_num_seqs(8)
    rows = s.step()
    assert len(rows.req_ids) == 32 and rows.preempted == []   # nobody evicted
    while len(s.running) > 8:
        rows = s.step()
        assert rows.admitted == []
    with pytest.raises(ValueError):
        s.set_max_num_seqs(0)


def test_decode_wants_one_token_and_prefill_is_chunked():
    s = oracle.Scheduler(8, 100, 16, list(range(100)))
    s.add(0, 250, 3)
    r1 = s.step()
    r2 = s.step()
    r3 = s.step()
    assert (r1.q_lens.tolist(), r2.q_lens.tolist(), r3.q_lens.tolist()) == ([100], [100], [50])
    r4 = s.step()
    assert r4.q_lens.tolist() == [1] and r4.context_lens.tolist() == [251]


def test_abort_frees_every_block():
    s, _ = _trace_sched(num_blocks=3000, cap=64)
    for _ in range(4):
        s.step()
    victim = s.running[3].req_id
    s.abort(victim)
    held = [b for r in s.running for b in r.blocks]
    assert len(held) + len(s.free) == s.num_blocks
    assert victim not in [r.req_id for r in s.running]


def test_no_preemption_when_pool_is_large():
    s, reqs = _trace_sched(num_blocks=20000, cap=256, n=256)
    while not s.done():
        s.step()
    assert s.num_preemptions == 0
    assert s.max_batch == 256


# --- allocation and scheduling-unit variants ("The allocator is the other half", "The boundary: when this
# is worth nothing"): the orderings the page reports, checked on the trace workload --------------------

def _policy_run(alloc, unit, declared=1.0, num_blocks=5000, cap=256, spread=True):
    reqs = synth.trace_requests(0) if spread else synth.trace_requests(0, out_lo=256, out_hi=256)
    s = oracle.Scheduler(cap, 8192, 16, synth.block_permutation(num_blocks, 0), alloc, unit)
    for r in reqs:
        s.add(r.req_id, r.prompt_len, r.max_output, int(round(declared * r.max_output)))
    while not s.done():
        s.step()
        assert s.steps < 100000
    assert all(r.num_output == r.max_output for r in s.by_id.values())
    return s


def test_reservation_never_preempts_and_costs_batch_and_live_cache():
    on_demand = _policy_run(oracle.ON_DEMAND, oracle.PASS)
    assert on_demand.num_preemptions > 0                       # this pool is under pressure on demand
    live = []
    batches = []
    for factor in (1.0, 2.0, 4.0, 8.0):
        r = _policy_run(oracle.RESERVE, oracle.PASS, declared=factor)
        assert r.num_preemptions == 0 and r.recomputed_tokens == 0
        live.append(r.live_tokens / r.held_slots)
        batches.append(r.max_batch)
    # declaring more than is used lowers the live share of held cache and the largest batch
    assert all(a > b for a, b in zip(live, live[1:])), live
    assert all(a >= b for a, b in zip(batches, batches[1:])) and batches[0] > batches[-1], batches
    # on demand, held cache is live up to the partly filled last block of each request; a reservation holds
    # a request's whole output from admission, so even an exact declaration (1x) leaves part of it empty
    # until the outputs arrive -- how much depends on the output/prompt mix (long outputs here)
    assert on_demand.live_tokens / on_demand.held_slots > 0.95 > live[0] > 0.5
    assert on_demand.max_batch > batches[0]


def test_request_level_scheduling_waits_for_the_slowest_member():
    for alloc in (oracle.ON_DEMAND, oracle.RESERVE):
        per_pass = _policy_run(alloc, oracle.PASS, num_blocks=20000, cap=64)
        per_req = _policy_run(alloc, oracle.REQUEST, num_blocks=20000, cap=64)
        assert per_req.tokens_scheduled == per_pass.tokens_scheduled   # the same work...
        assert per_req.steps > 1.3 * per_pass.steps                    # ...in many more passes
        # with equal outputs the batch ends together and the unit barely matters
        eq_pass = _policy_run(alloc, oracle.PASS, num_blocks=20000, cap=64, spread=False)
        eq_req = _policy_run(alloc, oracle.REQUEST, num_blocks=20000, cap=64, spread=False)
        assert eq_req.steps <= 1.1 * eq_pass.steps


def test_request_level_admits_only_while_the_batch_forms():
    s = oracle.Scheduler(8, 8192, 16, list(range(4000)), oracle.ON_DEMAND, oracle.REQUEST)
    for r in synth.trace_requests(3, n=40):
        s.add(r.req_id, r.prompt_len, r.max_output)
    closed = False
    while not s.done():
        running_before = len(s.running)
        rows = s.step()
        if running_before and closed:
            assert rows.admitted == []                # a running batch that has lost a member takes nobody
        closed = bool(rows.finished) or (closed and bool(s.running))


# --- prefix caching of recompute after preemption ("What the scheduler does on one step": the recompute is
# "partly refundable ... a race, not a guarantee") ------------------------------------------------------

def test_prefix_hits_are_the_requests_own_untouched_blocks():
    reqs = synth.trace_requests(0)
    s = oracle.Scheduler(256, 8192, 16, synth.block_permutation(5000, 0), prefix_caching=True)
    for r in reqs:
        s.add(r.req_id, r.prompt_len, r.max_output)
    held_at_preemption = {}
    hits_seen = 0
    while not s.done():
        blocks_before = {r.req_id: list(r.blocks) for r in s.running}
        hits_before = s.prefix_hit_tokens
        rows = s.step()
        for rid in rows.preempted:
            held_at_preemption[rid] = blocks_before[rid]
        for b, rid in enumerate(rows.req_ids.tolist()):
            if rid in rows.admitted and rid in held_at_preemption:
                start = int(rows.context_lens[b] - rows.q_lens[b])
                assert start % 16 == 0 and start < int(rows.context_lens[b])
                reused = rows.block_tables[b][: start // 16].tolist()
                # a prefix of the blocks it held when it was preempted, in the same logical order
                assert reused == held_at_preemption[rid][: len(reused)]
                hits_seen += len(reused)
        assert s.prefix_hit_tokens - hits_before == 16 * sum(
            int(rows.context_lens[b] - rows.q_lens[b]) // 16 for b, rid in enumerate(rows.req_ids.tolist())
            if rid in rows.admitted)
    assert hits_seen > 0 and 0 < s.prefix_hit_tokens <= s.recomputed_tokens
    assert all(r.num_output == r.max_output for r in s.by_id.values())


def test_prefix_caching_only_removes_recompute():
    """The same workload with and without the cache: the same outputs, fewer prefill tokens."""
    runs = []
    for pc in (False, True):
        s = oracle.Scheduler(256, 8192, 16, synth.block_permutation(5000, 0), prefix_caching=pc)
        for r in synth.trace_requests(0):
            s.add(r.req_id, r.prompt_len, r.max_output)
        while not s.done():
            s.step()
        runs.append(s)
    off, on = runs
    assert on.prefix_hit_tokens > 0 and off.prefix_hit_tokens == 0
    assert on.tokens_scheduled < off.tokens_scheduled
    with pytest.raises(ValueError):
        oracle.Scheduler(4, 64, 16, list(range(8)), oracle.RESERVE, prefix_caching=True)
