"""The C++ host scheduler (pkv_sched_*) against the oracle's restatement, step by step, bit for bit."""
import json
import os

import numpy as np
import pytest

import oracle
from continuous_batching_paged_ragged_gb300 import synth
from continuous_batching_paged_ragged_gb300.pkv import PkvError, Scheduler

TRACES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sched_traces.json")))["traces"]


def _compare_runs(native, ref, max_steps=100000):
    n = 0
    while not ref.done():
        a = native.step()
        b = ref.step()
        assert a["req_ids"].tolist() == b.req_ids.tolist()
        assert np.array_equal(a["q_lens"], b.q_lens)
        assert np.array_equal(a["context_lens"], b.context_lens)
        assert np.array_equal(a["block_tables"], b.block_tables)
        assert np.array_equal(a["slot_mapping"], b.slot_mapping)
        assert a["query_start_loc"].tolist() == [0] + np.cumsum(b.q_lens).tolist()
        assert a["preempted"] == b.preempted and a["admitted"] == b.admitted
        assert sorted(a["finished"]) == sorted(b.finished)
        n += 1
        assert n < max_steps
    assert native.done()
    st = native.stats()
    assert st["steps"] == ref.steps and st["preemptions"] == ref.num_preemptions
    assert st["recomputed_tokens"] == ref.recomputed_tokens
    assert st["recomputed_prompt_tokens"] == ref.recomputed_prompt_tokens
    assert st["max_batch"] == ref.max_batch and st["batch_sum"] == ref.batch_sum
    assert (st["live_tokens"], st["held_slots"]) == (ref.live_tokens, ref.held_slots)
    assert st["prefix_hit_tokens"] == ref.prefix_hit_tokens
    assert native.free_list() == list(ref.free)
    return st


_ALLOC = {oracle.ON_DEMAND: 0, oracle.RESERVE: 1}
_UNIT = {oracle.PASS: 0, oracle.REQUEST: 1}


@pytest.mark.parametrize("trace", TRACES, ids=[t["name"] for t in TRACES])
def test_hand_worked_traces(built, trace):
    alloc, unit = trace.get("alloc", oracle.ON_DEMAND), trace.get("unit", oracle.PASS)
    pc = trace.get("prefix_caching", False)
    native = Scheduler(trace["max_num_seqs"], trace["token_budget"], trace["block_size"], len(trace["free_blocks"]),
                       trace["free_blocks"], alloc=_ALLOC[alloc], unit=_UNIT[unit], prefix_caching=pc)
    ref = oracle.Scheduler(trace["max_num_seqs"], trace["token_budget"], trace["block_size"], trace["free_blocks"],
                           alloc, unit, pc)
    for req in trace["requests"]:
        native.add(*req)
        ref.add(*req)
    _compare_runs(native, ref)


@pytest.mark.parametrize("alloc,unit,factor,num_blocks,cap", [
    (oracle.RESERVE, oracle.PASS, 1.0, 5000, 256), (oracle.RESERVE, oracle.PASS, 4.0, 5000, 256),
    (oracle.ON_DEMAND, oracle.REQUEST, 1.0, 20000, 64), (oracle.RESERVE, oracle.REQUEST, 2.0, 20000, 64),
    (oracle.ON_DEMAND, oracle.REQUEST, 1.0, 5000, 256)])
def test_policy_variants_match_oracle(built, alloc, unit, factor, num_blocks, cap):
    reqs = synth.trace_requests(0)
    perm = synth.block_permutation(num_blocks, 0)
    native = Scheduler(cap, 8192, 16, num_blocks, perm, alloc=_ALLOC[alloc], unit=_UNIT[unit])
    ref = oracle.Scheduler(cap, 8192, 16, perm, alloc, unit)
    for r in reqs:
        d = int(round(factor * r.max_output))
        native.add(r.req_id, r.prompt_len, r.max_output, d)
        ref.add(r.req_id, r.prompt_len, r.max_output, d)
    st = _compare_runs(native, ref)
    if alloc == oracle.RESERVE:
        assert st["preemptions"] == 0


@pytest.mark.parametrize("num_blocks,cap", [(20000, 256), (20000, 64), (5000, 256), (5000, 64), (1500, 512)])
def test_trace_workload_matches_oracle(built, num_blocks, cap):
    """The scheduler-driven trace (256 requests, lognormal prompts, U[50,781] outputs, budget 8192)."""
    reqs = synth.trace_requests(0)
    perm = synth.block_permutation(num_blocks, 0)
    native = Scheduler(cap, 8192, 16, num_blocks, perm)
    ref = oracle.Scheduler(cap, 8192, 16, perm)
    for r in reqs:
        native.add(r.req_id, r.prompt_len, r.max_output)
        ref.add(r.req_id, r.prompt_len, r.max_output)
    st = _compare_runs(native, ref)
    if num_blocks == 5000 and cap == 256:
        assert st["preemptions"] > 0


def test_argument_errors(built):
    with pytest.raises(PkvError):
        Scheduler(0, 8192, 16, 100)
    with pytest.raises(PkvError):
        Scheduler(4, 8192, 16, 100, alloc=7)
    r = Scheduler(4, 64, 16, 4, alloc=1)
    with pytest.raises(PkvError):
        r.add(1, 10, 2, 1)          # declared below the real output budget
    with pytest.raises(PkvError):
        r.add(1, 10, 2, 60)         # a reservation of 5 blocks never fits 4
    r.add(1, 10, 2, 20)
    with pytest.raises(PkvError):
        Scheduler(4, 8192, 16, 3, [0, 0, 1])
    s = Scheduler(4, 64, 16, 4)
    with pytest.raises(PkvError):
        s.add(1, 100, 1)            # can never fit 4 blocks of 16
    s.add(1, 10, 2)
    with pytest.raises(PkvError):
        s.add(1, 10, 2)             # duplicate id
    with pytest.raises(PkvError):
        s.abort(99)
    with pytest.raises(PkvError):
        s.set_max_num_seqs(0)


def test_abort_and_drain(built):
    reqs = synth.trace_requests(1, n=40)
    s = Scheduler(32, 8192, 16, 4000, synth.block_permutation(4000, 1))
    for r in reqs:
        s.add(r.req_id, r.prompt_len, r.max_output)
    for _ in range(3):
        s.step()
    s.abort(reqs[0].req_id)
    s.abort(reqs[35].req_id)        # still waiting
    st = s.stats()
    assert st["running"] == 31 and st["waiting"] == 40 - 32 - 1
    s.set_max_num_seqs(4)
    rows = s.step()
    assert len(rows["req_ids"]) == 31 and rows["preempted"] == []
    while not s.done():
        s.step()
    assert s.stats()["free_blocks"] == 4000


@pytest.mark.parametrize("num_blocks,cap", [(5000, 256), (3000, 64), (1500, 512)])
def test_prefix_caching_matches_oracle(built, num_blocks, cap):
    reqs = synth.trace_requests(0)
    perm = synth.block_permutation(num_blocks, 0)
    native = Scheduler(cap, 8192, 16, num_blocks, perm, prefix_caching=True)
    ref = oracle.Scheduler(cap, 8192, 16, perm, prefix_caching=True)
    for r in reqs:
        native.add(r.req_id, r.prompt_len, r.max_output)
        ref.add(r.req_id, r.prompt_len, r.max_output)
    st = _compare_runs(native, ref)
    assert st["prefix_hit_tokens"] > 0


def _compare_step(a, b):
    assert a["req_ids"].tolist() == b.req_ids.tolist()
    assert np.array_equal(a["q_lens"], b.q_lens) and np.array_equal(a["context_lens"], b.context_lens)
    assert np.array_equal(a["block_tables"], b.block_tables)
    assert np.array_equal(a["slot_mapping"], b.slot_mapping)
    assert a["preempted"] == b.preempted and a["admitted"] == b.admitted
    assert sorted(a["finished"]) == sorted(b.finished)


@pytest.mark.parametrize("seed", range(40))
def test_random_workloads_with_arrivals_aborts_and_cap_changes(built, seed):
    """Small random pools (heavy preemption), budgets, block sizes and every policy; requests arriving during
    the run, aborts of live requests and max_num_seqs changes between passes: the C++ scheduler and the oracle
    agree pass by pass, and at the end every block is back in the same free-list order."""
    rng = np.random.default_rng(1000 + seed)
    bs = int(rng.choice([1, 4, 16]))
    nb = int(rng.integers(8, 200))
    budget = int(rng.integers(4, 300))
    cap = int(rng.integers(1, 24))
    alloc = [oracle.ON_DEMAND, oracle.RESERVE][int(rng.integers(0, 2))]
    unit = [oracle.PASS, oracle.REQUEST][int(rng.integers(0, 2))]
    pc = alloc == oracle.ON_DEMAND and bool(rng.integers(0, 2))
    perm = [int(x) for x in rng.permutation(nb)]
    native = Scheduler(cap, budget, bs, nb, perm, alloc=_ALLOC[alloc], unit=_UNIT[unit], prefix_caching=pc)
    ref = oracle.Scheduler(cap, budget, bs, perm, alloc, unit, pc)
    next_id, live = 0, set()

    def arrive():
        nonlocal next_id
        room = nb * bs
        prompt = int(rng.integers(1, max(2, room // 3)))
        out = int(rng.integers(1, max(2, room // 4)))
        declared = out + int(rng.integers(0, 3 * out + 1))
        worst = prompt + (declared if alloc == oracle.RESERVE else out)
        if -(-worst // bs) > nb:
            return
        native.add(next_id, prompt, out, declared)
        ref.add(next_id, prompt, out, declared)
        live.add(next_id)
        next_id += 1

    for _ in range(int(rng.integers(1, 12))):
        arrive()
    for n in range(20000):
        if ref.done() and n > 60:
            break
        if n < 60:
            r = rng.random()
            if r < 0.25:
                arrive()
            elif r < 0.30 and live:
                victim = int(rng.choice(sorted(live)))
                native.abort(victim)
                ref.abort(victim)
                live.discard(victim)
            elif r < 0.35:
                c = int(rng.integers(1, 24))
                native.set_max_num_seqs(c)
                ref.set_max_num_seqs(c)
        a, b = native.step(), ref.step()
        _compare_step(a, b)
        live -= set(a["finished"])
    assert ref.done() and native.done()
    st = native.stats()
    assert (st["steps"], st["preemptions"], st["recomputed_tokens"]) == (ref.steps, ref.num_preemptions,
                                                                        ref.recomputed_tokens)
    assert (st["live_tokens"], st["held_slots"], st["prefix_hit_tokens"]) == (ref.live_tokens, ref.held_slots,
                                                                             ref.prefix_hit_tokens)
    assert native.free_list() == list(ref.free) and len(ref.free) == nb
