"""Scheduler oracle: a plain restatement of the per-pass schedule() the pages describe.

Test infrastructure only (see the package docstring).  Follows "Continuous Batching Is Not a Bigger
Batch" (deepconcepts.dev), section "What the scheduler does on one step":

* Phase one walks the running requests in arrival order.  Each wants num_tokens - num_computed_tokens
  (one while decoding, the rest of the prompt while prefilling), capped by the pass's token budget:
  chunked prefill, no separate prefill phase.
* For each it allocates the blocks those tokens need.  On failure it pops the LAST running request
  (the newest), frees its blocks, marks it PREEMPTED, resets num_computed_tokens to 0 and prepends it to
  the waiting queue; then it retries.  If the popped request is the one being scheduled, phase one ends
  (reading: the pages show only the pop; this is the plain consequence).
* Phase two admits from the head of the waiting queue, only if the pass preempted nobody, while the
  token budget lasts and while the running count is below max_num_seqs -- the cap is read only there
  ("Saturation and Capacity", section "Runtime capacity control": lowering it drains, never evicts).
* Blocks are 16-token units handed out on demand from a free list
  (same page, sections "Where the batch size actually comes from" and "The allocator is the other half").

Readings where the pages are silent (listed in the design notes): the waiting queue is strict FIFO with
head-of-line blocking (an unallocatable head stops admission for the pass); a pass that computes a
request's last known token yields one output token; a request finishes when its outputs reach its
budget and frees its blocks the same pass; freed blocks go to the tail of the free list in block-table
order; the token budget is shared by both phases.

Two variants from the same page, section "The allocator is the other half" and "The boundary: when this
is worth nothing":

* Allocation RESERVE (Orca): a request is admitted only if its worst case fits -- the page's
  n_rsrv + max_tokens <= n_slots, here counted in blocks: ceil((prompt + declared output) / block_size)
  free blocks, all taken at admission and returned when the request finishes.  An admitted request can
  never run out of cache, so this policy never preempts.  The declared output is what the client claims
  (at least its real budget).
* Unit REQUEST (static batching): a batch forms when nothing runs; requests join it while it forms, and
  it stops taking members at the first pass in which one of them finishes -- from then on it runs to its
  slowest member.  (Reading: with chunked prefill a batch cannot form in a single pass; "forms the batch
  once" is read as "admits only until its first member completes".)
* Reported with both: the share of held cache that holds a token, summed over passes after each pass --
  tokens whose K/V a running request holds over the slots of the blocks it holds.

And prefix caching for recompute after preemption (same page, "What the scheduler does on one step": the
recompute "is partly refundable: if prefix caching is on and the freed blocks have not been evicted from
the cache by the time the request comes back, the recompute is a cache hit instead"):

* When a request is preempted, each of its full blocks (all 16 slots computed) stays registered as holding
  that request's block j while it sits in the free list; handing the block to any request evicts it.  Its
  blocks return to the free list last block first, so that its prefix is evicted last (reading).
* When the request is admitted again, it takes back the longest prefix j = 0, 1, ... of its still
  registered blocks (leaving at least one token to compute) and counts those tokens as computed; the rest
  is recomputed.  A hit the remaining allocation cannot accompany is not taken (head-of-line blocking as
  usual).  On demand only: a reserving scheduler never preempts.
"""
from __future__ import annotations

import collections
import dataclasses
from typing import Deque, List, Optional, Sequence

import numpy as np

from .paging import slot_of

WAITING, RUNNING, PREEMPTED, FINISHED = "WAITING", "RUNNING", "PREEMPTED", "FINISHED"
ON_DEMAND, RESERVE = "on_demand", "reserve"   # block allocation policies
PASS, REQUEST = "pass", "request"             # units of scheduling


@dataclasses.dataclass(eq=False)
class Request:
    req_id: int
    prompt_len: int
    max_output: int
    declared_output: int = 0      # output the client claims (RESERVE sizes the reservation by it)
    num_computed: int = 0
    num_output: int = 0
    status: str = WAITING
    blocks: List[int] = dataclasses.field(default_factory=list)

    @property
    def num_tokens(self) -> int:
        """Tokens whose K/V the request needs: the prompt plus outputs generated so far."""
        return self.prompt_len + self.num_output


@dataclasses.dataclass
class StepRows:
    """The ragged batch one pass hands to the GPU, rows in scheduling order."""
    req_ids: np.ndarray        # int64 [B]
    q_lens: np.ndarray         # int32 [B]
    context_lens: np.ndarray   # int32 [B]  num_computed before the pass + q_len
    block_tables: np.ndarray   # int32 [B, max_blocks], -1 padded
    slot_mapping: np.ndarray   # int64 [T]
    preempted: List[int]
    admitted: List[int]
    finished: List[int]


class Scheduler:
    def __init__(self, max_num_seqs: int, token_budget: int, block_size: int, free_blocks: Sequence[int],
                 alloc: str = ON_DEMAND, unit: str = PASS, prefix_caching: bool = False):
        if max_num_seqs < 1:
            raise ValueError("max_num_seqs must be at least 1")
        if token_budget < 1 or block_size < 1:
            raise ValueError("token_budget and block_size must be positive")
        if alloc not in (ON_DEMAND, RESERVE) or unit not in (PASS, REQUEST):
            raise ValueError("unknown policy")
        if prefix_caching and alloc != ON_DEMAND:
            raise ValueError("prefix caching refunds recompute after preemption; a reserving scheduler never preempts")
        self.alloc = alloc
        self.unit = unit
        self.batch_open = False
        self.prefix_caching = prefix_caching
        self.cached = {}          # (req_id, j) -> a free block still holding that request's full block j
        self.block_key = {}       # block -> (req_id, j) for those blocks
        self.prefix_hit_tokens = 0
        self.max_num_seqs = max_num_seqs
        self.token_budget = token_budget
        self.block_size = block_size
        self.num_blocks = len(free_blocks)
        self.free: Deque[int] = collections.deque(int(b) for b in free_blocks)
        self.running: List[Request] = []
        self.waiting: Deque[Request] = collections.deque()
        self.by_id = {}
        # statistics
        self.steps = 0
        self.num_preemptions = 0
        self.recomputed_tokens = 0
        self.recomputed_prompt_tokens = 0
        self.max_batch = 0
        self.batch_sum = 0
        self.tokens_scheduled = 0
        self.live_tokens = 0      # summed over passes: tokens held by running requests after the pass
        self.held_slots = 0       # summed over passes: slots of the blocks running requests hold

    # --- allocator -----------------------------------------------------------------------------------
    def _reservation(self, req: Request) -> int:
        return -(-(req.prompt_len + req.declared_output) // self.block_size)

    def _admit_blocks(self, req: Request, budget: int) -> int:
        """Blocks at admission: the whole reservation (RESERVE), or the request's cached prefix and those its
        first new tokens need.  Returns the new tokens of the pass, 0 if it cannot be admitted."""
        if self.alloc == RESERVE:
            need = self._reservation(req)
            if need > len(self.free):
                return 0
            req.blocks = [self._take() for _ in range(need)]
            return min(req.num_tokens - req.num_computed, budget)
        hits = self._prefix_hits(req)
        start = len(hits) * self.block_size
        num_new = min(req.num_tokens - start, budget)
        need = -(-(start + num_new) // self.block_size) - len(hits)
        if need > len(self.free) - len(hits):
            return 0
        for b in hits:
            self.free.remove(b)
            del self.cached[self.block_key.pop(b)]
        req.blocks = hits
        req.num_computed = start
        self.prefix_hit_tokens += start
        self._allocate(req, num_new)
        return num_new

    def _take(self) -> int:
        """The free list's head; a block handed out no longer holds what it cached."""
        b = self.free.popleft()
        key = self.block_key.pop(b, None)
        if key is not None:
            del self.cached[key]
        return b

    def _allocate(self, req: Request, num_new: int) -> bool:
        need = -(-(req.num_computed + num_new) // self.block_size) - len(req.blocks)
        if need > len(self.free):
            return False
        for _ in range(max(need, 0)):
            req.blocks.append(self._take())
        return True

    def _free(self, req: Request, keep: bool = False) -> None:
        """Return the blocks to the free list's tail; keep=True registers the full ones for prefix caching."""
        if keep and self.prefix_caching:
            for j, b in enumerate(req.blocks):
                if (j + 1) * self.block_size <= req.num_computed:
                    self.cached[(req.req_id, j)] = b
                    self.block_key[b] = (req.req_id, j)
            # last block first: the allocator hands out the free list's head, so the request's prefix --
            # what its readmission can reuse -- is evicted last
            self.free.extend(reversed(req.blocks))
        else:
            self.free.extend(req.blocks)
        req.blocks = []

    def _prefix_hits(self, req: Request) -> List[int]:
        hits = []
        while self.prefix_caching and req.num_computed == 0:
            b = self.cached.get((req.req_id, len(hits)))
            if b is None or (len(hits) + 1) * self.block_size > req.num_tokens - 1:
                break
            hits.append(b)
        return hits

    # --- requests ------------------------------------------------------------------------------------
    def add(self, req_id: int, prompt_len: int, max_output: int, declared_output: Optional[int] = None) -> None:
        if prompt_len < 1 or max_output < 1:
            raise ValueError("prompt_len and max_output must be positive")
        declared = max_output if declared_output is None else declared_output
        if declared < max_output:
            raise ValueError("the declared output cannot be below the real budget")
        req = Request(req_id, prompt_len, max_output, declared)
        self.by_id[req_id] = req
        self.waiting.append(req)

    def abort(self, req_id: int) -> None:
        """A cancelled request leaves no blocks behind ("An advertised batch limit proves nothing until
        sampled", section "Counting jobs while they run")."""
        req = self.by_id.pop(req_id)
        if req in self.running:
            self.running.remove(req)
        if req in self.waiting:
            self.waiting.remove(req)
        self._free(req)
        req.status = FINISHED

    def set_max_num_seqs(self, n: int) -> None:
        if n < 1:
            raise ValueError("max_num_seqs must be at least 1")
        self.max_num_seqs = n

    def done(self) -> bool:
        return not self.running and not self.waiting

    # --- one pass ------------------------------------------------------------------------------------
    def step(self) -> StepRows:
        budget = self.token_budget
        scheduled = []          # (request, num_new, num_computed before the pass)
        preempted: List[Request] = []
        admitted: List[int] = []
        if self.unit == REQUEST and not self.running:
            self.batch_open = True          # nothing runs: a new batch forms

        # phase one: running requests, arrival order
        i = 0
        while i < len(self.running) and budget > 0:
            req = self.running[i]
            num_new = min(req.num_tokens - req.num_computed, budget)
            schedulable = True
            while not self._allocate(req, num_new):
                victim = self.running.pop()
                self._free(victim, keep=True)
                victim.status = PREEMPTED
                self.recomputed_tokens += victim.num_computed
                self.recomputed_prompt_tokens += min(victim.num_computed, victim.prompt_len)
                victim.num_computed = 0
                self.waiting.appendleft(victim)
                preempted.append(victim)
                if victim is req:
                    schedulable = False
                    break
            if not schedulable:
                break
            scheduled.append((req, num_new, req.num_computed))
            budget -= num_new
            i += 1

        # phase two: admission, only when nothing was preempted (and, per request, while the batch forms)
        if not preempted and (self.unit == PASS or self.batch_open):
            while self.waiting and budget > 0:
                if len(self.running) >= self.max_num_seqs:
                    break
                req = self.waiting[0]
                num_new = self._admit_blocks(req, budget)
                if num_new == 0:
                    break
                self.waiting.popleft()
                req.status = RUNNING
                self.running.append(req)
                admitted.append(req.req_id)
                scheduled.append((req, num_new, req.num_computed))
                budget -= num_new

        rows = self._rows(scheduled)
        rows.preempted = [r.req_id for r in preempted]
        rows.admitted = admitted
        self.num_preemptions += len(preempted)

        # the forward pass has run: advance each scheduled request
        finished = []
        for req, num_new, _ in scheduled:
            req.num_computed += num_new
            if req.num_computed == req.num_tokens:
                req.num_output += 1
                if req.num_output >= req.max_output:
                    self.running.remove(req)
                    self._free(req)
                    req.status = FINISHED
                    finished.append(req.req_id)
        rows.finished = finished
        if finished:
            self.batch_open = False             # a member completed: the batch takes no more
        self.live_tokens += sum(r.num_computed for r in self.running)
        self.held_slots += sum(len(r.blocks) for r in self.running) * self.block_size
        self.steps += 1
        self.max_batch = max(self.max_batch, len(scheduled))
        self.batch_sum += len(scheduled)
        self.tokens_scheduled += int(rows.q_lens.sum()) if len(scheduled) else 0
        return rows

    def _rows(self, scheduled) -> StepRows:
        B = len(scheduled)
        bs = self.block_size
        # a row's table lists the blocks its context occupies (a reservation may hold more)
        used = [-(-(start + num_new) // bs) for _, num_new, start in scheduled]
        max_blocks = max(used + [1])
        req_ids = np.zeros(B, dtype=np.int64)
        q_lens = np.zeros(B, dtype=np.int32)
        ctx = np.zeros(B, dtype=np.int32)
        bt = np.full((B, max_blocks), -1, dtype=np.int32)
        slots = []
        for b, (req, num_new, start) in enumerate(scheduled):
            req_ids[b] = req.req_id
            q_lens[b] = num_new
            ctx[b] = start + num_new
            bt[b, : used[b]] = req.blocks[: used[b]]
            for p in range(start, start + num_new):
                slots.append(slot_of(req.blocks, p, bs))
        return StepRows(req_ids, q_lens, ctx, bt, np.asarray(slots, dtype=np.int64), [], [], [])
