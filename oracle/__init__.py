"""CPU oracle for the paged ragged attention step -- TEST INFRASTRUCTURE, not part of the product.

Plain, slow, obviously correct NumPy code in float64, single-threaded in spirit (no blocking, no fusion,
no reordering beyond the definitions it restates).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It shares no code with the
CUDA path: it never imports the ``continuous_batching_paged_ragged_gb300`` package and that package never
imports it.  Inputs reach it as arrays built by the seeded generator module (``synth``).

Pages it follows (cited by title and section in each function):

* "Continuous Batching Is Not a Bigger Batch" (deepconcepts.dev) -- the per-pass scheduler
  (section "What the scheduler does on one step"), KV sizing and 16-token blocks
  (section "Where the batch size actually comes from"), on-demand paged allocation
  (section "The allocator is the other half").
* "Static batching" (danielfleming.xyz) -- KV bytes per token for Qwen2.5-1.5B (section
  "What I expected") and the motivation for paged, unpadded storage (sections "Ragged batches" and
  "Bottleneck, and what follows").
* "An advertised batch limit proves nothing until sampled" (a8q9.cn) -- long-context KV arithmetic
  (section "Context math sets the ceiling the fields ignore").
* "Saturation and Capacity" (inference-lab) -- max_num_seqs gates admission only and must be >= 1
  (section "Runtime capacity control").
* The 8-bit cache (``oracle.fp8``): quantize the cache when memory is the cap ("Continuous Batching Is
  Not a Bigger Batch", section "Checking it on a real system"); 8-bit KV halves the raw bytes, scales on
  top ("An advertised batch limit proves nothing until sampled", section "Context math sets the ceiling
  the fields ignore").  The E4M3 format is the OCP 8-bit floating point specification's.

Every function here is pinned by a ``-m "not gpu"`` test against something other than itself (a library
routine, a closed form, values the pages print, or brute force); see ``tests/test_oracle_*.py``.
"""
from .attention import attention_row, attention_batch, round_fp16
from .paging import (kv_bytes_per_token, kv_bytes_for_window, pool_blocks_for_bytes, blocks_for_tokens,
                     max_resident_sequences, cache_bytes, slot_of, slot_mapping_for_batch, append_reference)
from . import fp8
from .scheduler import ON_DEMAND, PASS, REQUEST, RESERVE, Request, Scheduler, StepRows

__all__ = [
    "attention_row", "attention_batch", "round_fp16",
    "kv_bytes_per_token", "kv_bytes_for_window", "pool_blocks_for_bytes", "blocks_for_tokens",
    "max_resident_sequences", "cache_bytes", "slot_of", "slot_mapping_for_batch", "append_reference",
    "fp8", "Request", "Scheduler", "StepRows", "ON_DEMAND", "RESERVE", "PASS", "REQUEST",
]
