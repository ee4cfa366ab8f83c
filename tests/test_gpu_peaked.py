"""GPU parity on peaked softmax inputs, on the fp16 and the 8-bit cache.

The seeded generator's values give scores of about N(0, 1), so a row's running maximum settles within its
first keys and every softmax weight sits within a few powers of two of the largest.  These cases push the
arithmetic where that never goes (the oracle's one-hot pin -- a dominant key -- applied to the kernels):

* decode rows with queries scaled by 8 (scores spanning tens of log2 units) and a dominant key (a copy of
  the query, scaled) in the first block, in a last partial block, in the last split of a multi-split row,
  at the row's own new position, and in the last split of a row merged by the long-context merge;
* chunked-prefill rows whose queries are all aligned with keys placed past the first 128-key tile, with
  growing weights, so that a row's running maximum grows by more than 2^8 after its first tile (the tile
  kernel's lazy rescale of O and of the running sum) and, between rescales, by less (weights up to 2^8
  held in fp16).

Every case is compared element by element with the fp64 oracle over the same host values.
"""
import math

import numpy as np
import pytest

from continuous_batching_paged_ragged_gb300 import pkv, synth
from helpers_gpu import assert_close, host_rows, oracle_host_row, row_slice, run_host_values, score_span_log2

pytestmark = pytest.mark.gpu

KV = [pytest.param(pkv.PKV_KV_F16, id="fp16"), pytest.param(pkv.PKV_KV_E4M3, id="e4m3")]

# decode rows: (cached tokens, where the dominant key sits); one new token each
DECODE_ROWS = [(400, "first_block"), (699, "last_partial_block"), (1499, "last_split"), (300, "own_position"),
               (16400, "last_of_33_splits"), (37, "none")]


def _dominant_position(where: str, ctx: int):
    return {"first_block": 3, "last_partial_block": ctx - 5, "last_split": ctx - 200, "own_position": ctx - 1,
            "last_of_33_splits": ctx - 100, "none": None}[where]


@pytest.mark.parametrize("kv", KV)
@pytest.mark.parametrize("hq,hkv,d", [(12, 2, 128), (16, 4, 256), (4, 1, 64)])
def test_peaked_decode_rows(cuda, built, kv, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached = [c for c, _ in DECODE_ROWS]
    batch = synth.custom_batch(shape, cached, [1] * len(cached), seed=41)
    rows = host_rows(batch, 0)
    G = hq // hkv
    for (c, where), row in zip(DECODE_ROWS, rows):
        q, k, _ = row
        q *= np.float16(8)                         # exact: a power of two, far from the fp16 range's end
        j = _dominant_position(where, c + 1)
        if j is not None:
            for g in range(hkv):
                k[j, g] = q[0, g * G] * np.float16(0.5)   # scores of thousands of log2 units for head g * G
        assert score_span_log2(q, k).max() >= 20
    assert ((batch.context_lens[4] + 15) // 16 + 31) // 32 == 33    # the long-context merge path
    pool, ds, outs = run_host_values(batch, [0], {0: rows}, kv_dtype=kv)
    for b, (c, where) in enumerate(DECODE_ROWS):
        assert_close(row_slice(batch, outs[0], b), oracle_host_row(rows[b], kv), f"{(hq, hkv, d)} row {b} {where}")


# chunked-prefill rows (cached, new tokens); the last has more than 24 K/V tiles (two key chunks, merged)
PREFILL_ROWS = [(300, 64), (0, 400), (1000, 40), (3500, 32)]
# aligned keys: (position, weight) -- the key is weight * the (shared) query of its group's first head
ALIGNED = [(130, 0.75), (200, 1.25), (260, 2.0), (275, 2.4), (290, 3.0), (1800, 3.5), (2100, 4.0)]


def _lazy_rescale_reached(q: np.ndarray, k: np.ndarray) -> bool:
    """Whether some (query, head) sees a score past the first 128 keys above the first tile's maximum by more
    than 8 log2 units (the tile kernel's lazy-rescale threshold)."""
    ql, hq, d = q.shape
    g = hq // k.shape[1]
    ctx = k.shape[0]
    for i in range(0, ql, 7):
        last = ctx - ql + i
        if last < 128:
            continue
        for h in range(hq):
            s = k[:last + 1, h // g, :].astype(np.float64) @ q[i, h].astype(np.float64) / math.sqrt(d) / math.log(2)
            if s[128:].max() > s[:128].max() + 8:
                return True
    return False


@pytest.mark.parametrize("kv", KV)
@pytest.mark.parametrize("hq,hkv,d", [(12, 2, 128), (8, 8, 64), (16, 4, 128)])
def test_prefill_rows_whose_max_grows_past_the_first_tile(cuda, built, kv, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached, qls = zip(*PREFILL_ROWS)
    batch = synth.custom_batch(shape, cached, qls, seed=43)
    rows = host_rows(batch, 0)
    G = hq // hkv
    reached = False
    for b, row in enumerate(rows):
        q, k, _ = row
        q[:] = q[0]                                  # every position asks the same question
        for pos, w in ALIGNED:
            if pos < k.shape[0]:
                for g in range(hkv):
                    k[pos, g] = (q[0, g * G].astype(np.float32) * np.float32(w)).astype(np.float16)
        reached = reached or _lazy_rescale_reached(q, k)
    assert reached
    pool, ds, outs = run_host_values(batch, [0], {0: rows}, kv_dtype=kv)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_host_row(rows[b], kv), f"{(hq, hkv, d)} row {b} {PREFILL_ROWS[b]}")


@pytest.mark.parametrize("kv", KV)
def test_peaked_rows_through_the_fused_call(cuda, built, kv):
    """The same kind of values through pkv_attention_append: decode rows only (the append fused into the
    decode launch), the dominant key being this pass's own token in one row."""
    shape = synth.Shape(1, 12, 2, 128)
    rows_spec = [(400, "first_block"), (699, "last_partial_block"), (300, "own_position"), (1499, "last_split")]
    batch = synth.custom_batch(shape, [c for c, _ in rows_spec], [1] * len(rows_spec), seed=47)
    rows = host_rows(batch, 0)
    for (c, where), row in zip(rows_spec, rows):
        q, k, _ = row
        q *= np.float16(8)
        j = _dominant_position(where, c + 1)
        for g in range(2):
            k[j, g] = q[0, g * 6] * np.float16(0.5)
    pool, ds, outs = run_host_values(batch, [0], {0: rows}, kv_dtype=kv, fused=True)
    for b, (c, where) in enumerate(rows_spec):
        assert_close(row_slice(batch, outs[0], b), oracle_host_row(rows[b], kv), f"row {b} {where}")
