"""GPU: the 8-bit cache (E4M3 codes, one power-of-two scale per cached row).

The append's codes and scale bytes are bit-exact against the oracle's quantizer; attention over the cache
matches the oracle's attention over the dequantized values within the fp16 tolerance; the fused call gives
bit for bit the cache and outputs of append-then-attention; rows are batch-invariant; the long-context
merge and every supported head shape are covered."""
import numpy as np
import pytest
import torch

from oracle import fp8
from continuous_batching_paged_ragged_gb300 import pkv, synth, workload
from helpers_gpu import assert_close, oracle_row_8bit, poison, row_slice, run_batch

pytestmark = pytest.mark.gpu

E4M3 = pkv.PKV_KV_E4M3


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _rows_of_many_magnitudes(rng, n, hkv, d):
    """fp16 [n, hkv, d]: normal values scaled per row over 2^-20 .. 2^12, plus an all-zero row, a row that
    peaks exactly at 448, one at the fp16 maximum and one of fp16 subnormals."""
    mags = np.exp2(rng.uniform(-20, 12, size=(n, hkv, 1)))
    x = (rng.standard_normal((n, hkv, d)) * mags).astype(np.float16)
    x[0, 0] = 0
    x[1, 0, :] = np.float16(0.5)
    x[1, 0, 3] = np.float16(448.0)
    x[2, -1, :] = rng.uniform(-1, 1, d).astype(np.float16)
    x[2, -1, 5] = np.float16(65504.0)
    x[3, 0] = (rng.integers(-1000, 1000, d) * 2.0 ** -24).astype(np.float16)
    return x


@pytest.mark.parametrize("d", [64, 128, 256])
def test_append_codes_and_scales_bit_exact(cuda, built, d):
    rng = np.random.default_rng(d)
    hkv, nb, T = 2, 9, 40
    pool = pkv.Pool(1, 2 * hkv, hkv, d, nb, kv_dtype=E4M3)
    pool.cache_view().zero_()
    pool.scales_view().zero_()
    k = _rows_of_many_magnitudes(rng, T, hkv, d)
    v = _rows_of_many_magnitudes(rng, T, hkv, d)[::-1].copy()
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[7] = -1
    pkv.pkv_append(pool.handle, 0, torch.from_numpy(k).to(cuda), torch.from_numpy(v).to(cuda),
                   torch.from_numpy(slots).to(cuda), T)
    torch.cuda.synchronize()
    assert pool.check() == 0
    ck = np.zeros((nb, hkv, 16, d), np.uint8)
    cv = np.zeros_like(ck)
    sc = np.zeros((nb, hkv, 2, 16), np.uint8)
    fp8.append_reference_8bit(ck, cv, sc, k, v, slots)
    assert np.array_equal(pool.layer(0, 0).cpu().numpy(), ck)
    assert np.array_equal(pool.layer(0, 1).cpu().numpy(), cv)
    assert np.array_equal(pool.scales_view()[0].cpu().numpy(), sc)


def test_append_out_of_range_slot_is_reported(cuda, built):
    pool = pkv.Pool(1, 4, 2, 64, 4, kv_dtype=E4M3)
    k = torch.ones(2, 2, 64, dtype=torch.float16, device=cuda)
    slots = torch.tensor([4 * 16, 3], dtype=torch.int64, device=cuda)
    pkv.pkv_append(pool.handle, 0, k, k, slots, 2)
    torch.cuda.synchronize()
    assert pool.check() & pkv.PKV_DEVERR_SLOT_RANGE


ROWS = [(0, 1), (1, 1), (15, 1), (16, 1), (255, 1), (511, 1), (512, 1), (700, 1), (1023, 1), (16, 3), (0, 33),
        (240, 17), (500, 12), (1020, 6)]
SHAPES = [(12, 2, 128), (4, 2, 64), (16, 4, 256), (8, 8, 128), (8, 1, 128), (16, 2, 64), (4, 1, 256)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
def test_attention_over_8bit_cache(cuda, built, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached, qls = zip(*ROWS)
    batch = synth.custom_batch(shape, cached, qls, seed=31)
    pool, ds, outs = run_batch(batch, [0], kv_dtype=E4M3)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row_8bit(batch, 0, b), f"{(hq, hkv, d)} row {b} {ROWS[b]}")


@pytest.mark.parametrize("rows", [
    [(300, 1), (17, 1), (0, 1), (255, 1), (256, 1), (700, 1), (15, 1)],     # decode rows
    [(300, 1), (40, 3), (0, 7), (255, 2), (16, 1), (900, 4)],               # short chunks
    [(200, 1), (0, 40), (50, 1)],                                           # a chunk of 40: append first
])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_fused_equals_append_then_attention(cuda, built, rows, d):
    shape = synth.Shape(2, 2 * 6 if d != 256 else 8, 2, d)
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=17)
    pa, _, oa = run_batch(batch, [0, 1], kv_dtype=E4M3, fused=False)
    pb, _, ob = run_batch(batch, [0, 1], kv_dtype=E4M3, fused=True)
    if max(qls) < 16:
        assert pkv.pkv_last_launch_count(pb.handle) == 1   # the append ran inside the decode launch
    assert _same(pa.cache_view(), pb.cache_view())
    assert _same(pa.scales_view(), pb.scales_view())
    for layer in (0, 1):
        assert _same(oa[layer], ob[layer])
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, ob[layer], b), oracle_row_8bit(batch, layer, b), f"layer {layer} row {b}")


def test_cache_written_by_attention_matches_oracle_quantizer(cuda, built):
    """The fused call's own writes: every token appended this pass holds the oracle's codes and scales."""
    shape = synth.Shape(1, 12, 2, 128)
    batch = synth.custom_batch(shape, [300, 40, 0, 17], [1, 3, 5, 1], seed=23)
    pool, ds, _ = run_batch(batch, [0], kv_dtype=E4M3, fused=True)
    codes_k = pool.layer(0, 0).cpu().numpy()
    codes_v = pool.layer(0, 1).cpu().numpy()
    scales = pool.scales_view()[0].cpu().numpy()
    slots = ds.slot_mapping.cpu().numpy()
    req, pos = batch.token_req_pos()
    k = synth.token_values(synth.KIND_K, batch.seed, 0, req, pos, 2, 128)
    v = synth.token_values(synth.KIND_V, batch.seed, 0, req, pos, 2, 128)
    for t, s in enumerate(slots):
        for h in range(2):
            c, sb = fp8.quantize_row(k[t, h])
            assert np.array_equal(codes_k[s // 16, h, s % 16], c) and scales[s // 16, h, 0, s % 16] == sb
            c, sb = fp8.quantize_row(v[t, h])
            assert np.array_equal(codes_v[s // 16, h, s % 16], c) and scales[s // 16, h, 1, s % 16] == sb


def test_batched_equals_each_row_alone(cuda, built):
    shape = synth.Shape(1, 12, 2, 128)
    cached, qls = [300, 17, 650, 1, 0, 255], [1, 1, 1, 1, 20, 1]
    full = synth.custom_batch(shape, cached, qls, seed=4)
    _, _, of = run_batch(full, [0], kv_dtype=E4M3)
    for b in range(len(cached)):
        alone = synth.custom_batch(shape, [cached[b]], [qls[b]], seed=4, req_ids=[full.req_ids[b]])
        _, _, oa = run_batch(alone, [0], kv_dtype=E4M3)
        assert torch.equal(oa[0].view(torch.int16),
                           torch.from_numpy(row_slice(full, of[0], b)).to(cuda).view(torch.int16))


@pytest.mark.parametrize("split_blocks", [1, 3, 16])
def test_split_size_does_not_change_the_answer(cuda, built, split_blocks):
    shape = synth.Shape(1, 12, 2, 128)
    batch = synth.custom_batch(shape, [1000, 37, 400, 0], [1, 1, 5, 12], seed=2)
    pool, ds, outs = run_batch(batch, [0], split_blocks=split_blocks, kv_dtype=E4M3)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row_8bit(batch, 0, b), f"split {split_blocks} row {b}")


def test_long_context_merge(cuda, built):
    """Contexts of more than 32 splits take the separate merge launch."""
    shape = synth.Shape(1, 16, 4, 256)
    batch = synth.custom_batch(shape, [20000, 9000, 100], [1, 1, 1], seed=9)
    pool, ds, outs = run_batch(batch, [0], kv_dtype=E4M3)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row_8bit(batch, 0, b), f"row {b}")


def test_many_launches_on_one_plan(cuda, built):
    rng = np.random.default_rng(5)
    rows = 512
    ctx = rng.integers(2, 770, size=rows)
    shape = synth.Shape(2, 12, 2, 128)
    batch = synth.custom_batch(shape, ctx - 1, np.ones(rows, dtype=np.int64), seed=13)
    pool = workload.make_pool(batch, kv_dtype=E4M3)
    poison(pool)
    workload.prefill_cache(pool, batch, [0, 1])
    ds = workload.upload(batch, pool)
    qs, ks, vs = workload.step_inputs(ds, [0, 1])
    outs = [torch.full_like(q, float("nan")) for q in qs]
    attn = workload.Attention(pool, ds)
    attn.plan()
    for i in range(24):
        attn.run_append(i % 2, qs[i % 2], ks[i % 2], vs[i % 2], outs[i % 2])
    torch.cuda.synchronize()
    assert pool.check() == 0
    for layer in (0, 1):
        for b in range(0, rows, 23):
            assert_close(row_slice(batch, outs[layer], b), oracle_row_8bit(batch, layer, b), f"layer {layer} row {b}")


def test_qwen_decode_full_size_sampled(cuda, built):
    """The benchmark's workload on an 8-bit cache through the fused call: 256 rows, every row on both layers
    of a 2-layer pool."""
    batch = synth.qwen_decode(0)
    batch.shape = synth.Shape(2, 12, 2, 128)
    pool, ds, outs = run_batch(batch, [0, 1], kv_dtype=E4M3, fused=True)
    for layer in (0, 1):
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, outs[layer], b), oracle_row_8bit(batch, layer, b), f"layer {layer} row {b}")


# chunked-prefill rows: the tile kernel over the fp16 shadow of their blocks (head_dim 64, 128 and 256)
PREFILL_ROWS = [(0, 16), (0, 21), (0, 128), (0, 129), (5, 43), (127, 16), (1000, 64), (2047, 200), (16, 250)]
PREFILL_SHAPES = [(12, 2, 128), (8, 8, 64), (8, 1, 128), (16, 4, 128), (4, 2, 64), (8, 8, 128), (16, 4, 256)]


@pytest.mark.parametrize("hq,hkv,d", PREFILL_SHAPES)
def test_prefill_rows_over_8bit_cache(cuda, built, hq, hkv, d):
    shape = synth.Shape(1, hq, hkv, d)
    cached, qls = zip(*PREFILL_ROWS)
    batch = synth.custom_batch(shape, cached, qls, seed=41)
    pool, ds, outs = run_batch(batch, [0], kv_dtype=E4M3)
    for b in range(batch.num_seqs):
        assert_close(row_slice(batch, outs[0], b), oracle_row_8bit(batch, 0, b),
                     f"{(hq, hkv, d)} row {b} {PREFILL_ROWS[b]}")


def test_prefill_and_decode_rows_fused_call(cuda, built):
    """Decode rows, short chunks and long chunks in one pass through pkv_attention_append, two layers: the
    cache gets the append's codes, the long chunks read the shadow, the rest the codes."""
    shape = synth.Shape(2, 12, 2, 128)
    rows = [(300, 1), (0, 40), (17, 1), (700, 15), (64, 16), (3000, 1), (250, 333), (1, 1)]
    cached, qls = zip(*rows)
    batch = synth.custom_batch(shape, cached, qls, seed=8)
    pa, _, oa = run_batch(batch, [0, 1], kv_dtype=E4M3, fused=False)
    pb, _, ob = run_batch(batch, [0, 1], kv_dtype=E4M3, fused=True)
    assert _same(pa.cache_view(), pb.cache_view()) and _same(pa.scales_view(), pb.scales_view())
    for layer in (0, 1):
        assert _same(oa[layer], ob[layer])
        for b in range(batch.num_seqs):
            assert_close(row_slice(batch, ob[layer], b), oracle_row_8bit(batch, layer, b), f"layer {layer} row {b}")


def test_mixed_step_full_size_sampled(cuda, built):
    """The mixed pass (83 decode rows, chunks of 2048 on 0 and 1024 on 3072) on an 8-bit cache: decode rows
    and sampled query tokens of the chunks against the oracle, each over its own causal context."""
    batch = synth.mixed_step(0)
    batch.shape = synth.Shape(1, batch.shape.num_q_heads, batch.shape.num_kv_heads, batch.shape.head_dim)
    pool, ds, outs = run_batch(batch, [0], kv_dtype=E4M3)
    s = batch.shape
    for b in range(batch.num_seqs):
        ql, ctx, req = int(batch.q_lens[b]), int(batch.context_lens[b]), int(batch.req_ids[b])
        got = row_slice(batch, outs[0], b)
        if ql == 1:
            if b % 9 == 0:
                assert_close(got, oracle_row_8bit(batch, 0, b), f"row {b}")
            continue
        k, v = synth.sequence_kv(batch.seed, 0, req, ctx, s.num_kv_heads, s.head_dim)
        kq = fp8.dequantize_rows(*fp8.quantize_rows(k))
        vq = fp8.dequantize_rows(*fp8.quantize_rows(v))
        for i in (0, 1, 127, 128, ql // 2, ql - 1):
            pos = ctx - ql + i
            q = synth.token_values(synth.KIND_Q, batch.seed, 0, np.array([req]), np.array([pos]), s.num_q_heads,
                                   s.head_dim)
            from oracle import attention_row
            ref = attention_row(q, kq[: pos + 1], vq[: pos + 1])
            assert_close(got[i:i + 1], ref, f"row {b} token {i}")
