"""Pins for the attention oracle against things other than itself (no GPU).

* a library routine: torch's scaled_dot_product_attention in float64 (textbook softmax(QK^T/sqrt(d))V,
  with its own GQA expansion and its own causal mask for the square case);
* a dense brute-force matrix form with an explicit bottom-right mask;
* closed forms: ctx = 1 gives V exactly, equal keys give the mean of V, constant V gives the constant,
  one dominant key gives its value;
* invariances: key order (a decode query sees a set, not a sequence), chunking of a prompt, batching.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from continuous_batching_paged_ragged_gb300 import synth


def _rand(rng, *shape):
    return rng.standard_normal(shape).astype(np.float16)


def _sdpa(q, k, v, causal):
    # q [L, Hq, d], k/v [S, Hkv, d] -> [L, Hq, d]; torch expects [B, H, L, d]
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv,d,ctx", [(4, 2, 64, 1), (4, 2, 64, 9), (12, 2, 128, 37), (16, 4, 256, 20)])
def test_decode_matches_sdpa(hq, hkv, d, ctx):
    rng = np.random.default_rng(ctx * 7 + d)
    q, k, v = _rand(rng, 1, hq, d), _rand(rng, ctx, hkv, d), _rand(rng, ctx, hkv, d)
    ref = _sdpa(q, k, v, causal=False)
    np.testing.assert_allclose(oracle.attention_row(q, k, v), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 64, 5), (6, 2, 32, 23), (8, 8, 16, 17)])
def test_full_prefill_matches_sdpa_causal(hq, hkv, d, n):
    """q_len == ctx: the bottom-right causal reading coincides with the textbook square causal mask."""
    rng = np.random.default_rng(n)
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    ref = _sdpa(q, k, v, causal=True)
    np.testing.assert_allclose(oracle.attention_row(q, k, v), ref, rtol=0, atol=1e-12)


def test_dense_bruteforce_chunk_over_cache():
    """A chunk on top of cached tokens, written as dense matrices with an explicit mask."""
    rng = np.random.default_rng(3)
    hq, hkv, d, ctx, qn = 6, 3, 16, 29, 7
    q, k, v = _rand(rng, qn, hq, d), _rand(rng, ctx, hkv, d), _rand(rng, ctx, hkv, d)
    qf, kf, vf = (x.astype(np.float64) for x in (q, k, v))
    ref = np.zeros((qn, hq, d))
    cached = ctx - qn
    mask = np.arange(ctx)[None, :] <= (cached + np.arange(qn))[:, None]      # [qn, ctx]
    for h in range(hq):
        kh, vh = kf[:, h // (hq // hkv)], vf[:, h // (hq // hkv)]
        s = qf[:, h] @ kh.T / math.sqrt(d)
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref[:, h] = (p / p.sum(axis=1, keepdims=True)) @ vh
    np.testing.assert_allclose(oracle.attention_row(q, k, v), ref, rtol=0, atol=1e-12)


def test_ctx_one_returns_v_exactly():
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 1, 4, 64), _rand(rng, 1, 2, 64), _rand(rng, 1, 2, 64)
    out = oracle.attention_row(q, k, v)
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // 2].astype(np.float64))
        assert np.array_equal(oracle.round_fp16(out[0, h]), v[0, h // 2])


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    ctx = 13
    q = _rand(rng, 1, 4, 32)
    k = np.repeat(_rand(rng, 1, 2, 32), ctx, axis=0)
    v = _rand(rng, ctx, 2, 32)
    out = oracle.attention_row(q, k, v)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[:, h // 2].astype(np.float64).mean(axis=0), atol=1e-14)


def test_constant_values_give_the_constant():
    rng = np.random.default_rng(4)
    q, k = _rand(rng, 3, 4, 32), _rand(rng, 11, 2, 32)
    v = np.full((11, 2, 32), np.float16(0.375))
    np.testing.assert_allclose(oracle.attention_row(q, k, v), 0.375, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(5)
    d = 64
    q = _rand(rng, 1, 2, d)
    k = (_rand(rng, 20, 1, d) * np.float16(0.01)).astype(np.float16)
    k[11, 0] = (q[0, 0] * np.float16(8)).astype(np.float16)   # score of key 11 for head 0 dominates
    v = _rand(rng, 20, 1, d)
    out = oracle.attention_row(q, k, v)
    np.testing.assert_allclose(out[0, 0], v[11, 0].astype(np.float64), atol=1e-6)


def test_gqa_group_is_contiguous():
    """Heads 0..G-1 read KV head 0: giving KV head 1 huge values must not change heads 0..G-1."""
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 1, 6, 16), _rand(rng, 9, 2, 16), _rand(rng, 9, 2, 16)
    a = oracle.attention_row(q, k, v)
    v2 = v.copy()
    v2[:, 1] = np.float16(100)
    b = oracle.attention_row(q, k, v2)
    np.testing.assert_array_equal(a[:, :3], b[:, :3])
    np.testing.assert_allclose(b[:, 3:], 100.0, atol=1e-12)


def test_decode_invariant_to_key_order():
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 1, 4, 32), _rand(rng, 40, 2, 32), _rand(rng, 40, 2, 32)
    perm = rng.permutation(40)
    np.testing.assert_allclose(oracle.attention_row(q, k, v), oracle.attention_row(q, k[perm], v[perm]),
                               atol=1e-13)


def test_chunked_prefill_equals_full_prefill():
    """A prompt consumed in chunks (each chunk over the cache of the ones before) gives the same rows
    as one full prefill -- this pins the chunk's causal offset."""
    rng = np.random.default_rng(8)
    n, hq, hkv, d = 26, 4, 2, 16
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    full = oracle.attention_row(q, k, v)
    cuts = [0, 5, 6, 17, 26]
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = oracle.attention_row(q[a:b], k[:b], v[:b])
        np.testing.assert_allclose(part, full[a:b], atol=1e-13)


def test_batch_equals_rows_alone():
    """The pages' parity method: a ragged batch gives each row what it gets alone at batch 1."""
    shape = synth.Shape(1, 4, 2, 32)
    rng = np.random.default_rng(9)
    ctxs, qls = [5, 17, 1, 33], [1, 4, 1, 33]
    qsl = np.concatenate([[0], np.cumsum(qls)])
    q = _rand(rng, int(qsl[-1]), 4, 32)
    ks = [_rand(rng, c, 2, 32) for c in ctxs]
    vs = [_rand(rng, c, 2, 32) for c in ctxs]
    out = oracle.attention_batch(q, ks, vs, qsl)
    for b in range(4):
        alone = oracle.attention_batch(q[qsl[b]:qsl[b + 1]], [ks[b]], [vs[b]], [0, qls[b]])
        np.testing.assert_array_equal(out[qsl[b]:qsl[b + 1]], alone)
    assert shape.block_size == 16


def test_rejects_more_queries_than_context():
    rng = np.random.default_rng(10)
    with pytest.raises(AssertionError):
        oracle.attention_row(_rand(rng, 3, 2, 8), _rand(rng, 2, 1, 8), _rand(rng, 2, 1, 8))
