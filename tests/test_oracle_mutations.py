"""The attention pins are sensitive: each plausible mistake planted in a copy of the oracle fails one.

Mistakes are planted here, on the CPU, in a local re-implementation with switches; the real oracle is
untouched.  Each mutant must be caught by at least one of the pin checks used in test_oracle_attention.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _mutant(kind):
    def attn(q, k, v):
        q_len, hq, d = q.shape
        ctx, hkv, _ = k.shape
        group = hq // hkv
        scale = 1.0 / d if kind == "scale_1_over_d" else 1.0 / math.sqrt(d)
        out = np.zeros((q_len, hq, d))
        for i in range(q_len):
            last = ctx - q_len + i
            if kind == "causal_off_by_one":
                last -= 1
            if kind == "top_left_causal":
                last = i
            for h in range(hq):
                g = h % hkv if kind == "gqa_interleaved" else h // group
                kk = v if kind == "k_v_swapped" else k
                vv = k if kind == "k_v_swapped" else v
                s = kk[: max(last, 0) + 1, g].astype(np.float64) @ q[i, h].astype(np.float64) * scale
                w = np.exp(s - s.max())
                if kind != "no_normalisation":
                    w /= w.sum()
                out[i, h] = w @ vv[: max(last, 0) + 1, g].astype(np.float64)
        return out
    return attn


def _sdpa(q, k, v, causal):
    t = lambda x: torch.from_numpy(x.astype(np.float64)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


def _pins_pass(attn):
    rng = np.random.default_rng(0)
    r = lambda *s: rng.standard_normal(s).astype(np.float16)
    # decode vs library routine
    q, k, v = r(1, 6, 32), r(19, 2, 32), r(19, 2, 32)
    if not np.allclose(attn(q, k, v), _sdpa(q, k, v, False), atol=1e-12):
        return False
    # full prefill vs library causal routine
    q, k, v = r(9, 6, 32), r(9, 2, 32), r(9, 2, 32)
    if not np.allclose(attn(q, k, v), _sdpa(q, k, v, True), atol=1e-12):
        return False
    # chunk over cache equals the matching rows of the full prefill
    q, k, v = r(14, 4, 16), r(14, 2, 16), r(14, 2, 16)
    if not np.allclose(attn(q[9:], k, v), attn(q, k, v)[9:], atol=1e-12):
        return False
    return True


def test_unmutated_copy_passes():
    assert _pins_pass(_mutant("none"))
    assert _pins_pass(oracle.attention_row)


@pytest.mark.parametrize("kind", ["scale_1_over_d", "causal_off_by_one", "top_left_causal", "gqa_interleaved",
                                  "k_v_swapped", "no_normalisation"])
def test_planted_mistake_is_caught(kind):
    assert not _pins_pass(_mutant(kind))
