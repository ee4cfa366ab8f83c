"""The seeded input generator: published Philox4x32-10 answers and the value distribution."""
import numpy as np

from continuous_batching_paged_ragged_gb300 import synth


def test_philox_known_answers():
    """Known-answer vectors distributed with the Random123 reference implementation of Philox4x32-10."""
    cases = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in cases:
        got = synth.philox4x32_10(*ctr, *key)
        assert tuple(int(x) for x in got) == want


def test_values_are_a_pure_function_of_their_coordinates():
    a = synth.token_values(synth.KIND_K, 7, 3, [5, 9], [100, 0], 2, 64)
    b = synth.token_values(synth.KIND_K, 7, 3, [9, 5, 5], [0, 100, 1], 2, 64)
    assert np.array_equal(a[0], b[1]) and np.array_equal(a[1], b[0])
    c = synth.token_values(synth.KIND_V, 7, 3, [5], [100], 2, 64)
    assert not np.array_equal(a[0], c[0])


def test_distribution_is_near_standard_normal():
    v = synth.token_values(synth.KIND_Q, 0, 0, np.arange(512), np.zeros(512), 4, 128).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    assert np.abs(v).max() <= np.sqrt(3) * 2 + 1e-3


def test_workload_recipes():
    b = synth.tiny_decode(0)
    assert b.cached_lens.tolist() == [7, 16, 33, 50] and b.context_lens.tolist() == [8, 17, 34, 51]
    assert b.num_blocks == 64 and sorted(b.block_perm.tolist()) == list(range(64))
    q = synth.qwen_decode(0)
    assert q.num_seqs == 256 and 257 <= q.context_lens.min() and q.context_lens.max() <= 769
    need = sum(-(-int(c) // 16) for c in q.context_lens)
    assert q.num_blocks == int(np.ceil(1.25 * need))
    m = synth.mixed_step(0)
    assert m.num_tokens == 3155 and m.q_lens[-2:].tolist() == [2048, 1024]
    assert m.context_lens[-2:].tolist() == [2048, 4096]
    reqs = synth.trace_requests(0)
    assert len(reqs) == 256 and all(16 <= r.prompt_len <= 4096 and 50 <= r.max_output <= 781 for r in reqs)
