"""The seeded input generator: published SplitMix64 outputs, determinism,
slices, moments and workload structure."""
import numpy as np

import synth


def test_splitmix64_published_outputs():
    # first outputs of SplitMix64 started at state 0
    out = synth.splitmix64(0, 0, 2)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_values_are_slice_independent():
    key = synth.stream_key(7, synth.STREAM_K_POOL)
    whole = synth.normal_bf16(key, 0, 5000)
    assert np.array_equal(whole[1234:2345], synth.normal_bf16(key, 1234, 1111))


def test_moments_and_range():
    x = synth.bf16_bits_to_f32(synth.normal_bf16(synth.stream_key(3, 1), 0, 1 << 18)).astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.var() - 1.0) < 0.01
    assert np.max(np.abs(x)) <= 2 * np.sqrt(3) + 1e-2


def test_pool_pages_match_whole_pool():
    w = synth.build("phi3_tiny")
    pool = w.pool("k")
    pages = np.array([5, 0, 63])
    got = w.pool_pages("k", 3, pages)
    for i, pg in enumerate(pages):
        assert np.array_equal(got[i], pool[3, pg * 64:(pg + 1) * 64])


def test_workload_structure():
    for name in sorted(synth.WORKLOADS):
        w = synth.build(name, scale=0.05)
        tp, tr = w.token_positions(), w.token_rows()
        assert len(tp) == w.T
        # every token's page exists and lies in the pool
        for p, r in zip(tp, tr):
            page = w.table[r, p // 64]
            assert 0 <= page < w.num_pages
        # distinct tokens write distinct slots
        slots = {(int(w.table[r, p // 64]) * 64 + int(p) % 64) for p, r in zip(tp, tr)}
        assert len(slots) == w.T


def test_shared_prefix_pages():
    w = synth.build("qwen3", scale=0.2)
    for b in range(w.B):
        for b2 in range(b - b % 16, min(w.B, b - b % 16 + 16)):
            s = min(8, int(w.dec_positions[b]) // 64, int(w.dec_positions[b2]) // 64)
            assert np.array_equal(w.table[b, :s], w.table[b2, :s])
        # the page a row writes is never shared
        wp = w.table[b, int(w.dec_positions[b]) // 64]
        assert np.sum(w.table == wp) == 1
