"""The seeded input generator: determinism, stream independence, layout of a batch."""
import math

import numpy as np

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0: the first outputs of Vigna's reference generator
    # (state += 0x9E3779B97F4A7C15, then the mix) are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    z = W._mix64(np.array([0x9E3779B97F4A7C15, (2 * 0x9E3779B97F4A7C15) % 2**64], dtype=np.uint64))
    assert int(z[0]) == 0xE220A8397B1DCDAF
    assert int(z[1]) == 0x6E789E6AA1B965F4


def test_draws_are_deterministic_and_chunk_independent():
    a = W.normal_bf16(3, W.STREAM_Q, 10_001)
    b = W.normal_bf16(3, W.STREAM_Q, 10_001)
    np.testing.assert_array_equal(a, b)
    # a prefix of a longer draw is the shorter draw
    np.testing.assert_array_equal(W.normal_bf16(3, W.STREAM_Q, 5_000), a[:5_000])
    assert not np.array_equal(W.normal_bf16(3, W.STREAM_KBLK, 100), a[:100])


def test_normal_moments():
    x = W.bf16_to_f64(W.normal_bf16(0, W.STREAM_CTXK, 400_000))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_bf16_round_trip_and_rounding():
    v = np.array([1.0, -2.5, 3.140625, 0.0, 1e-3])
    np.testing.assert_array_equal(W.bf16_to_f64(W.f64_to_bf16(v))[:4], [1.0, -2.5, 3.140625, 0.0])
    assert W.f64_to_bf16(np.array([1.0 + 2 ** -8]))[0] == 0x3F80  # tie to even
    assert W.f64_to_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82


def test_batch_layout_follows_the_runner():
    cfg = W.CONFIGS["qwen3_0p6b"]
    b = W.make_batch(cfg)
    c = b.ctx_lens.astype(int)
    assert len(c) == 8 and c.min() >= 512 and c.max() <= 2048
    np.testing.assert_array_equal(np.diff(b.query_start_loc), 16)
    np.testing.assert_array_equal(np.diff(b.ctx_start_loc), c)
    for r in range(8):
        # context positions 0..C-1, block positions C..C+B-1
        np.testing.assert_array_equal(b.ctx_pos[b.ctx_start_loc[r]:b.ctx_start_loc[r + 1]], np.arange(c[r]))
        np.testing.assert_array_equal(b.positions[16 * r:16 * (r + 1)], c[r] + np.arange(16))
    w = W.bf16_to_f64(b.q_norm_w)
    assert w.min() >= 0.5 and w.max() <= 1.5
    assert b.q.shape == (128, 16, 128) and b.ctx_k_raw.shape == (c.sum(), 8, 128)


def test_ragged_lengths_are_log_uniform_in_range():
    c = W.context_lengths(W.CONFIGS["ragged"]).astype(float)
    assert c.min() >= 1024 and c.max() <= 32768 and len(c) == 64
    # log-uniform: the mean of log C sits near the middle of [ln 1024, ln 32768]
    assert abs(np.log(c).mean() - 0.5 * (math.log(1024) + math.log(32768))) < 0.35
