"""Pins of the f64 oracle to facts fixed by the mathematics of the method.

Each test ties one part of the oracle (RMSNorm, NeoX rotary, the ragged key set,
the masks, GQA, the softmax-weighted sum) to a closed form, an invariant, a special
case or a second, differently structured computation, so that a dropped term, a
wrong sign or index or a transposed operand in the oracle fails at least one.

Definitions (vllm.cpp, qwen3_dflash.cpp and qwen3.cpp): per-head RMSNorm over
head_dim in the plain form (RmsNormArgs{eps, false}) BEFORE NeoX RoPE; context K
normed and rotated at context positions, V raw; each request's block rows attend
over [context ; block] of that request, bidirectionally on full-attention layers
and causally with a sliding window on SWA layers.
"""
import math

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W

BF_ONE = 0x3F80  # bf16 bits of 1.0
BF_ZERO = 0x0000


def bf(x):
    return W.f64_to_bf16(np.asarray(x, dtype=np.float64))


def small_cfg(hq=4, hkv=2, dh=64, causal=False, window=0, block=4):
    return W.Config("pin", 0, block, hq, hkv, dh, causal=causal, window=window, ctx_len=0)


def stored_ctx_k(b):
    """Context keys as the draft model stores them: normed, rotated, bf16."""
    return oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, b.cfg.eps, b.cfg.theta)[1]


def attn(b, ctx_k=None, fn=oracle.block_attention, **kw):
    c = b.cfg
    args = dict(eps=c.eps, theta=c.theta, causal=c.causal, window=c.window)
    args.update(kw)
    return fn(b.q, b.k_blk, b.v_blk, stored_ctx_k(b) if ctx_k is None else ctx_k, b.ctx_v,
              b.query_start_loc, b.ctx_start_loc, b.ctx_lens, b.positions, b.q_norm_w, b.k_norm_w, **args)


# ---------------------------------------------------------------- RMSNorm
def test_rms_norm_constant_vector_closed_form():
    # x = c * 1  =>  y_i = w_i * c / sqrt(c^2 + eps)
    dh, c, eps = 64, 0.5, 1e-6
    x = np.full((1, 1, dh), bf([c])[0], dtype=np.uint16)
    w = bf(np.linspace(0.5, 1.5, dh))
    y = oracle.rms_norm(x, w, eps)[0, 0]
    expect = W.bf16_to_f64(w) * c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(y, expect, rtol=1e-15, atol=0)


def test_rms_norm_mean_square_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = bf(rng.normal(size=(3, 5, 128)))
    ones = bf(np.ones(128))
    y = oracle.rms_norm(x, ones, 0.0)
    np.testing.assert_allclose((y ** 2).mean(axis=-1), 1.0, rtol=1e-13)
    # doubling a bf16 vector is exact, and with eps = 0 the norm ignores scale
    x2 = bf(2.0 * W.bf16_to_f64(x))
    np.testing.assert_allclose(oracle.rms_norm(x2, ones, 0.0), y, rtol=1e-14, atol=1e-15)
    # with eps > 0: mean(y^2) = ms / (ms + eps)
    eps = 0.25
    ye = oracle.rms_norm(x, ones, eps)
    ms = (W.bf16_to_f64(x) ** 2).mean(axis=-1)
    np.testing.assert_allclose((ye ** 2).mean(axis=-1), ms / (ms + eps), rtol=1e-13)


def test_rms_norm_weight_is_elementwise():
    rng = np.random.default_rng(2)
    x = bf(rng.normal(size=(2, 1, 64)))
    w = bf(rng.uniform(0.5, 1.5, size=64))
    y1 = oracle.rms_norm(x, bf(np.ones(64)), 1e-6)
    yw = oracle.rms_norm(x, w, 1e-6)
    np.testing.assert_allclose(yw, y1 * W.bf16_to_f64(w), rtol=1e-14)


# ---------------------------------------------------------------- NeoX RoPE
@pytest.mark.parametrize("dh,theta", [(4, 10000.0), (64, 1e6), (128, 1e6)])
def test_rope_basis_vectors_neox_pairing_and_frequencies(dh, theta):
    # e_i (i < Dh/2) rotates in the plane (i, i + Dh/2) by pos * theta^(-2i/Dh);
    # e_{i+Dh/2} rotates the other way round: (-sin, cos).
    half = dh // 2
    pos = np.array([0, 1, 7, 4095, 32783], dtype=np.int32)
    for i in range(half):
        for first in (True, False):
            x = np.zeros((len(pos), 1, dh))
            x[:, 0, i if first else i + half] = 1.0
            y = oracle.rope_neox(x, pos, theta)[:, 0]
            a = pos.astype(np.float64) * theta ** (-2.0 * i / dh)
            expect = np.zeros_like(y)
            if first:
                expect[:, i], expect[:, i + half] = np.cos(a), np.sin(a)
            else:
                expect[:, i], expect[:, i + half] = -np.sin(a), np.cos(a)
            np.testing.assert_allclose(y, expect, atol=1e-12)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(6, 3, 128))
    y0 = oracle.rope_neox(x, np.zeros(6, np.int32), 1e6)
    np.testing.assert_array_equal(y0, x)
    pos = rng.integers(0, 40000, size=6).astype(np.int32)
    y = oracle.rope_neox(x, pos, 1e6)
    pair = lambda v: v[..., :64] ** 2 + v[..., 64:] ** 2
    np.testing.assert_allclose(pair(y), pair(x), rtol=1e-12)


def test_rope_composition_and_relative_position():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(1, 1, 128))
    k = rng.normal(size=(1, 1, 128))
    th = 1e6
    R = lambda v, p: oracle.rope_neox(v, np.array([p], np.int32), th)
    # R_a R_b = R_(a+b)
    np.testing.assert_allclose(R(R(q, 300), 4000), R(q, 4300), atol=1e-10)
    # <R_m q, R_n k> depends only on m - n
    for m, n in [(10, 3), (5000, 4993), (20007, 20000)]:
        np.testing.assert_allclose(np.sum(R(q, m) * R(k, n)), np.sum(R(q, m - n) * k), rtol=1e-10, atol=1e-10)


def test_norm_then_rope_order():
    # norm is applied first: norm_rope == rope(norm(x)), and != norm of rope with w != 1
    rng = np.random.default_rng(5)
    x = bf(rng.normal(size=(4, 2, 64)))
    w = bf(rng.uniform(0.5, 1.5, size=64))
    pos = np.array([3, 9, 100, 2000], np.int32)
    y = oracle.norm_rope(x, w, pos, 1e-6, 1e6)
    np.testing.assert_allclose(y, oracle.rope_neox(oracle.rms_norm(x, w, 1e-6), pos, 1e6), rtol=1e-14, atol=1e-15)
    # the elementwise weight does not commute with the rotation, so the order matters
    rot = oracle.rope_neox(W.bf16_to_f64(x), pos, 1e6)
    ms = (rot ** 2).mean(axis=-1, keepdims=True)
    other = rot / np.sqrt(ms + 1e-6) * W.bf16_to_f64(w)
    assert np.abs(other - y).max() > 1e-3


def test_round_bf16_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5 - 2 ** -7, 3e-3, 0.0])
    bits = oracle.round_bf16(vals)
    back = W.bf16_to_f64(bits)
    # ties go to the even neighbour; others to the nearest bf16
    np.testing.assert_array_equal(back[:3], [1.0, 1.0, 1.0 + 2 ** -6])
    assert back[3] == 1.0
    rng = np.random.default_rng(6)
    x = rng.normal(size=10000)
    r = W.bf16_to_f64(oracle.round_bf16(x))
    ulp = 2.0 ** (np.floor(np.log2(np.abs(x))) - 7)
    assert np.all(np.abs(r - x) <= ulp / 2 + 1e-300)


# ---------------------------------------------------------------- attention
def test_single_block_token_without_context_returns_v():
    # C = 0, B = 1: the only allowed key is the token itself, so out = v exactly
    cfg = small_cfg(hq=4, hkv=2, block=1)
    b = W.make_batch(cfg, ctx_lens=[0], block_lens=[1], seed=11)
    out = attn(b)
    v = W.bf16_to_f64(b.v_blk)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], v[0, h // 2])


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_weights_sum_to_one(causal, window):
    # V == 1 everywhere => every output is exactly the sum of the softmax weights
    cfg = small_cfg(causal=causal, window=window)
    b = W.make_batch(cfg, ctx_lens=[7, 0, 13], block_lens=[4, 3, 5], seed=12)
    b.v_blk[:] = BF_ONE
    b.ctx_v[:] = BF_ONE
    out = attn(b)
    np.testing.assert_allclose(out, 1.0, atol=1e-13)


def allowed_keys(c, nb, b_idx, causal, window):
    """Combined key indices a block query may see (explicit enumeration of the mask)."""
    i = c + b_idx
    keys = []
    for j in range(c + nb):
        if causal and j > i:
            continue
        if window > 0 and not (i - j < window):
            continue
        keys.append(j)
    return keys


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 1), (True, 4), (True, 9), (True, 100)])
def test_zero_query_gives_mean_of_allowed_values(causal, window):
    # q = 0 => RMSNorm(q) = 0 => all scores 0 => uniform weights over the allowed keys.
    # Pins the ragged key set (context rows at ctx_start_loc, live length ctx_lens,
    # then the block rows), the mask, and the GQA head -> kv head map.
    cfg = small_cfg(hq=6, hkv=2, causal=causal, window=window)
    ctx_lens = [5, 0, 9, 3]
    blocks = [4, 2, 0, 6]
    b = W.make_batch(cfg, ctx_lens=ctx_lens, block_lens=blocks, seed=13)
    # give the context segments slack: capacity > live length for request 0 and 3
    cap = [8, 0, 9, 4]
    csl = np.concatenate([[0], np.cumsum(cap)]).astype(np.int32)
    ck = np.zeros((csl[-1], 2, 64), np.uint16)
    cv = np.zeros((csl[-1], 2, 64), np.uint16)
    old = b.ctx_start_loc
    for r in range(4):
        ck[csl[r]:csl[r] + ctx_lens[r]] = b.ctx_k_raw[old[r]:old[r + 1]]
        cv[csl[r]:csl[r] + ctx_lens[r]] = b.ctx_v[old[r]:old[r + 1]]
        cv[csl[r] + ctx_lens[r]:csl[r + 1]] = bf(1e4)  # slack rows must never be read
    b.ctx_k_raw, b.ctx_v, b.ctx_start_loc = ck, cv, csl
    b.ctx_pos = np.zeros(csl[-1], np.int32)
    b.q[:] = BF_ZERO
    out = attn(b)
    v_ctx, v_blk = W.bf16_to_f64(b.ctx_v), W.bf16_to_f64(b.v_blk)
    for r in range(4):
        c, nb, q0 = ctx_lens[r], blocks[r], b.query_start_loc[r]
        for bi in range(nb):
            keys = allowed_keys(c, nb, bi, causal, window)
            for h in range(6):
                kvh = h // 3
                rows = [v_ctx[csl[r] + j, kvh] if j < c else v_blk[q0 + j - c, kvh] for j in keys]
                np.testing.assert_allclose(out[q0 + bi, h], np.mean(rows, axis=0), rtol=1e-13, atol=1e-13)


def test_gqa_head_to_kv_head_mapping():
    # kv head k carries V == k + 1; query head h must return h // G + 1 (contiguous groups)
    cfg = small_cfg(hq=8, hkv=2, dh=64)
    b = W.make_batch(cfg, ctx_lens=[6, 3], block_lens=[3, 2], seed=14)
    for k in range(2):
        b.v_blk[:, k] = bf(k + 1.0)
        b.ctx_v[:, k] = bf(k + 1.0)
    out = attn(b)
    for h in range(8):
        np.testing.assert_allclose(out[:, h], h // 4 + 1.0, rtol=1e-13)


def test_two_keys_closed_form():
    # C = 1, B = 1, bidirectional: out = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1
    cfg = small_cfg(hq=2, hkv=1, dh=64)
    b = W.make_batch(cfg, ctx_lens=[1], block_lens=[1], seed=15)
    c = b.cfg
    qh = oracle.norm_rope(b.q, b.q_norm_w, b.positions, c.eps, c.theta)[0]
    kb = oracle.norm_rope(b.k_blk, b.k_norm_w, b.positions, c.eps, c.theta)[0, 0]
    ck = stored_ctx_k(b)
    k0 = W.bf16_to_f64(ck)[0, 0]
    v0, v1 = W.bf16_to_f64(b.ctx_v)[0, 0], W.bf16_to_f64(b.v_blk)[0, 0]
    out = attn(b, ctx_k=ck)
    sc = 1.0 / math.sqrt(64)
    for h in range(2):
        s0, s1 = sc * qh[h] @ k0, sc * qh[h] @ kb
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(out[0, h], p0 * v0 + (1.0 - p0) * v1, rtol=1e-12, atol=1e-14)


def test_default_scale_is_inverse_sqrt_head_dim_and_sharp_limit():
    cfg = small_cfg(hq=4, hkv=2, dh=64)
    b = W.make_batch(cfg, ctx_lens=[9], block_lens=[3], seed=16)
    ck = stored_ctx_k(b)
    np.testing.assert_array_equal(attn(b, ctx_k=ck), attn(b, ctx_k=ck, scale=1.0 / 8.0))
    # a huge scale turns softmax into argmax: the output is the V row of the best key
    out = attn(b, ctx_k=ck, scale=1e6)
    c = b.cfg
    qh = oracle.norm_rope(b.q, b.q_norm_w, b.positions, c.eps, c.theta)
    kb = oracle.norm_rope(b.k_blk, b.k_norm_w, b.positions, c.eps, c.theta)
    keys = np.concatenate([W.bf16_to_f64(ck), kb], axis=0)
    vals = np.concatenate([W.bf16_to_f64(b.ctx_v), W.bf16_to_f64(b.v_blk)], axis=0)
    for t in range(3):
        for h in range(4):
            j = int(np.argmax(keys[:, h // 2] @ qh[t, h]))
            np.testing.assert_allclose(out[t, h], vals[j, h // 2], atol=1e-9)


def test_block_permutation_equivariance_bidirectional():
    cfg = small_cfg(hq=4, hkv=2, dh=64)
    b = W.make_batch(cfg, ctx_lens=[10], block_lens=[6], seed=17)
    ck = stored_ctx_k(b)
    out = attn(b, ctx_k=ck)
    perm = np.array([3, 0, 5, 1, 4, 2])
    b.q, b.k_blk, b.v_blk, b.positions = b.q[perm], b.k_blk[perm], b.v_blk[perm], b.positions[perm]
    out_p = attn(b, ctx_k=ck)
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 6)])
def test_common_position_shift_invariance(causal, window):
    # Stored context keys are bf16, whose rounding depends on the position, so the exact
    # invariance is checked on block keys, which the oracle rotates in f64.
    cfg = small_cfg(hq=4, hkv=2, dh=128, causal=causal, window=window)
    b = W.make_batch(cfg, ctx_lens=[0, 0], block_lens=[12, 7], seed=18)
    out = attn(b)
    assert not np.allclose(out[:, 0], out[:, 0].mean(axis=0))  # the rotation matters
    b.positions = b.positions + 9973
    np.testing.assert_allclose(attn(b), out, rtol=1e-9, atol=1e-9)


def test_wide_window_equals_plain_causal():
    cfg = small_cfg(hq=4, hkv=2, causal=True)
    b = W.make_batch(cfg, ctx_lens=[11, 4], block_lens=[5, 3], seed=19)
    ck = stored_ctx_k(b)
    np.testing.assert_array_equal(attn(b, ctx_k=ck, window=16), attn(b, ctx_k=ck, window=0))
    assert not np.allclose(attn(b, ctx_k=ck, window=6), attn(b, ctx_k=ck, window=0))


def test_output_is_linear_in_v():
    cfg = small_cfg(hq=4, hkv=2)
    b1 = W.make_batch(cfg, ctx_lens=[8], block_lens=[4], seed=20)
    ck = stored_ctx_k(b1)
    o1 = attn(b1, ctx_k=ck)
    b2 = W.make_batch(cfg, ctx_lens=[8], block_lens=[4], seed=20)
    b2.v_blk = bf(2.0 * W.bf16_to_f64(b1.v_blk))
    b2.ctx_v = bf(2.0 * W.bf16_to_f64(b1.ctx_v))
    np.testing.assert_allclose(attn(b2, ctx_k=ck), 2.0 * o1, rtol=1e-13)


@pytest.mark.parametrize("hq,hkv,dh,causal,window", [
    (4, 2, 64, False, 0), (4, 4, 64, False, 0), (8, 2, 128, False, 0),
    (4, 1, 64, True, 0), (6, 2, 64, True, 3), (4, 2, 128, True, 7),
])
def test_streaming_matches_materialised_brute_force(hq, hkv, dh, causal, window):
    # the streaming oracle (block rows only) against the draft model's materialised form
    # (combined buffers, dense score matrix over all rows, IndexSelect of block rows)
    cfg = small_cfg(hq=hq, hkv=hkv, dh=dh, causal=causal, window=window)
    b = W.make_batch(cfg, ctx_lens=[9, 0, 4, 17], block_lens=[5, 3, 0, 4], seed=21)
    ck = stored_ctx_k(b)
    fast = attn(b, ctx_k=ck)
    slow = attn(b, ctx_k=ck, fn=oracle.block_attention_dense)
    np.testing.assert_allclose(fast, slow, rtol=1e-12, atol=1e-13)


def test_sampled_rows_equal_full_output():
    cfg = small_cfg(hq=4, hkv=2, causal=True, window=5)
    b = W.make_batch(cfg, ctx_lens=[9, 3], block_lens=[4, 6], seed=22)
    ck = stored_ctx_k(b)
    full = attn(b, ctx_k=ck)
    st = np.array([0, 3, 4, 9, 7], np.int32)
    sh = np.array([3, 0, 2, 1, 3], np.int32)
    c = b.cfg
    samp = oracle.block_attention_sampled(st, sh, b.q, b.k_blk, b.v_blk, ck, b.ctx_v, b.query_start_loc,
                                          b.ctx_start_loc, b.ctx_lens, b.positions, b.q_norm_w, b.k_norm_w,
                                          eps=c.eps, theta=c.theta, causal=True, window=5)
    np.testing.assert_array_equal(samp, full[st, sh])


def test_rejects_window_without_causal_and_bad_heads():
    cfg = small_cfg(hq=4, hkv=2)
    b = W.make_batch(cfg, ctx_lens=[3], block_lens=[2], seed=23)
    with pytest.raises(ValueError):
        attn(b, causal=False, window=4)
    b.k_blk = b.k_blk[:, :1].copy()
    b.v_blk = b.v_blk[:, :1].copy()
    b.ctx_k_raw = np.zeros((3, 3, 64), np.uint16)
    b.ctx_v = np.zeros((3, 3, 64), np.uint16)
    with pytest.raises(ValueError):  # Hq = 4 is not a multiple of Hkv = 3
        oracle.block_attention(b.q, np.zeros((2, 3, 64), np.uint16), np.zeros((2, 3, 64), np.uint16),
                               b.ctx_k_raw, b.ctx_v, b.query_start_loc, b.ctx_start_loc, b.ctx_lens,
                               b.positions, b.q_norm_w, b.k_norm_w)
