"""Pins of the oracle's paged-context addressing (CPU).

Paging changes only where a request's context rows live: row j of request r is row
j % page_size of page block_table[r, j // page_size]. The paged oracle must therefore equal
the contiguous oracle, bit for bit, on the rows it gathers, whatever the page order, and must
never read rows past a request's live length.
"""
from __future__ import annotations

import numpy as np

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests.util import to_pages as _to_pages

NAN_BF16 = np.uint16(0x7FC0)


def _batch():
    cfg = W.Config(name="paged_pin", num_reqs=3, block=16, hq=4, hkv=2, dh=64, ctx_uniform=(20, 90), seed=3)
    b = W.make_batch(cfg)
    ck = oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, cfg.eps, cfg.theta)[1]
    return b, ck


def _contiguous(b, ck, **kw):
    return oracle.block_attention(b.q, b.k_blk, b.v_blk, ck, b.ctx_v, b.query_start_loc, b.ctx_start_loc, b.ctx_lens,
                                  b.positions, b.q_norm_w, b.k_norm_w, **kw)


def _paged(b, kp, vp, bt, page_size, **kw):
    return oracle.block_attention_paged(b.q, b.k_blk, b.v_blk, kp, vp, bt, b.query_start_loc, b.ctx_lens,
                                        b.positions, b.q_norm_w, b.k_norm_w, page_size, **kw)


def test_gather_follows_the_block_table_by_hand():
    pool = np.arange(4 * 16, dtype=np.uint16).reshape(4, 16, 1, 1)
    rows, starts = oracle.gather_paged_context(pool, np.array([[2, 0, 3], [1, 0, 0]], dtype=np.int32),
                                               np.array([20, 5], dtype=np.int32), 16)
    want = list(range(32, 48)) + list(range(0, 4)) + list(range(16, 21))
    assert rows.reshape(-1).tolist() == want
    assert starts.tolist() == [0, 20, 25]


def test_identity_paging_equals_contiguous():
    b, ck = _batch()
    n_pages = sum((int(l) + 15) // 16 for l in b.ctx_lens)
    order = np.arange(n_pages)
    kp, bt = _to_pages(ck, b.ctx_start_loc, b.ctx_lens, 16, order)
    vp, _ = _to_pages(b.ctx_v, b.ctx_start_loc, b.ctx_lens, 16, order)
    assert np.array_equal(_paged(b, kp, vp, bt, 16), _contiguous(b, ck))


def test_permuted_pages_and_other_page_sizes_equal_contiguous():
    b, ck = _batch()
    want = _contiguous(b, ck, causal=True, window=37)
    rng = np.random.default_rng(7)
    for ps in (16, 32, 64):
        n_pages = sum((int(l) + ps - 1) // ps for l in b.ctx_lens)
        order = rng.permutation(n_pages)
        kp, bt = _to_pages(ck, b.ctx_start_loc, b.ctx_lens, ps, order)
        vp, _ = _to_pages(b.ctx_v, b.ctx_start_loc, b.ctx_lens, ps, order)
        assert np.array_equal(_paged(b, kp, vp, bt, ps, causal=True, window=37), want), ps


def test_rows_past_the_live_length_are_never_read():
    b, ck = _batch()
    n_pages = sum((int(l) + 15) // 16 for l in b.ctx_lens)
    order = np.arange(n_pages)[::-1]
    kp, bt = _to_pages(ck, b.ctx_start_loc, b.ctx_lens, 16, order, fill=NAN_BF16)
    vp, _ = _to_pages(b.ctx_v, b.ctx_start_loc, b.ctx_lens, 16, order, fill=NAN_BF16)
    got = _paged(b, kp, vp, bt, 16)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, _contiguous(b, ck))
