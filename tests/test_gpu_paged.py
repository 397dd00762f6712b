"""dflash_block_attention_paged on the GPU: context K/V in page pools behind a block table.

Parity with the paged oracle (which gathers the rows by the block table and takes the plain
attention definition), bit-identity with the contiguous entry point where the tiling is the
same, and the device-side check of block-table entries.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu

NAN_BF16 = np.uint16(0x7FC0)


def _paged_inputs(b: W.Batch, ck_bits: np.ndarray, page_size: int, seed: int = 11, fill=NAN_BF16):
    n_pages = sum((int(l) + page_size - 1) // page_size for l in b.ctx_lens)
    order = np.random.default_rng(seed).permutation(max(1, n_pages))
    kp, bt = U.to_pages(ck_bits, b.ctx_start_loc, b.ctx_lens, page_size, order, fill)
    vp, _ = U.to_pages(b.ctx_v, b.ctx_start_loc, b.ctx_lens, page_size, order, fill)
    return kp, vp, bt


def _gpu_paged(b: W.Batch, kp, vp, bt, out_dtype=0, flags=0, max_ctx_len=None, **kw):
    import speculative_decoding_draft_rmsnorm_gb300 as D
    c = b.cfg
    args = dict(eps=c.eps, theta=c.theta, causal=c.causal, window=c.window)
    args.update(kw)
    out = D.block_attention_paged(
        U.bf16_dev(b.q), U.bf16_dev(b.k_blk), U.bf16_dev(b.v_blk), U.bf16_dev(kp), U.bf16_dev(vp), U.i32_dev(bt),
        U.i32_dev(b.query_start_loc), U.i32_dev(b.ctx_lens), U.i32_dev(b.positions), U.bf16_dev(b.q_norm_w),
        U.bf16_dev(b.k_norm_w), max_ctx_len=max_ctx_len or int(max(1, b.ctx_lens.max(initial=0))),
        max_block_len=int(max(1, b.block_lens.max(initial=0))), out_dtype=out_dtype, flags=flags, **args)
    return out


def _oracle_paged(b: W.Batch, kp, vp, bt, page_size, **kw):
    c = b.cfg
    args = dict(eps=c.eps, theta=c.theta, causal=c.causal, window=c.window)
    args.update(kw)
    return oracle.block_attention_paged(b.q, b.k_blk, b.v_blk, kp, vp, bt, b.query_start_loc, b.ctx_lens, b.positions,
                                        b.q_norm_w, b.k_norm_w, page_size, **args)


CASES = [
    ("qwen3_0p6b", 16, {}),
    ("qwen3_0p6b", 64, {}),
    ("qwen3_0p6b", 128, {}),                  # one box brings a whole 128-key tile
    ("swa_small", 16, {}),                    # window start not on a page boundary
    ("swa_small", 128, {}),
    ("tiny", 16, {}),
    ("ragged_small", 32, {}),
]


def _cfg(name: str) -> W.Config:
    if name == "swa_small":
        return dataclasses.replace(W.CONFIGS["swa"], num_reqs=3, ctx_len=2500, window=1003)
    if name == "ragged_small":
        return dataclasses.replace(W.CONFIGS["ragged"], num_reqs=6, ctx_loguniform=(100, 3000))
    return W.CONFIGS[name]


@pytest.mark.parametrize("name,page_size,kw", CASES)
def test_paged_matches_oracle_bf16(name, page_size, kw):
    cfg = _cfg(name)
    b = W.make_batch(cfg)
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, page_size)
    got = U.dev_to_f64(_gpu_paged(b, kp, vp, bt, flags=1 if cfg.force_split else 0))
    U.assert_close_bf16(got, _oracle_paged(b, kp, vp, bt, page_size), f"{name} ps={page_size}")


@pytest.mark.parametrize("name,page_size", [("qwen3_0p6b", 16), ("swa_small", 16), ("tiny", 16),
                                            ("ragged_small", 32), ("swa_small", 128)])
def test_paged_matches_oracle_f32(name, page_size):
    cfg = _cfg(name)
    b = W.make_batch(cfg)
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, page_size)
    got = U.dev_to_f64(_gpu_paged(b, kp, vp, bt, out_dtype=1, flags=1 if cfg.force_split else 0))
    U.assert_close_f32(got, _oracle_paged(b, kp, vp, bt, page_size), f"{name} ps={page_size} f32")


@pytest.mark.parametrize("flags", [0, 1, 2])
def test_paged_equals_contiguous(flags):
    # Without a window both entry points cut every request into the same key tiles. Whole
    # groups per CTA (flag 2) give the same bits; with splitting the grids may differ (the
    # paged call's context bound counts whole pages), so split points, and the rounding of
    # the merge, may differ by one bf16 step.
    b = W.make_batch(W.CONFIGS["qwen3_0p6b"])
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, 16)
    got = _gpu_paged(b, kp, vp, bt, flags=flags)
    want = U.gpu_attention(b, ck, flags=flags)
    if flags == 2:
        assert np.array_equal(U.dev_bits(got), U.dev_bits(want))
    else:
        g, w = U.dev_to_f64(got), U.dev_to_f64(want)
        assert np.all(np.abs(g - w) <= np.maximum(np.abs(g), np.abs(w)) * 2.0 ** -7 + 1e-30)


def test_bad_block_table_entry_is_reported_and_unused_entries_are_not_read():
    import speculative_decoding_draft_rmsnorm_gb300 as D
    b = W.make_batch(W.CONFIGS["qwen3_0p6b"])
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, 16)
    n = b.query_start_loc.shape[0] - 1
    c = b.cfg
    dev = dict(q=U.bf16_dev(b.q), kb=U.bf16_dev(b.k_blk), vb=U.bf16_dev(b.v_blk), kp=U.bf16_dev(kp),
               vp=U.bf16_dev(vp), qsl=U.i32_dev(b.query_start_loc), cl=U.i32_dev(b.ctx_lens),
               pos=U.i32_dev(b.positions), qw=U.bf16_dev(b.q_norm_w), kw=U.bf16_dev(b.k_norm_w))
    max_ctx = int(b.ctx_lens.max())
    ws = D.alloc_workspace(D.workspace_size(n, b.q.shape[0], c.hq, c.hkv, c.dh, kp.shape[0] * 16, max_ctx, 16))

    def run(table):
        D.block_attention_paged(dev["q"], dev["kb"], dev["vb"], dev["kp"], dev["vp"], U.i32_dev(table), dev["qsl"],
                                dev["cl"], dev["pos"], dev["qw"], dev["kw"], max_ctx_len=max_ctx, max_block_len=16,
                                workspace=ws, eps=c.eps, theta=c.theta)

    # entries past each request's live pages are -1 already (see to_pages): never read
    assert (bt == -1).any()
    run(bt)
    D.check_error(ws)
    bad = bt.copy()
    bad[1, 0] = kp.shape[0] + 5
    run(bad)
    with pytest.raises(D.DFlashError) as e:
        D.check_error(ws)
    assert e.value.code == D.ERR_DEVICE_METADATA
    run(bt)  # the error word is per call
    D.check_error(ws)


def test_paged_rejects_unsupported_page_size_and_short_table():
    import torch
    import speculative_decoding_draft_rmsnorm_gb300 as D
    b = W.make_batch(W.CONFIGS["tiny"])
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, 16)
    kp24 = np.zeros((kp.shape[0], 24) + kp.shape[2:], dtype=np.uint16)
    with pytest.raises(D.DFlashError) as e:
        _gpu_paged(b, kp24, kp24, bt)
    assert e.value.code == D.ERR_UNSUPPORTED
    with pytest.raises(D.DFlashError) as e:
        _gpu_paged(b, kp, vp, bt, max_ctx_len=bt.shape[1] * 16 + 1)
    assert e.value.code == D.ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_pool_smaller_than_the_block_table_width():
    # a block table sized for the longest context a request may reach (64 pages of 16 rows)
    # over a pool that holds fewer pages than that: each request's live rows fit in its pages,
    # so every request is computed and nothing is reported
    import torch
    import speculative_decoding_draft_rmsnorm_gb300 as D
    cfg = dataclasses.replace(W.CONFIGS["qwen3_0p6b"], num_reqs=3)
    b = W.make_batch(cfg, ctx_lens=[100, 37, 0], block_lens=[16, 16, 5])
    ck = U.stored_ctx_k(b)
    kp, vp, bt = _paged_inputs(b, ck, 16)
    wide = np.full((bt.shape[0], 64), -1, dtype=np.int32)  # room for 1024 rows per request
    wide[:, :bt.shape[1]] = bt
    assert kp.shape[0] < wide.shape[1]  # the pool has fewer pages than a table row
    ws = D.alloc_workspace(D.workspace_size(3, b.q.shape[0], cfg.hq, cfg.hkv, cfg.dh, kp.shape[0] * 16, 1024, 16))
    got = _gpu_paged(b, kp, vp, wide, max_ctx_len=1024, workspace=ws)
    torch.cuda.synchronize()
    D.check_error(ws)
    U.assert_close_bf16(U.dev_to_f64(got), _oracle_paged(b, kp, vp, wide, 16), "pool narrower than the table")
