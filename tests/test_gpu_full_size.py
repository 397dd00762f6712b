"""Full-size parity: every block row and head of all five workloads against the f64 oracle.

The benchmarked path -- dflash_context_kv building the context store, then
dflash_block_attention (ragged with the split forced, as benchmarked) -- runs on each
workload at its full size, and every output element is compared with the oracle: bf16
output within max|diff| 1.5e-2 and mean|diff| 2e-3 (end to end: the GPU-built store
against the oracle's exact context keys), f32 output within 2e-4 (both sides given the
same stored bf16 keys, so the comparison isolates the attention). The paged call with
16-row pages (the pages' own page size) runs on the Qwen3-4B-shaped and the sliding-window
layers in both output types. The oracle of each workload is computed once per module
and reused.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu

ALL = ["tiny", "qwen3_0p6b", "qwen3_4b", "swa", "ragged"]


def D():
    import speculative_decoding_draft_rmsnorm_gb300 as lib
    return lib


@functools.lru_cache(maxsize=1)
def _case(name):
    """(batch, the oracle's stored context-key bits, the oracle's output); one workload at a time."""
    b = W.make_batch(W.CONFIGS[name])
    ck = U.stored_ctx_k(b)
    return b, ck, U.oracle_attention(b, ck)


def _flags(c):
    return D().FLAG_FORCE_SPLIT if c.force_split else 0


@pytest.mark.parametrize("name", ALL)
def test_full_size_every_row_bf16(name):
    import torch
    b, _, want = _case(name)
    c = b.cfg
    ctx_k = torch.empty(b.ctx_k_raw.shape, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), ctx_k, status=status,
                   eps=c.eps, theta=c.theta)
    ws = D().alloc_workspace(D().workspace_size(c.num_reqs, b.q.shape[0], c.hq, c.hkv, c.dh, b.ctx_k_raw.shape[0],
                                                int(b.ctx_lens.max()), int(b.block_lens.max()), c.causal, c.window,
                                                D().OUT_BF16, _flags(c)))
    out = U.gpu_attention(b, ctx_k_dev=ctx_k, flags=_flags(c), workspace=ws)
    torch.cuda.synchronize()
    D().check_error(ws)
    assert status.item() == 0
    got = U.dev_to_f64(out)
    U.assert_close_bf16(got, want, f"{name}, all {got.shape[0]} block rows x {got.shape[1]} heads")


@pytest.mark.parametrize("name", ["qwen3_4b", "swa", "ragged"])
def test_full_size_every_row_f32(name):
    import torch
    b, ck, want = _case(name)
    c = b.cfg
    out = U.gpu_attention(b, ck, out_dtype=D().OUT_F32, flags=_flags(c))
    torch.cuda.synchronize()
    U.assert_close_f32(U.dev_to_f64(out), want, f"{name} f32, every row")


@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("name", ["qwen3_4b", "swa"])
def test_full_size_paged_16_row_pages(name, out_dtype):
    # the layer with its context in 16-row pages handed out in shuffled order (for the sliding
    # window, its first context tile starts on the page boundary below the window's first key)
    import torch
    b, ck, want_contig = _case(name)
    c, ps = b.cfg, 16
    order = np.random.default_rng(5).permutation(sum((int(l) + ps - 1) // ps for l in b.ctx_lens))
    pool_k, bt = U.to_pages(ck, b.ctx_start_loc, b.ctx_lens, ps, order)
    pool_v, _ = U.to_pages(b.ctx_v, b.ctx_start_loc, b.ctx_lens, ps, order)
    want = oracle.block_attention_paged(b.q, b.k_blk, b.v_blk, pool_k, pool_v, bt, b.query_start_loc, b.ctx_lens,
                                        b.positions, b.q_norm_w, b.k_norm_w, ps, eps=c.eps, theta=c.theta,
                                        causal=c.causal, window=c.window)
    assert np.array_equal(want, want_contig)  # the paged oracle is the contiguous one on gathered rows
    out = D().block_attention_paged(U.bf16_dev(b.q), U.bf16_dev(b.k_blk), U.bf16_dev(b.v_blk), U.bf16_dev(pool_k),
                                    U.bf16_dev(pool_v), U.i32_dev(bt), U.i32_dev(b.query_start_loc),
                                    U.i32_dev(b.ctx_lens), U.i32_dev(b.positions), U.bf16_dev(b.q_norm_w),
                                    U.bf16_dev(b.k_norm_w), max_ctx_len=int(b.ctx_lens.max()), max_block_len=c.block,
                                    eps=c.eps, theta=c.theta, causal=c.causal, window=c.window,
                                    out_dtype=out_dtype)
    torch.cuda.synchronize()
    got = U.dev_to_f64(out)
    if out_dtype:
        U.assert_close_f32(got, want, f"{name} paged16 f32")
    else:
        U.assert_close_bf16(got, want, f"{name} paged16 bf16")
