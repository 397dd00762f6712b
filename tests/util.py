"""Helpers shared by the tests: move a seeded batch to the GPU, run the oracle on it."""
from __future__ import annotations

import numpy as np

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W

# GPU vs f64 oracle, per output element
BF16_MAX_ABS = 1.5e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 2e-4


def bf16_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def i32_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        return W.bf16_to_f64(bits).reshape(t.shape)
    return t.double().cpu().numpy()


def dev_bits(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def stored_ctx_k(b: W.Batch) -> np.ndarray:
    import oracle
    return oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, b.cfg.eps, b.cfg.theta)[1]


def oracle_attention(b: W.Batch, ctx_k_bits: np.ndarray, **kw) -> np.ndarray:
    import oracle
    c = b.cfg
    args = dict(eps=c.eps, theta=c.theta, causal=c.causal, window=c.window)
    args.update(kw)
    return oracle.block_attention(b.q, b.k_blk, b.v_blk, ctx_k_bits, b.ctx_v, b.query_start_loc, b.ctx_start_loc,
                                  b.ctx_lens, b.positions, b.q_norm_w, b.k_norm_w, **args)


def gpu_attention(b: W.Batch, ctx_k_bits=None, ctx_k_dev=None, out_dtype=0, flags=0, **kw):
    import speculative_decoding_draft_rmsnorm_gb300 as D
    c = b.cfg
    ck = ctx_k_dev if ctx_k_dev is not None else bf16_dev(ctx_k_bits)
    args = dict(eps=c.eps, theta=c.theta, causal=c.causal, window=c.window,
                max_ctx_len=int(max(1, b.ctx_lens.max(initial=0))))
    args.update(kw)
    return D.block_attention(
        bf16_dev(b.q), bf16_dev(b.k_blk), bf16_dev(b.v_blk), ck, bf16_dev(b.ctx_v), i32_dev(b.query_start_loc),
        i32_dev(b.ctx_start_loc), i32_dev(b.ctx_lens), i32_dev(b.positions), bf16_dev(b.q_norm_w),
        bf16_dev(b.k_norm_w), max_block_len=int(max(1, b.block_lens.max(initial=0))), out_dtype=out_dtype,
        flags=flags, **args)


def assert_close_bf16(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    d = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert d.max() <= BF16_MAX_ABS, f"{what}: max|diff| {d.max():.3e} > {BF16_MAX_ABS}"
    assert d.mean() <= BF16_MEAN_ABS, f"{what}: mean|diff| {d.mean():.3e} > {BF16_MEAN_ABS}"


def assert_close_f32(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    d = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert d.max() <= F32_MAX_ABS, f"{what}: max|diff| {d.max():.3e} > {F32_MAX_ABS}"


def to_pages(rows: np.ndarray, starts: np.ndarray, lens: np.ndarray, page_size: int, order, fill=np.uint16(0)):
    """Lays request r's first lens[r] rows (rows[starts[r]:]) into pages of a pool; the k-th page
    allocated (in request order) is pool page order[k]. Returns (pool, block_table) with unused
    block-table entries -1."""
    n = len(lens)
    pages_per = [(int(l) + page_size - 1) // page_size for l in lens]
    total = max(1, sum(pages_per))
    max_pages = max(1, max(pages_per, default=1))
    pool = np.full((total, page_size) + rows.shape[1:], fill, dtype=rows.dtype)
    bt = np.full((n, max_pages), -1, dtype=np.int32)
    k = 0
    for r in range(n):
        for p in range(pages_per[r]):
            page = int(order[k])
            k += 1
            bt[r, p] = page
            lo = p * page_size
            hi = min(int(lens[r]), lo + page_size)
            pool[page, : hi - lo] = rows[starts[r] + lo: starts[r] + hi]
    return pool, bt
