"""CUDA-graph capture of the two entry points, compared with eager calls.

The attention call allocates nothing, reads every length from device arrays and derives its
schedule on the device, so one captured call serves later steps whose lengths change (within the
bounds it was captured with): a replay must equal an eager call on the same data, bit for bit.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu


def _device_batch(b: W.Batch):
    import speculative_decoding_draft_rmsnorm_gb300 as D
    c = b.cfg
    t = dict(q=U.bf16_dev(b.q), k_blk=U.bf16_dev(b.k_blk), v_blk=U.bf16_dev(b.v_blk),
             ctx_k=U.bf16_dev(U.stored_ctx_k(b)), ctx_v=U.bf16_dev(b.ctx_v), qsl=U.i32_dev(b.query_start_loc),
             csl=U.i32_dev(b.ctx_start_loc), clen=U.i32_dev(b.ctx_lens), pos=U.i32_dev(b.positions),
             qw=U.bf16_dev(b.q_norm_w), kw=U.bf16_dev(b.k_norm_w))
    max_ctx = int(b.ctx_lens.max())
    max_blk = int(b.block_lens.max())
    n = b.query_start_loc.shape[0] - 1
    need = D.workspace_size(n, b.q.shape[0], c.hq, c.hkv, c.dh, b.ctx_k_raw.shape[0], max_ctx, max_blk,
                            c.causal, c.window, D.OUT_BF16, 0)
    return t, max_ctx, max_blk, D.alloc_workspace(need)


def _attend(t, b, max_ctx, max_blk, ws, out):
    import speculative_decoding_draft_rmsnorm_gb300 as D
    c = b.cfg
    return D.block_attention(t["q"], t["k_blk"], t["v_blk"], t["ctx_k"], t["ctx_v"], t["qsl"], t["csl"], t["clen"],
                             t["pos"], t["qw"], t["kw"], max_ctx_len=max_ctx, max_block_len=max_blk, out=out,
                             workspace=ws, eps=c.eps, theta=c.theta, causal=c.causal, window=c.window)


@pytest.mark.parametrize("name", ["qwen3_0p6b", "swa_small"])
def test_block_attention_graph_replay_matches_eager(name):
    import torch
    import speculative_decoding_draft_rmsnorm_gb300 as D
    if name == "swa_small":
        cfg = dataclasses.replace(W.CONFIGS["swa"], num_reqs=4, ctx_len=3000, window=1000)
    else:
        cfg = W.CONFIGS[name]
    b = W.make_batch(cfg)
    t, max_ctx, max_blk, ws = _device_batch(b)
    shape = (b.q.shape[0], cfg.hq, cfg.dh)
    eager = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    _attend(t, b, max_ctx, max_blk, ws, eager)  # also the warm-up before capture
    torch.cuda.synchronize()

    replay = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _attend(t, b, max_ctx, max_blk, ws, replay)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))
    D.check_error(ws)

    # new values in the captured buffers: other queries, and context lengths that shrink or stay
    # (the captured bounds hold), i.e. what a later draft step hands to the same graph
    gen = torch.Generator(device="cuda").manual_seed(1)
    t["q"].copy_(torch.randn(t["q"].shape, device="cuda", generator=gen).to(torch.bfloat16))
    new_lens = np.maximum(b.ctx_lens - np.arange(b.ctx_lens.shape[0], dtype=np.int32) * 37, 0).astype(np.int32)
    t["clen"].copy_(torch.from_numpy(new_lens).cuda())
    g.replay()
    _attend(t, b, max_ctx, max_blk, ws, eager)
    torch.cuda.synchronize()
    assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))
    D.check_error(ws)
    # and the replayed result is the attention over the new lengths
    nb = dataclasses.replace(b, ctx_lens=new_lens, q=U.dev_bits(t["q"]).reshape(b.q.shape))
    U.assert_close_bf16(U.dev_to_f64(replay), U.oracle_attention(nb, U.stored_ctx_k(b)), f"{name} replay")


def test_context_kv_graph_replay_matches_eager():
    import torch
    import speculative_decoding_draft_rmsnorm_gb300 as D
    cfg = W.CONFIGS["qwen3_0p6b"]
    b = W.make_batch(cfg)
    n_ctx = b.ctx_k_raw.shape[0]
    rows = 64
    k_new = U.bf16_dev(b.ctx_k_raw[:rows])
    v_new = U.bf16_dev(b.ctx_v[:rows])
    pos = U.i32_dev(b.ctx_pos[:rows])
    kw = U.bf16_dev(b.k_norm_w)
    slot = U.i32_dev(np.arange(rows, dtype=np.int32) * 3)
    store_e = torch.zeros((n_ctx, cfg.hkv, cfg.dh), dtype=torch.bfloat16, device="cuda")
    store_ve = torch.zeros_like(store_e)
    D.context_kv(k_new, pos, kw, store_e, v=v_new, ctx_v=store_ve, slot=slot, eps=cfg.eps, theta=cfg.theta)
    torch.cuda.synchronize()

    store_g = torch.zeros_like(store_e)
    store_vg = torch.zeros_like(store_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        D.context_kv(k_new, pos, kw, store_g, v=v_new, ctx_v=store_vg, slot=slot, eps=cfg.eps, theta=cfg.theta)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(store_g.view(torch.int16), store_e.view(torch.int16))
    assert torch.equal(store_vg.view(torch.int16), store_ve.view(torch.int16))
    # other slots on replay: rows land where the device array says
    slot.copy_(torch.arange(rows, dtype=torch.int32, device="cuda") * 3 + 1)
    g.replay()
    D.context_kv(k_new, pos, kw, store_e, v=v_new, ctx_v=store_ve, slot=slot, eps=cfg.eps, theta=cfg.theta)
    torch.cuda.synchronize()
    assert torch.equal(store_g.view(torch.int16), store_e.view(torch.int16))
    assert torch.equal(store_vg.view(torch.int16), store_ve.view(torch.int16))
