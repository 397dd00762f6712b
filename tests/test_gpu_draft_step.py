"""The draft step's integer-side calls on the GPU, against the oracle.

dflash_paged_append (qwen3_dflash.cpp, AppendContextKVDevice): rows land where the oracle puts
them, V bit for bit, K within one bf16 ulp of the exact projection (and almost always its
nearest bf16), lengths advanced on the device; with the attention behind it, the appended
store gives the oracle's attention. dflash_prepare_inputs (PrepareDflashInputs): integer
outputs bit-exact, padding included.
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


def D():
    import speculative_decoding_draft_rmsnorm_gb300 as lib
    return lib


def _store(n_req, lens, counts, ps, max_pages, hkv, dh, seed):
    """Random page ownership: every request gets max_pages distinct pages of a shuffled pool."""
    rng = np.random.default_rng(seed)
    pages = n_req * max_pages + 3
    bt = rng.permutation(pages)[:n_req * max_pages].reshape(n_req, max_pages).astype(np.int32)
    pool_k = np.full((pages, ps, hkv, dh), NAN_BF16, dtype=np.uint16)
    pool_v = pool_k.copy()
    nsl = np.zeros(n_req + 1, dtype=np.int32)
    nsl[1:] = np.cumsum(counts)
    return bt, pool_k, pool_v, nsl


def _k_ok(got_bits, exact, want_bits):
    got = W.bf16_to_f64(got_bits)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(got - exact) <= ulp + 2.0 ** -17), "an appended key is off by more than one bf16 ulp"
    assert np.mean(got_bits == want_bits) > 0.999


@pytest.mark.parametrize("dh,ps", [(128, 16), (64, 16), (128, 5)])
def test_paged_append_matches_oracle(dh, ps):
    import torch
    hkv, n_req = 4, 7
    rng = np.random.default_rng(dh + ps)
    lens = rng.integers(0, 300, n_req).astype(np.int32)
    counts = rng.integers(0, 40, n_req)
    counts[2] = 0  # a request with nothing to append
    max_pages = (int((lens + counts).max()) + ps - 1) // ps + 1
    bt, pk, pv, nsl = _store(n_req, lens, counts, ps, max_pages, hkv, dh, seed=1)
    n = int(nsl[-1])
    k_raw = W.normal_bf16(2, 0, n * hkv * dh).reshape(n, hkv, dh)
    v = W.normal_bf16(2, 1, n * hkv * dh).reshape(n, hkv, dh)
    w = W.uniform_bf16(2, 2, dh, 0.5, 1.5)
    want_k, want_v, want_lens, bad = oracle.paged_append(pk, pv, bt, lens, nsl, k_raw, v, w, ps)
    assert not bad
    dk, dv, dl = U.bf16_dev(pk), U.bf16_dev(pv), U.i32_dev(lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D().paged_append(U.bf16_dev(k_raw), U.i32_dev(nsl), dl, U.i32_dev(bt), U.bf16_dev(w), dk, v=U.bf16_dev(v),
                     v_pool=dv, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert dl.cpu().numpy().tolist() == want_lens.tolist()
    assert np.array_equal(U.dev_bits(dv).reshape(pv.shape), want_v)
    got_k = U.dev_bits(dk).reshape(pk.shape)
    written = ~np.all(want_k == NAN_BF16, axis=(2, 3))  # rows the oracle wrote
    assert np.array_equal(got_k[~written], want_k[~written])
    # the exact projection of every written row, from its source row and position
    src, pos, where = [], [], []
    for r in range(n_req):
        for i in range(int(counts[r])):
            p = int(lens[r]) + i
            src.append(int(nsl[r]) + i)
            pos.append(p)
            where.append((int(bt[r, p // ps]), p % ps))
    exact, _ = oracle.context_kv(k_raw[src], np.array(pos, dtype=np.int32), w, 1e-6, 1e6)
    got_rows = np.stack([got_k[a, b] for a, b in where])
    want_rows = np.stack([want_k[a, b] for a, b in where])
    _k_ok(got_rows, exact, want_rows)


def test_paged_append_equals_context_kv_with_the_same_slots():
    # the same kernel arithmetic: only the row -> (position, slot) mapping differs
    import torch
    hkv, dh, ps, n_req = 8, 128, 16, 5
    lens = np.array([0, 17, 100, 3, 64], dtype=np.int32)
    counts = np.array([16, 16, 1, 30, 16])
    max_pages = 10
    bt, pk, pv, nsl = _store(n_req, lens, counts, ps, max_pages, hkv, dh, seed=3)
    n = int(nsl[-1])
    k_raw = U.bf16_dev(W.normal_bf16(4, 0, n * hkv * dh).reshape(n, hkv, dh))
    v = U.bf16_dev(W.normal_bf16(4, 1, n * hkv * dh).reshape(n, hkv, dh))
    w = U.bf16_dev(W.uniform_bf16(4, 2, dh, 0.5, 1.5))
    pos = np.concatenate([lens[r] + np.arange(counts[r]) for r in range(n_req)]).astype(np.int32)
    req = np.repeat(np.arange(n_req), counts)
    slot = (bt[req, pos // ps].astype(np.int64) * ps + pos % ps).astype(np.int32)
    a_k, a_v = U.bf16_dev(pk), U.bf16_dev(pv)
    D().paged_append(k_raw, U.i32_dev(nsl), U.i32_dev(lens), U.i32_dev(bt), w, a_k, v=v, v_pool=a_v)
    b_k, b_v = U.bf16_dev(pk), U.bf16_dev(pv)
    D().context_kv(k_raw, U.i32_dev(pos), w, b_k.view(-1, hkv, dh), v=v, ctx_v=b_v.view(-1, hkv, dh),
                   slot=U.i32_dev(slot))
    torch.cuda.synchronize()
    assert torch.equal(a_k.view(torch.int16), b_k.view(torch.int16))
    assert torch.equal(a_v.view(torch.int16), b_v.view(torch.int16))


def _attention_args(b):
    c = b.cfg
    return dict(q=U.bf16_dev(b.q), k_blk=U.bf16_dev(b.k_blk), v_blk=U.bf16_dev(b.v_blk),
                qsl=U.i32_dev(b.query_start_loc), pos=U.i32_dev(b.positions), qw=U.bf16_dev(b.q_norm_w),
                kw=U.bf16_dev(b.k_norm_w), eps=c.eps, theta=c.theta)


def test_prefill_then_decode_appends_feed_the_attention():
    # a store filled by a long first append and a 16-row second one, then attention of the
    # next block over it, with the device lengths the appends left as ctx_lens
    import torch
    cfg = dataclasses.replace(W.CONFIGS["qwen3_0p6b"], num_reqs=5)
    b = W.make_batch(cfg)
    c, ps = b.cfg, 16
    n_req = len(b.ctx_lens)
    first = np.maximum(b.ctx_lens.astype(np.int64) - 16, 0)
    second = b.ctx_lens.astype(np.int64) - first
    max_pages = (int(b.ctx_lens.max()) + ps - 1) // ps
    bt, pk, pv, _ = _store(n_req, np.zeros(n_req), first, ps, max_pages, c.hkv, c.dh, seed=5)
    rows = [np.arange(int(b.ctx_start_loc[r]), int(b.ctx_start_loc[r]) + int(first[r])) for r in range(n_req)]
    rows2 = [np.arange(int(b.ctx_start_loc[r]) + int(first[r]), int(b.ctx_start_loc[r + 1])) for r in range(n_req)]
    i1, i2 = np.concatenate(rows), np.concatenate(rows2)
    nsl1 = np.concatenate([[0], np.cumsum(first)]).astype(np.int32)
    nsl2 = np.concatenate([[0], np.cumsum(second)]).astype(np.int32)
    lens0 = np.zeros(n_req, dtype=np.int32)
    ok1 = oracle.paged_append(pk, pv, bt, lens0, nsl1, b.ctx_k_raw[i1], b.ctx_v[i1], b.k_norm_w, ps, c.eps, c.theta)
    ok2 = oracle.paged_append(ok1[0], ok1[1], bt, ok1[2], nsl2, b.ctx_k_raw[i2], b.ctx_v[i2], b.k_norm_w, ps, c.eps,
                              c.theta)
    assert ok2[2].tolist() == b.ctx_lens.tolist()
    dk, dv, lens = U.bf16_dev(pk), U.bf16_dev(pv), U.i32_dev(lens0)
    w, dbt = U.bf16_dev(b.k_norm_w), U.i32_dev(bt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for idx, nsl in [(i1, nsl1), (i2, nsl2)]:
        D().paged_append(U.bf16_dev(b.ctx_k_raw[idx]), U.i32_dev(nsl), lens, dbt, w, dk, v=U.bf16_dev(b.ctx_v[idx]),
                         v_pool=dv, status=status, eps=c.eps, theta=c.theta)
    a = _attention_args(b)
    out = D().block_attention_paged(a["q"], a["k_blk"], a["v_blk"], dk, dv, dbt, a["qsl"], lens, a["pos"], a["qw"],
                                    a["kw"], max_ctx_len=int(b.ctx_lens.max()), max_block_len=16, eps=c.eps,
                                    theta=c.theta)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert lens.cpu().numpy().tolist() == b.ctx_lens.tolist()
    want = oracle.block_attention_paged(b.q, b.k_blk, b.v_blk, ok2[0], ok2[1], bt, b.query_start_loc, ok2[2],
                                        b.positions, b.q_norm_w, b.k_norm_w, ps, eps=c.eps, theta=c.theta)
    U.assert_close_bf16(U.dev_to_f64(out), want, "append + paged attention")


def test_paged_append_reports_rows_past_the_table_and_bad_start_locations():
    import torch
    hkv, dh, ps = 2, 64, 16
    lens = np.array([20, 0], dtype=np.int32)
    counts = np.array([20, 5])
    bt, pk, pv, nsl = _store(2, lens, counts, ps, 2, hkv, dh, seed=6)  # 32 rows per request
    n = int(nsl[-1])
    k_raw = W.normal_bf16(7, 0, n * hkv * dh).reshape(n, hkv, dh)
    v = W.normal_bf16(7, 1, n * hkv * dh).reshape(n, hkv, dh)
    w = W.uniform_bf16(7, 2, dh, 0.5, 1.5)
    want_k, want_v, want_lens, bad = oracle.paged_append(pk, pv, bt, lens, nsl, k_raw, v, w, ps)
    assert bad
    dk, dv, dl = U.bf16_dev(pk), U.bf16_dev(pv), U.i32_dev(lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D().paged_append(U.bf16_dev(k_raw), U.i32_dev(nsl), dl, U.i32_dev(bt), U.bf16_dev(w), dk, v=U.bf16_dev(v),
                     v_pool=dv, status=status)
    torch.cuda.synchronize()
    assert status.item() & D().STATUS_METADATA
    # request 0 (20 rows after 20, a 32-row table) does not fit: nothing of it is written and its
    # length stays; request 1 appends its 5 rows
    assert dl.cpu().numpy().tolist() == want_lens.tolist() == [20, 5]
    assert np.array_equal(U.dev_bits(dv).reshape(pv.shape), want_v)
    assert np.array_equal(U.dev_bits(dk).reshape(pk.shape)[bt[0]], pk[bt[0]])  # request 0's pages untouched
    # start locations past the rows: no length moves
    status.zero_()
    dl2 = U.i32_dev(lens)
    D().paged_append(U.bf16_dev(k_raw), U.i32_dev(np.array([0, 5, n + 1], dtype=np.int32)), dl2, U.i32_dev(bt),
                     U.bf16_dev(w), U.bf16_dev(pk), status=status)
    torch.cuda.synchronize()
    assert status.item() & D().STATUS_METADATA
    assert dl2.cpu().numpy().tolist() == lens.tolist()


def test_captured_append_and_attention_grow_the_context_on_every_replay():
    # one graph (append the step's new rows, attend with the device lengths) replayed twice:
    # the second replay sees the rows the first appended
    import torch
    cfg = dataclasses.replace(W.CONFIGS["qwen3_0p6b"], num_reqs=4)
    b = W.make_batch(cfg)
    c, ps, step = b.cfg, 16, 16
    n_req = len(b.ctx_lens)
    base = b.ctx_lens.astype(np.int64) - 2 * step  # stored before the two replays
    assert base.min() >= 0
    max_pages = (int(b.ctx_lens.max()) + ps - 1) // ps
    bt, pk, pv, _ = _store(n_req, base, base, ps, max_pages, c.hkv, c.dh, seed=8)
    # the stored part, appended eagerly (untimed set-up)
    nsl0 = np.concatenate([[0], np.cumsum(base)]).astype(np.int32)
    i0 = np.concatenate([np.arange(int(b.ctx_start_loc[r]), int(b.ctx_start_loc[r] + base[r])) for r in range(n_req)])
    dk, dv, lens = U.bf16_dev(pk), U.bf16_dev(pv), U.i32_dev(np.zeros(n_req, dtype=np.int32))
    w, dbt = U.bf16_dev(b.k_norm_w), U.i32_dev(bt)
    D().paged_append(U.bf16_dev(b.ctx_k_raw[i0]), U.i32_dev(nsl0), lens, dbt, w, dk, v=U.bf16_dev(b.ctx_v[i0]),
                     v_pool=dv, eps=c.eps, theta=c.theta)
    o = oracle.paged_append(pk, pv, bt, np.zeros(n_req, dtype=np.int32), nsl0, b.ctx_k_raw[i0], b.ctx_v[i0],
                            b.k_norm_w, ps, c.eps, c.theta)

    def step_rows(j):
        return np.concatenate([np.arange(int(b.ctx_start_loc[r] + base[r] + j * step),
                                         int(b.ctx_start_loc[r] + base[r] + (j + 1) * step)) for r in range(n_req)])

    nsl = U.i32_dev(np.arange(n_req + 1, dtype=np.int32) * step)
    k_in = U.bf16_dev(b.ctx_k_raw[step_rows(0)])
    v_in = U.bf16_dev(b.ctx_v[step_rows(0)])
    a = _attention_args(b)
    ws = D().alloc_workspace(D().workspace_size(n_req, b.q.shape[0], c.hq, c.hkv, c.dh, dk.shape[0] * ps,
                                                int(b.ctx_lens.max()), 16))
    out = torch.empty(b.q.shape, dtype=torch.bfloat16, device="cuda")

    def body():
        D().paged_append(k_in, nsl, lens, dbt, w, dk, v=v_in, v_pool=dv, eps=c.eps, theta=c.theta)
        D().block_attention_paged(a["q"], a["k_blk"], a["v_blk"], dk, dv, dbt, a["qsl"], lens, a["pos"], a["qw"],
                                  a["kw"], max_ctx_len=int(b.ctx_lens.max()), max_block_len=16, out=out,
                                  workspace=ws, eps=c.eps, theta=c.theta)

    # warm-up on a scratch copy of the store state, then capture
    saved = (dk.clone(), dv.clone(), lens.clone())
    body()
    torch.cuda.synchronize()
    dk.copy_(saved[0]), dv.copy_(saved[1]), lens.copy_(saved[2])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    torch.cuda.synchronize()
    for j in range(2):
        k_in.copy_(U.bf16_dev(b.ctx_k_raw[step_rows(j)]))
        v_in.copy_(U.bf16_dev(b.ctx_v[step_rows(j)]))
        g.replay()
        torch.cuda.synchronize()
        o = oracle.paged_append(o[0], o[1], bt, o[2], np.arange(n_req + 1) * step, b.ctx_k_raw[step_rows(j)],
                                b.ctx_v[step_rows(j)], b.k_norm_w, ps, c.eps, c.theta)
        assert lens.cpu().numpy().tolist() == o[2].tolist()
        want = oracle.block_attention_paged(b.q, b.k_blk, b.v_blk, o[0], o[1], bt, b.query_start_loc, o[2],
                                            b.positions, b.q_norm_w, b.k_norm_w, ps, eps=c.eps, theta=c.theta)
        U.assert_close_bf16(U.dev_to_f64(out), want, f"replay {j}")
    D().check_error(ws)
    assert lens.cpu().numpy().tolist() == b.ctx_lens.tolist()


# ------------------------------------------------------------------ input preparation
def _prep_dev(pb: W.PrepareBatch):
    import torch
    t = {k: U.i32_dev(getattr(pb, k)) for k in ("idx_mapping", "target_query_start_loc", "num_rejected",
                                                 "num_sampled", "last_sampled", "next_prefill_tokens",
                                                 "block_table")}
    t["target_positions"] = torch.from_numpy(np.ascontiguousarray(pb.target_positions, dtype=np.int64)).cuda()
    return t


def _prep_gpu(pb: W.PrepareBatch, status=None, out=None):
    import torch
    t = _prep_dev(pb)
    if out is None:  # garbage first: every entry must be written
        out = D().prepare_inputs(**t, **pb.scalars())
        for v in out.values():
            v.fill_(12345)
    res = D().prepare_inputs(**t, **pb.scalars(), out=out, status=status)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def _prep_oracle(pb: W.PrepareBatch):
    return oracle.prepare_dflash_inputs(pb.idx_mapping, pb.target_query_start_loc, pb.num_rejected, pb.num_sampled,
                                        pb.last_sampled, pb.next_prefill_tokens, pb.target_positions,
                                        pb.block_table, **pb.scalars())


PREP_CASES = [
    dict(seed=0, num_reqs=1),
    dict(seed=1, num_reqs=37),
    dict(seed=2, num_reqs=37, sample_from_anchor=True),
    dict(seed=3, num_reqs=64, prefill_frac=0.9, max_prefill_chunk=2048),      # long prefill chunks
    dict(seed=4, num_reqs=20, max_model_len=20000, stride=900),                # both clamps
    dict(seed=5, num_reqs=256, max_num_reqs=256, max_num_tokens=4096),         # no padding rows
    dict(seed=6, num_reqs=9, block_size=32, max_num_reqs=300, max_num_tokens=8192),  # much padding
]


@pytest.mark.parametrize("case", PREP_CASES, ids=[str(i) for i in range(len(PREP_CASES))])
def test_prepare_inputs_bit_exact(case):
    import torch
    pb = W.make_prepare_batch(**case)
    want = _prep_oracle(pb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _prep_gpu(pb, status=status)
    assert status.item() == 0
    assert set(got) == set(want)
    for k in want:
        assert got[k].dtype == want[k].dtype, k
        assert np.array_equal(got[k], want[k]), k


def test_prepare_inputs_reports_bad_metadata():
    import torch
    pb = W.make_prepare_batch(7, 8)
    pb.idx_mapping = pb.idx_mapping.copy()
    pb.idx_mapping[3] = pb.max_num_reqs  # a request state outside the table
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _prep_gpu(pb, status=status)
    assert status.item() & D().STATUS_METADATA
    pb = W.make_prepare_batch(7, 8)
    pb.num_rejected = pb.num_rejected.copy()
    pb.num_rejected[0] = int(pb.target_query_start_loc[1]) + 1  # accepted end before the first token
    status.zero_()
    _prep_gpu(pb, status=status)
    assert status.item() & D().STATUS_METADATA


def test_prepare_inputs_graph_replay_with_new_values():
    import torch
    pb = W.make_prepare_batch(8, 16)
    t = _prep_dev(pb)
    out = D().prepare_inputs(**t, **pb.scalars())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        D().prepare_inputs(**t, **pb.scalars(), out=out)
    # the next step: other rejections, samples and positions, same shapes
    pb2 = W.make_prepare_batch(9, 16)
    same = pb2.target_query_start_loc[-1] == pb.target_query_start_loc[-1]
    if not same:  # keep the captured sizes: reuse the first batch's token layout
        pb2 = dataclasses.replace(pb2, target_query_start_loc=pb.target_query_start_loc,
                                  target_positions=pb.target_positions + 7,
                                  num_rejected=np.minimum(pb2.num_rejected,
                                                          np.diff(pb.target_query_start_loc) - 1).astype(np.int32))
    for k, v in _prep_dev(pb2).items():
        t[k].copy_(v)
    g.replay()
    torch.cuda.synchronize()
    want = _prep_oracle(pb2)
    for k in want:
        assert np.array_equal(out[k].cpu().numpy(), want[k]), k


def test_prepare_inputs_context_arrays_longer_than_the_scored_tokens():
    pb = W.make_prepare_batch(10, 6)
    n_tgt = int(pb.target_query_start_loc[-1])
    pb.target_positions = np.concatenate([pb.target_positions, np.full(9, 777, dtype=np.int64)])
    want = oracle.prepare_dflash_inputs(pb.idx_mapping, pb.target_query_start_loc, pb.num_rejected, pb.num_sampled,
                                        pb.last_sampled, pb.next_prefill_tokens, pb.target_positions, pb.block_table,
                                        num_target_tokens=n_tgt + 9, **pb.scalars())
    got = _prep_gpu(pb)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_paged_append_without_values_writes_keys_only():
    import torch
    hkv, dh, ps, n_req = 2, 128, 16, 3
    lens = np.array([5, 0, 40], dtype=np.int32)
    counts = np.array([16, 3, 16])
    bt, pk, pv, nsl = _store(n_req, lens, counts, ps, 5, hkv, dh, seed=12)
    n = int(nsl[-1])
    k_raw = W.normal_bf16(13, 0, n * hkv * dh).reshape(n, hkv, dh)
    w = W.uniform_bf16(13, 2, dh, 0.5, 1.5)
    want_k, _, want_lens, _ = oracle.paged_append(pk, pv, bt, lens, nsl, k_raw, None, w, ps)
    dk, dl = U.bf16_dev(pk), U.i32_dev(lens)
    D().paged_append(U.bf16_dev(k_raw), U.i32_dev(nsl), dl, U.i32_dev(bt), U.bf16_dev(w), dk)
    torch.cuda.synchronize()
    assert dl.cpu().numpy().tolist() == want_lens.tolist()
    got_k = U.dev_bits(dk).reshape(pk.shape)
    written = ~np.all(want_k == NAN_BF16, axis=(2, 3))
    assert written.sum() == n
    assert np.array_equal(got_k[~written], want_k[~written])
    assert np.mean(got_k[written] == want_k[written]) > 0.999


def test_paged_append_more_requests_than_staged_start_locations():
    # past 1024 requests the row kernel searches the start locations in global memory, and the
    # length kernel's one block loops over the requests
    import torch
    hkv, dh, ps, n_req = 1, 64, 16, 1100
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 40, n_req).astype(np.int32)
    counts = rng.integers(0, 3, n_req)
    bt, pk, pv, nsl = _store(n_req, lens, counts, ps, 3, hkv, dh, seed=32)
    n = int(nsl[-1])
    k_raw = W.normal_bf16(33, 0, n * hkv * dh).reshape(n, hkv, dh)
    v = W.normal_bf16(33, 1, n * hkv * dh).reshape(n, hkv, dh)
    w = W.uniform_bf16(33, 2, dh, 0.5, 1.5)
    want_k, want_v, want_lens, bad = oracle.paged_append(pk, pv, bt, lens, nsl, k_raw, v, w, ps)
    assert not bad
    dk, dv, dl = U.bf16_dev(pk), U.bf16_dev(pv), U.i32_dev(lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D().paged_append(U.bf16_dev(k_raw), U.i32_dev(nsl), dl, U.i32_dev(bt), U.bf16_dev(w), dk, v=U.bf16_dev(v),
                     v_pool=dv, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert dl.cpu().numpy().tolist() == want_lens.tolist()
    assert np.array_equal(U.dev_bits(dv).reshape(pv.shape), want_v)
    got_k = U.dev_bits(dk).reshape(pk.shape)
    written = ~np.all(want_k == NAN_BF16, axis=(2, 3))
    assert written.sum() == n
    assert np.array_equal(got_k[~written], want_k[~written])
    # every written row within one bf16 ulp of the exact projection of its source row
    src, pos, where = [], [], []
    for r in range(n_req):
        for i in range(int(counts[r])):
            p = int(lens[r]) + i
            src.append(int(nsl[r]) + i)
            pos.append(p)
            where.append((int(bt[r, p // ps]), p % ps))
    exact, _ = oracle.context_kv(k_raw[src], np.array(pos, dtype=np.int32), w, 1e-6, 1e6)
    _k_ok(np.stack([got_k[a, b] for a, b in where]), exact, np.stack([want_k[a, b] for a, b in where]))
