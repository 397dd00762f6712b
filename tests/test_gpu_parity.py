"""GPU parity: the CUDA path (through the C ABI) against the f64 oracle.

Tolerances per output element: bf16 output max|diff| <= 1.5e-2 and mean|diff| <= 2e-3;
f32 output max|diff| <= 2e-4. The context-K store is checked against the exact value:
every stored bf16 is within one bf16 ulp of it and almost all are its nearest bf16.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu


def D():
    import speculative_decoding_draft_rmsnorm_gb300 as lib
    return lib


def cfg(hq=4, hkv=2, dh=64, causal=False, window=0, block=16, seed=0):
    return W.Config("t", 0, block, hq, hkv, dh, causal=causal, window=window, ctx_len=0, seed=seed)


# ------------------------------------------------------------------ context K/V store
@pytest.mark.parametrize("hkv,dh,n", [(2, 64, 200), (8, 128, 1000), (3, 128, 37)])
def test_context_kv_matches_oracle(hkv, dh, n):
    import torch
    c = cfg(hq=hkv, hkv=hkv, dh=dh)
    b = W.make_batch(c, ctx_lens=[n], block_lens=[1], seed=3)
    pos = (np.arange(n) * 37 + 5).astype(np.int32)  # positions up to ~37k
    exact, want_bits = oracle.context_kv(b.ctx_k_raw, pos, b.k_norm_w, c.eps, c.theta)
    out = torch.empty((n, hkv, dh), dtype=torch.bfloat16, device="cuda")
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(pos), U.bf16_dev(b.k_norm_w), out, eps=c.eps, theta=c.theta)
    got_bits = U.dev_bits(out).reshape(exact.shape)
    got = W.bf16_to_f64(got_bits).reshape(exact.shape)
    # one bf16 ulp of the exact value, plus the absolute error of the f32 rotation of
    # normalised values (|x^| < ~8): where cos/sin terms cancel, the result is tiny and
    # its own ulp is smaller than that f32 error
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(got - exact) <= ulp + 2.0 ** -17), "a stored key is off by more than one bf16 ulp"
    assert np.mean(got_bits == want_bits) > 0.999


def test_context_kv_slots_copy_v_and_leave_other_rows():
    import torch
    c = cfg(hq=2, hkv=2, dh=128)
    b = W.make_batch(c, ctx_lens=[40], block_lens=[1], seed=4)
    cap = 100
    slots = np.random.default_rng(0).permutation(cap)[:40].astype(np.int32)
    store_k = torch.full((cap, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    store_v = torch.full((cap, 2, 128), -3.0, dtype=torch.bfloat16, device="cuda")
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), store_k,
                   v=U.bf16_dev(b.ctx_v), ctx_v=store_v, slot=U.i32_dev(slots), eps=c.eps, theta=c.theta)
    exact, _ = oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, c.eps, c.theta)
    gk = U.dev_to_f64(store_k)
    gv = U.dev_bits(store_v).reshape(cap, 2, 128)
    np.testing.assert_allclose(gk[slots], exact, atol=2e-2, rtol=1e-2)
    np.testing.assert_array_equal(gv[slots], b.ctx_v)
    rest = np.setdiff1d(np.arange(cap), slots)
    assert np.all(gk[rest] == 7.0)
    assert np.all(W.bf16_to_f64(gv[rest]) == -3.0)


def test_context_kv_reports_out_of_range_slots():
    # a row whose slot is outside the store is not written and sets the status word; the
    # other rows land as usual
    import torch
    c = cfg(hq=2, hkv=2, dh=64)
    b = W.make_batch(c, ctx_lens=[6], block_lens=[1], seed=14)
    cap = 8
    slots = np.array([0, 8, 3, -1, 7, 2], dtype=np.int32)
    store = torch.full((cap, 2, 64), 5.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), store,
                   slot=U.i32_dev(slots), status=status, eps=c.eps, theta=c.theta)
    torch.cuda.synchronize()
    assert status.item() & D().STATUS_METADATA
    _, want = oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, c.eps, c.theta)
    got = U.dev_bits(store).reshape(cap, 2, 64)
    ok = [i for i, s in enumerate(slots) if 0 <= s < cap]
    assert np.mean(got[slots[ok]] == want[ok]) > 0.99
    rest = np.setdiff1d(np.arange(cap), slots[ok])
    assert np.all(W.bf16_to_f64(got[rest]) == 5.0)
    # in-range slots only: the word stays clear
    status.zero_()
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), store,
                   slot=U.i32_dev(np.arange(6, dtype=np.int32)), status=status, eps=c.eps, theta=c.theta)
    torch.cuda.synchronize()
    assert status.item() == 0


def test_context_kv_append_in_pieces_is_bit_identical():
    # per-row independence: appending rows in chunks gives the bits of one call
    import torch
    c = cfg(hq=8, hkv=8, dh=128)
    b = W.make_batch(c, ctx_lens=[300], block_lens=[1], seed=5)
    whole = torch.empty((300, 8, 128), dtype=torch.bfloat16, device="cuda")
    D().context_kv(U.bf16_dev(b.ctx_k_raw), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), whole)
    pieces = torch.empty_like(whole)
    k = U.bf16_dev(b.ctx_k_raw)
    pos = U.i32_dev(b.ctx_pos)
    w = U.bf16_dev(b.k_norm_w)
    for lo, hi in [(0, 1), (1, 17), (17, 150), (150, 300)]:
        slot = torch.arange(lo, hi, dtype=torch.int32, device="cuda")
        D().context_kv(k[lo:hi].contiguous(), pos[lo:hi].contiguous(), w, pieces, slot=slot)
    assert torch.equal(whole.view(torch.int16), pieces.view(torch.int16))


def test_context_kv_in_place():
    import torch
    c = cfg(hq=8, hkv=8, dh=64)
    b = W.make_batch(c, ctx_lens=[64], block_lens=[1], seed=6)
    buf = U.bf16_dev(b.ctx_k_raw)
    ref = torch.empty_like(buf)
    D().context_kv(buf.clone(), U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), ref)
    D().context_kv(buf, U.i32_dev(b.ctx_pos), U.bf16_dev(b.k_norm_w), buf)
    assert torch.equal(ref.view(torch.int16), buf.view(torch.int16))


# ------------------------------------------------------------------ block attention, small
SMALL_CASES = [
    # (name, hq, hkv, dh, causal, window, ctx_lens, block_lens)
    ("tiny_cfg", 4, 2, 64, False, 0, [64], [16]),
    ("gqa4_dh128", 32, 8, 128, False, 0, [300, 129, 128, 5], [16, 16, 16, 16]),
    ("mha", 8, 8, 128, False, 0, [200, 1], [16, 3]),
    ("no_context", 4, 2, 64, False, 0, [0, 0, 7], [16, 5, 1]),
    ("ragged_blocks", 16, 8, 128, False, 0, [257, 0, 1000, 33], [1, 17, 5, 16]),
    ("empty_request", 8, 4, 128, False, 0, [50, 60, 70], [4, 0, 9]),
    ("causal", 8, 2, 128, True, 0, [130, 7], [16, 9]),
    ("swa", 32, 8, 128, True, 200, [1000, 150, 4], [16, 16, 16]),
    ("swa_w1", 4, 2, 64, True, 1, [20, 3], [5, 4]),
    ("swa_w_lt_block", 4, 2, 64, True, 6, [40], [16]),
    ("two_qtiles", 16, 4, 128, False, 0, [300, 10], [20, 33]),
    ("g8_qtiles", 64, 8, 64, True, 50, [400], [20]),
    ("g16", 32, 2, 128, False, 0, [700, 5, 260], [16, 7, 16]),    # 4 tokens a query tile
    ("g32_causal", 64, 2, 64, True, 0, [300, 129], [16, 3]),       # 2 tokens a query tile
    ("mqa_g64", 64, 1, 128, True, 100, [500, 0, 64], [16, 9, 5]),  # one kv head, 1 token a query tile
    ("long_blocks", 8, 2, 128, True, 0, [900, 40], [150, 130]),    # 2 block-key tiles (3 in f32), 10 query tiles
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
def test_block_attention_small_bf16(case):
    name, hq, hkv, dh, causal, window, cl, bl = case
    b = W.make_batch(cfg(hq, hkv, dh, causal, window, seed=7), ctx_lens=cl, block_lens=bl)
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck))
    U.assert_close_bf16(got, want, name)


F32_CASES = [c for c in SMALL_CASES if c[0] in ("tiny_cfg", "gqa4_dh128", "no_context", "ragged_blocks", "causal",
                                               "swa", "swa_w1", "two_qtiles", "g8_qtiles", "mqa_g64",
                                               "long_blocks")]


@pytest.mark.parametrize("case", F32_CASES, ids=[c[0] for c in F32_CASES])
def test_block_attention_small_f32(case):
    # f32 output runs on split hi+lo bf16 operands (q^, block k^ and P), so it must sit
    # within 2e-4 of the exact result even where few keys make every weight count
    name, hq, hkv, dh, causal, window, cl, bl = case
    b = W.make_batch(cfg(hq, hkv, dh, causal, window, seed=17), ctx_lens=cl, block_lens=bl)
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck, out_dtype=1))
    U.assert_close_f32(got, want, name)


@pytest.mark.parametrize("flags", [1, 2])
def test_f32_split_and_unsplit(flags):
    b = W.make_batch(cfg(32, 8, 128, seed=18), ctx_lens=[1500, 0, 2000], block_lens=[16, 16, 16])
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck, out_dtype=1, flags=flags))
    U.assert_close_f32(got, want, f"f32 flags={flags}")


@pytest.mark.parametrize("flags", [1, 2])
def test_split_and_unsplit_paths_both_match(flags):
    b = W.make_batch(cfg(32, 8, 128, seed=8), ctx_lens=[1500, 700, 2000], block_lens=[16, 16, 16])
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck, flags=flags))
    U.assert_close_bf16(got, want, f"flags={flags}")


@pytest.mark.parametrize("ctx,cap", [(300, 32768), (8000, 32768), (3000, 3000)])
def test_store_capacity_far_above_the_lengths(ctx, cap):
    # the grid is sized from the host bounds (store capacity, max lengths); with live lengths
    # far below them there are fewer tiles than CTAs (ctx 300 in segments of 32768: 16 tiles
    # for 129 CTAs, every group split over 4 CTAs) or under 4 tiles a CTA (ctx 8000), where
    # the schedule leaves the cost-balanced split; every split group must still merge from
    # exactly its contributors
    import dataclasses
    import speculative_decoding_draft_rmsnorm_gb300 as lib
    full = W.make_batch(cfg(8, 2, 128, seed=21), ctx_lens=[cap, cap], block_lens=[16, 16])
    b = dataclasses.replace(full, ctx_lens=np.array([ctx, ctx - 1], dtype=np.int32))
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    plan = lib.plan(2, 32, 8, 2, 128, b.ctx_k_raw.shape[0], cap, 16)
    got = U.dev_to_f64(U.gpu_attention(b, ck, max_ctx_len=cap))
    U.assert_close_bf16(got, want, f"ctx {ctx} in segments of {cap} ({plan['ctas']} CTAs)")


@pytest.mark.parametrize("flags", [0, 1, 2])
def test_more_than_256_requests(flags):
    # the schedule is built 256 requests at a time past 256 requests (an even split of the tiles)
    rng = np.random.default_rng(23)
    n = 300
    ctx = rng.integers(0, 400, n)
    ctx[::17] = 0
    blk = rng.integers(1, 17, n)
    b = W.make_batch(cfg(8, 2, 64, seed=23), ctx_lens=ctx, block_lens=blk)
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck, flags=flags))
    U.assert_close_bf16(got, want, f"300 requests flags={flags}")


def test_context_slack_rows_are_never_read():
    # the segment holds more rows than ctx_lens says; the extra rows are NaN and must
    # not reach the output (neither through K scores nor through V with weight 0)
    b = W.make_batch(cfg(32, 8, 128, seed=9), ctx_lens=[130, 77], block_lens=[16, 16])
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    csl = np.array([0, 200, 300], np.int32)
    nan = np.uint16(0x7FC0)
    kk = np.full((300, 8, 128), nan, np.uint16)
    vv = np.full((300, 8, 128), nan, np.uint16)
    old = b.ctx_start_loc
    for r in range(2):
        n = b.ctx_lens[r]
        kk[csl[r]:csl[r] + n] = ck[old[r]:old[r] + n]
        vv[csl[r]:csl[r] + n] = b.ctx_v[old[r]:old[r] + n]
    b.ctx_start_loc, b.ctx_v = csl, vv
    got = U.dev_to_f64(U.gpu_attention(b, kk))
    U.assert_close_bf16(got, want, "slack")


def test_zero_query_gives_mean_of_values():
    # q = 0 -> uniform weights; the GPU must average exactly the allowed V rows
    b = W.make_batch(cfg(8, 2, 128, True, 40, seed=10), ctx_lens=[100, 3], block_lens=[16, 7])
    b.q[:] = 0
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck))
    U.assert_close_bf16(got, want, "zero-q")


def test_scale_override():
    b = W.make_batch(cfg(8, 4, 64, seed=11), ctx_lens=[90], block_lens=[16])
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck, scale=0.3)
    got = U.dev_to_f64(U.gpu_attention(b, ck, scale=0.3))
    U.assert_close_bf16(got, want, "scale")


def test_bad_device_metadata_is_reported_not_faulted():
    import torch
    lib = D()
    b = W.make_batch(cfg(8, 4, 128, seed=12), ctx_lens=[50, 60], block_lens=[16, 16])
    ck = U.stored_ctx_k(b)
    b.ctx_lens = np.array([50, 999], np.int32)  # more live rows than the segment holds
    ws = lib.alloc_workspace(lib.workspace_size(2, 32, 8, 4, 128, 110, 2000, 16))
    out = lib.block_attention(U.bf16_dev(b.q), U.bf16_dev(b.k_blk), U.bf16_dev(b.v_blk), U.bf16_dev(ck),
                              U.bf16_dev(b.ctx_v), U.i32_dev(b.query_start_loc), U.i32_dev(b.ctx_start_loc),
                              U.i32_dev(b.ctx_lens), U.i32_dev(b.positions), U.bf16_dev(b.q_norm_w),
                              U.bf16_dev(b.k_norm_w), max_ctx_len=2000, max_block_len=16, workspace=ws)
    torch.cuda.synchronize()
    with pytest.raises(lib.DFlashError) as e:
        lib.check_error(ws)
    assert e.value.code == lib.ERR_DEVICE_METADATA
    # the valid request was still computed
    want = U.oracle_attention(W.make_batch(cfg(8, 4, 128, seed=12), ctx_lens=[50, 60], block_lens=[16, 16]), ck)
    U.assert_close_bf16(U.dev_to_f64(out)[:16], want[:16], "valid request")


def test_empty_batch_is_a_no_op():
    import torch
    lib = D()
    z16 = torch.zeros((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = lib.block_attention(z16, torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(1, dtype=torch.int32, device="cuda"),
                              torch.zeros(1, dtype=torch.int32, device="cuda"),
                              torch.zeros(0, dtype=torch.int32, device="cuda"),
                              torch.zeros(0, dtype=torch.int32, device="cuda"),
                              torch.ones(64, dtype=torch.bfloat16, device="cuda"),
                              torch.ones(64, dtype=torch.bfloat16, device="cuda"), max_ctx_len=0, max_block_len=1)
    assert out.shape == (0, 4, 64)


@pytest.mark.parametrize("flags", [0, 1, 2])
def test_more_requests_than_one_schedule_scan(flags):
    # past 1024 requests every CTA scans the requests in several chunks (an even split of the
    # tiles, and a second pass to find its segments)
    rng = np.random.default_rng(29)
    n = 1100
    ctx = rng.integers(0, 300, n)
    ctx[::13] = 0
    blk = rng.integers(1, 17, n)
    b = W.make_batch(cfg(8, 2, 64, seed=29), ctx_lens=ctx, block_lens=blk)
    ck = U.stored_ctx_k(b)
    want = U.oracle_attention(b, ck)
    got = U.dev_to_f64(U.gpu_attention(b, ck, flags=flags))
    U.assert_close_bf16(got, want, f"1100 requests flags={flags}")
