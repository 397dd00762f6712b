"""Pins of the paged-append oracle (CPU).

vllm.cpp qwen3_dflash.cpp, AppendContextKVDevice: new context rows of a request continue its
stored context, project like every other context row (k_norm, then NeoX RoPE at their
positions, V raw), land at their paged slots, and the request's length grows by their count.
The store built this way is the contiguous store with its rows placed in pages, so identity
paging must give exactly the contiguous context K/V of the same rows.
"""
from __future__ import annotations

import numpy as np

import oracle
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W

FILL = np.uint16(0x7FC0)


def _rows(n, hkv=2, dh=64, seed=4):
    k = W.normal_bf16(seed, 0, n * hkv * dh).reshape(n, hkv, dh)
    v = W.normal_bf16(seed, 1, n * hkv * dh).reshape(n, hkv, dh)
    w = W.uniform_bf16(seed, 2, dh, 0.5, 1.5)
    return k, v, w


def _pool(pages, ps, hkv=2, dh=64):
    return np.full((pages, ps, hkv, dh), FILL, dtype=np.uint16)


def test_rows_land_by_hand():
    # two requests, pages of 2 rows. Request 0 holds 3 rows and appends 2: positions 3 and 4,
    # i.e. page index 1 (id 0) row 1 and page index 2 (id 2) row 0. Request 1 is empty and
    # appends 3: positions 0, 1, 2 -> page id 1 rows 0 and 1, page id 3 row 0.
    k, _, w = _rows(5, hkv=1)
    v = np.stack([np.full((1, 64), t + 1, dtype=np.uint16) for t in range(5)])
    kp, vp, lens, bad = oracle.paged_append(_pool(5, 2, hkv=1), _pool(5, 2, hkv=1), [[4, 0, 2], [1, 3, -1]], [3, 0],
                                            [0, 2, 5], k, v, w, 2)
    assert not bad
    assert lens.tolist() == [5, 3]
    want_v = {(0, 1): 1, (2, 0): 2, (1, 0): 3, (1, 1): 4, (3, 0): 5}
    for pg in range(5):
        for off in range(2):
            got = vp[pg, off, 0]
            assert np.all(got == want_v.get((pg, off), FILL)), (pg, off)
            assert np.all(np.isnan(W.bf16_to_f64(kp[pg, off]))) == ((pg, off) not in want_v)


def test_identity_paging_gives_the_contiguous_store():
    # one request, pages handed out in order from an empty store: page p holds positions
    # [p * ps, (p + 1) * ps), so the pool read row by row is the contiguous context store
    n, ps = 77, 16
    k, v, w = _rows(n)
    pages = (n + ps - 1) // ps
    kp, vp, lens, bad = oracle.paged_append(_pool(pages, ps), _pool(pages, ps), [list(range(pages))], [0], [0, n],
                                            k, v, w, ps, eps=1e-6, theta=1e6)
    assert not bad and lens.tolist() == [n]
    want_k = oracle.context_kv(k, np.arange(n, dtype=np.int32), w, 1e-6, 1e6)[1]
    assert np.array_equal(kp.reshape(-1, 2, 64)[:n], want_k)
    assert np.array_equal(vp.reshape(-1, 2, 64)[:n], v)


def test_appending_in_two_steps_equals_one_step():
    n, ps = 50, 16
    k, v, w = _rows(n)
    bt = [[3, 0, 2, 1], [7, 5, 4, 6]]
    one = oracle.paged_append(_pool(8, ps), _pool(8, ps), bt, [5, 0], [0, 20, 50], k, v, w, ps)
    # step 1: 13 rows of request 0, 11 of request 1; step 2: the rest
    idx1 = list(range(0, 13)) + list(range(20, 31))
    idx2 = list(range(13, 20)) + list(range(31, 50))
    a = oracle.paged_append(_pool(8, ps), _pool(8, ps), bt, [5, 0], [0, 13, 24], k[idx1], v[idx1], w, ps)
    b = oracle.paged_append(a[0], a[1], bt, a[2], [0, 7, 26], k[idx2], v[idx2], w, ps)
    assert np.array_equal(one[0], b[0]) and np.array_equal(one[1], b[1])
    assert one[2].tolist() == b[2].tolist() == [25, 30]
    assert not (one[3] or a[3] or b[3])


def test_a_request_that_does_not_fit_changes_nothing():
    # the page's capacity check comes before any write: a request whose new rows run past its
    # block table, or onto a page id outside the pool, writes none of them and keeps its length
    k, v, w = _rows(6)
    # a 2-page table (4 rows of 2) holding 3 rows: position 3 would fit, 4 and 5 do not
    kp, vp, lens, bad = oracle.paged_append(_pool(4, 2), _pool(4, 2), [[0, 1]], [3], [0, 3], k[:3], v[:3], w, 2)
    assert bad and lens.tolist() == [3]
    assert np.all(vp == FILL) and np.all(kp == FILL)
    # exactly full: positions 3 only
    kp, vp, lens, bad = oracle.paged_append(_pool(4, 2), _pool(4, 2), [[0, 1]], [3], [0, 1], k[:1], v[:1], w, 2)
    assert not bad and lens.tolist() == [4] and np.array_equal(vp[1, 1], v[0])
    # a page id outside the pool on the second page only: the first page's row is not written either
    kp, vp, lens, bad = oracle.paged_append(_pool(4, 2), _pool(4, 2), [[2, 9]], [1], [0, 2], k[:2], v[:2], w, 2)
    assert bad and lens.tolist() == [1] and np.all(vp == FILL)
    # start locations that run past the rows: nothing happens
    kp, vp, lens, bad = oracle.paged_append(_pool(4, 2), _pool(4, 2), [[0, 1]], [0], [0, 7], k, v, w, 2)
    assert bad and lens.tolist() == [0] and np.all(vp == FILL)


def test_the_requests_that_fit_append_as_if_alone():
    # request 1 overflows its 2-page table; requests 0 and 2 must come out as an append of
    # just their rows, and request 1's pages and length stay as they were
    ps = 4
    k, v, w = _rows(17)
    bt = [[0, 1], [2, 3], [4, 5]]
    lens = [1, 5, 0]
    nsl = [0, 6, 10, 17]  # request 1 appends 4 rows after 5: positions 5..8, past 8 rows
    kp, vp, out_lens, bad = oracle.paged_append(_pool(6, ps), _pool(6, ps), bt, lens, nsl, k, v, w, ps)
    assert bad and out_lens.tolist() == [7, 5, 7]
    idx = list(range(0, 6)) + list(range(10, 17))
    alone = oracle.paged_append(_pool(6, ps), _pool(6, ps), [[0, 1], [4, 5]], [1, 0], [0, 6, 13], k[idx], v[idx], w,
                                ps)
    assert not alone[3]
    assert np.array_equal(kp, alone[0]) and np.array_equal(vp, alone[1])
    assert np.all(vp[2:4] == FILL) and np.all(kp[2:4] == FILL)
