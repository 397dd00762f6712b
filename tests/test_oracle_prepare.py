"""Pins of the draft-step input preparation oracle (CPU).

vllm.cpp qwen3_dflash.cpp, PrepareDflashInputs: the expected arrays of the two worked cases
below were derived by hand from the rules in the oracle's docstring (slot = page id * block
size + position mod block size, the query block after the last accepted token, the sample
map, the padding); the random cases check properties that hold for every batch.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle.prepare_inputs import PrepareError
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W


def _run(**kw):
    args = dict(kw)
    arrays = [args.pop(k) for k in ("idx_mapping", "target_query_start_loc", "num_rejected", "num_sampled",
                                    "last_sampled", "next_prefill_tokens", "target_positions", "block_table")]
    return oracle.prepare_dflash_inputs(*arrays, **args)


def test_worked_case_two_requests():
    # request 0 (state 2): context positions 5, 6, 7, one rejected, so the last accepted
    # position is 6; it sampled, so its bonus token is last_sampled[2] = 12; its queries sit at
    # 7, 8, 9 (pages 1, 2, 2 of its table: page ids 4, 9, 9). Request 1 (state 0): positions
    # 2, 3, none rejected, nothing sampled: bonus next_prefill_tokens[0] = 20, queries at
    # 4, 5, 6 (page 1: id 8).
    o = _run(idx_mapping=[2, 0], target_query_start_loc=[0, 3, 5], num_rejected=[1, 0], num_sampled=[1, 0],
             last_sampled=[10, 11, 12], next_prefill_tokens=[20, 21, 22], target_positions=[5, 6, 7, 2, 3],
             block_table=[[7, 4, 9], [1, 8, 3]], num_query_per_req=3, num_speculative_steps=2, block_size=4,
             max_num_reqs=3, max_num_tokens=8, max_model_len=12, parallel_drafting_token_id=99,
             sample_from_anchor=False)
    want = {
        "input_ids": [12, 99, 99, 20, 99, 99],
        "query_positions": [7, 8, 9, 4, 5, 6],
        "query_start_loc": [0, 3, 6, 6],
        "seq_lens": [10, 7, 0],
        "query_slot_mapping": [19, 36, 37, 32, 33, 34, -1, -1],
        "context_positions": [5, 6, 7, 2, 3],
        "context_slot_mapping": [17, 18, 19, 6, 7],
        "sample_indices": [1, 2, 4, 5, 0, 0],
        "sample_pos": [8, 9, 5, 6, 0, 0],
        "sample_idx_mapping": [2, 2, 0, 0, -1, -1],
    }
    assert set(o) == set(want)
    for k, v in want.items():
        assert o[k].tolist() == v, k


def test_worked_case_clamps_and_anchor_sampling():
    # one request, pages of 4, a table of 2 pages: queries at 8, 9, 10 lie past the table and
    # take its last page (id 1); their positions clamp to max_model_len - 1 = 8, their slots do
    # not. Sampling from the anchor: every query row is sampled, at its position + 1.
    o = _run(idx_mapping=[0], target_query_start_loc=[0, 2], num_rejected=[0], num_sampled=[1], last_sampled=[5],
             next_prefill_tokens=[6], target_positions=[6, 7], block_table=[[3, 1]], num_query_per_req=3,
             num_speculative_steps=3, block_size=4, max_num_reqs=1, max_num_tokens=3, max_model_len=9,
             parallel_drafting_token_id=99, sample_from_anchor=True)
    want = {
        "input_ids": [5, 99, 99], "query_positions": [8, 8, 8], "query_start_loc": [0, 3], "seq_lens": [11],
        "query_slot_mapping": [4, 5, 6], "context_positions": [6, 7], "context_slot_mapping": [6, 7],
        "sample_indices": [0, 1, 2], "sample_pos": [9, 10, 11], "sample_idx_mapping": [0, 0, 0],
    }
    for k, v in want.items():
        assert o[k].tolist() == v, k


@pytest.mark.parametrize("anchor", [False, True])
def test_random_batches_satisfy_the_rules(anchor):
    b = W.make_prepare_batch(5, 24, sample_from_anchor=anchor, max_model_len=1 << 30)
    o = _run(**b.__dict__)
    n, nq, ns, bs = len(b.idx_mapping), b.num_query_per_req, b.num_speculative_steps, b.block_size
    qsl = b.target_query_start_loc
    assert np.array_equal(o["context_positions"], b.target_positions)
    for r in range(n):
        s = b.idx_mapping[r]
        last = int(b.target_positions[qsl[r + 1] - b.num_rejected[r] - 1])
        qp = o["query_positions"][r * nq:(r + 1) * nq]
        assert qp.tolist() == list(range(last + 1, last + 1 + nq))
        assert o["seq_lens"][r] == qp[-1] + 1
        bonus = b.last_sampled[s] if b.num_sampled[r] > 0 else b.next_prefill_tokens[s]
        assert o["input_ids"][r * nq] == bonus
        assert np.all(o["input_ids"][r * nq + 1:(r + 1) * nq] == b.parallel_drafting_token_id)
        # slots: the page that holds the position, at its offset
        for p, sl in zip(qp, o["query_slot_mapping"][r * nq:(r + 1) * nq]):
            assert sl == int(b.block_table[r, p // bs]) * bs + p % bs
        for t in range(qsl[r], qsl[r + 1]):
            p = int(b.target_positions[t])
            assert o["context_slot_mapping"][t] == int(b.block_table[r, p // bs]) * bs + p % bs
        first = 0 if anchor else 1
        rows = o["sample_indices"][r * ns:(r + 1) * ns]
        assert rows.tolist() == list(range(r * nq + first, r * nq + nq))
        assert np.array_equal(o["sample_pos"][r * ns:(r + 1) * ns], o["query_positions"][rows] + (1 if anchor else 0))
        assert np.all(o["sample_idx_mapping"][r * ns:(r + 1) * ns] == s)
    assert np.all(o["query_start_loc"][:n] == np.arange(n) * nq)
    assert np.all(o["query_start_loc"][n:] == n * nq)
    assert np.all(o["seq_lens"][n:] == 0)
    assert np.all(o["query_slot_mapping"][n * nq:] == -1)
    assert np.all(o["sample_idx_mapping"][n * ns:] == -1)
    assert np.all(o["sample_indices"][n * ns:] == 0) and np.all(o["sample_pos"][n * ns:] == 0)


def test_identity_block_table_gives_the_position_as_slot():
    # one contiguous run of pages per request, in order: slot = base + position
    b = W.make_prepare_batch(9, 12)
    stride = b.block_table.shape[1]
    b.block_table = (np.arange(12)[:, None] * stride + np.arange(stride)[None, :]).astype(np.int32)
    o = _run(**b.__dict__)
    req = np.searchsorted(b.target_query_start_loc, np.arange(len(b.target_positions)), side="right") - 1
    assert np.array_equal(o["context_slot_mapping"], req * stride * b.block_size + b.target_positions)


def test_rejecting_more_tokens_moves_the_query_block_back():
    b = W.make_prepare_batch(3, 16, prefill_frac=0.0)
    o1 = _run(**b.__dict__)
    counts = np.diff(b.target_query_start_loc)
    before = b.num_rejected.astype(np.int64)
    b.num_rejected = np.minimum(before + 1, counts - 1).astype(np.int32)
    o2 = _run(**b.__dict__)
    nq = b.num_query_per_req
    moved = b.num_rejected - before  # 1 where one more token was rejected (positions are consecutive)
    assert moved.sum() > 0
    shift = np.repeat(moved, nq)
    assert np.array_equal(o1["query_positions"] - o2["query_positions"], shift)
    assert np.array_equal(o1["seq_lens"][:16] - o2["seq_lens"][:16], moved)


def test_more_sampled_rows_than_steps_and_negative_positions_are_rejected():
    b = W.make_prepare_batch(1, 4)
    kw = dict(b.__dict__)
    kw["num_speculative_steps"] = b.num_query_per_req - 2
    with pytest.raises(PrepareError):
        _run(**kw)
    kw = dict(b.__dict__)
    kw["target_positions"] = b.target_positions.copy()
    kw["target_positions"][0] = -1
    with pytest.raises(PrepareError):
        _run(**kw)


def test_context_arrays_longer_than_the_scored_tokens_end_in_zeros():
    # a caller may size the context arrays for a larger batch; entries past the last request's
    # tokens belong to no request and are written as 0
    b = W.make_prepare_batch(4, 5)
    n_tgt = int(b.target_query_start_loc[-1])
    kw = dict(b.__dict__)
    kw["target_positions"] = np.concatenate([b.target_positions, np.full(7, 12345, dtype=np.int64)])
    o = _run(**kw, num_target_tokens=n_tgt + 7)
    base = _run(**b.__dict__)
    assert np.array_equal(o["context_positions"][:n_tgt], base["context_positions"])
    assert np.array_equal(o["context_slot_mapping"][:n_tgt], base["context_slot_mapping"])
    assert np.all(o["context_positions"][n_tgt:] == 0) and np.all(o["context_slot_mapping"][n_tgt:] == 0)
