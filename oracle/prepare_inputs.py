"""Oracle of the DFlash draft step's input preparation (pure integer, plain Python loops).

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the smoke check and the
benchmark's CPU leg call it.

qwen3_dflash.cpp, PrepareDflashInputs (a host restatement of vLLM's
_prepare_dflash_inputs_kernel): before a draft step, every request r of the batch gets

  * its context (the target tokens of this step that were scored, target_query_start_loc[r]
    .. target_query_start_loc[r+1]) re-addressed: each token keeps its target position and
    gets the draft KV slot of that position;
  * a query block of num_query_per_req tokens at the positions right after the last accepted
    token (the last context token that was not rejected): the first carries the bonus token
    (the token sampled last, or the next prefill token when nothing was sampled), the others
    the parallel-drafting (mask) token; positions are clamped to max_model_len - 1, slots
    are taken from the unclamped position;
  * its draft sequence length, last accepted position + 1 + num_query_per_req;
  * the map of the block rows whose outputs are sampled: the rows from offset 1 on (or from
    offset 0 when sampling from the anchor), the position each sample stands for (the row's
    position, plus one when sampling from the anchor) and the request state it belongs to.

A slot is block_table[r, min(pos // block_size, stride - 1)] * block_size + pos % block_size.
Entries past the live requests are padded so that a captured graph can replay with fewer
requests: query_start_loc repeats the end of the last query block, seq_lens 0, sample rows
(0, 0, -1), query slots -1 (vLLM's PAD_SLOT_ID).

Readings where the page leaves a step open (each is stated in the design notes):
  * dtypes follow vLLM: positions and slots int64, token ids, lengths and indices int32;
  * a request has at most num_speculative_steps sampled rows (num_query_per_req minus the
    sample offset <= num_speculative_steps); with fewer, its remaining sample rows stay 0;
  * positions are >= 0 (floor and truncating division then agree);
  * the request state index addresses last_sampled and next_prefill_tokens.
"""
from __future__ import annotations

import numpy as np

PAD_SLOT_ID = -1


class PrepareError(ValueError):
    pass


def prepare_dflash_inputs(idx_mapping, target_query_start_loc, num_rejected, num_sampled, last_sampled,
                          next_prefill_tokens, target_positions, block_table, *, num_query_per_req: int,
                          num_speculative_steps: int, block_size: int, max_num_reqs: int, max_num_tokens: int,
                          max_model_len: int, parallel_drafting_token_id: int, sample_from_anchor: bool,
                          num_target_tokens: int | None = None) -> dict:
    """The prepared draft inputs as a dict of numpy arrays (see the module docstring).

    block_table is [>= num_reqs, stride]. num_target_tokens sizes the context arrays; by
    default it is target_query_start_loc[-1] (entries past that are 0).
    """
    idx_mapping = [int(x) for x in idx_mapping]
    qsl = [int(x) for x in target_query_start_loc]
    n = len(idx_mapping)
    nq, ns, bs = int(num_query_per_req), int(num_speculative_steps), int(block_size)
    bt = np.asarray(block_table, dtype=np.int64)
    stride = bt.shape[1]
    pos_in = np.asarray(target_positions, dtype=np.int64)
    n_tgt = qsl[-1] if num_target_tokens is None else int(num_target_tokens)
    off0 = 0 if sample_from_anchor else 1
    if n <= 0 or len(qsl) != n + 1 or n > max_num_reqs or n * nq > max_num_tokens or nq - off0 > ns:
        raise PrepareError("sizes")
    if qsl[0] < 0 or qsl[-1] > n_tgt or any(qsl[r + 1] < qsl[r] for r in range(n)):
        raise PrepareError("target_query_start_loc")

    def slot_of(r: int, pos: int) -> int:
        if pos < 0:
            raise PrepareError("negative position")
        page = min(pos // bs, stride - 1)
        return int(bt[r, page]) * bs + pos % bs

    out = {
        "input_ids": np.zeros(n * nq, dtype=np.int32),
        "query_positions": np.zeros(n * nq, dtype=np.int64),
        "query_start_loc": np.zeros(max_num_reqs + 1, dtype=np.int32),
        "seq_lens": np.zeros(max_num_reqs, dtype=np.int32),
        "query_slot_mapping": np.zeros(max_num_tokens, dtype=np.int64),
        "context_positions": np.zeros(n_tgt, dtype=np.int64),
        "context_slot_mapping": np.zeros(n_tgt, dtype=np.int64),
        "sample_indices": np.zeros(max_num_reqs * ns, dtype=np.int32),
        "sample_pos": np.zeros(max_num_reqs * ns, dtype=np.int64),
        "sample_idx_mapping": np.zeros(max_num_reqs * ns, dtype=np.int32),
    }
    for r in range(n):
        state = idx_mapping[r]
        if not 0 <= state < len(last_sampled) or not 0 <= state < len(next_prefill_tokens):
            raise PrepareError("request state index")
        first, end = qsl[r], qsl[r + 1]
        accepted_end = end - int(num_rejected[r])  # one past the last accepted context token
        if not 0 < accepted_end <= n_tgt:
            raise PrepareError("rejected count")
        last_pos = int(pos_in[accepted_end - 1])
        bonus = int(last_sampled[state]) if int(num_sampled[r]) > 0 else int(next_prefill_tokens[state])

        # the context tokens keep their positions and get their slots
        for t in range(first, end):
            p = int(pos_in[t])
            out["context_positions"][t] = p
            out["context_slot_mapping"][t] = slot_of(r, p)

        # the query block right after the last accepted token
        for k in range(nq):
            row = r * nq + k
            p = last_pos + 1 + k
            out["input_ids"][row] = bonus if k == 0 else parallel_drafting_token_id
            out["query_positions"][row] = min(p, max_model_len - 1)
            out["query_slot_mapping"][row] = slot_of(r, p)
            if k >= off0:
                s = r * ns + (k - off0)
                out["sample_indices"][s] = row
                out["sample_pos"][s] = p + 1 if sample_from_anchor else p
                out["sample_idx_mapping"][s] = state

        out["query_start_loc"][r] = r * nq
        out["seq_lens"][r] = last_pos + 1 + nq

    # padding past the live requests
    out["query_start_loc"][n:] = n * nq
    out["sample_idx_mapping"][n * ns:] = -1
    out["query_slot_mapping"][n * nq:] = PAD_SLOT_ID
    return out
