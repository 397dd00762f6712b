"""Writes the oracle regression fixtures in this folder.

The pages this path follows print no worked example, so these fixtures pin the
oracle to its own earlier output: a change to its arithmetic shows up as a diff
here and has to be justified. The script calls only the oracle and the seeded
input generator; nothing here comes from the CUDA path.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from speculative_decoding_draft_rmsnorm_gb300 import workloads as W  # noqa: E402

CASES = {
    # configuration 1 of the workload table: one request, C=64, B=16, Hq=4, Hkv=2, Dh=64
    "tiny_bidirectional": dict(cfg="tiny"),
    # a small ragged SWA case: causal with window 5, three requests, one with no context
    "small_swa": dict(cfg=None, hq=4, hkv=2, dh=64, causal=True, window=5, ctx=[9, 0, 6], blk=[4, 3, 5]),
}


def run_case(spec):
    if spec["cfg"]:
        b = W.make_batch(W.CONFIGS[spec["cfg"]])
    else:
        cfg = W.Config("golden", 0, 4, spec["hq"], spec["hkv"], spec["dh"], causal=spec["causal"],
                       window=spec["window"], ctx_len=0, seed=5)
        b = W.make_batch(cfg, ctx_lens=spec["ctx"], block_lens=spec["blk"])
    c = b.cfg
    _, ck16 = oracle.context_kv(b.ctx_k_raw, b.ctx_pos, b.k_norm_w, c.eps, c.theta)
    out = oracle.block_attention(b.q, b.k_blk, b.v_blk, ck16, b.ctx_v, b.query_start_loc, b.ctx_start_loc,
                                 b.ctx_lens, b.positions, b.q_norm_w, b.k_norm_w, eps=c.eps, theta=c.theta,
                                 causal=c.causal, window=c.window)
    return b, ck16, out


def summarise(b, ck16, out):
    t, hq, dh = out.shape
    picks = [(0, 0), (t // 2, hq - 1), (t - 1, hq // 2)]
    return {
        "shape": list(out.shape),
        "sum": float(out.sum()),
        "abs_sum": float(np.abs(out).sum()),
        "rows": {f"{i},{h}": [float(v) for v in out[i, h, :8]] for i, h in picks},
        "ctx_k_bits_sum": int(ck16.astype(np.int64).sum()),
    }


def main():
    for name, spec in CASES.items():
        data = summarise(*run_case(spec))
        data["source"] = ("oracle/dflash_oracle.c on the seeded inputs of "
                          "speculative_decoding_draft_rmsnorm_gb300/workloads.py; written by make_golden.py")
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(data, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
