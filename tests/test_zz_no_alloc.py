"""The no-allocation entry point against the regular one.

dflash_block_attention_noalloc serves callers that cannot allocate device memory (a
host that owns all device memory, code inside another allocator's callback, static
memory plans): its scratch is an array compiled into the library. This test calls it
through the C ABI twice in a row -- the second call runs on scratch the first one left
behind -- and checks both outputs against dflash_block_attention with a caller
workspace, within the bf16 tolerance the parity tests use. This file is collected last.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import speculative_decoding_draft_rmsnorm_gb300 as D
    lib = D.load()
    fn = lib.dflash_block_attention_noalloc
    P, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [P] * 11 + [I32, I64, I32, I32, I32, I64, I32, I32, F32, F32, F32, I32, I32, I32, P, I32, P]
    fn.restype = I32
    return D, lib, fn


@pytest.mark.parametrize("case", [
    ("gqa4", 32, 8, 128, False, 0, [700, 40, 2000], [16, 16, 16]),
    ("swa_dh64", 8, 4, 64, True, 96, [300, 5], [16, 9]),
])
def test_noalloc_matches_workspace_entry_point_twice(case):
    import torch
    D, lib, fn = _noalloc_fn()
    name, hq, hkv, dh, causal, window, cl, bl = case
    outs = []
    for seed in (31, 32):  # two calls in a row, different inputs
        b = W.make_batch(W.Config(name, 0, 16, hq, hkv, dh, causal=causal, window=window, ctx_len=0, seed=seed),
                         ctx_lens=cl, block_lens=bl)
        ck = U.stored_ctx_k(b)
        want = U.dev_to_f64(U.gpu_attention(b, ck))
        dev = dict(q=U.bf16_dev(b.q), k=U.bf16_dev(b.k_blk), v=U.bf16_dev(b.v_blk), ck=U.bf16_dev(ck),
                   cv=U.bf16_dev(b.ctx_v), qsl=U.i32_dev(b.query_start_loc), csl=U.i32_dev(b.ctx_start_loc),
                   cl=U.i32_dev(b.ctx_lens), pos=U.i32_dev(b.positions), qw=U.bf16_dev(b.q_norm_w),
                   kw=U.bf16_dev(b.k_norm_w))
        t = b.q.shape[0]
        out = torch.empty((t, hq, dh), dtype=torch.bfloat16, device="cuda")
        rc = fn(*(dev[k].data_ptr() for k in ("q", "k", "v", "ck", "cv", "qsl", "csl", "cl", "pos", "qw", "kw")),
                len(cl), t, hq, hkv, dh, ck.shape[0], max(cl), max(bl), b.cfg.eps, b.cfg.theta, 0.0, int(causal),
                window, 0, out.data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, lib.dflash_last_error().decode()
        torch.cuda.synchronize()
        got = U.dev_to_f64(out)
        U.assert_close_bf16(got, want, f"{name} seed {seed}")
        outs.append(got)
    assert not np.array_equal(outs[0], outs[1])


def test_noalloc_rejects_calls_beyond_its_scratch():
    import torch
    D, lib, fn = _noalloc_fn()
    # 8192 block rows x 64 heads x 128 dims of normed q alone exceed the 32 MiB scratch
    t, hq, hkv, dh = 8192, 64, 8, 128
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(*([z.data_ptr()] * 11), 1, t, hq, hkv, dh, 0, 0, t, 1e-6, 1e6, 0.0, 0, 0, 0, z.data_ptr(), 0,
            torch.cuda.current_stream().cuda_stream)
    assert rc == D.ERR_WORKSPACE
    assert b"32" in lib.dflash_last_error() or b"scratch" in lib.dflash_last_error()
