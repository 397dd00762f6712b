"""The no-allocation entry point against the regular one and the oracle.

dflash_block_attention_noalloc serves callers that cannot allocate device memory (a host
that owns all device memory, code inside another allocator's callback, static memory
plans): its scratch is an array compiled into the library. This test calls it through the
C ABI twice in a row -- the second call runs on scratch the first one left behind -- and
requires each output to equal, bit for bit, dflash_block_attention's on a caller workspace
(the same kernels, grid and inputs), and to sit within the bf16 tolerance of the f64
oracle. Device-side errors of a noalloc call are read back through
dflash_block_attention_noalloc_check_error. This file is collected last.
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
    chk = lib.dflash_block_attention_noalloc_check_error
    chk.argtypes = [P]
    chk.restype = I32
    return D, lib, fn, chk


def _call(fn, b, ck, out, ctx_lens=None):
    import torch
    c = b.cfg
    dev = [U.bf16_dev(b.q), U.bf16_dev(b.k_blk), U.bf16_dev(b.v_blk), U.bf16_dev(ck), U.bf16_dev(b.ctx_v),
           U.i32_dev(b.query_start_loc), U.i32_dev(b.ctx_start_loc),
           U.i32_dev(b.ctx_lens if ctx_lens is None else ctx_lens), U.i32_dev(b.positions), U.bf16_dev(b.q_norm_w),
           U.bf16_dev(b.k_norm_w)]
    t, hq, dh = b.q.shape
    rc = fn(*(x.data_ptr() for x in dev), len(b.ctx_lens), t, hq, c.hkv, dh, ck.shape[0],
            int(max(1, b.ctx_lens.max())), int(b.block_lens.max()), c.eps, c.theta, 0.0, int(c.causal), c.window, 0,
            out.data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
    return rc, dev


@pytest.mark.parametrize("case", [
    ("gqa4", 32, 8, 128, False, 0, [700, 40, 2000], [16, 16, 16]),
    ("swa_dh64", 8, 4, 64, True, 96, [300, 5], [16, 9]),
])
def test_noalloc_equals_workspace_entry_point_twice(case):
    import torch
    D, lib, fn, chk = _noalloc_fn()
    name, hq, hkv, dh, causal, window, cl, bl = case
    outs = []
    for seed in (31, 32):  # two calls in a row, different inputs
        b = W.make_batch(W.Config(name, 0, 16, hq, hkv, dh, causal=causal, window=window, ctx_len=0, seed=seed),
                         ctx_lens=cl, block_lens=bl)
        ck = U.stored_ctx_k(b)
        ref = U.gpu_attention(b, ck)
        out = torch.empty((b.q.shape[0], hq, dh), dtype=torch.bfloat16, device="cuda")
        rc, _ = _call(fn, b, ck, out)
        assert rc == 0, lib.dflash_last_error().decode()
        torch.cuda.synchronize()
        assert chk(torch.cuda.current_stream().cuda_stream) == 0, lib.dflash_last_error().decode()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{name} seed {seed}: bits differ"
        got = U.dev_to_f64(out)
        U.assert_close_bf16(got, U.oracle_attention(b, ck), f"{name} seed {seed} vs oracle")
        outs.append(got)
    assert not np.array_equal(outs[0], outs[1])


def test_noalloc_device_errors_are_readable():
    # a ctx_lens entry above its segment is skipped on the device and recorded in the built-in
    # scratch; the reader reports it, and the next good call clears it
    import torch
    D, lib, fn, chk = _noalloc_fn()
    b = W.make_batch(W.Config("bad", 0, 16, 8, 4, 128, ctx_len=0, seed=33), ctx_lens=[50, 60], block_lens=[16, 16])
    ck = U.stored_ctx_k(b)
    out = torch.zeros((32, 8, 128), dtype=torch.bfloat16, device="cuda")
    rc, _ = _call(fn, b, ck, out, ctx_lens=np.array([50, 999], np.int32))
    assert rc == 0
    assert chk(torch.cuda.current_stream().cuda_stream) == D.ERR_DEVICE_METADATA
    U.assert_close_bf16(U.dev_to_f64(out)[:16], U.oracle_attention(b, ck)[:16], "the valid request")
    rc, _ = _call(fn, b, ck, out)
    assert rc == 0
    assert chk(torch.cuda.current_stream().cuda_stream) == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    import torch
    D, lib, fn, chk = _noalloc_fn()
    # 8192 block rows x 64 heads x 128 dims of normed q alone exceed the 32 MiB scratch
    t, hq, hkv, dh = 8192, 64, 8, 128
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(*([z.data_ptr()] * 11), 1, t, hq, hkv, dh, 0, 0, t, 1e-6, 1e6, 0.0, 0, 0, 0, z.data_ptr(), 0,
            torch.cuda.current_stream().cuda_stream)
    assert rc == D.ERR_WORKSPACE
    assert b"scratch" in lib.dflash_last_error()
