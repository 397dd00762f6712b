"""A bounded device wait that runs out, and the call after it.

Every mbarrier wait of the attention kernel gives up after a time limit, records
DFLASH_ERR_DEVICE_TIMEOUT in the workspace's error word and unwinds: the other roles of
the CTA see the shared abort flag and stop, the producer waits (bounded) for the copies it
issued, the MMA thread for the MMAs it issued, and the CTA frees its tensor memory and
exits. Nothing here faults or hangs the GPU: the test library is the product's sources
built with DFLASH_WAIT_TEST, where a wait gives up after 5 ms and a hook makes one CTA's
producer skip one V tile's copy, so the consumer's wait on that tile runs out. The test
asserts that the call returns within a second, that dflash_check_error reports the
timeout, and that the next call on the same workspace, with the hook off, is bit-identical
to the product library's and within tolerance of the f64 oracle.
"""
import ctypes
import time

import numpy as np
import pytest

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from tests import util as U

pytestmark = pytest.mark.gpu


def _test_lib():
    import speculative_decoding_draft_rmsnorm_gb300 as D
    from speculative_decoding_draft_rmsnorm_gb300 import _build
    D.load()  # the product library (built by the package's build step, with this one)
    if not _build.up_to_date(_build.WAIT_TEST_LIB_PATH):
        _build.build()
    lib = ctypes.CDLL(_build.WAIT_TEST_LIB_PATH)
    P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.dflash_block_attention.restype = I32
    lib.dflash_block_attention.argtypes = ([P] * 11 + [I32, I64, I32, I32, I32, I64, I32, I32, F32, F32, F32,
                                                       I32, I32, I32, P, P, SZ, I32, P])
    lib.dflash_check_error.restype = I32
    lib.dflash_check_error.argtypes = [P, P]
    lib.dflash_last_error.restype = ctypes.c_char_p
    lib.dflash_test_withhold_v_tile.restype = I32
    lib.dflash_test_withhold_v_tile.argtypes = [I32, I32]
    return D, lib


def _call(lib, b, ck, out, ws, flags):
    import torch
    c = b.cfg
    dev = [U.bf16_dev(b.q), U.bf16_dev(b.k_blk), U.bf16_dev(b.v_blk), ck, U.bf16_dev(b.ctx_v),
           U.i32_dev(b.query_start_loc), U.i32_dev(b.ctx_start_loc), U.i32_dev(b.ctx_lens), U.i32_dev(b.positions),
           U.bf16_dev(b.q_norm_w), U.bf16_dev(b.k_norm_w)]
    t, hq, dh = b.q.shape
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.dflash_block_attention(*(x.data_ptr() for x in dev), len(b.ctx_lens), t, hq, c.hkv, dh, ck.shape[0],
                                    int(b.ctx_lens.max()), int(b.block_lens.max()), c.eps, c.theta, 0.0,
                                    int(c.causal), c.window, 0, out.data_ptr(), ws.data_ptr(), ws.numel(), flags,
                                    stream)
    return rc, stream


@pytest.mark.parametrize("which", ["first_cta", "middle_cta_split"])
def test_a_wait_that_runs_out_reports_a_timeout_and_the_next_call_is_correct(which):
    import torch
    D, lib = _test_lib()
    b = W.make_batch(W.Config("wait", 0, 16, 32, 8, 128, ctx_len=0, seed=41), ctx_lens=[900, 300, 2000],
                     block_lens=[16, 16, 16])
    c = b.cfg
    flags = D.FLAG_FORCE_SPLIT if which == "middle_cta_split" else 0
    ck = U.bf16_dev(U.stored_ctx_k(b))
    args = (len(b.ctx_lens), b.q.shape[0], c.hq, c.hkv, c.dh, ck.shape[0], int(b.ctx_lens.max()),
            int(b.block_lens.max()), c.causal, c.window, D.OUT_BF16, flags)
    plan = D.plan(*args)
    ws = D.alloc_workspace(D.workspace_size(*args))
    out = torch.zeros((b.q.shape[0], c.hq, c.dh), dtype=torch.bfloat16, device="cuda")
    cta = 0 if which == "first_cta" else int(plan["ctas"]) // 2  # its first V tile is withheld
    tile = 0
    assert lib.dflash_test_withhold_v_tile(cta, tile) == 0
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rc, stream = _call(lib, b, ck, out, ws, flags)
        assert rc == 0, lib.dflash_last_error().decode()
        torch.cuda.synchronize()
        took = time.perf_counter() - t0
        assert lib.dflash_check_error(ws.data_ptr(), stream) == D.ERR_DEVICE_TIMEOUT
        assert b"wait" in lib.dflash_last_error()
        assert took < 1.0, f"the timed-out call took {took:.3f} s"
    finally:
        assert lib.dflash_test_withhold_v_tile(-1, -1) == 0
    # the context is usable and the workspace serves the next call: error word cleared, output right
    rc, stream = _call(lib, b, ck, out, ws, flags)
    assert rc == 0
    torch.cuda.synchronize()
    assert lib.dflash_check_error(ws.data_ptr(), stream) == 0, lib.dflash_last_error().decode()
    ref = U.gpu_attention(b, ctx_k_dev=ck, flags=flags)  # the product library
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    U.assert_close_bf16(U.dev_to_f64(out), U.oracle_attention(b, U.stored_ctx_k(b)), "after the timeout")
