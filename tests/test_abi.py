"""The C-ABI library: it loads, exports every entry point include/dflash.h declares, and
rejects bad host arguments before touching a device (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_draft_rmsnorm_gb300 as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names += re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", text)
    return names


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ["dflash_context_kv", "dflash_block_attention", "dflash_block_attention_workspace_size",
              "dflash_check_error", "dflash_last_error", "dflash_version"]:
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    lib = D.load()
    raw = ctypes.CDLL(D.lib_path())
    for n in declared_symbols():
        assert hasattr(raw, n), f"{n} is declared in include/ but not exported"
    assert lib.dflash_version() >> 16 == 1
    # the test build's hook (a withheld copy, see test_gpu_wait_timeout.py) is not in the product
    assert not hasattr(raw, "dflash_test_withhold_v_tile")


def test_wait_test_library_is_the_product_plus_the_hook():
    from speculative_decoding_draft_rmsnorm_gb300 import _build
    if not _build.up_to_date(_build.WAIT_TEST_LIB_PATH):
        _build.build()
    raw = ctypes.CDLL(_build.WAIT_TEST_LIB_PATH)
    assert hasattr(raw, "dflash_test_withhold_v_tile")
    for n in declared_symbols():
        assert hasattr(raw, n), n


def _attn(**over):
    lib = D.load()
    a = dict(num_reqs=1, total_q=16, hq=4, hkv=2, dh=64, total_ctx=64, max_ctx=64, max_blk=16, eps=1e-6,
             theta=1e6, scale=0.0, causal=0, window=0, out_dtype=0, flags=0)
    a.update(over)
    fake = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    return lib.dflash_block_attention(*([fake] * 11), a["num_reqs"], a["total_q"], a["hq"], a["hkv"], a["dh"],
                                      a["total_ctx"], a["max_ctx"], a["max_blk"], a["eps"], a["theta"], a["scale"],
                                      a["causal"], a["window"], a["out_dtype"], fake, fake, 1 << 20, a["flags"], None)


@pytest.mark.parametrize("over,code", [
    (dict(hq=6, hkv=4), D.ERR_INVALID_ARG),         # Hq not a multiple of Hkv
    (dict(dh=96), D.ERR_UNSUPPORTED),               # head_dim outside {64, 128}
    (dict(hq=130, hkv=1), D.ERR_UNSUPPORTED),       # group larger than a query tile
    (dict(window=8, causal=0), D.ERR_INVALID_ARG),  # window only with causal
    (dict(causal=2), D.ERR_INVALID_ARG),
    (dict(out_dtype=7), D.ERR_INVALID_ARG),
    (dict(total_q=-1), D.ERR_INVALID_ARG),
    (dict(flags=3), D.ERR_INVALID_ARG),             # force and forbid split together
    (dict(eps=-1.0), D.ERR_INVALID_ARG),
    (dict(max_blk=0), D.ERR_INVALID_ARG),
])
def test_attention_rejects_bad_host_arguments(over, code):
    lib = D.load()
    assert _attn(**over) == code
    assert lib.dflash_last_error()  # a message is set


def test_context_kv_rejects_bad_host_arguments():
    lib = D.load()
    fake = ctypes.c_void_p(256)
    assert lib.dflash_context_kv(fake, None, fake, fake, None, 10, 2, 96, 1e-6, 1e6, fake, None, 10, None, None) == \
        D.ERR_UNSUPPORTED
    assert lib.dflash_context_kv(fake, None, fake, fake, None, 11, 2, 64, 1e-6, 1e6, fake, None, 10, None, None) == \
        D.ERR_INVALID_ARG
    assert lib.dflash_context_kv(fake, None, fake, fake, None, 0, 2, 64, 1e-6, 1e6, fake, None, 10, None, None) == 0


def test_header_declares_the_draft_step_entry_points():
    names = declared_symbols()
    assert "dflash_paged_append" in names and "dflash_prepare_inputs" in names


def test_paged_append_rejects_bad_host_arguments():
    lib = D.load()
    f = ctypes.c_void_p(256)

    def call(n_req=2, n=8, hkv=2, dh=64, ps=16, max_pages=4, pages=8, eps=1e-6, theta=1e6):
        return lib.dflash_paged_append(f, f, f, f, f, f, n_req, n, hkv, dh, ps, max_pages, pages, eps, theta, f, f,
                                       None, None)

    assert call(dh=96) == D.ERR_UNSUPPORTED
    assert call(ps=0) == D.ERR_INVALID_ARG
    assert call(max_pages=0) == D.ERR_INVALID_ARG
    assert call(hkv=0) == D.ERR_INVALID_ARG
    assert call(n=-1) == D.ERR_INVALID_ARG
    assert call(theta=0.0) == D.ERR_INVALID_ARG
    assert call(n_req=0) == 0  # nothing to do, nothing enqueued


def test_prepare_inputs_rejects_bad_host_arguments():
    lib = D.load()
    f = ctypes.c_void_p(256)

    def call(n=4, n_tgt=40, nq=16, ns=15, bs=16, max_reqs=8, max_tok=64, mml=4096, anchor=0, stride=8):
        return lib.dflash_prepare_inputs(f, f, f, f, f, f, f, f, stride, n, n_tgt, nq, ns, bs, max_reqs, max_tok, mml,
                                         7, anchor, *([f] * 10), None, None)

    assert call(n=0) == D.ERR_INVALID_ARG
    assert call(max_reqs=3) == D.ERR_INVALID_ARG          # more requests than request slots
    assert call(max_tok=63) == D.ERR_INVALID_ARG          # query rows do not fit
    assert call(ns=14) == D.ERR_INVALID_ARG               # 15 sampled rows per request, 14 steps
    assert call(anchor=1) == D.ERR_INVALID_ARG            # sampling from the anchor: 16 rows, 15 steps
    assert call(anchor=2) == D.ERR_INVALID_ARG
    assert call(bs=0) == D.ERR_INVALID_ARG
    assert call(stride=0) == D.ERR_INVALID_ARG
    assert call(n_tgt=-1) == D.ERR_INVALID_ARG
