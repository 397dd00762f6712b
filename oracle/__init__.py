"""Python face of the f64 C oracle for DFlash draft block attention.

TEST INFRASTRUCTURE: only the tests, the package smoke check and the benchmark's
CPU-baseline leg import this module. The CUDA library never does, and this module
imports nothing from it.

Every function takes bf16 tensors as uint16 bit patterns (numpy) and int32
metadata, and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (plain C11, OpenMP, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I32, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            attn = [P] * 11 + [I32, I64, I32, I32, I32, I64, D, D, D, I32, I32]
            sig = {
                "orc_num_threads": [],
                "orc_rms_norm_rows": [P, P, I64, I32, I32, D, P],
                "orc_rope_neox_rows": [P, P, I64, I32, I32, D, P],
                "orc_norm_rope": [P, P, P, I64, I32, I32, D, D, P],
                "orc_round_bf16": [P, I64, P],
                "orc_context_kv": [P, P, P, I64, I32, I32, D, D, P, P],
                "orc_block_attention": attn + [P],
                "orc_block_attention_sampled": attn + [I64, P, P, P],
                "orc_block_attention_dense": attn + [P],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _u16(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name} failed with code {rc}")


def num_threads() -> int:
    return int(_load().orc_num_threads())


def rms_norm(x, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis of bf16 x [..., Dh]; w None means all ones."""
    x = _u16(x)
    dh = x.shape[-1]
    rows = x.size // dh
    y = np.empty(x.shape, dtype=np.float64)
    _check(_load().orc_rms_norm_rows(_p(x), _p(_u16(w)), rows, 1, dh, eps, _p(y)), "rms_norm")
    return y


def rope_neox(x, pos, theta: float) -> np.ndarray:
    """NeoX rotary embedding of double x [T, H, Dh] at pos [T]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    t, h, dh = x.shape
    y = np.empty_like(x)
    _check(_load().orc_rope_neox_rows(_p(x), _p(_i32(pos)), t, h, dh, theta, _p(y)), "rope_neox")
    return y


def norm_rope(x, w, pos, eps: float, theta: float) -> np.ndarray:
    """RMSNorm then NeoX RoPE of bf16 x [T, H, Dh] at pos [T]."""
    x = _u16(x)
    t, h, dh = x.shape
    y = np.empty(x.shape, dtype=np.float64)
    _check(_load().orc_norm_rope(_p(x), _p(_u16(w)), _p(_i32(pos)), t, h, dh, eps, theta, _p(y)), "norm_rope")
    return y


def round_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _check(_load().orc_round_bf16(_p(x), x.size, _p(out)), "round_bf16")
    return out


def context_kv(k_raw, ctx_pos, k_norm_w, eps: float, theta: float):
    """Stored context keys: (exact f64 values, their bf16 bits), both [n_ctx, Hkv, Dh]."""
    k_raw = _u16(k_raw)
    n, hkv, dh = k_raw.shape
    out = np.empty(k_raw.shape, dtype=np.float64)
    out16 = np.empty(k_raw.shape, dtype=np.uint16)
    _check(_load().orc_context_kv(_p(k_raw), _p(_i32(ctx_pos)), _p(_u16(k_norm_w)), n, hkv, dh, eps, theta,
                                  _p(out), _p(out16)), "context_kv")
    return out, out16


def _attn_args(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens, positions,
               q_norm_w, k_norm_w, eps, theta, scale, causal, window):
    arrs = [_u16(q), _u16(k_blk), _u16(v_blk), _u16(ctx_k), _u16(ctx_v), _i32(query_start_loc),
            _i32(ctx_start_loc), _i32(ctx_lens), _i32(positions), _u16(q_norm_w), _u16(k_norm_w)]
    t, hq, dh = arrs[0].shape
    hkv = arrs[1].shape[1]
    n_req = len(arrs[5]) - 1
    total_ctx = arrs[3].shape[0]
    args = [_p(a) for a in arrs] + [n_req, t, hq, hkv, dh, total_ctx, eps, theta, scale, int(causal), int(window)]
    return arrs, args, (t, hq, dh)


def block_attention(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens, positions,
                    q_norm_w, k_norm_w, eps=1e-6, theta=1e6, scale=0.0, causal=False, window=0) -> np.ndarray:
    """Attention output of every block row, [T, Hq, Dh] float64. ctx_k are stored keys."""
    keep, args, shape = _attn_args(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens,
                                   positions, q_norm_w, k_norm_w, eps, theta, scale, causal, window)
    out = np.empty(shape, dtype=np.float64)
    _check(_load().orc_block_attention(*args, _p(out)), "block_attention")
    return out


def block_attention_sampled(samples_t, samples_h, q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc,
                            ctx_lens, positions, q_norm_w, k_norm_w, eps=1e-6, theta=1e6, scale=0.0, causal=False,
                            window=0) -> np.ndarray:
    """Attention output for the listed (block row, head) samples, [n, Dh] float64."""
    keep, args, shape = _attn_args(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens,
                                   positions, q_norm_w, k_norm_w, eps, theta, scale, causal, window)
    st, sh = _i32(samples_t), _i32(samples_h)
    out = np.empty((len(st), shape[2]), dtype=np.float64)
    _check(_load().orc_block_attention_sampled(*args, len(st), _p(st), _p(sh), _p(out)), "block_attention_sampled")
    return out


def block_attention_dense(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens, positions,
                          q_norm_w, k_norm_w, eps=1e-6, theta=1e6, scale=0.0, causal=False, window=0) -> np.ndarray:
    """Brute force over the materialised [context; block] sequences, [T, Hq, Dh] float64."""
    keep, args, shape = _attn_args(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens,
                                   positions, q_norm_w, k_norm_w, eps, theta, scale, causal, window)
    out = np.empty(shape, dtype=np.float64)
    _check(_load().orc_block_attention_dense(*args, _p(out)), "block_attention_dense")
    return out


def gather_paged_context(pool, block_table, ctx_lens, page_size: int):
    """The context rows of every request, gathered from a page pool, and their offsets.

    pool [num_pages, page_size, Hkv, Dh]; block_table [N, max_pages]. Request r's context row j
    is row j % page_size of page block_table[r, j // page_size] (the paged layout of the
    DFlash draft's KV store). Returns (rows [sum ctx_lens, Hkv, Dh], ctx_start_loc [N+1]).
    """
    pool = np.asarray(pool)
    bt = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(ctx_lens, dtype=np.int64)
    starts = np.zeros(len(lens) + 1, dtype=np.int32)
    starts[1:] = np.cumsum(lens)
    rows = np.empty((int(starts[-1]),) + pool.shape[2:], dtype=pool.dtype)
    for r, n in enumerate(lens):
        for j in range(int(n)):
            rows[starts[r] + j] = pool[bt[r, j // page_size], j % page_size]
    return rows, starts


def block_attention_paged(q, k_blk, v_blk, k_pool, v_pool, block_table, query_start_loc, ctx_lens, positions,
                          q_norm_w, k_norm_w, page_size: int, **kw) -> np.ndarray:
    """block_attention with the context read from page pools through a block table."""
    ck, starts = gather_paged_context(k_pool, block_table, ctx_lens, page_size)
    cv, _ = gather_paged_context(v_pool, block_table, ctx_lens, page_size)
    return block_attention(q, k_blk, v_blk, ck, cv, query_start_loc, starts, ctx_lens, positions, q_norm_w,
                           k_norm_w, **kw)


def paged_append(k_pool, v_pool, block_table, seq_lens, new_start_loc, k_raw, v, k_norm_w, page_size: int,
                 eps: float = 1e-6, theta: float = 1e6):
    """Appends every request's new context rows to its pages and advances its length.

    qwen3_dflash.cpp, AppendContextKVDevice (the paged draft KV store): the new rows of a
    request sit at the positions that follow its stored context, [L, L + count) with L its
    current length; each is projected as PrecomputeContextKVDevice does (k_norm, then NeoX
    RoPE at that position, stored in bf16; V raw) and lands at row p % page_size of page
    block_table[r, p // page_size]; the length then grows by count.

    Rows new_start_loc[r] .. new_start_loc[r+1] of k_raw / v belong to request r; rows
    outside [new_start_loc[0], new_start_loc[N]) belong to none and are ignored. The page
    checks the store's capacity before it writes anything and leaves the store as it was
    when the rows do not fit; per request the same holds here: if any new row of a request
    would fall past its block table (page index >= max_pages) or on a page id outside the
    pool, none of that request's rows is written, its length does not move, and the
    returned flag is set. The other requests append as usual. new_start_loc must be
    nondecreasing, start at >= 0 and end at <= len(k_raw); otherwise nothing changes and
    the flag is set.

    Returns (k_pool, v_pool, seq_lens, flag): new arrays, the inputs are not modified.
    """
    kp = np.array(k_pool, dtype=np.uint16, copy=True)
    vp = np.array(v_pool, dtype=np.uint16, copy=True)
    lens = np.array(seq_lens, dtype=np.int64, copy=True)
    nsl = np.asarray(new_start_loc, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    k_raw = _u16(k_raw)
    v = _u16(v)
    n = k_raw.shape[0]
    n_req = len(nsl) - 1
    num_pages, max_pages = kp.shape[0], bt.shape[1]
    if nsl[0] < 0 or nsl[n_req] > n or np.any(np.diff(nsl) < 0):
        return kp, vp, lens.astype(np.int32), True
    flag = False
    rows, dst_page, dst_off, pos = [], [], [], []
    for r in range(n_req):
        count = int(nsl[r + 1] - nsl[r])
        if count == 0:
            continue
        # the request's rows and their destinations, all checked before any is written
        mine = []
        for i in range(count):
            p = int(lens[r]) + i
            if p < 0 or p // page_size >= max_pages:
                break
            page = int(bt[r, p // page_size])
            if page < 0 or page >= num_pages:
                break
            mine.append((int(nsl[r]) + i, page, p % page_size, p))
        if len(mine) < count:
            flag = True
            continue
        for row, page, off, p in mine:
            rows.append(row)
            dst_page.append(page)
            dst_off.append(off)
            pos.append(p)
        lens[r] += count
    if rows:
        k16 = context_kv(k_raw[rows], np.array(pos, dtype=np.int32), k_norm_w, eps, theta)[1]
        for j, (pg, off) in enumerate(zip(dst_page, dst_off)):
            kp[pg, off] = k16[j]
            if v is not None:
                vp[pg, off] = v[rows[j]]
    return kp, vp, lens.astype(np.int32), flag


from .prepare_inputs import prepare_dflash_inputs  # noqa: E402  (pure integer, no C part)
