"""GB300 (sm_103a) DFlash draft block attention: Python binding of libdflash_gb300.so.

The binding only marshals arguments: every step of the path (context-K norm+RoPE, the
fused q/k prologue, block attention, split-KV combine) runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. There is no CPU or
PyTorch fallback: if the library cannot be built or loaded, every call raises.

Entry points mirror include/dflash.h:
    context_kv(...)          -> dflash_context_kv
    paged_append(...)        -> dflash_paged_append
    prepare_inputs(...)      -> dflash_prepare_inputs
    block_attention(...)     -> dflash_block_attention
    workspace_size(...)      -> dflash_block_attention_workspace_size
    check_error(workspace)   -> dflash_check_error
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["load", "lib_path", "context_kv", "paged_append", "prepare_inputs", "STATUS_METADATA", "block_attention", "block_attention_paged", "workspace_size", "plan",
           "alloc_workspace",
           "check_error", "DFlashError", "OUT_BF16", "OUT_F32", "FLAG_FORCE_SPLIT", "FLAG_NO_SPLIT",
           "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_WORKSPACE", "ERR_CUDA", "ERR_DEVICE_TIMEOUT",
           "ERR_DEVICE_METADATA"]

OUT_BF16, OUT_F32 = 0, 1
STATUS_METADATA = 2  # bit ORed into the status word of context_kv / paged_append / prepare_inputs
FLAG_FORCE_SPLIT, FLAG_NO_SPLIT = 1, 2
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_DEVICE_METADATA = \
    -1, -2, -3, -4, -5, -6

_lock = threading.Lock()
_lib = None


class DFlashError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"dflash error {code}: {message}")
        self.code = code


def lib_path() -> str:
    from . import _build
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Loads the library (building it in-tree with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        if not _build.up_to_date():
            if not build_if_missing:
                raise RuntimeError(f"{_build.LIB_PATH} is not built; run __graft_entry__.build()")
            _build.build()
        lib = ctypes.CDLL(_build.LIB_PATH)
        P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.dflash_last_error.restype = ctypes.c_char_p
        lib.dflash_last_error.argtypes = []
        lib.dflash_version.restype = I32
        lib.dflash_version.argtypes = []
        lib.dflash_context_kv.restype = I32
        lib.dflash_context_kv.argtypes = [P, P, P, P, P, I64, I32, I32, F32, F32, P, P, I64, P, P]
        lib.dflash_block_attention_workspace_size.restype = SZ
        lib.dflash_block_attention_workspace_size.argtypes = [I32, I64, I32, I32, I32, I64, I32, I32, I32, I32, I32, I32]
        lib.dflash_block_attention.restype = I32
        lib.dflash_block_attention.argtypes = ([P] * 11 + [I32, I64, I32, I32, I32, I64, I32, I32, F32, F32, F32,
                                                           I32, I32, I32, P, P, SZ, I32, P])
        lib.dflash_block_attention_paged.restype = I32
        lib.dflash_block_attention_paged.argtypes = ([P] * 6 + [I64, I32, I32] + [P] * 5 +
                                                     [I32, I64, I32, I32, I32, I32, I32, F32, F32, F32, I32, I32,
                                                      I32, P, P, SZ, I32, P])
        lib.dflash_block_attention_plan.restype = I32
        lib.dflash_block_attention_plan.argtypes = [I32, I64, I32, I32, I32, I64, I32, I32, I32, I32, I32, I32, P]
        lib.dflash_check_error.restype = I32
        lib.dflash_check_error.argtypes = [P, P]
        lib.dflash_paged_append.restype = I32
        lib.dflash_paged_append.argtypes = [P] * 6 + [I32, I64, I32, I32, I32, I32, I64, F32, F32, P, P, P, P]
        lib.dflash_prepare_inputs.restype = I32
        lib.dflash_prepare_inputs.argtypes = ([P] * 8 + [I32, I32, I64, I32, I32, I32, I32, I32, I64, I32, I32] +
                                              [P] * 12)
        _lib = lib
        return lib


def _raise(rc: int) -> None:
    if rc != 0:
        raise DFlashError(rc, load().dflash_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(name, t, dtype, shape=None):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def context_kv(k_raw, ctx_pos, k_norm_w, ctx_k, *, v=None, ctx_v=None, slot=None, status=None, eps=1e-6,
               theta=1e6, stream=None) -> None:
    """Writes rope(rmsnorm(k_raw)) into ctx_k (and v into ctx_v) at rows `slot` (or 0..n-1).

    status: an optional int32 device word that receives STATUS_METADATA when a slot is out of
    range (that row is not written)."""
    import torch
    n, hkv, dh = k_raw.shape
    _check_tensor("k_raw", k_raw, torch.bfloat16)
    _check_tensor("v", v, torch.bfloat16, (n, hkv, dh))
    _check_tensor("ctx_pos", ctx_pos, torch.int32, (n,))
    _check_tensor("k_norm_w", k_norm_w, torch.bfloat16, (dh,))
    _check_tensor("slot", slot, torch.int32, (n,))
    _check_tensor("ctx_k", ctx_k, torch.bfloat16)
    _check_tensor("ctx_v", ctx_v, torch.bfloat16, None if ctx_v is None else tuple(ctx_k.shape))
    _check_tensor("status", status, torch.int32, (1,))
    if tuple(ctx_k.shape[1:]) != (hkv, dh):
        raise ValueError("ctx_k must be [capacity, Hkv, Dh]")
    rc = load().dflash_context_kv(_ptr(k_raw), _ptr(v), _ptr(ctx_pos), _ptr(k_norm_w), _ptr(slot), n, hkv, dh,
                                  float(eps), float(theta), _ptr(ctx_k), _ptr(ctx_v), ctx_k.shape[0], _ptr(status),
                                  _stream(stream))
    _raise(rc)


def paged_append(k_raw, new_start_loc, seq_lens, block_table, k_norm_w, k_pool, *, v=None, v_pool=None,
                 status=None, eps=1e-6, theta=1e6, stream=None) -> None:
    """Appends the new rows of every request to its pages and advances seq_lens on the device.

    k_raw / v [n, Hkv, Dh] bf16; new_start_loc [N+1], seq_lens [N] (in/out), block_table
    [N, max_pages] int32; k_pool / v_pool [num_pages, page_size, Hkv, Dh] bf16; status: an
    optional int32 device word that receives STATUS_METADATA on bad metadata.
    """
    import torch
    n, hkv, dh = k_raw.shape
    nr = new_start_loc.shape[0] - 1
    _check_tensor("k_raw", k_raw, torch.bfloat16)
    _check_tensor("v", v, torch.bfloat16, (n, hkv, dh))
    _check_tensor("new_start_loc", new_start_loc, torch.int32, (nr + 1,))
    _check_tensor("seq_lens", seq_lens, torch.int32, (nr,))
    _check_tensor("block_table", block_table, torch.int32)
    _check_tensor("k_norm_w", k_norm_w, torch.bfloat16, (dh,))
    _check_tensor("k_pool", k_pool, torch.bfloat16)
    _check_tensor("v_pool", v_pool, torch.bfloat16, None if v_pool is None else tuple(k_pool.shape))
    _check_tensor("status", status, torch.int32, (1,))
    if k_pool.dim() != 4 or tuple(k_pool.shape[2:]) != (hkv, dh):
        raise ValueError("k_pool must be [num_pages, page_size, Hkv, Dh]")
    if block_table.dim() != 2 or block_table.shape[0] != nr:
        raise ValueError("block_table must be [N, max_pages_per_req]")
    if (v is None) != (v_pool is None):
        raise ValueError("pass v and v_pool together")
    rc = load().dflash_paged_append(
        _ptr(k_raw), _ptr(v), _ptr(new_start_loc), _ptr(seq_lens), _ptr(block_table), _ptr(k_norm_w), nr, n, hkv,
        dh, k_pool.shape[1], block_table.shape[1], k_pool.shape[0], float(eps), float(theta), _ptr(k_pool),
        _ptr(v_pool), _ptr(status), _stream(stream))
    _raise(rc)


PREPARE_OUTPUTS = ("input_ids", "query_positions", "query_start_loc", "seq_lens", "query_slot_mapping",
                   "context_positions", "context_slot_mapping", "sample_indices", "sample_pos", "sample_idx_mapping")


def prepare_inputs(idx_mapping, target_query_start_loc, num_rejected, num_sampled, last_sampled,
                   next_prefill_tokens, target_positions, block_table, *, num_query_per_req, num_speculative_steps,
                   block_size, max_num_reqs, max_num_tokens, max_model_len, parallel_drafting_token_id,
                   sample_from_anchor, out=None, status=None, stream=None) -> dict:
    """The draft step's prepared inputs (dict of device tensors named as PREPARE_OUTPUTS).

    idx_mapping, num_rejected, num_sampled [N], target_query_start_loc [N+1], last_sampled,
    next_prefill_tokens [max_num_reqs], block_table [N, stride]: int32; target_positions int64.
    `out` may hold preallocated outputs (same names), e.g. for graph capture.
    """
    import torch
    n = idx_mapping.shape[0]
    dev = idx_mapping.device
    n_tgt = target_positions.shape[0]
    nq, ns = int(num_query_per_req), int(num_speculative_steps)
    for name, ten, shp in [("idx_mapping", idx_mapping, (n,)), ("target_query_start_loc", target_query_start_loc,
                                                               (n + 1,)),
                           ("num_rejected", num_rejected, (n,)), ("num_sampled", num_sampled, (n,)),
                           ("last_sampled", last_sampled, (max_num_reqs,)),
                           ("next_prefill_tokens", next_prefill_tokens, (max_num_reqs,)),
                           ("block_table", block_table, None)]:
        _check_tensor(name, ten, torch.int32, shp)
    _check_tensor("target_positions", target_positions, torch.int64, (n_tgt,))
    _check_tensor("status", status, torch.int32, (1,))
    if block_table.dim() != 2 or block_table.shape[0] < n:
        raise ValueError("block_table must be [>= N, stride]")
    i32, i64 = torch.int32, torch.int64
    spec = {"input_ids": (i32, n * nq), "query_positions": (i64, n * nq), "query_start_loc": (i32, max_num_reqs + 1),
            "seq_lens": (i32, max_num_reqs), "query_slot_mapping": (i64, max_num_tokens),
            "context_positions": (i64, n_tgt), "context_slot_mapping": (i64, n_tgt),
            "sample_indices": (i32, max_num_reqs * ns), "sample_pos": (i64, max_num_reqs * ns),
            "sample_idx_mapping": (i32, max_num_reqs * ns)}
    out = dict(out or {})
    for k, (dt, size) in spec.items():
        if k not in out:
            out[k] = torch.empty(size, dtype=dt, device=dev)
        _check_tensor(k, out[k], dt, (size,))
    rc = load().dflash_prepare_inputs(
        _ptr(idx_mapping), _ptr(target_query_start_loc), _ptr(num_rejected), _ptr(num_sampled), _ptr(last_sampled),
        _ptr(next_prefill_tokens), _ptr(target_positions), _ptr(block_table), block_table.stride(0), n, n_tgt, nq,
        ns, int(block_size), int(max_num_reqs), int(max_num_tokens), int(max_model_len),
        int(parallel_drafting_token_id), int(bool(sample_from_anchor)), *[_ptr(out[k]) for k in PREPARE_OUTPUTS],
        _ptr(status), _stream(stream))
    _raise(rc)
    return out


def workspace_size(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, causal=False, window=0,
                   out_dtype=OUT_BF16, flags=0) -> int:
    n = load().dflash_block_attention_workspace_size(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len,
                                                     max_block_len, int(causal), int(window), out_dtype, flags)
    if n == 0:
        _raise(ERR_INVALID_ARG)
    return int(n)


def plan(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, causal=False, window=0,
         out_dtype=OUT_BF16, flags=0) -> dict:
    """How a call with these arguments runs: launches, tiles per split, unit bound, CTAs."""
    arr = (ctypes.c_int64 * 5)()
    _raise(load().dflash_block_attention_plan(num_reqs, total_q, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len,
                                              int(causal), int(window), out_dtype, flags, arr))
    return {"launches": arr[0], "tiles_per_split": arr[1], "units_max": arr[2], "ctas": arr[3],
            "workspace_bytes": arr[4] * 256}


def alloc_workspace(nbytes: int, device=None):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def block_attention(q, k_blk, v_blk, ctx_k, ctx_v, query_start_loc, ctx_start_loc, ctx_lens, positions, q_norm_w,
                    k_norm_w, *, max_ctx_len, max_block_len, out=None, workspace=None, eps=1e-6, theta=1e6,
                    scale=0.0, causal=False, window=0, out_dtype=OUT_BF16, flags=0, stream=None):
    """Block attention of every block row over [context ; block] of its request.

    Shapes: q [T, Hq, Dh], k_blk / v_blk [T, Hkv, Dh], ctx_k / ctx_v [total_ctx, Hkv, Dh] (bf16);
    query_start_loc / ctx_start_loc [N+1], ctx_lens [N], positions [T] (int32).
    Returns `out` [T, Hq, Dh] (bf16, or f32 with out_dtype=OUT_F32).
    """
    import torch
    t, hq, dh = q.shape
    hkv = k_blk.shape[1]
    n = query_start_loc.shape[0] - 1
    total_ctx = ctx_k.shape[0]
    for name, ten, shp in [("q", q, None), ("k_blk", k_blk, (t, hkv, dh)), ("v_blk", v_blk, (t, hkv, dh)),
                           ("ctx_k", ctx_k, (total_ctx, hkv, dh)), ("ctx_v", ctx_v, (total_ctx, hkv, dh)),
                           ("q_norm_w", q_norm_w, (dh,)), ("k_norm_w", k_norm_w, (dh,))]:
        _check_tensor(name, ten, torch.bfloat16, shp)
    for name, ten, shp in [("query_start_loc", query_start_loc, (n + 1,)), ("ctx_start_loc", ctx_start_loc, (n + 1,)),
                           ("ctx_lens", ctx_lens, (n,)), ("positions", positions, (t,))]:
        _check_tensor(name, ten, torch.int32, shp)
    odt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((t, hq, dh), dtype=odt, device=q.device)
    _check_tensor("out", out, odt, (t, hq, dh))
    need = workspace_size(n, t, hq, hkv, dh, total_ctx, max_ctx_len, max_block_len, causal, window, out_dtype, flags)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    _check_tensor("workspace", workspace, torch.uint8)
    rc = load().dflash_block_attention(
        _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(ctx_k), _ptr(ctx_v), _ptr(query_start_loc), _ptr(ctx_start_loc),
        _ptr(ctx_lens), _ptr(positions), _ptr(q_norm_w), _ptr(k_norm_w), n, t, hq, hkv, dh, total_ctx,
        int(max_ctx_len), int(max_block_len), float(eps), float(theta), float(scale), int(causal), int(window),
        out_dtype, _ptr(out), _ptr(workspace), workspace.numel(), flags, _stream(stream))
    _raise(rc)
    return out


def block_attention_paged(q, k_blk, v_blk, k_pool, v_pool, block_table, query_start_loc, ctx_lens, positions,
                          q_norm_w, k_norm_w, *, max_ctx_len, max_block_len, out=None, workspace=None, eps=1e-6,
                          theta=1e6, scale=0.0, causal=False, window=0, out_dtype=OUT_BF16, flags=0, stream=None):
    """block_attention with the context in page pools.

    k_pool / v_pool [num_pages, page_size, Hkv, Dh] bf16; block_table [N, max_pages_per_req] int32
    (request r's context row j is row j % page_size of page block_table[r, j // page_size]).
    """
    import torch
    t, hq, dh = q.shape
    hkv = k_blk.shape[1]
    n = query_start_loc.shape[0] - 1
    num_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    max_pages = block_table.shape[1] if block_table.dim() == 2 else 0
    for name, ten, shp in [("q", q, None), ("k_blk", k_blk, (t, hkv, dh)), ("v_blk", v_blk, (t, hkv, dh)),
                           ("k_pool", k_pool, (num_pages, page_size, hkv, dh)),
                           ("v_pool", v_pool, (num_pages, page_size, hkv, dh)),
                           ("q_norm_w", q_norm_w, (dh,)), ("k_norm_w", k_norm_w, (dh,))]:
        _check_tensor(name, ten, torch.bfloat16, shp)
    for name, ten, shp in [("block_table", block_table, (n, max_pages)), ("query_start_loc", query_start_loc, (n + 1,)),
                           ("ctx_lens", ctx_lens, (n,)), ("positions", positions, (t,))]:
        _check_tensor(name, ten, torch.int32, shp)
    odt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((t, hq, dh), dtype=odt, device=q.device)
    _check_tensor("out", out, odt, (t, hq, dh))
    need = workspace_size(n, t, hq, hkv, dh, num_pages * page_size, max_ctx_len, max_block_len, causal, window,
                          out_dtype, flags)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    _check_tensor("workspace", workspace, torch.uint8)
    rc = load().dflash_block_attention_paged(
        _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), num_pages, page_size,
        max_pages, _ptr(query_start_loc), _ptr(ctx_lens), _ptr(positions), _ptr(q_norm_w), _ptr(k_norm_w), n, t, hq,
        hkv, dh, int(max_ctx_len), int(max_block_len), float(eps), float(theta), float(scale), int(causal),
        int(window), out_dtype, _ptr(out), _ptr(workspace), workspace.numel(), flags, _stream(stream))
    _raise(rc)
    return out


def check_error(workspace, stream=None) -> None:
    """Raises DFlashError if the last attention call on `workspace` recorded a device error."""
    _raise(load().dflash_check_error(_ptr(workspace), _stream(stream)))
