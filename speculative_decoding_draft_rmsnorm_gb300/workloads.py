"""Seeded synthetic workloads for DFlash draft block attention.

This module only *draws* inputs: lengths, bf16 tensors and the integer metadata that
describes a ragged batch.  It holds none of the method's arithmetic (no norm, no
rotary, no softmax), so the CUDA path and the f64 oracle can both consume its bytes.

Random numbers come from one counter-based generator, SplitMix64 (S. Vigna's
published finaliser over a Weyl sequence), turned into uniforms in (0, 1] and into
normals with the Box-Muller transform.  Every tensor has its own stream, so drawing
one array never shifts another.

The batch layout follows vllm.cpp's DFlash draft (qwen3_dflash.cpp,
ForwardWithCtxKVDev and runner.cpp, propose_drafts_dflash): request r owns C_r
context rows (positions 0..C_r-1) and a block of B_r draft rows (an anchor plus
mask tokens, positions C_r..C_r+B_r-1); block rows of all requests are packed by
``query_start_loc`` and context rows by ``ctx_start_loc``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import math
import os
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# Stream ids, in the documented generation order.
STREAM_LENGTHS, STREAM_Q, STREAM_KBLK, STREAM_VBLK, STREAM_CTXK, STREAM_CTXV, STREAM_QW, STREAM_KW = range(8)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (uint64 arithmetic wraps modulo 2**64)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x632BE59BD9B4E019 + stream * 0xD1B54A32D192ED03) & (2**64 - 1)], dtype=np.uint64)
        return _mix64(s)[0]


def uniform(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of a stream as doubles in (0, 1]."""
    base = _stream_base(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        x = _mix64(base + idx * _GOLDEN)
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _normal_chunk(seed: int, stream: int, first_pair: int, n_pairs: int) -> np.ndarray:
    u = uniform(seed, stream, 2 * first_pair, 2 * n_pairs)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = 2.0 * math.pi * u[1::2]
    out = np.empty(2 * n_pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Rounds to bfloat16 bit patterns (via float32, both steps round-to-nearest-even)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_bf16(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` draws of N(0, 1), rounded to bf16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    n_pairs = (n + 1) // 2
    starts = list(range(0, n_pairs, _CHUNK))

    def work(p0: int) -> None:
        cnt = min(_CHUNK, n_pairs - p0)
        v = _normal_chunk(seed, stream, p0, cnt)
        lo = 2 * p0
        hi = min(n, lo + 2 * cnt)
        out[lo:hi] = f64_to_bf16(v[: hi - lo])

    if len(starts) <= 1:
        for p0 in starts:
            work(p0)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    return out


def uniform_bf16(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    return f64_to_bf16(lo + (hi - lo) * uniform(seed, stream, 0, n))


@dataclass
class Config:
    """One synthetic workload: shapes, mask mode and how context lengths are drawn."""

    name: str
    num_reqs: int
    block: int
    hq: int
    hkv: int
    dh: int
    causal: bool = False
    window: int = 0
    ctx_len: int | None = None          # fixed context length
    ctx_uniform: tuple[int, int] | None = None     # integer uniform [lo, hi]
    ctx_loguniform: tuple[int, int] | None = None  # floor(exp(U(ln lo, ln hi)))
    force_split: bool = False
    eps: float = 1e-6
    theta: float = 1e6
    seed: int = 0
    note: str = ""


CONFIGS: dict[str, Config] = {
    "tiny": Config("tiny", 1, 16, 4, 2, 64, ctx_len=64,
                   note="1 request, C=64, B=16, Hq=4, Hkv=2, Dh=64, bidirectional"),
    "qwen3_0p6b": Config("qwen3_0p6b", 8, 16, 16, 8, 128, ctx_uniform=(512, 2048),
                         note="Qwen3-0.6B-shaped layer, 8 requests, C~U[512,2048], B=16"),
    "qwen3_4b": Config("qwen3_4b", 32, 16, 32, 8, 128, ctx_len=4096,
                       note="Qwen3-4B-shaped layer, 32 requests, C=4096, B=16"),
    "swa": Config("swa", 16, 16, 32, 8, 128, ctx_len=16384, causal=True, window=4096,
                  note="SWA layer, 16 requests, C=16384, B=16, causal, window 4096"),
    "ragged": Config("ragged", 64, 16, 32, 8, 128, ctx_loguniform=(1024, 32768), force_split=True,
                     note="64 requests, C log-uniform in [1024,32768], B=16, split-KV"),
}


def context_lengths(cfg: Config) -> np.ndarray:
    if cfg.ctx_len is not None:
        return np.full(cfg.num_reqs, cfg.ctx_len, dtype=np.int64)
    u = uniform(cfg.seed, STREAM_LENGTHS, 0, cfg.num_reqs)
    if cfg.ctx_uniform is not None:
        lo, hi = cfg.ctx_uniform
        return np.minimum(lo + np.floor(u * (hi - lo + 1)).astype(np.int64), hi)
    if cfg.ctx_loguniform is not None:
        lo, hi = cfg.ctx_loguniform
        c = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
        return np.clip(c, lo, hi)
    raise ValueError("config has no context-length rule")


@dataclass
class Batch:
    """Host copy of one ragged batch; every tensor is bf16 bits (uint16) or int32."""

    cfg: Config
    ctx_lens: np.ndarray          # int32 [N]   live context rows per request
    block_lens: np.ndarray        # int32 [N]
    query_start_loc: np.ndarray   # int32 [N+1] block rows of request r: qsl[r]..qsl[r+1]
    ctx_start_loc: np.ndarray     # int32 [N+1] context segment of request r
    positions: np.ndarray         # int32 [T]   block-token positions
    ctx_pos: np.ndarray           # int32 [sum C] context-token positions
    q: np.ndarray                 # bf16 [T, Hq, Dh]   raw (pre-norm) queries
    k_blk: np.ndarray             # bf16 [T, Hkv, Dh]  raw block keys
    v_blk: np.ndarray             # bf16 [T, Hkv, Dh]
    ctx_k_raw: np.ndarray         # bf16 [sum C, Hkv, Dh] raw context keys
    ctx_v: np.ndarray             # bf16 [sum C, Hkv, Dh]
    q_norm_w: np.ndarray          # bf16 [Dh]
    k_norm_w: np.ndarray          # bf16 [Dh]
    extra: dict = field(default_factory=dict)

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def total_ctx(self) -> int:
        return int(self.ctx_start_loc[-1])


def make_batch(cfg: Config, ctx_lens=None, block_lens=None, seed: int | None = None) -> Batch:
    """Draws a batch in the fixed order: lengths, q, k_blk, v_blk, ctx k, ctx v, q_norm_w, k_norm_w."""
    if seed is not None:
        cfg = Config(**{**cfg.__dict__, "seed": seed})
    c = np.asarray(context_lengths(cfg) if ctx_lens is None else ctx_lens, dtype=np.int64)
    b = np.full(len(c), cfg.block, dtype=np.int64) if block_lens is None else np.asarray(block_lens, dtype=np.int64)
    n = len(c)
    qsl = np.zeros(n + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(b)
    csl = np.zeros(n + 1, dtype=np.int64)
    csl[1:] = np.cumsum(c)
    t, ct = int(qsl[-1]), int(csl[-1])
    positions = np.concatenate([c[r] + np.arange(b[r]) for r in range(n)]) if t else np.zeros(0, np.int64)
    ctx_pos = np.concatenate([np.arange(c[r]) for r in range(n)]) if ct else np.zeros(0, np.int64)
    s = cfg.seed
    return Batch(
        cfg=cfg,
        ctx_lens=c.astype(np.int32), block_lens=b.astype(np.int32),
        query_start_loc=qsl.astype(np.int32), ctx_start_loc=csl.astype(np.int32),
        positions=positions.astype(np.int32), ctx_pos=ctx_pos.astype(np.int32),
        q=normal_bf16(s, STREAM_Q, t * cfg.hq * cfg.dh).reshape(t, cfg.hq, cfg.dh),
        k_blk=normal_bf16(s, STREAM_KBLK, t * cfg.hkv * cfg.dh).reshape(t, cfg.hkv, cfg.dh),
        v_blk=normal_bf16(s, STREAM_VBLK, t * cfg.hkv * cfg.dh).reshape(t, cfg.hkv, cfg.dh),
        ctx_k_raw=normal_bf16(s, STREAM_CTXK, ct * cfg.hkv * cfg.dh).reshape(ct, cfg.hkv, cfg.dh),
        ctx_v=normal_bf16(s, STREAM_CTXV, ct * cfg.hkv * cfg.dh).reshape(ct, cfg.hkv, cfg.dh),
        q_norm_w=uniform_bf16(s, STREAM_QW, cfg.dh, 0.5, 1.5),
        k_norm_w=uniform_bf16(s, STREAM_KW, cfg.dh, 0.5, 1.5),
    )


# ---------------------------------------------------------------- draft-step input preparation
STREAM_PREP = 8


@dataclass
class PrepareBatch:
    """Integer inputs of one draft step's input preparation (vllm.cpp qwen3_dflash.cpp,
    PrepareDflashInputs): the target tokens scored this step per request, how many were
    rejected, the sampled / next-prefill token of each request state and the block tables."""
    idx_mapping: np.ndarray             # int32 [N] request state of each batch row
    target_query_start_loc: np.ndarray  # int32 [N+1]
    num_rejected: np.ndarray            # int32 [N]
    num_sampled: np.ndarray             # int32 [N]
    last_sampled: np.ndarray            # int32 [max_num_reqs] per request state
    next_prefill_tokens: np.ndarray     # int32 [max_num_reqs] per request state
    target_positions: np.ndarray        # int64 [num_target_tokens]
    block_table: np.ndarray             # int32 [N, stride]
    num_query_per_req: int
    num_speculative_steps: int
    block_size: int
    max_num_reqs: int
    max_num_tokens: int
    max_model_len: int
    parallel_drafting_token_id: int
    sample_from_anchor: bool

    def scalars(self) -> dict:
        return dict(num_query_per_req=self.num_query_per_req, num_speculative_steps=self.num_speculative_steps,
                    block_size=self.block_size, max_num_reqs=self.max_num_reqs, max_num_tokens=self.max_num_tokens,
                    max_model_len=self.max_model_len, parallel_drafting_token_id=self.parallel_drafting_token_id,
                    sample_from_anchor=self.sample_from_anchor)


def make_prepare_batch(seed: int, num_reqs: int, block: int = 16, sample_from_anchor: bool = False,
                       prefill_frac: float = 0.25, max_prefill_chunk: int = 512, max_start: int = 30000,
                       block_size: int = 16, max_model_len: int = 32768, stride: int | None = None,
                       max_num_reqs: int | None = None, max_num_tokens: int | None = None,
                       vocab: int = 151936) -> PrepareBatch:
    """Draws a batch: each request is a decode step (the target scored the previous block of up
    to `block` tokens and rejected some of them) or, with probability prefill_frac, a prefill
    chunk (nothing rejected, sampled only if it was the last chunk). Positions continue a
    context of a uniformly drawn length below max_start; request states are a random subset of
    max_num_reqs; page ids are distinct and shuffled."""
    n = int(num_reqs)
    max_num_reqs = n + 3 if max_num_reqs is None else int(max_num_reqs)
    max_num_tokens = n * block + 5 if max_num_tokens is None else int(max_num_tokens)
    if stride is None:
        stride = (max_start + max_prefill_chunk + 2 * block + block_size - 1) // block_size
    u = uniform(seed, STREAM_PREP, 0, 5 * n)
    counts = np.zeros(n, dtype=np.int64)
    rejected = np.zeros(n, dtype=np.int64)
    sampled = np.zeros(n, dtype=np.int64)
    start = np.zeros(n, dtype=np.int64)
    for r in range(n):
        a, b_, c_, d_, e_ = u[5 * r:5 * r + 5]
        start[r] = int(d_ * max_start)
        if a < prefill_frac:
            counts[r] = 1 + int(b_ * (max_prefill_chunk - 1))
            sampled[r] = 1 if c_ < 0.5 else 0
        else:
            counts[r] = 1 + int(b_ * (block - 1e-9))
            rejected[r] = int(c_ * (counts[r] - 1e-9))
            sampled[r] = 1 if e_ < 0.9 else 0
    qsl = np.zeros(n + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(counts)
    positions = np.concatenate([start[r] + np.arange(counts[r]) for r in range(n)]).astype(np.int64)
    states = np.argsort(uniform(seed, STREAM_PREP + 1, 0, max_num_reqs), kind="stable")[:n]
    tokens = (uniform(seed, STREAM_PREP + 2, 0, 2 * max_num_reqs) * vocab).astype(np.int64).clip(0, vocab - 1)
    pages = np.argsort(uniform(seed, STREAM_PREP + 3, 0, n * stride), kind="stable").reshape(n, stride)
    return PrepareBatch(
        idx_mapping=states.astype(np.int32), target_query_start_loc=qsl.astype(np.int32),
        num_rejected=rejected.astype(np.int32), num_sampled=sampled.astype(np.int32),
        last_sampled=tokens[:max_num_reqs].astype(np.int32),
        next_prefill_tokens=tokens[max_num_reqs:].astype(np.int32), target_positions=positions,
        block_table=pages.astype(np.int32), num_query_per_req=block,
        num_speculative_steps=block if sample_from_anchor else block - 1, block_size=block_size,
        max_num_reqs=max_num_reqs, max_num_tokens=max_num_tokens, max_model_len=max_model_len,
        parallel_drafting_token_id=vocab - 1, sample_from_anchor=bool(sample_from_anchor))
