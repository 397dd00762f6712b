#!/usr/bin/env python3
"""Benchmark of the DFlash draft block-attention hot path on GB300.

One step = one pass of the whole path over one synthetic batch, as a draft step runs it:
  1. the rows appended to each request's context this step (the previous block, B rows
     per request) are normed, rotated and scattered into the device-resident context K/V
     store: dflash_context_kv with explicit slots (contiguous store), or, with --paged,
     dflash_paged_append, which derives positions and page slots on the device and
     advances the device lengths;
  2. dflash_block_attention (or _paged): q/k norm + RoPE prologue, block attention of
     every block row over [context ; block] of its request, split-KV combine.
The context store is device state that persists across steps (it is built once,
untimed), as the draft model keeps it resident. The two integer-side calls of a draft
step (paged append, input preparation) are also timed on their own ("draft_step_ops").

Metric: K/V HBM GB/s of block attention (algorithmic bytes: each allowed context or
block key's K and V read once per (request, kv head)), with TFLOP/s and the fraction
of the GB300 roofline beside it. L2 is flushed (256 MB write) before every step,
outside the timed events.

The timed step runs the largest workload (ragged: 64 requests, contexts log-uniform in
[1024, 32768]) by default. The same JSON line also carries, each timed the same way with its
own clock record: "per_workload" (the Qwen3-4B-shaped layer and the sliding-window layer),
"context_store" (dflash_context_kv building the whole context store) and "draft_step_ops".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W  # noqa: E402
from speculative_decoding_draft_rmsnorm_gb300.sharding import max_over_ranks  # noqa: E402

METRIC = "DFlash block-attn TFLOP/s and K/V HBM GB/s, % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- accounting
def algorithmic_counts(cfg: W.Config, ctx_lens, block_lens) -> dict:
    """Keys each (request, kv head) must read, allowed (query, key) pairs, bytes and flops.

    A key counts once per (request, kv head) if some block row of the request may attend
    to it (window-masked context keys are not counted). Bytes: bf16 K and V of those
    keys. Flops: 4 * Dh per allowed (query row, key) pair and query head (QK^T and PV).
    """
    keys = 0
    pairs = 0
    for c, b in zip(ctx_lens, block_lens):
        c, b = int(c), int(b)
        if b == 0:
            continue
        if not cfg.causal:
            keys += c + b
            pairs += b * (c + b)
            continue
        w = cfg.window if cfg.window > 0 else c + b + 1
        keys += (c + b) - max(0, c - w + 1)
        for i in range(c, c + b):
            pairs += i + 1 - max(0, i - w + 1)
    return {"keys": keys, "pairs": pairs, "kv_bytes": keys * cfg.hkv * cfg.dh * 4,
            "flops": 4 * cfg.dh * pairs * cfg.hq}


def describe(cfg: W.Config, ctx_lens, paged: int = 0, world: int = 1) -> dict:
    """The workload's config dict, the same in both arms."""
    mask = "bidirectional" if not cfg.causal else (f"causal, window {cfg.window}" if cfg.window else "causal")
    if cfg.ctx_len is not None:
        c = str(cfg.ctx_len)
    elif cfg.ctx_uniform is not None:
        c = f"U[{cfg.ctx_uniform[0]},{cfg.ctx_uniform[1]}] (sum {int(sum(ctx_lens))})"
    else:
        c = f"log-uniform[{cfg.ctx_loguniform[0]},{cfg.ctx_loguniform[1]}] (sum {int(sum(ctx_lens))})"
    return {"workload": cfg.name + ": " + cfg.note, "requests": cfg.num_reqs, "ctx_len": c, "block": cfg.block,
            "hq": cfg.hq, "hkv": cfg.hkv, "dh": cfg.dh, "mask": mask, "seed": cfg.seed,
            "split_kv": "forced" if cfg.force_split else "balanced schedule",
            "appended_rows_per_request": cfg.block,
            "l2": "flushed before every step (256 MB write, outside the timed events)",
            "context": (f"paged: {paged}-row pages in shuffled order, block table per request; the step's append "
                        "(dflash_paged_append) advances the device lengths the attention reads, and they are put "
                        "back between steps outside the timed events" if paged else "contiguous segments"),
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"])}, "of measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "of fallback"


# the sources of the three launches of one attention call (prologue, attention, combine)
ATTENTION_SOURCES = ("api.cu", "attention.cu", "internal.h", "norm_rope.cuh", "ptx.cuh")


def _code_only(text: str) -> str:
    """The source without comments and blank lines, so that editing a comment keeps the hash."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip() if '"' not in line else line.rstrip()
        if code.strip():
            out.append(code)
    return "\n".join(out)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_draft_rmsnorm_gb300", "csrc")
    for name in ATTENTION_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu capture, if the kernels are unchanged."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("source_hash") != kernel_source_hash():
            return None
        return d.get("per_launch_bytes", {}).get(workload)
    except Exception:
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        """Starts nvidia-smi (one sample every 20 ms) and waits, up to 3 s, for its first
        sample, so that the record covers the work launched after this returns."""
        import threading
        self.proc = None
        self.dev = device_index
        self.lines: list[str] = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        first = threading.Event()

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line)
                first.set()
            first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(timeout=3.0)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.03)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        self.thread.join(timeout=2)
        out = "".join(self.lines)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm
class Step:
    """Device-resident inputs of one step and the two library calls that make it."""

    def __init__(self, lib, b: W.Batch, flags: int, page_size: int = 0):
        import numpy as np
        import torch
        self.lib, self.b, self.cfg, self.flags, self.page_size = lib, b, b.cfg, flags, page_size
        c = b.cfg

        def d16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

        def d32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()

        self.d16, self.d32 = d16, d32
        # rows appended this step: the last min(B, C) context rows of every request
        idx = []
        appended = np.zeros(c.num_reqs, dtype=np.int64)
        for r in range(c.num_reqs):
            a = min(int(b.block_lens[r]), int(b.ctx_lens[r]))
            appended[r] = a
            end = int(b.ctx_start_loc[r]) + int(b.ctx_lens[r])
            idx.extend(range(end - a, end))
        self.new_idx = np.array(idx, dtype=np.int64)
        # store row of every context row: itself (contiguous), or its page slot in a pool whose
        # pages are handed out in a shuffled order (paged)
        n_ctx = b.ctx_k_raw.shape[0]
        if page_size:
            pages_per = [(int(l) + page_size - 1) // page_size for l in b.ctx_lens]
            n_pages = max(1, sum(pages_per))
            order = np.random.default_rng(c.seed + 1).permutation(n_pages)
            self.block_table = np.full((c.num_reqs, max(1, max(pages_per))), -1, dtype=np.int32)
            store_row = np.zeros(n_ctx, dtype=np.int64)
            k = 0
            for r in range(c.num_reqs):
                for p in range(pages_per[r]):
                    self.block_table[r, p] = order[k]
                    k += 1
                base = int(b.ctx_start_loc[r])
                j = np.arange(int(b.ctx_lens[r]))
                store_row[base + j] = self.block_table[r, j // page_size].astype(np.int64) * page_size + j % page_size
            store_rows = n_pages * page_size
        else:
            store_row = np.arange(n_ctx, dtype=np.int64)
            store_rows = n_ctx
        self.store_rows = store_rows
        self.host = {
            "k_new": np.ascontiguousarray(b.ctx_k_raw[self.new_idx]),
            "v_new": np.ascontiguousarray(b.ctx_v[self.new_idx]),
            "q": b.q, "k_blk": b.k_blk, "v_blk": b.v_blk, "positions": b.positions, "qsl": b.query_start_loc,
        }
        if page_size:
            # the step's append derives positions and slots on the device from the stored
            # lengths and the block table, and advances the lengths the attention then reads
            nsl = np.zeros(c.num_reqs + 1, dtype=np.int32)
            nsl[1:] = np.cumsum(appended)
            self.host.update({"nsl": nsl, "bt": self.block_table,
                              "lens_before": (b.ctx_lens.astype(np.int64) - appended).astype(np.int32)})
        else:
            self.host.update({"pos_new": np.ascontiguousarray(b.ctx_pos[self.new_idx]).astype(np.int32),
                              "slot": store_row[self.new_idx].astype(np.int32), "csl": b.ctx_start_loc,
                              "clen": b.ctx_lens})
        self.dev = {k: (d16(v) if v.dtype == np.uint16 else d32(v)) for k, v in self.host.items()}
        # device lengths of the paged store (the attention's ctx_lens); set by reset()
        self.seq_lens = d32(b.ctx_lens) if page_size else None
        self.q_norm_w, self.k_norm_w = d16(b.q_norm_w), d16(b.k_norm_w)
        # the resident context store, built once (untimed): keys normed + rotated into their
        # store rows by the append kernel itself, values copied there
        hkv, dh = c.hkv, c.dh
        self.ctx_k = torch.empty((store_rows, hkv, dh), dtype=torch.bfloat16, device="cuda")
        self.ctx_v = torch.zeros((store_rows, hkv, dh), dtype=torch.bfloat16, device="cuda")
        lib.context_kv(d16(b.ctx_k_raw), d32(b.ctx_pos), self.k_norm_w, self.ctx_k, v=d16(b.ctx_v), ctx_v=self.ctx_v,
                       slot=d32(store_row.astype(np.int32)), eps=c.eps, theta=c.theta)
        self.max_ctx = int(max(1, b.ctx_lens.max(initial=0)))
        self.max_blk = int(max(1, b.block_lens.max(initial=0)))
        t, hq, dh = b.q.shape
        self.out = torch.empty((t, hq, dh), dtype=torch.bfloat16, device="cuda")
        self.args = (b.cfg.num_reqs, t, hq, c.hkv, dh, store_rows, self.max_ctx, self.max_blk, c.causal,
                     c.window, lib.OUT_BF16, flags)
        self.plan = lib.plan(*self.args)
        self.ws = lib.alloc_workspace(lib.workspace_size(*self.args))
        torch.cuda.synchronize()

    def reset(self):
        """Puts the stored lengths back to their value before this step's append, so that every
        step is the same step (outside the timed events, like the L2 flush)."""
        if self.page_size:
            self.seq_lens.copy_(self.dev["lens_before"])

    def append(self, dev=None):
        d = dev or self.dev
        c = self.cfg
        if self.page_size:
            ps = self.page_size
            self.lib.paged_append(d["k_new"], d["nsl"], self.seq_lens, d["bt"], self.k_norm_w,
                                  self.ctx_k.view(-1, ps, c.hkv, c.dh), v=d["v_new"],
                                  v_pool=self.ctx_v.view(-1, ps, c.hkv, c.dh), eps=c.eps, theta=c.theta)
            return
        self.lib.context_kv(d["k_new"], d["pos_new"], self.k_norm_w, self.ctx_k, v=d["v_new"], ctx_v=self.ctx_v,
                            slot=d["slot"], eps=c.eps, theta=c.theta)

    def attend(self, dev=None):
        d = dev or self.dev
        c = self.cfg
        if self.page_size:
            ps = self.page_size
            self.lib.block_attention_paged(
                d["q"], d["k_blk"], d["v_blk"], self.ctx_k.view(-1, ps, c.hkv, c.dh),
                self.ctx_v.view(-1, ps, c.hkv, c.dh), d["bt"], d["qsl"], self.seq_lens, d["positions"], self.q_norm_w,
                self.k_norm_w, max_ctx_len=self.max_ctx, max_block_len=self.max_blk, out=self.out,
                workspace=self.ws, eps=c.eps, theta=c.theta, causal=c.causal, window=c.window, flags=self.flags)
            return
        self.lib.block_attention(d["q"], d["k_blk"], d["v_blk"], self.ctx_k, self.ctx_v, d["qsl"], d["csl"],
                                 d["clen"], d["positions"], self.q_norm_w, self.k_norm_w, max_ctx_len=self.max_ctx,
                                 max_block_len=self.max_blk, out=self.out, workspace=self.ws, eps=c.eps,
                                 theta=c.theta, causal=c.causal, window=c.window, flags=self.flags)

    def launches_per_step(self) -> int:
        return (2 if self.page_size else 1) + int(self.plan["launches"])


def gpu_spin(seconds: float) -> None:
    """Queues a kernel that keeps the GPU busy for about `seconds` (SM clock cycles at the
    maximum clock), so that the host can queue the following launches ahead of the GPU."""
    import torch
    torch.cuda._sleep(int(seconds * 2.07e9))


def timed_steps(st: "Step", flush, stream, steps: int, warmup: int, barrier, dev_index: int,
                window_s: float) -> tuple[list, list, dict | None]:
    """Warm-up, then `steps` timed steps (CUDA events around the append and the attention
    call, L2 flushed before each step outside the events), then a clock window: the same
    step repeated for about `window_s` seconds, untimed by the result but sampled, so that the
    nvidia-smi record (20 ms period) spans the timed steps with enough samples. Returns the
    per-step and per-call times (ms) and the clock record (with the window's mean step time
    and time x MHz)."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        st.reset()
        st.append()
        st.attend()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev_index)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    # untimed GPU work queued first (a spin of about 0.3 ms per step to come), so that the host
    # has queued every timed step before the GPU reaches the first one: the host's own time per
    # step (Python argument checks, tensor-map encoding, launches) then never shows up as GPU
    # idle time between the events
    gpu_spin(0.3e-3 * steps)
    for i in range(steps):
        flush.zero_()
        st.reset()
        ev[i][0].record(stream)
        st.append()
        ev[i][1].record(stream)
        st.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    attn_ms = [e[1].elapsed_time(e[2]) for e in ev]
    # clock window
    win_ms, n_win = 0.0, 0
    if window_s > 0:
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_win = max(1, int(window_s * 1e3 / max(1e-3, statistics.mean(step_ms) + 0.08)))
        w0.record(stream)
        for _ in range(n_win):
            flush.zero_()
            st.reset()
            st.append()
            st.attend()
        w1.record(stream)
        torch.cuda.synchronize()
        win_ms = w0.elapsed_time(w1)
    clk = clocks.stop()
    if clk is not None and n_win:
        per = win_ms / n_win
        clk["window"] = {"steps": n_win, "ms_per_step_incl_flush": per,
                         "us_x_mhz_per_step": per * 1e3 * clk["sm_mhz"]}
    return step_ms, attn_ms, clk


def attention_entry(cfg: W.Config, b: W.Batch, attn_ms: list, peaks: dict, peak_note: str, paged: int,
                    clk) -> dict:
    counts = algorithmic_counts(cfg, b.ctx_lens, b.block_lens)
    avg_s = statistics.mean(attn_ms) / 1e3
    achieved = counts["kv_bytes"] / avg_s / 1e9
    return {
        "bound": "hbm",
        "kernel": "dflash_block_attention call (prologue + attention + combine launches)",
        "achieved": achieved,
        "peak": peaks["hbm_gbs"],
        "unit": "GB/s",
        "frac": achieved / peaks["hbm_gbs"],
        "peak_source": peak_note,
        "traffic": recorded_traffic(cfg.name + (f"_paged{paged}" if paged else "")),
        "algorithmic_bytes_per_launch": counts["kv_bytes"],
        "call_us": avg_s * 1e6,
        "tensor_tflops": counts["flops"] / avg_s / 1e12,
        "tensor_frac": counts["flops"] / avg_s / 1e12 / peaks["bf16_tflops"],
        **({"clocks": clk} if clk is not None else {}),
    }


def time_context_store(lib, b: W.Batch, st: "Step", flush, stream, steps: int, peaks: dict, peak_note: str) -> dict:
    """dflash_context_kv over the whole context (every row of the store: K normed + rotated,
    V copied), timed on its own: algorithmic bytes = K and V read and written, 4 * rows * Hkv *
    Dh * 2 B."""
    import numpy as np
    import torch
    c = b.cfg
    k_raw = st.d16(b.ctx_k_raw)
    v_raw = st.d16(b.ctx_v)
    pos = st.d32(b.ctx_pos)
    n = b.ctx_k_raw.shape[0]
    ck = torch.empty((n, c.hkv, c.dh), dtype=torch.bfloat16, device="cuda")
    cv = torch.empty_like(ck)
    call = lambda: lib.context_kv(k_raw, pos, st.k_norm_w, ck, v=v_raw, ctx_v=cv, eps=c.eps, theta=c.theta)  # noqa: E731
    for _ in range(3):
        flush.zero_()
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    gpu_spin(0.2e-3 * steps)
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    nbytes = 4 * n * c.hkv * c.dh * 2
    achieved = nbytes / (us * 1e-6) / 1e9
    del k_raw, v_raw, ck, cv
    return {"kernel": "dflash_context_kv (norm_rope_kernel), the whole context store", "rows": int(n),
            "us": us, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_note,
            "algorithmic_bytes_per_launch": nbytes}


def run_gpu(args, b: W.Batch, rank: int, world: int) -> dict | None:
    import numpy as np
    import torch
    import speculative_decoding_draft_rmsnorm_gb300 as lib

    lib.load(build_if_missing=False)
    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    cfg = b.cfg
    flags = lib.FLAG_FORCE_SPLIT if cfg.force_split else 0
    st = Step(lib, b, flags, args.paged)
    counts = algorithmic_counts(cfg, b.ctx_lens, b.block_lens)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    peaks, peak_note = load_peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    step_ms, attn_ms, clk = timed_steps(st, flush, stream, args.steps, args.warmup, barrier, dev_index,
                                        args.clock_window)
    lib.check_error(st.ws)
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, device="cuda")

    roof = attention_entry(cfg, b, attn_ms, peaks, peak_note, args.paged, None)
    res = {
        "metric": METRIC,
        "value": world * counts["kv_bytes"] * args.steps / (total_ms / 1e3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": describe(cfg, b.ctx_lens, args.paged, world),
        "tflops": world * counts["flops"] * args.steps / (total_ms / 1e3) / 1e12,
        "attention_ms": statistics.mean(attn_ms),
        "append_ms": statistics.mean(s - a for s, a in zip(step_ms, attn_ms)),
        "roofline": roof,
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clk,
        "plan": st.plan,
    }
    if args.step_only:
        return res

    # ---- end to end through the public API with host buffers (pinned), copies timed: the step's
    # host inputs sit in one pinned buffer and go to the device in one copy (staging.HostStaging)
    from speculative_decoding_draft_rmsnorm_gb300.staging import HostStaging
    staging = HostStaging(st.host)
    out_host = torch.empty(st.out.shape, dtype=torch.bfloat16).pin_memory()
    h2d = staging.nbytes
    d2h = out_host.numel() * out_host.element_size()
    device_lens = st.seq_lens
    if st.page_size:  # the lengths before the append arrive with the inputs and are advanced in place
        st.seq_lens = staging.views["lens_before"]

    def e2e_step():
        staging.upload(stream)
        st.append(staging.views)
        st.attend(staging.views)
        out_host.copy_(st.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for _ in range(3):
        flush.zero_()
    for i in range(args.steps):
        flush.zero_()
        eev[i][0].record(stream)
        e2e_step()
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(e[0].elapsed_time(e[1]) for e in eev)
    st.seq_lens = device_lens

    res["e2e"] = {"value": world * counts["kv_bytes"] * args.steps / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "host_inputs": "one pinned staging buffer, one host-to-device copy per step"}
    res["context_store"] = time_context_store(lib, b, st, flush, stream, args.steps, peaks, peak_note)
    res["draft_step_ops"] = time_draft_ops(lib, b, flush, stream, args.steps)
    del st, staging
    torch.cuda.empty_cache()
    # ---- the other long-context workloads of the target (Qwen3-4B-shaped and SWA layers),
    # each timed the same way with its own clock record
    if not args.paged and not args.no_per_workload:
        per = {}
        for name in ("qwen3_4b", "swa", "ragged"):
            if name == cfg.name:
                continue
            bw = W.make_batch(W.CONFIGS[name])
            sw = Step(lib, bw, lib.FLAG_FORCE_SPLIT if bw.cfg.force_split else 0, 0)
            _, am, ck = timed_steps(sw, flush, stream, args.steps, args.warmup, barrier, dev_index,
                                    args.clock_window)
            lib.check_error(sw.ws)
            per[name] = {"config": describe(bw.cfg, bw.ctx_lens, 0, world),
                         "roofline": attention_entry(bw.cfg, bw, am, peaks, peak_note, 0, ck)}
            del sw
            torch.cuda.empty_cache()
        res["per_workload"] = per
    return res


def time_draft_ops(lib, b: W.Batch, flush, stream, steps: int) -> dict:
    """The two integer-side calls of a draft step on a batch of this workload's requests,
    each timed on its own (CUDA events around each call, L2 flushed before each):

      paged_append: every request appends B rows (the previous block) after its context
        into 16-row pages; bytes = rows read (K and V) + rows written (K and V).
      prepare_inputs: decode-step metadata of the same requests (each scored a block of up
        to B target tokens and rejected some); bytes = every input and output array.
    Both move kilobytes to a few MB, so their time is launch latency, not bandwidth.
    """
    import numpy as np
    import torch
    c = b.cfg
    n, blk, ps = c.num_reqs, c.block, 16
    d32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()  # noqa: E731

    def timed(fn, reset=None):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for _ in range(3):
            if reset:
                reset()
            fn()
        gpu_spin(0.2e-3 * steps)
        for i in range(steps):
            flush.zero_()
            if reset:
                reset()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3  # us

    # paged append: B rows per request after a context of ctx_lens[r] rows
    lens0 = b.ctx_lens.astype(np.int64)
    first_page = lens0 // ps
    last_page = (lens0 + blk - 1) // ps
    max_pages = int(last_page.max()) + 1
    bt = np.zeros((n, max_pages), dtype=np.int32)
    nxt = 0
    for r in range(n):
        for p in range(int(first_page[r]), int(last_page[r]) + 1):
            bt[r, p] = nxt
            nxt += 1
    pool_k = torch.zeros((nxt, ps, c.hkv, c.dh), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    rows = n * blk
    k_new = torch.randn((rows, c.hkv, c.dh), device="cuda").to(torch.bfloat16)
    v_new = torch.randn_like(k_new)
    w = torch.ones(c.dh, dtype=torch.bfloat16, device="cuda")
    nsl = d32(np.arange(n + 1) * blk)
    base, lens, dbt = d32(lens0), d32(lens0), d32(bt)
    append_us = timed(lambda: lib.paged_append(k_new, nsl, lens, dbt, w, pool_k, v=v_new, v_pool=pool_v,
                                               eps=c.eps, theta=c.theta), reset=lambda: lens.copy_(base))
    append_bytes = 2 * 2 * rows * c.hkv * c.dh * 2 + (n + 1) * 4 + 2 * n * 4

    # input preparation for the same requests
    pb = W.make_prepare_batch(c.seed, n, block=blk, prefill_frac=0.0)
    t = {k: d32(getattr(pb, k)) for k in ("idx_mapping", "target_query_start_loc", "num_rejected", "num_sampled",
                                          "last_sampled", "next_prefill_tokens", "block_table")}
    t["target_positions"] = torch.from_numpy(pb.target_positions.astype(np.int64)).cuda()
    out = lib.prepare_inputs(**t, **pb.scalars())
    prep_us = timed(lambda: lib.prepare_inputs(**t, **pb.scalars(), out=out))
    prep_bytes = sum(v.numel() * v.element_size() for v in list(t.values()) + list(out.values()))
    return {
        "paged_append": {"us": append_us, "rows": rows, "bytes": append_bytes,
                         "gb_per_s": append_bytes / (append_us * 1e-6) / 1e9, "launches": 2,
                         "bound": "launch latency (a few MB)"},
        "prepare_inputs": {"us": prep_us, "requests": n, "target_tokens": int(pb.target_query_start_loc[-1]),
                           "bytes": prep_bytes, "launches": 1, "bound": "launch latency (kilobytes)"},
    }


# ---------------------------------------------------------------- oracle (CPU)
def oracle_sample(b_full: W.Batch, budget_s: float):
    """Times the f64 oracle on a bounded prefix of the workload's requests.

    Returns (seconds, kv_bytes of the sample, description, cores). The context store
    of the sample is built by the oracle first (untimed); the timed part is the step:
    the appended rows' store write plus block attention.
    """
    import numpy as np
    import oracle

    def sub_batch(b: W.Batch, k: int) -> W.Batch:
        q1, c1 = int(b.query_start_loc[k]), int(b.ctx_start_loc[k])
        return W.Batch(cfg=b.cfg, ctx_lens=b.ctx_lens[:k], block_lens=b.block_lens[:k],
                       query_start_loc=b.query_start_loc[:k + 1], ctx_start_loc=b.ctx_start_loc[:k + 1],
                       positions=b.positions[:q1], ctx_pos=b.ctx_pos[:c1], q=b.q[:q1], k_blk=b.k_blk[:q1],
                       v_blk=b.v_blk[:q1], ctx_k_raw=b.ctx_k_raw[:c1], ctx_v=b.ctx_v[:c1], q_norm_w=b.q_norm_w,
                       k_norm_w=b.k_norm_w)

    cfg = b_full.cfg
    lens = b_full.ctx_lens.astype(np.int64)

    def time_step(sb: W.Batch) -> float:
        c = sb.cfg
        _, store = oracle.context_kv(sb.ctx_k_raw, sb.ctx_pos, sb.k_norm_w, c.eps, c.theta)
        idx = []
        for r in range(len(sb.ctx_lens)):
            a = min(int(sb.block_lens[r]), int(sb.ctx_lens[r]))
            end = int(sb.ctx_start_loc[r]) + int(sb.ctx_lens[r])
            idx.extend(range(end - a, end))
        idx = np.array(idx, dtype=np.int64)
        t0 = time.perf_counter()
        _, new16 = oracle.context_kv(sb.ctx_k_raw[idx], sb.ctx_pos[idx], sb.k_norm_w, c.eps, c.theta)
        store[idx] = new16
        oracle.block_attention(sb.q, sb.k_blk, sb.v_blk, store, sb.ctx_v, sb.query_start_loc, sb.ctx_start_loc,
                               sb.ctx_lens, sb.positions, sb.q_norm_w, sb.k_norm_w, eps=c.eps, theta=c.theta,
                               causal=c.causal, window=c.window)
        return time.perf_counter() - t0

    t1 = time_step(sub_batch(b_full, 1))
    k = int(max(1, min(cfg.num_reqs, math.floor(budget_s / max(t1, 1e-3)))))
    sb = sub_batch(b_full, k)
    secs = time_step(sb) if k > 1 else t1
    cnt = algorithmic_counts(cfg, sb.ctx_lens, sb.block_lens)
    desc = f"first {k} of {cfg.num_reqs} requests (context lengths {int(lens[:k].sum())} rows in all)"
    return secs, cnt["kv_bytes"], desc, oracle.num_threads(), sb, time_step


def cpu_baseline(b: W.Batch) -> dict:
    secs, nbytes, desc, cores, _, _ = oracle_sample(b, budget_s=12.0)
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc,
            "seconds": secs}


def run_reference(args, b: W.Batch) -> dict:
    # each step: the oracle on a bounded sample sized so that the whole run takes minutes
    cfg = b.cfg
    per_step_budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    secs, nbytes, desc, cores, sb, time_step = oracle_sample(b, per_step_budget)
    for _ in range(max(0, args.warmup - 1)):
        time_step(sb)
    times = [time_step(sb) for _ in range(args.steps)]
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": describe(cfg, b.ctx_lens, args.paged, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ragged", choices=sorted(W.CONFIGS),
                    help="the timed step's workload (default: the largest, the ragged long-context batch)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip timing the other long-context workloads beside the main one")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step alone: no end-to-end, context-store, draft-op, per-workload or CPU lines "
                         "(for profiling: fewer launches and allocations)")
    ap.add_argument("--clock-window", type=float, default=0.3,
                    help="seconds of repeated steps after the timed ones, sampled for the clock record")
    ap.add_argument("--paged", type=int, default=0, choices=[0, 16, 32, 64, 128],
                    help="context in a page pool of this many rows per page (shuffled page order); 0: contiguous")
    args = ap.parse_args()
    if args.step_only:
        args.no_per_workload = args.no_cpu_baseline = True
        args.clock_window = 0.0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = W.CONFIGS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, W.make_batch(cfg))), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    b = W.make_batch(cfg)
    res = run_gpu(args, b, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(b)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
