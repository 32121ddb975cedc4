#!/usr/bin/env python
"""Benchmark of the generalized paged-attention hot path on one GB300.

One *step* is one pass of the whole path over one batch of synthetic input:
  block_copy  (copy-on-write of shared blocks before they are written),
  kv_append   (the step's new tokens into their slots),
  pa_forward  (attention of every sequence's new tokens over its cached-plus-new context).

Workloads (``--workload``):
  decode13b   (default) 64 sequences, Llama-2-13B attention shape (40 MHA heads, d=128), bf16,
              block 16, q_len 1, context U{512..4096}, blocks scattered in a pool with 10% free;
              6 sequences fork (copy-on-write of their partially filled last block).
              Metric: algorithmic HBM bytes / step time, GB/s.  The line also carries the metric's
              prefill half, measured in the same process with the same --steps / --warmup:
              "mixed_prefill" (the mixed_gqa workload) and "long_prefill" (longprefill), each with
              its own value (TFLOP/s), roofline, cpu_baseline, e2e and clocks
              (--headline-only leaves them out).
  decode13b_fp8  the same batch with FP8 E4M3 K/V caches (scale 1/32 for K and V): half the K/V
              bytes per token.  Metric: GB/s (of the 8-bit bytes); the line also gives tokens/s.
  mixed_gqa   32 resumed conversations (history U{1024..16384}, new turn U{16..512}) + 32 decode
              sequences, GQA 32/8, d=128, bf16, block 32.  Metric: attention TFLOP/s (causal-exact).
  mixed_gqa_fp8  the mixed_gqa batch with FP8 E4M3 K/V caches (scale 1/32): the resumed turns'
              blocks widened to bf16 in workspace scratch, then the tcgen05 kernel; decode rows on
              the CUDA-core E4M3 kernel.  Metric: TFLOP/s.
  longprefill 8 x (16384 cached + 2048 new), 40 MHA heads, d=128, bf16, block 16, ConvKV-style
              turn segments.  Metric: attention TFLOP/s.
  kvmove      40-layer 5120-hidden fp16 pool (8 layers resident), 64 sessions: append, 10%
              copy-on-write copies, swap-in of 8 sessions from a pinned host pool, layer by
              layer.  Metric: GB/s moved (read + write).
  swap_pipeline  the mixed_gqa batch as 8 layers; before each layer's attention the earliest 1/8
              of every resumed conversation's history comes back from pinned host memory, layer
              by layer, overlapped with the attention of the layer before (copy-engine transfer
              into a staging slot + block_copy scatter).  Metric: attention TFLOP/s of all layers
              with the swap-in inside the step; the JSON line also carries the serial schedule,
              each half alone, the gather-kernel variant and swap-out.
  decode13b_kitty  the decode13b batch over 2-bit K/V pages of 128 tokens with 32 of 128 key
              channels at 4 bits (Kitty), the last n % 128 tokens of each sequence in a bf16
              residual page; per step one appended token per sequence and one page quantised.
              Metric: GB/s (of the page records and residual bytes); the line also gives tokens/s.
  layout      the decode13b batch on one layer of an 8-layer pool kept block-first (all layers of
              a block contiguous) and layer-first; swap-in of 8 sessions in both layouts, by the
              gather kernel and by one copy-engine transfer per contiguous segment.  Metric: decode
              KV GB/s on the block-first pool.

``--impl reference`` times the float64 CPU oracle (the only reference implementation: the pages
publish no code) on a bounded sample of the same workload and prints the same JSON line.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path has no
exchange step); the time is the max over ranks and ``value`` sums the ranks' work.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_generalized_gb300 import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "paged_kv_cache_generalized_gb300", "csrc")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def measured_traffic(workload, algorithmic_bytes):
    """DRAM bytes of one launch of the dominant kernel: the ratio (traffic / algorithmic bytes)
    from the last ncu capture of this workload's kernel, scaled to this launch; None when the
    kernel sources changed since that capture (or there is none)."""
    import hashlib

    try:
        with open(TRAFFIC_FILE) as f:
            entry = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, None
    if not entry:
        return None, None
    h = hashlib.sha256()
    for name in entry["sources"]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != entry["source_sha"]:
        return None, "kernel changed since the ncu capture"
    return entry["ratio"] * algorithmic_bytes, entry["captured_case"]


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
            return self
        # the sampler is live once its first line arrives; the timed region starts after that,
        # and only lines from then on count
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.lines = []
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            # a timed region shorter than the sampling interval still gets the sample taken
            # right after it
            t0 = time.time()
            while not self.lines and time.time() - t0 < 0.5 and self.proc.poll() is None:
                time.sleep(0.01)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# Workloads on the device
# ------------------------------------------------------------------------------------------------
def attn_flops(ctx, ql, hq, d):
    """Causal-exact attention FLOPs: 4 * d * Hq per (query, visible key) pair (QK^T and PV)."""
    c = ctx.astype(np.float64)
    q = ql.astype(np.float64)
    pairs = (q * c + q * (q + 1) / 2).sum()
    return 4.0 * d * hq * pairs


TC_MIN_ROWS = 16   # query rows per KV head from which a sequence takes the tensor-core kernel


def tc_rows(batch):
    """Mask of the sequences libpagedkv runs on its tcgen05 kernel (q_len x GQA group >= 16 query
    rows per KV head, in a batch of a supported shape, scale > 0, same-dtype caches)."""
    g = batch.num_q_heads // batch.num_kv_heads
    if not _tc_enabled(batch) or batch.total_q <= batch.num_seqs:
        return np.zeros(batch.num_seqs, bool)
    return batch.q_lens.astype(np.int64) * g >= TC_MIN_ROWS


def _tc_enabled(batch):
    """Whether libpagedkv routes this batch's multi-token turns to its tensor-core kernel (bf16 or
    f16, head_dim 128, a GQA group dividing 128, blocks of 16..128 tokens)."""
    g = batch.num_q_heads // batch.num_kv_heads
    return (batch.dtype in ("bf16", "f16") and batch.head_dim == 128 and 128 % g == 0
            and 16 <= batch.block_size <= 128)


def attn_accounting(batch, cow_frac=0.0, seed=0, kv8=False):
    """Host-only accounting of one attention step over ``batch``: the copy-on-write fork pairs
    (a fraction of sequences copy their partially filled last block to a free block) and the
    step's algorithmic bytes and FLOPs.  Both arms of the bench use it, so their configs agree."""
    B = batch.block_size
    n = batch.seq_lens
    used = np.zeros(batch.num_blocks, bool)
    for i in range(batch.num_seqs):
        used[batch.block_tables[i, :(n[i] + B - 1) // B]] = True
    free = np.flatnonzero(~used)
    rng = np.random.default_rng(seed)
    k = min(int(round(cow_frac * batch.num_seqs)), len(free))
    forks = rng.choice(batch.num_seqs, k, replace=False) if k else np.zeros(0, np.int64)
    pairs = np.array([[batch.block_tables[i, (n[i] - 1) // B], free[j]] for j, i in enumerate(forks)],
                     dtype=np.int64).reshape(-1, 2)
    es = 4 if batch.dtype == "f32" else 2
    ek = 1 if kv8 else es                           # bytes of one cached element
    Hq, Hkv, d = batch.num_q_heads, batch.num_kv_heads, batch.head_dim
    T = batch.total_q
    nb = (n + B - 1) // B
    tc = tc_rows(batch)
    return {"pairs": pairs,
            "bytes_attn_tc": float(n[tc].sum() * Hkv * d * ek * 2 + 2 * batch.q_lens[tc].sum() * Hq * d * es
                                   + nb[tc].sum() * 4 + tc.sum() * 8),
            "bytes_attn": float(n.sum() * Hkv * d * ek * 2 + 2 * T * Hq * d * es + nb.sum() * 4 + batch.num_seqs * 8),
            "bytes_append": float(2 * T * Hkv * d * (es + ek) + 8 * T),
            "bytes_copy": float(len(pairs) * 2 * 2 * Hkv * B * d * ek + pairs.size * 8),
            "flops": attn_flops(batch.ctx_lens, batch.q_lens, Hq, d),
            "flops_tc": attn_flops(batch.ctx_lens[tc], batch.q_lens[tc], Hq, d),
            "pool_bytes": 2 * int(np.prod(batch.k_cache.shape)) * ek}


def kitty_record_bytes(promoted, head_dim=128):
    """Bytes of one (page, KV head) record of the 2-bit page format, from its documented layout:
    K scale and minimum per channel, V scale and minimum per token (float32), 32 promoted-id
    bytes, 2-bit K low bits and V codes of 128 tokens, and the promoted channels' high bits."""
    T = 128
    return 4 * 2 * head_dim + 4 * 2 * T + 32 + T * head_dim // 4 + T * promoted // 4 + T * head_dim // 4


def kitty_accounting(batch, R=None):
    """Host-only accounting of one 2-bit page decode step (append, one page quantised, attention)."""
    T = 128
    R = R or kitty_record_bytes(batch.promoted, batch.head_dim)
    S, Hq, Hkv, d = batch.num_seqs, batch.num_q_heads, batch.num_kv_heads, batch.head_dim
    n = batch.ctx_lens.astype(np.int64) + 1
    nfull, tail = n // T, n % T
    es = 2
    return {"bytes_attn": float((nfull * Hkv * R).sum() + (tail * Hkv * d * es * 2).sum()
                                + 2 * S * Hq * d * es + ((n + T - 1) // T).sum() * 4 + S * 8),
            "bytes_append": float(2 * int((tail > 0).sum()) * Hkv * d * es * 2 + 8 * S),
            "bytes_copy": float(2 * Hkv * T * d * es + Hkv * R + 16),
            "flops": attn_flops(batch.ctx_lens, batch.q_lens, Hq, d),
            "pool_bytes": batch.num_pages * Hkv * R + 2 * int(np.prod(batch.res_k.shape)) * es}


# (copy-on-write fraction, seed of the fork draw) of the attention workloads
ATTN_COW = {"decode13b": (0.1, 2), "decode13b_fp8": (0.1, 2), "mixed_gqa": (0.0, 3), "mixed_gqa_fp8": (0.0, 3),
            "longprefill": (0.0, 4)}


def workload_batch(name, args):
    """The workload's synthetic host-side batch (or KV-movement plan), the same in both arms."""
    seqs = getattr(args, "seqs", None)
    if name in ("decode13b", "decode13b_fp8", "layout"):
        return W.decode13b(seed=2, num_seqs=seqs or 64, poison=False)
    if name == "decode13b_kitty":
        return W.decode13b_kitty(seed=2, num_seqs=seqs or 64)
    if name in ("mixed_gqa", "mixed_gqa_fp8", "swap_pipeline"):
        half = (seqs or 64) // 2
        return W.mixed_gqa(seed=3, n_resume=half, n_decode=half, poison=False)
    if name == "longprefill":
        return W.longprefill(seed=4, num_seqs=seqs or 8, poison=False)
    if name == "kvmove":
        sessions = seqs or 64
        return W.kvmove_plan(seed=5, num_layers=args.layers, num_sessions=sessions,
                             swap_sessions=max(1, sessions // 8))
    raise ValueError(name)


def kvmove_accounting(plan):
    L, hkv, B, d = plan.num_layers, plan.num_kv_heads, plan.block_size, plan.head_dim
    T = len(plan.slot_mapping)
    bb = plan.block_bytes
    return {"bytes_cow": float(len(plan.cow_pairs) * 2 * L * bb * 2),
            "bytes_append": float(2 * L * T * hkv * d * 2 * 2 + 8 * T),
            "bytes_swap": float(len(plan.swap_pairs) * 2 * L * bb * 2),
            "pool_bytes": L * 2 * plan.num_blocks * hkv * B * d * 2}


def workload_config(name, args, world, batch):
    """The JSON line's ``config``: what the workload is and its sizes, computed on the host from
    the batch alone, so that the native and the reference arm print the same dict."""
    cfg = {"workload": workload_text(name, args)}
    if name in ATTN_COW:
        a = attn_accounting(batch, *ATTN_COW[name], kv8=name.endswith("fp8"))
        cfg["l2"] = "inputs larger than L2 (KV pool %.2f GB resident)" % (a["pool_bytes"] / 1e9)
        cfg["bytes_per_step"] = a["bytes_attn"] + a["bytes_append"] + a["bytes_copy"]
        cfg["attn_flops_per_step"] = a["flops"]
    elif name == "decode13b_kitty":
        a = kitty_accounting(batch)
        cfg["l2"] = "inputs larger than L2 (page records + residual pages %.2f GB resident)" % (a["pool_bytes"] / 1e9)
        cfg["bytes_per_step"] = a["bytes_attn"] + a["bytes_append"] + a["bytes_copy"]
        cfg["attn_flops_per_step"] = a["flops"]
    elif name == "kvmove":
        a = kvmove_accounting(batch)
        cfg["layers_resident"] = batch.num_layers
        cfg["l2"] = "inputs larger than L2 (pool %.1f GB)" % (a["pool_bytes"] / 1e9)
        cfg["bytes_per_step"] = a["bytes_cow"] + a["bytes_append"] + a["bytes_swap"]
        cfg["cow_pairs"] = len(batch.cow_pairs)
        cfg["swap_blocks"] = len(batch.swap_pairs)
        cfg["append_tokens"] = len(batch.slot_mapping)
    elif name == "swap_pipeline":
        cfg["layers_resident"] = args.layers
        cfg["l2"] = "inputs larger than L2 (%d-layer pool of the mixed batch)" % args.layers
        cfg["attn_flops_per_step"] = args.layers * attn_flops(batch.ctx_lens, batch.q_lens,
                                                              batch.num_q_heads, batch.head_dim)
    elif name == "layout":
        cfg["layers"] = args.layers
        cfg["l2"] = "inputs larger than L2 (two %d-layer pools of the decode batch)" % args.layers
    cfg["parallelism"] = f"replicas x{world}"
    return cfg


class AttnStep:
    """block_copy + pa_forward_append (the new tokens' K/V into their slots, then the attention)
    over one AttnBatch, all inputs resident on the GPU."""

    def __init__(self, batch: W.AttnBatch, dev, cow_frac=0.0, seed=0, kv8=False):
        import torch
        import paged_kv_cache_generalized_gb300 as pkg

        self.pkg, self.torch, self.b, self.dev = pkg, torch, batch, dev
        # 8-bit caches: E4M3 codes of value / scale; a scale of 1/32 puts N(0,1) values in the
        # format's normal range (|x| / scale <= 448 for |x| <= 14)
        self.kv8 = kv8
        self.ks = self.vs = (1.0 / 32) if kv8 else None
        tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[batch.dtype]
        self.tdt = tdt

        def up(x, dt=None):
            t = torch.from_numpy(np.ascontiguousarray(x))
            if dt is not None and dt != torch.float32:
                t = t.view(torch.int16).view(dt)
            return t

        self.host = {
            "q": up(batch.q, tdt).pin_memory(),
            "k_new": up(batch.k_new, tdt).pin_memory(),
            "v_new": up(batch.v_new, tdt).pin_memory(),
            "slots": up(batch.slot_mapping).pin_memory(),
            "bt": up(batch.block_tables).pin_memory(),
            "ctx": up(batch.ctx_lens).pin_memory(),
            "ql": up(batch.q_lens).pin_memory(),
        }
        acct = attn_accounting(batch, cow_frac, seed, kv8)
        pairs = acct["pairs"]
        self.host["pairs"] = up(pairs).pin_memory()
        self.dev_in = {k2: v.to(dev) for k2, v in self.host.items()}
        # K and V caches are the two planes of one pool, so one block_copy moves both
        if kv8:
            self.pool = torch.empty((2,) + batch.k_cache.shape, dtype=torch.uint8, device=dev)
            for i, x in enumerate((batch.k_cache, batch.v_cache)):
                xf = up(x, tdt).to(dev).float() / self.ks
                self.pool[i].copy_(xf.to(torch.float8_e4m3fn).view(torch.uint8))
                del xf
        else:
            self.pool = torch.empty((2,) + batch.k_cache.shape, dtype=tdt, device=dev)
            self.pool[0].copy_(up(batch.k_cache, tdt))
            self.pool[1].copy_(up(batch.v_cache, tdt))
        self.k_cache, self.v_cache = self.pool[0], self.pool[1]
        self.out = torch.empty_like(self.dev_in["q"])
        self.out_host = torch.empty_like(self.host["q"]).pin_memory()
        self.ws = torch.empty(max(256, pkg.forward_workspace_size(self.dev_in["q"], self.k_cache,
                                                                 self.dev_in["bt"], self.dev_in["ctx"])),
                              dtype=torch.uint8, device=dev)
        self.bytes_attn, self.bytes_append = acct["bytes_attn"], acct["bytes_append"]
        self.bytes_copy, self.flops = acct["bytes_copy"], acct["flops"]
        self.flops_tc, self.bytes_attn_tc = acct["flops_tc"], acct["bytes_attn_tc"]
        T = batch.total_q
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host.values())
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        # block_copy (if any fork) + the planner (whose extra blocks write the new tokens; E4M3
        # caches take a quantising append launch of their own) + the decode kernel (which merges
        # its own splits) (+ the tensor-core kernel when some turn takes it, after the widening
        # of its E4M3 blocks; the workspace holds scratch for all of them)
        self.has_tc = bool(tc_rows(batch).any())
        self.launches_per_step = ((1 if len(pairs) else 0) + (1 if kv8 else 0) + 2 + (1 if self.has_tc else 0)
                                  + (1 if self.has_tc and kv8 else 0))

    def _copy(self, inp):
        if inp["pairs"].shape[0]:
            self.pkg.block_copy(self.pool, self.pool, inp["pairs"])

    def step(self, ev=None):
        """One step; ``ev`` = (call start, call stop, tc start, tc stop, decode start, decode stop)
        events, the last four recorded by the library around its kernels."""
        inp = self.dev_in
        self._copy(inp)
        if ev is not None:
            self.pkg.set_timing_events(tc=(ev[2], ev[3]) if self.has_tc else None, cc=(ev[4], ev[5]))
            ev[0].record()
        self.pkg.pa_forward_append(inp["q"], inp["k_new"], inp["v_new"], inp["slots"], self.k_cache,
                                   self.v_cache, inp["bt"], inp["ctx"], inp["ql"], self.b.scale, out=self.out,
                                   workspace=self.ws, k_scale=self.ks, v_scale=self.vs)
        if ev is not None:
            ev[1].record()
            self.pkg.set_timing_events()

    def e2e_step(self):
        for k2, v in self.host.items():
            self.dev_in[k2].copy_(v, non_blocking=True)
        self.step()
        self.out_host.copy_(self.out, non_blocking=True)

    def decode_alone_ms(self, warmup=3, reps=20):
        """Median time of pa_forward over the sequences that do not take the tensor-core kernel
        alone (same device caches, their rows of q), outside the timed steps: the decode part's
        own rate, which the mixed call's bracket cannot give (there the decode kernel waits for the
        SMs the tensor-core kernel holds).  None when every sequence takes the tensor-core kernel."""
        torch = self.torch
        dec = np.flatnonzero(~tc_rows(self.b))
        if not self.has_tc or len(dec) == 0:
            return None
        cu = np.concatenate([[0], np.cumsum(self.b.q_lens.astype(np.int64))])
        rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in dec])
        sel = torch.from_numpy(dec).to(self.dev)
        q = self.dev_in["q"][torch.from_numpy(rows).to(self.dev)].contiguous()
        bt = self.dev_in["bt"][sel].contiguous()
        ctx, ql = self.dev_in["ctx"][sel].contiguous(), self.dev_in["ql"][sel].contiguous()
        ws = torch.empty(max(256, self.pkg.forward_workspace_size(q, self.k_cache, bt, ctx)),
                         dtype=torch.uint8, device=self.dev)
        out = torch.empty_like(q)

        def call():
            self.pkg.pa_forward(q, self.k_cache, self.v_cache, bt, ctx, ql, self.b.scale, out=out,
                                workspace=ws, k_scale=self.ks, v_scale=self.vs)

        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            call()
            e[1].record()
            torch.cuda.synchronize()
            ts.append(e[0].elapsed_time(e[1]))
        return float(np.median(ts))


class KittyStep:
    """kv_append + kv_quantize_pages + pa_forward_kitty over one KittyBatch (2-bit pages with
    promoted 4-bit key channels), all inputs resident on the GPU.  The step appends each
    sequence's new token into its residual page (the token's own values: the append is
    idempotent) and quantises one residual page into a spare record: with 64 sequences a page
    fills every 2 steps on average, so one page per step is the amortised quantisation cost."""

    def __init__(self, batch: W.KittyBatch, dev):
        import torch
        import paged_kv_cache_generalized_gb300 as pkg

        self.pkg, self.torch, self.b, self.dev = pkg, torch, batch, dev
        self.kv8 = False
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[batch.dtype]
        S, Hq, Hkv, d, P = batch.num_seqs, batch.num_q_heads, batch.num_kv_heads, batch.head_dim, batch.promoted
        T = 128
        R = pkg.kitty_record_bytes(P)

        def up(x, dt=None):
            t = torch.from_numpy(np.ascontiguousarray(x))
            if dt is not None:
                t = t.view(torch.int16).view(dt)
            return t

        n = batch.ctx_lens.astype(np.int64) + 1
        nfull, tail = n // T, n % T
        slots = np.full(S, -1, np.int64)
        k_new = np.zeros((S, Hkv, d), np.uint16)
        v_new = np.zeros((S, Hkv, d), np.uint16)
        for i in range(S):
            if tail[i]:
                rid = int(batch.block_tables[i, nfull[i]])
                slots[i] = rid * T + tail[i] - 1
                k_new[i] = batch.res_k[rid, :, tail[i] - 1]
                v_new[i] = batch.res_v[rid, :, tail[i] - 1]
        spare = np.setdiff1d(np.arange(batch.num_pages), batch.pairs[:, 1])[0]
        self.host = {
            "q": up(batch.q, tdt).pin_memory(),
            "k_new": up(k_new, tdt).pin_memory(),
            "v_new": up(v_new, tdt).pin_memory(),
            "slots": up(slots).pin_memory(),
            "bt": up(batch.block_tables).pin_memory(),
            "ctx": up(batch.ctx_lens).pin_memory(),
            "ql": up(batch.q_lens).pin_memory(),
            "qpair": up(np.array([[0, spare]], np.int64)).pin_memory(),
        }
        self.dev_in = {k2: v.to(dev) for k2, v in self.host.items()}
        self.pages = torch.zeros((batch.num_pages, Hkv, R), dtype=torch.uint8, device=dev)
        sk, sv = up(batch.stage_k, tdt).to(dev), up(batch.stage_v, tdt).to(dev)
        pkg.kv_quantize_pages(sk, sv, up(batch.pairs).to(dev), self.pages, P)
        # one staging page pair stays for the per-step quantisation
        self.stage_k, self.stage_v = sk[:1].clone(), sv[:1].clone()
        del sk, sv
        self.res_k, self.res_v = up(batch.res_k, tdt).to(dev), up(batch.res_v, tdt).to(dev)
        self.pool = self.pages
        self.out = torch.empty_like(self.dev_in["q"])
        self.out_host = torch.empty_like(self.host["q"]).pin_memory()
        need = pkg.kitty_workspace_size(self.dev_in["q"], self.pages, self.res_k, self.dev_in["bt"], P)
        self.ws = torch.empty(max(256, need), dtype=torch.uint8, device=dev)
        acct = kitty_accounting(batch, R)
        self.bytes_attn, self.bytes_append = acct["bytes_attn"], acct["bytes_append"]
        self.bytes_copy, self.flops = acct["bytes_copy"], acct["flops"]
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host.values())
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        self.launches_per_step = 3          # kv_append, kv_quantize_pages, the decode kernel
        self.kernel_name = "pa_forward_kitty (persistent decode kernel over 2-bit page records + residual pages)"
        self.bound_note = ("bound by instruction issue, not HBM: 288 mixed-precision FMAs and 144 ANDs per "
                           "(key, head) at 16 warps per SM, 65% issue-active under ncu; frac is of HBM bytes")
        self.dtype_label = f"bf16 q/out, 2-bit K/V with {P} of 128 key channels at 4 bits, fp32 accumulate"
        self.pool_bytes = acct["pool_bytes"]

    def step(self, ev=None):
        inp = self.dev_in
        self.pkg.kv_append(inp["k_new"], inp["v_new"], inp["slots"], self.res_k, self.res_v)
        self.pkg.kv_quantize_pages(self.stage_k, self.stage_v, inp["qpair"], self.pages, self.b.promoted)
        if ev is not None:
            ev[0].record()
        self.pkg.pa_forward_kitty(inp["q"], self.pages, self.res_k, self.res_v, inp["bt"], inp["ctx"],
                                  inp["ql"], self.b.promoted, self.b.scale, out=self.out, workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def e2e_step(self):
        for k2, v in self.host.items():
            self.dev_in[k2].copy_(v, non_blocking=True)
        self.step()
        self.out_host.copy_(self.out, non_blocking=True)


class KVMoveStep:
    """KV movement over a multi-layer fp16 pool [L, 2, num_blocks, Hkv, B, d] resident on the GPU:
    block_copy of the copy-on-write pairs (every resident layer, K and V), kv_append of every
    session's new tokens into all layers, then the swap-in of host-staged sessions layer by layer
    (one block_copy per layer from a page-locked host pool)."""

    def __init__(self, plan: W.KVMovePlan, dev):
        import torch
        import paged_kv_cache_generalized_gb300 as pkg

        self.pkg, self.torch, self.plan, self.dev = pkg, torch, plan, dev
        L, nb, hkv, B, d = plan.num_layers, plan.num_blocks, plan.num_kv_heads, plan.block_size, plan.head_dim
        g = torch.Generator(device=dev)
        g.manual_seed(plan.seed)
        # values do not matter for timing (bit-exactness is tested on the same kernels elsewhere)
        self.pool = torch.empty((L, 2, nb, hkv, B, d), dtype=torch.float16, device=dev)
        self.pool.view(torch.int16).random_(generator=g)
        T = len(plan.slot_mapping)
        self.new = torch.empty((L, 2, T, hkv, d), dtype=torch.float16, device=dev)
        self.new.view(torch.int16).random_(generator=g)
        host_dev = torch.empty((L, 2, plan.num_host_blocks, hkv, B, d), dtype=torch.float16, device=dev)
        host_dev.view(torch.int16).random_(generator=g)
        self.host_pool = host_dev.cpu().pin_memory()
        del host_dev
        self.cow = torch.from_numpy(plan.cow_pairs).to(dev)
        self.swap = torch.from_numpy(plan.swap_pairs).to(dev)
        self.slots = torch.from_numpy(plan.slot_mapping).to(dev)
        self.cow_planes = self.pool.view(L * 2, nb, hkv, B, d)
        acct = kvmove_accounting(plan)
        self.bytes_cow, self.bytes_append, self.bytes_swap = acct["bytes_cow"], acct["bytes_append"], acct["bytes_swap"]
        self.flops = 0.0
        self.launches_per_step = 1 + 1 + L
        self.h2d_bytes = self.bytes_swap / 2 + self.new.numel() * 2 + 8 * T + plan.cow_pairs.nbytes + plan.swap_pairs.nbytes
        self.d2h_bytes = 0
        self.out = None

    def step(self, ev=None):
        pkg, L = self.pkg, self.plan.num_layers
        if ev is not None:
            ev[0].record()
        pkg.block_copy(self.cow_planes, self.cow_planes, self.cow)
        if ev is not None:
            ev[1].record()
        pkg.kv_append(self.new[:, 0], self.new[:, 1], self.slots, self.pool[:, 0], self.pool[:, 1])
        if ev is not None:
            ev[2].record()
        for layer in range(L):
            pkg.block_copy(self.host_pool[layer], self.pool[layer], self.swap)
        if ev is not None:
            ev[3].record()

    def e2e_step(self):
        # the step's host inputs: new tokens, slot map, pair lists (the swap source is already host)
        self.step()


class SwapPipelineStep:
    """Layer-by-layer swap-in overlapped with attention: L layers of the mixed GQA batch in a device
    pool [L, 2 (K,V), num_blocks, Hkv, B, d]; before layer l's attention, the earliest 1/8 of every
    resumed conversation's cached history (that layer's K and V of those blocks) comes back from a
    page-locked host pool [L, 2, Hn, Hkv, B, d]."""

    def __init__(self, batch: W.AttnBatch, dev, layers: int, frac: float = 0.125):
        import torch
        import paged_kv_cache_generalized_gb300 as pkg
        from paged_kv_cache_generalized_gb300 import swap as S

        self.pkg, self.S, self.torch, self.b, self.dev, self.L = pkg, S, torch, batch, dev, layers
        tdt = torch.bfloat16

        def up(x):
            return torch.from_numpy(np.ascontiguousarray(x)).view(torch.int16).view(tdt)

        self.pool = torch.empty((layers, 2) + batch.k_cache.shape, dtype=tdt, device=dev)
        kd, vd = up(batch.k_cache).to(dev), up(batch.v_cache).to(dev)
        for layer in range(layers):
            self.pool[layer, 0].copy_(kd)
            self.pool[layer, 1].copy_(vd)
        del kd, vd
        blocks = W.swap_plan(batch, frac)
        self.dev_blocks = torch.from_numpy(blocks).to(dev)
        self.hn = len(blocks)
        self.host = torch.empty((layers, 2, self.hn) + batch.k_cache.shape[1:], dtype=tdt).pin_memory()
        for layer in range(layers):
            self.host[layer].copy_(self.pool[layer][:, self.dev_blocks])
        self.host_out = torch.empty_like(self.host).pin_memory()
        self.hostin = {"q": up(batch.q).pin_memory(),
                       "bt": torch.from_numpy(batch.block_tables).pin_memory(),
                       "ctx": torch.from_numpy(batch.ctx_lens).pin_memory(),
                       "ql": torch.from_numpy(batch.q_lens).pin_memory()}
        self.din = {k: v.to(dev) for k, v in self.hostin.items()}
        self.out = torch.empty((layers,) + tuple(self.din["q"].shape), dtype=tdt, device=dev)
        self.out_host = torch.empty_like(self.out, device="cpu").pin_memory()
        self.ws = torch.empty(max(256, pkg.forward_workspace_size(self.din["q"], self.pool[0, 0],
                                                                 self.din["bt"], self.din["ctx"])),
                              dtype=torch.uint8, device=dev)
        self.block_bytes = int(np.prod(batch.k_cache.shape[1:])) * 2
        self.swap_bytes = float(layers * 2 * self.hn * self.block_bytes)   # host bytes per step
        self.flops = layers * attn_flops(batch.ctx_lens, batch.q_lens, batch.num_q_heads, batch.head_dim)
        self.copy_stream = torch.cuda.Stream(dev, priority=-1)
        self.out_stream = torch.cuda.Stream(dev, priority=0)

        # the schedules, built once (their tables and staging slots are reused every step)
        cur = torch.cuda.current_stream(dev)
        self.sw = {(m, ser): S.LayerSwapIn(self.host, self.pool, self.dev_blocks, mode=m,
                                           max_ctas=0 if ser else 32,
                                           copy_stream=cur if ser else self.copy_stream)
                   for m in ("staged", "gather") for ser in (False, True)}
        self.out_pairs = S.swap_out_pairs(self.dev_blocks)

    def attention(self, layer):
        d = self.din
        self.pkg.pa_forward(d["q"], self.pool[layer, 0], self.pool[layer, 1], d["bt"], d["ctx"], d["ql"],
                            self.b.scale, out=self.out[layer], workspace=self.ws)

    def attn_only(self):
        for layer in range(self.L):
            self.attention(layer)


    def run(self, mode, serial=False, attention=True):
        self.sw[(mode, serial)].run(self.attention if attention else None)

    def swap_out(self, stream=None, max_ctas=0):
        self.S.swap_out(self.pool, self.host_out, self.out_pairs, stream=stream, max_ctas=max_ctas)

    def e2e_step(self):
        for k, v in self.hostin.items():
            self.din[k].copy_(v, non_blocking=True)
        self.run("staged")
        self.out_host.copy_(self.out, non_blocking=True)


class LayoutStep:
    """The decode batch's attention on one layer of an L-layer pool kept in two layouts --
    layer-first [L, 2 (K,V), num_blocks, Hkv, B, d] and block-first [num_blocks, L, 2, Hkv, B, d]
    (every layer of a block contiguous, "KVキャッシュ管理の教科書" 第14章) -- and the swap-in of the
    blocks of some sessions from a page-locked host pool in either layout."""

    def __init__(self, batch: W.AttnBatch, dev, layers: int, swap_seqs: int = 8, memcpy_blocks: int = 64):
        import torch
        import paged_kv_cache_generalized_gb300 as pkg

        self.pkg, self.torch, self.b, self.dev, self.L = pkg, torch, batch, dev, layers
        tdt = torch.bfloat16
        blk = tuple(batch.k_cache.shape[1:])
        nb = batch.k_cache.shape[0]

        def up(x):
            return torch.from_numpy(np.ascontiguousarray(x)).view(torch.int16).view(tdt)

        self.mid = layers // 2
        self.lf = torch.empty((layers, 2, nb) + blk, dtype=tdt, device=dev)
        self.bf = torch.empty((nb, layers, 2) + blk, dtype=tdt, device=dev)
        kd, vd = up(batch.k_cache).to(dev), up(batch.v_cache).to(dev)
        self.lf[self.mid, 0].copy_(kd)
        self.lf[self.mid, 1].copy_(vd)
        self.bf[:, self.mid, 0].copy_(kd)
        self.bf[:, self.mid, 1].copy_(vd)
        del kd, vd
        self.din = {"q": up(batch.q).to(dev), "bt": torch.from_numpy(batch.block_tables).to(dev),
                    "ctx": torch.from_numpy(batch.ctx_lens).to(dev), "ql": torch.from_numpy(batch.q_lens).to(dev)}
        self.out = torch.empty_like(self.din["q"])
        self.ws = torch.empty(max(256, pkg.forward_workspace_size(self.din["q"], self.bf[:, 0, 0],
                                                                 self.din["bt"], self.din["ctx"])),
                              dtype=torch.uint8, device=dev)
        B = batch.block_size
        n = batch.seq_lens
        blocks = np.concatenate([batch.block_tables[i, :(int(n[i]) + B - 1) // B] for i in range(swap_seqs)])
        self.hn = len(blocks)
        self.dblocks = blocks.astype(np.int64)
        idx = np.arange(self.hn, dtype=np.int64)
        self.pairs = torch.from_numpy(np.stack([idx, self.dblocks], 1)).to(dev)
        self.host_lf = torch.zeros((layers, 2, self.hn) + blk, dtype=tdt).pin_memory()
        self.host_bf = torch.zeros((self.hn, layers, 2) + blk, dtype=tdt).pin_memory()
        self.plane_bytes = int(np.prod(blk)) * 2
        self.swap_bytes = float(self.hn * layers * 2 * self.plane_bytes)
        self.memcpy_blocks = min(memcpy_blocks, self.hn)
        es = 2
        self.bytes_attn = float(n.sum() * batch.num_kv_heads * batch.head_dim * es * 2 +
                                2 * batch.total_q * batch.num_q_heads * batch.head_dim * es +
                                ((n + B - 1) // B).sum() * 4 + batch.num_seqs * 8)

    def attention(self, layout):
        pool = self.lf[self.mid] if layout == "layer_first" else self.bf[:, self.mid].transpose(0, 1)
        d = self.din
        self.pkg.pa_forward(d["q"], pool[0], pool[1], d["bt"], d["ctx"], d["ql"], self.b.scale,
                            out=self.out, workspace=self.ws)

    def swap_gather(self, layout):
        if layout == "layer_first":      # one launch per layer; a block is Hkv*B*d per plane
            for layer in range(self.L):
                self.pkg.block_copy(self.host_lf[layer], self.lf[layer], self.pairs)
        else:                            # one launch; a block is every layer and plane at once
            self.pkg.block_copy(self.host_bf.unsqueeze(0), self.bf.unsqueeze(0), self.pairs)

    def swap_memcpy(self, layout):
        """One copy-engine transfer per contiguous segment (the first memcpy_blocks blocks):
        (block, layer, plane) segments layer-first, whole blocks block-first."""
        k = self.memcpy_blocks
        if layout == "layer_first":
            for j in range(k):
                t = int(self.dblocks[j])
                for layer in range(self.L):
                    for pl in range(2):
                        self.lf[layer, pl, t].copy_(self.host_lf[layer, pl, j], non_blocking=True)
        else:
            for j in range(k):
                self.bf[int(self.dblocks[j])].copy_(self.host_bf[j], non_blocking=True)


def h2d_peak_gbs(dev, nbytes=1 << 30, reps=5):
    """Page-locked host -> device copy bandwidth measured here (the swap-in roofline)."""
    import torch

    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9


def build_attn_step(name, dev, args):
    b = workload_batch(name, args)
    if name == "decode13b_kitty":
        return KittyStep(b, dev), b
    cow, seed = ATTN_COW[name]
    return AttnStep(b, dev, cow_frac=cow, seed=seed, kv8=name.endswith("fp8")), b


WORKLOAD_TEXT = {
    "decode13b": "decode13b: 64 seqs, 40 MHA heads, head_dim 128, bf16, block 16, q_len 1, "
                 "ctx U{512..4096}, pool +10% free, 6 copy-on-write forks per step",
    "decode13b_fp8": "decode13b_fp8: the decode13b batch with FP8 E4M3 K/V caches (scale 1/32 for K and V), "
                     "bf16 queries and outputs",
    "decode13b_kitty": "decode13b_kitty: the decode13b batch (64 seqs, 40 MHA heads, head_dim 128, ctx U{512..4096}) "
                       "over 2-bit K/V pages of 128 tokens with 32 of 128 key channels promoted to 4 bits "
                       "(Kitty), each sequence's last n % 128 tokens in a bf16 residual page; per step one "
                       "appended token per sequence and one page quantised",
    "mixed_gqa": "mixed_gqa: 32 resumed turns (ctx U{1024..16384}, q U{16..512}) + 32 decode "
                 "(ctx U{256..8192}), GQA 32/8, head_dim 128, bf16, block 32",
    "mixed_gqa_fp8": "mixed_gqa_fp8: the mixed_gqa batch with FP8 E4M3 K/V caches (scale 1/32 for K and V), "
                     "bf16 queries and outputs",
    "longprefill": "longprefill: 8 seqs x (16384 cached + 2048 new), 40 MHA heads, head_dim 128, "
                   "bf16, block 16, ConvKV turn segments 64..1024 tokens",
    "layout": "layout: the decode13b batch on one layer of an 8-layer pool, block-first [blocks, layers, K|V, heads, "
              "block, dim] against layer-first [layers, K|V, blocks, heads, block, dim]; swap-in of 8 sessions' "
              "blocks in either layout (gather kernel, and one copy-engine transfer per contiguous segment)",
    "swap_pipeline": "swap_pipeline: the mixed_gqa batch as 8 layers (GQA 32/8, head_dim 128, bf16, block 32); "
                     "before each layer's attention the earliest 1/8 of every resumed conversation's history "
                     "(that layer's K and V) is swapped in from pinned host memory, layer by layer, overlapped "
                     "with the previous layer's attention",
    "kvmove": "kvmove: 40-layer x 5120-hidden fp16 pool (0.78 MB/token), 8 layers resident, block 32, "
              "64 sessions U{512..8192} tokens, append U{1..256} tokens each, copy-on-write of 10% of "
              "blocks shared by U{2..4} sequences, swap-in of 8 sessions from pinned host memory, "
              "layer by layer",
}



def workload_text(name, args):
    """The workload's description; a run with --seqs / --layers says it is a reduced case."""
    t = WORKLOAD_TEXT[name]
    extra = []
    if getattr(args, "seqs", None):
        extra.append(f"--seqs {args.seqs}")
    if name == "kvmove" and getattr(args, "layers", None):
        extra.append(f"--layers {args.layers}")
    if extra:
        t += "; REDUCED case (" + ", ".join(extra) + "), not the headline workload"
    return t

# ------------------------------------------------------------------------------------------------
# Distributed helpers (independent replicas; timing barrier and max over ranks only)
# ------------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, use_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist

    dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def max_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ------------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ------------------------------------------------------------------------------------------------
def oracle_sample(b: W.AttnBatch, budget_s: float, max_rows=None):
    """Times the float64 oracle on rows of the workload (whole sequences, all heads, in order)
    until about ``budget_s`` seconds of work; returns (seconds, kv_bytes, flops, rows, threads)."""
    import oracle

    threads = oracle.max_threads()
    es = 4 if b.dtype == "f32" else 2
    order = np.argsort(-b.seq_lens, kind="stable")  # the longest first, then the rest
    rows, kv_bytes, flops = [], 0.0, 0.0
    t_total = 0.0
    done_rows = 0
    while t_total < budget_s:                        # whole passes over the batch if it is quick
        for i in order:
            seq_rows = [(i, j, h) for j in range(int(b.q_lens[i])) for h in range(b.num_q_heads)]
            if max_rows is not None and done_rows + len(seq_rows) > max_rows and done_rows:
                return t_total, kv_bytes, flops, rows, threads
            t0 = time.perf_counter()
            oracle.paged_attention_batch(b, rows=np.array(seq_rows, np.int64), threads=threads)
            t_total += time.perf_counter() - t0
            done_rows += len(seq_rows)
            c, q = int(b.ctx_lens[i]), int(b.q_lens[i])
            kv_bytes += (c + q) * b.num_kv_heads * b.head_dim * es * 2
            flops += attn_flops(np.array([c]), np.array([q]), b.num_q_heads, b.head_dim)
            rows.append(i)
            if t_total >= budget_s:
                break
    return t_total, kv_bytes, flops, rows, threads


def oracle_token_sample(b: W.AttnBatch, budget_s: float, tokens_per_call: int = 8):
    """Times the float64 oracle on query tokens (all heads each) drawn uniformly over the batch's
    new tokens, ``tokens_per_call`` per call, for about ``budget_s`` seconds: for batches whose
    single sequences take longer than the budget.  Returns (seconds, kv_bytes, flops, tokens,
    threads); FLOPs count 4 * d * Hq per visible key of each token, as in the GPU metric."""
    import oracle

    threads = oracle.max_threads()
    es = 4 if b.dtype == "f32" else 2
    rng = np.random.default_rng(0)
    cu = np.concatenate([[0], np.cumsum(b.q_lens)])
    T = int(cu[-1])
    t_total, kv_bytes, flops, toks = 0.0, 0.0, 0.0, []
    while t_total < budget_s:
        pick = rng.integers(0, T, tokens_per_call)
        seqs = np.searchsorted(cu, pick, side="right") - 1
        rows = np.array([(i, p - cu[i], h) for i, p in zip(seqs, pick) for h in range(b.num_q_heads)],
                        dtype=np.int64)
        t0 = time.perf_counter()
        oracle.paged_attention_batch(b, rows=rows, threads=threads)
        t_total += time.perf_counter() - t0
        for i, p in zip(seqs, pick):
            keys = int(b.ctx_lens[i]) + int(p - cu[i]) + 1
            kv_bytes += keys * b.num_kv_heads * b.head_dim * es * 2
            flops += 4.0 * b.head_dim * b.num_q_heads * keys
            toks.append(int(p))
    return t_total, kv_bytes, flops, toks, threads


def kitty_oracle_sample(b: W.KittyBatch, budget_s: float):
    """Times the oracle's decode attention over 2-bit pages (it dequantises every page of the
    sequence, then runs the float64 attention) on whole sequences of the batch, longest first,
    for about ``budget_s`` seconds; the oracle's own page records are made before the clock starts.
    Returns (seconds, bytes, flops, rows, threads)."""
    import oracle
    from oracle import kitty

    threads = oracle.max_threads()
    R = kitty.record_bytes(b.promoted)
    order = np.argsort(-b.ctx_lens, kind="stable")
    cache = {}
    t_total, nbytes, flops, rows = 0.0, 0.0, 0.0, []
    while t_total < budget_s:
        for i in order:
            i = int(i)
            n = int(b.ctx_lens[i]) + 1
            if i not in cache:
                recs = np.zeros((max(1, n // 128), b.num_kv_heads, R), np.uint8)
                bt = np.full((1, b.block_tables.shape[1]), -1, np.int32)
                for p_, sid in enumerate(b.page_of[i]):
                    for h in range(b.num_kv_heads):
                        f = kitty.quantize_page(oracle.widen_f32(b.stage_k[sid, h], b.dtype),
                                                oracle.widen_f32(b.stage_v[sid, h], b.dtype), b.promoted)
                        recs[p_, h] = kitty.pack_record(f)
                    bt[0, p_] = p_
                if n % 128:
                    bt[0, n // 128] = b.block_tables[i, n // 128]
                cache[i] = (recs, bt)
            recs, bt = cache[i]
            t0 = time.perf_counter()
            kitty.paged_attention(b.q[i:i + 1], recs, b.res_k, b.res_v, b.dtype, bt, b.ctx_lens[i:i + 1],
                                  b.q_lens[i:i + 1], b.num_q_heads, b.num_kv_heads, b.promoted, b.scale,
                                  threads=threads)
            t_total += time.perf_counter() - t0
            nbytes += (n // 128) * b.num_kv_heads * R + (n % 128) * b.num_kv_heads * b.head_dim * 4
            flops += attn_flops(b.ctx_lens[i:i + 1], b.q_lens[i:i + 1], b.num_q_heads, b.head_dim)
            rows.append(i)
            if t_total >= budget_s:
                break
    return t_total, nbytes, flops, rows, threads


def metric_for(name):
    if name == "kvmove":
        return ("KV movement GB/s (bytes read + written by copy-on-write, append and swap-in per step / step time)", "GB/s", True)
    if name == "decode13b":
        return ("paged-attn decode KV GB/s (algorithmic HBM bytes per step / step time)", "GB/s", True)
    if name == "decode13b_fp8":
        return ("paged-attn decode KV GB/s with FP8 E4M3 K/V caches (algorithmic HBM bytes per step / step "
                "time)", "GB/s", True)
    if name == "decode13b_kitty":
        return ("paged-attn decode KV GB/s over 2-bit pages with promoted 4-bit key channels (algorithmic "
                "HBM bytes per step / step time)", "GB/s", True)
    if name == "mixed_gqa_fp8":
        return ("paged-attn mixed-prefill TFLOP/s with FP8 E4M3 K/V caches (causal-exact attention FLOPs / "
                "step time)", "TFLOP/s", True)
    if name == "layout":
        return ("paged-attn decode KV GB/s on a block-first pool (one layer of L; all layers of a block "
                "contiguous)", "GB/s", True)
    if name == "swap_pipeline":
        return ("layer-pipelined swap-in + attention TFLOP/s (causal-exact attention FLOPs of all layers / "
                "step time, each layer's swap-in from host memory inside the step)", "TFLOP/s", True)
    return ("paged-attn mixed-prefill TFLOP/s (causal-exact attention FLOPs / step time)", "TFLOP/s", True)


def reference_attn(name, args, world, batch, per_step):
    """The oracle timed on the workload: ``args.warmup`` untimed and ``args.steps`` timed steps, each
    a bounded sample of about ``per_step`` seconds.  Returns (value, ms_per_step, sample text,
    threads)."""
    metric, unit, hib = metric_for(name)
    total = args.steps + args.warmup
    secs, kvb, fl, threads, desc = 0.0, 0.0, 0.0, 1, ""
    for s_ in range(total):
        if name == "longprefill":
            t, kb, f, rows, threads = oracle_token_sample(batch, per_step)
            desc = (f"float64 oracle rows of {len(rows)} query token(s) (all heads) drawn across the "
                    f"{name} batch per step, ~{per_step:.2f}s each")
        else:
            t, kb, f, rows, threads = oracle_sample(batch, per_step)
            desc = (f"float64 oracle rows of {len(rows)} sequence(s) (all heads, all new tokens) "
                    f"of the {name} batch per step, ~{per_step:.2f}s each")
        if s_ >= args.warmup:
            secs += t
            kvb += kb
            fl += f
    value = (kvb / secs / 1e9) if unit == "GB/s" else (fl / secs / 1e12)
    return value, secs / max(1, args.steps) * 1e3, desc, threads


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    metric, unit, hib = metric_for(name)
    batch = workload_batch(name, args)
    config = workload_config(name, args, world, batch)
    total = args.steps + args.warmup
    per_step = max(0.05, min(2.0, 150.0 / max(total, 1)))
    base = {"impl": "reference", "metric": metric, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic", "config": config}
    if name == "kvmove":
        secs, moved = 0.0, 0.0
        for s_ in range(total):
            t, mv, reps = kvmove_oracle_sample(batch, per_step)
            if s_ >= args.warmup:
                secs += t
                moved += mv
        value = moved / secs / 1e9
        line = dict(base, value=value, ms_per_step=secs / max(1, args.steps) * 1e3, dtype="f16",
                    cpu_baseline={"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                                  "sample": "numpy block copy of 64 copy-on-write pairs and append of 256 tokens per repetition"})
    elif name == "decode13b_kitty":
        secs, moved, nrows, threads = 0.0, 0.0, 0, 1
        for s_ in range(total):
            t, nb, _, rows, threads = kitty_oracle_sample(batch, per_step)
            if s_ >= args.warmup:
                secs += t
                moved += nb
                nrows += len(rows)
        value = moved / secs / 1e9
        line = dict(base, value=value, ms_per_step=secs / max(1, args.steps) * 1e3, dtype="f64",
                    cpu_baseline={"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                                  "sample": f"oracle decode attention over 2-bit pages (dequantise + float64 attention) "
                                            f"on {nrows} whole sequence(s), ~{per_step:.2f}s per step"})
    else:
        value, ms, desc, threads = reference_attn(name, args, world, batch, per_step)
        line = dict(base, value=value, ms_per_step=ms, dtype="f64",
                    cpu_baseline={"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": desc})
    line["e2e"] = {"value": line["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    if name == "decode13b" and not args.seqs and not args.headline_only:
        # the same prefill objects as the native line, with the oracle's numbers
        for sub, key in PREFILL_OBJECTS:
            sb = workload_batch(sub, args)
            sm, su, _ = metric_for(sub)
            sv, sms, sdesc, sth = reference_attn(sub, args, world, sb, max(0.05, per_step / 4))
            line[key] = {"metric": sm, "value": sv, "unit": su, "ms_per_step": sms, "dtype": "f64",
                         "config": workload_config(sub, args, world, sb),
                         "cpu_baseline": {"value": sv, "unit": su, "cores": sth, "kind": "oracle", "sample": sdesc},
                         "e2e": {"value": sv, "unit": su, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------
# Native (CUDA) arm
# ------------------------------------------------------------------------------------------------
def measure_attn_workload(name, args, dev, dist, world, local, peaks, peak_src, cpu_seconds):
    """Times ``args.steps`` steps of an attention workload (block_copy + kv_append + attention)
    after ``args.warmup`` untimed ones, with CUDA events on the launching stream and clock samples
    during the timed region, then the same step end to end (host inputs in, output back); returns
    the fields of the workload's JSON object (rank 0 also times the oracle on a sample)."""
    import torch

    metric, unit, hib = metric_for(name)
    step_obj, batch = build_attn_step(name, dev, args)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        step_obj.step()
    torch.cuda.synchronize()
    flags = step_obj.pkg.device_status()
    if flags:
        raise RuntimeError(f"{name}: device status after warm-up: {step_obj.pkg.status_names(flags)}")

    K = args.steps
    kernel_events = isinstance(step_obj, AttnStep)
    nev = 6 if kernel_events else 2
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(nev)) for _ in range(K)]
    for e in evs:                   # create every CUDA event before the timed region
        for x in e:
            x.record()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record()
        for i in range(K):
            step_obj.step(evs[i])
        stop.record()
        torch.cuda.synchronize()
    barrier(dist)
    elapsed_ms = start.elapsed_time(stop)
    attn_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    # the library-recorded brackets of its tensor-core and decode kernels
    tc_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / K if kernel_events and step_obj.has_tc else None
    cc_ms = sum(e[4].elapsed_time(e[5]) for e in evs) / K if kernel_events else None
    elapsed_ms = max_over_ranks(dist, elapsed_ms, dev)
    ms_step = elapsed_ms / K

    step_bytes = step_obj.bytes_attn + step_obj.bytes_append + step_obj.bytes_copy
    work = step_bytes if unit == "GB/s" else step_obj.flops
    scale_u = 1e9 if unit == "GB/s" else 1e12
    value = work * world / (ms_step * 1e-3) / scale_u

    # end to end through the public API: H2D of the step's inputs, the step, D2H of the output
    Ke = min(K, max(20, K // 5))
    for _ in range(3):
        step_obj.e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(Ke):
        step_obj.e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / Ke
    e2e_val = work * world / (e2e_ms * 1e-3) / scale_u
    dec_alone_ms = step_obj.decode_alone_ms() if kernel_events and unit != "GB/s" else None
    flags = step_obj.pkg.device_status()

    res = {"metric": metric, "unit": unit, "higher_is_better": hib, "value": value, "ms_per_step": ms_step,
           "attn_ms": attn_ms, "device_status": flags, "clocks": clocks.summary(),
           "gpu_launches": step_obj.launches_per_step * K,
           "dtype": getattr(step_obj, "dtype_label",
                            "bf16 q/out, e4m3 K/V, fp32 accumulate" if step_obj.kv8 else batch.dtype),
           "config": workload_config(name, args, world, batch),
           "query_tokens_per_s": getattr(batch, "total_q", batch.num_seqs) * world / (attn_ms * 1e-3),
           "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": step_obj.h2d_bytes,
                   "d2h_bytes_per_step": step_obj.d2h_bytes, "ms_per_step": e2e_ms}}
    if unit == "GB/s":
        # the decode kernel alone when the library bracketed it, else the whole attention call
        kern_ms = cc_ms if cc_ms else attn_ms
        achieved = step_obj.bytes_attn / (kern_ms * 1e-3) / 1e9
        traffic, tsrc = measured_traffic(name, step_obj.bytes_attn)
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "traffic_source": tsrc,
                "algorithmic_bytes": step_obj.bytes_attn, "kernel_ms": kern_ms,
                "kernel": getattr(step_obj, "kernel_name",
                                  "the decode kernel of pa_forward_append (split-KV, fused split merge), "
                                  "between events the library records around its launch"),
                "call_ms": attn_ms, "call_achieved": step_obj.bytes_attn / (attn_ms * 1e-3) / 1e9,
                "peak_source": f"hbm_gbs of {peak_src}"}
        if getattr(step_obj, "bound_note", None):
            roof["note"] = step_obj.bound_note
    else:
        pk = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        tflops, kern_ms = (step_obj.flops_tc, tc_ms) if tc_ms else (step_obj.flops, attn_ms)
        achieved = tflops / (kern_ms * 1e-3) / 1e12
        # DRAM bytes of the tensor-core kernel's launch (its own capture where the call also runs
        # the decode kernel, else the call's)
        tbytes = step_obj.bytes_attn_tc if tc_ms else step_obj.bytes_attn
        traffic, tsrc = measured_traffic(name + "_tc", tbytes)
        if tsrc is None:
            traffic, tsrc = measured_traffic(name, tbytes)
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                "frac": achieved / pk, "traffic": traffic, "traffic_source": tsrc,
                "algorithmic_flops": tflops, "kernel_ms": kern_ms,
                "kernel": ("tc_attention_kernel (tcgen05) on the turns it runs, between events the library "
                           "records around its launch"
                           + (" (on their E4M3 blocks widened to bf16 by a kernel before it, which the "
                              "call's time includes)" if step_obj.kv8 else "")) if tc_ms else
                          "the whole attention call (CUDA-core kernels: no turn of this batch takes the "
                          "tcgen05 kernel)",
                "call_ms": attn_ms, "call_flops": step_obj.flops,
                "call_achieved": step_obj.flops / (attn_ms * 1e-3) / 1e12,
                "decode_bracket_ms": cc_ms, "algorithmic_bytes": tbytes,
                "peak_source": f"bf16_tflops (burst) of {peak_src}"}
        if cc_ms and tc_ms and step_obj.bytes_attn > tbytes:
            # the decode rows' KV bytes over the decode kernel's bracket, which also holds its wait
            # for the SMs the tensor-core kernel's tail frees (the two kernels share the call)
            dec_bytes = step_obj.bytes_attn - tbytes
            roof["decode_part"] = {"algorithmic_bytes": dec_bytes, "bracket_ms": cc_ms,
                                   "achieved_gbs": dec_bytes / (cc_ms * 1e-3) / 1e9,
                                   "note": "bracket includes waiting for SMs held by the tensor-core kernel"}
            if dec_alone_ms:
                # the same rows in a call of their own (planner + decode kernel), after the steps
                a_gbs = dec_bytes / (dec_alone_ms * 1e-3) / 1e9
                roof["decode_part"].update({"alone_ms": dec_alone_ms, "alone_achieved_gbs": a_gbs,
                                            "alone_frac_hbm": a_gbs / peaks["hbm_gbs"]})
    res["roofline"] = roof
    del step_obj
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    res["cpu_baseline"] = None
    if world == 1 or dist.get_rank() == 0:
        if isinstance(batch, W.KittyBatch):
            t, kvb, fl, rows, threads = kitty_oracle_sample(batch, cpu_seconds)
            what = "oracle decode attention over 2-bit pages (dequantise + float64 attention)"
            unit_rows = "whole sequence(s)"
        elif batch.total_q > 4 * batch.num_seqs and name == "longprefill":
            t, kvb, fl, rows, threads = oracle_token_sample(batch, cpu_seconds)
            what = "float64 oracle"
            unit_rows = "query tokens (all heads) drawn across the batch"
        else:
            t, kvb, fl, rows, threads = oracle_sample(batch, cpu_seconds)
            what = "float64 oracle"
            unit_rows = "whole sequence(s)"
        cval = kvb / t / 1e9 if unit == "GB/s" else fl / t / 1e12
        res["cpu_baseline"] = {"value": cval, "unit": unit, "cores": threads, "kind": "oracle",
                               "sample": f"{what} on {len(rows)} {unit_rows} of the batch, repeated "
                                         f"passes allowed (all heads, all new tokens), {t:.1f}s; attention only"}
    return res


# The prefill workloads measured beside the decode headline: the metric's second half
PREFILL_OBJECTS = (("mixed_gqa", "mixed_prefill"), ("longprefill", "long_prefill"))


def run_native(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    peaks, peak_src = load_peaks()
    name = args.workload
    r = measure_attn_workload(name, args, dev, dist, world, local, peaks, peak_src, args.cpu_seconds)
    line = {"metric": r["metric"], "value": r["value"], "unit": r["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": r["higher_is_better"],
            "scaling": "weak", "vs_baseline": None, "dtype": r["dtype"], "data": "synthetic",
            "config": r["config"], "roofline": r["roofline"], "cpu_baseline": r["cpu_baseline"],
            "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "attn_ms": r["attn_ms"],
            "query_tokens_per_s": r["query_tokens_per_s"], "device_status": r["device_status"],
            "clocks": r["clocks"]}
    if name == "decode13b" and not args.seqs and not args.headline_only:
        # the headline metric's other half, measured in the same process with the same steps and
        # warm-up: attention TFLOP/s of the mixed multi-turn batch and of the long prefill
        for sub, key in PREFILL_OBJECTS:
            s = measure_attn_workload(sub, args, dev, dist, world, local, peaks, peak_src,
                                      max(1.0, args.cpu_seconds / 2))
            line[key] = {k: s[k] for k in ("metric", "value", "unit", "ms_per_step", "attn_ms", "dtype",
                                            "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                                            "query_tokens_per_s", "device_status", "clocks")}
    if rank == 0:
        print(json.dumps(line), flush=True)


def kvmove_oracle_sample(plan: W.KVMovePlan, budget_s: float):
    """Times the oracle's block copy and append (numpy) on a bounded sample of the KV-movement
    step: one layer's K and V planes holding only the blocks the sampled pairs and slots touch."""
    import oracle

    rng = np.random.default_rng(0)
    hkv, B, d = plan.num_kv_heads, plan.block_size, plan.head_dim
    moved, secs, reps = 0.0, 0.0, 0
    while secs < budget_s:
        cow = plan.cow_pairs[rng.choice(len(plan.cow_pairs), min(64, len(plan.cow_pairs)), replace=False)]
        ids = np.unique(cow.ravel())
        remap = {int(b): i for i, b in enumerate(ids)}
        pool = W.random_bits16((2, len(ids), hkv, B, d), reps)
        pairs = np.array([[remap[int(a)], remap[int(b)]] for a, b in cow], dtype=np.int64)
        t0 = time.perf_counter()
        oracle.block_copy(pool, pool, pairs)
        secs += time.perf_counter() - t0
        moved += len(pairs) * 2 * plan.block_bytes * 2
        sl = plan.slot_mapping[:256]
        blocks = np.unique(sl // B)
        bmap = {int(b): i for i, b in enumerate(blocks)}
        small_slots = np.array([bmap[int(x) // B] * B + int(x) % B for x in sl], dtype=np.int64)
        kc = W.random_bits16((len(blocks), hkv, B, d), reps + 1)
        new = W.random_bits16((len(sl), hkv, d), reps + 2)
        t0 = time.perf_counter()
        oracle.kv_append(new, new, small_slots, kc, kc, B)
        secs += time.perf_counter() - t0
        moved += 2 * len(sl) * hkv * d * 2 * 2
        reps += 1
    return secs, moved, reps


def run_native_kvmove(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    peaks, peak_src = load_peaks()
    metric, unit, hib = metric_for("kvmove")
    plan = workload_batch("kvmove", args)
    step_obj = KVMoveStep(plan, dev)
    h2d = h2d_peak_gbs(dev)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step_obj.step()
    torch.cuda.synchronize()
    flags = step_obj.pkg.device_status()
    if flags:
        raise RuntimeError(f"device status after warm-up: {step_obj.pkg.status_names(flags)}")
    K = args.steps
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record()
        for i in range(K):
            step_obj.step(evs[i])
        stop.record()
        torch.cuda.synchronize()
    barrier(dist)
    ms_step = max_over_ranks(dist, start.elapsed_time(stop), dev) / K
    cow_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    app_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    swap_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    step_bytes = step_obj.bytes_cow + step_obj.bytes_append + step_obj.bytes_swap
    value = step_bytes * world / (ms_step * 1e-3) / 1e9
    flags = step_obj.pkg.device_status()
    if rank != 0:
        return
    cow_gbs = step_obj.bytes_cow / (cow_ms * 1e-3) / 1e9
    traffic, tsrc = measured_traffic("kvmove", step_obj.bytes_cow)
    roof = {"bound": "hbm", "achieved": cow_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": cow_gbs / peaks["hbm_gbs"], "traffic": traffic, "traffic_source": tsrc,
            "traffic_note": "below the algorithmic bytes: a block shared by r sequences is copied r-1 times "
                            "and read from DRAM once; lines still dirty in L2 when the kernel ends are not counted",
            "algorithmic_bytes": step_obj.bytes_cow,
            "kernel": "block_copy (copy-on-write, device pool, all resident layers, K and V)",
            "peak_source": f"hbm_gbs of {peak_src}"}
    swap_gbs = step_obj.bytes_swap / 2 / (swap_ms * 1e-3) / 1e9
    t, moved, reps = kvmove_oracle_sample(plan, args.cpu_seconds)
    cpu = {"value": moved / t / 1e9, "unit": unit, "cores": 1, "kind": "oracle",
           "sample": f"numpy block copy of 64 copy-on-write pairs (one layer, K and V) and append of "
                     f"256 tokens, {reps} repetitions, {t:.1f}s"}
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": hib,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": workload_config("kvmove", args, world, plan),
            "roofline": roof,
            "swap_in": {"achieved": swap_gbs, "unit": "GB/s (host bytes read)", "peak": h2d,
                        "frac": swap_gbs / h2d, "peak_source": "pinned host->device copy measured in this run",
                        "ms": swap_ms},
            "append": {"ms": app_ms, "achieved": step_obj.bytes_append / (app_ms * 1e-3) / 1e9},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": step_obj.bytes_swap / 2,
                    "d2h_bytes_per_step": 0, "note": "the swap-in reads its blocks from pinned host memory inside the step"},
            "gpu_launches": step_obj.launches_per_step * K, "device_status": flags,
            "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def run_native_swap(args):
    """Layer-pipelined swap-in + attention (see SwapPipelineStep)."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    peaks, peak_src = load_peaks()
    metric, unit, hib = metric_for("swap_pipeline")
    batch = workload_batch("swap_pipeline", args)
    st = SwapPipelineStep(batch, dev, args.layers)
    h2d = h2d_peak_gbs(dev)
    K, Wm = args.steps, args.warmup

    def timed(fn, reps=K):
        for _ in range(Wm):
            fn()
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(dist, e0.elapsed_time(e1), dev) / reps

    modes = {
        "attn_only": st.attn_only,
        "swap_only_staged": lambda: st.run("staged", attention=False),
        "swap_only_gather": lambda: st.run("gather", serial=True, attention=False),
        "serial_staged": lambda: st.run("staged", serial=True),
        "pipelined_gather": lambda: st.run("gather"),
    }
    ms = {k: timed(f) for k, f in modes.items()}
    flags = st.pkg.device_status()
    if flags:
        raise RuntimeError(f"device status: {st.pkg.status_names(flags)}")
    # the headline schedule, with clock samples
    for _ in range(Wm):
        st.run("staged")
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(K):
            st.run("staged")
        e1.record()
        torch.cuda.synchronize()
    ms["pipelined_staged"] = max_over_ranks(dist, e0.elapsed_time(e1), dev) / K
    # swap-out (eviction) alone, and beside a swap-in (the swap-in on the higher-priority stream)
    ms["swap_out"] = timed(lambda: st.swap_out())

    def both():
        cur = torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(cur)
        st.copy_stream.wait_event(ev)
        st.out_stream.wait_event(ev)
        with torch.cuda.stream(st.out_stream):
            st.swap_out(stream=st.out_stream, max_ctas=152)
        st.sw[("gather", False)].run(None)
        done = torch.cuda.Event()
        done.record(st.out_stream)
        cur.wait_event(done)

    ms["swap_in_and_out"] = timed(both)
    e2e_ms = timed(st.e2e_step, max(5, K // 4))
    flags = st.pkg.device_status()
    if rank != 0:
        return
    Lr = st.L
    value = st.flops * world / (ms["pipelined_staged"] * 1e-3) / 1e12
    ideal = max(ms["attn_only"], st.swap_bytes / (h2d * 1e9) * 1e3)
    roof = {"bound": "tensor", "achieved": value / world, "peak": peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "unit": "TFLOP/s", "frac": value / world / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "traffic": None, "algorithmic_flops": st.flops,
            "kernel": f"{Lr} layers of pa_forward with each layer's staged swap-in (copy engine + block_copy scatter) inside the step",
            "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    swap_gb = st.swap_bytes / 1e9
    pipe = {"layers": Lr, "swapped_blocks_per_layer": st.hn, "swap_bytes_per_step": st.swap_bytes,
            "ms": {k: round(v, 4) for k, v in ms.items()},
            "swap_gbs": {"staged": swap_gb / (ms["swap_only_staged"] * 1e-3),
                         "gather": swap_gb / (ms["swap_only_gather"] * 1e-3)},
            "swap_out_gbs": swap_gb / (ms["swap_out"] * 1e-3),
            "swap_in_and_out_gbs": 2 * swap_gb / (ms["swap_in_and_out"] * 1e-3),
            "h2d_peak_gbs": h2d, "h2d_peak_source": "pinned host->device copy measured in this run",
            "ideal_ms": ideal, "frac_of_ideal": ideal / ms["pipelined_staged"],
            "hidden_fraction": (ms["serial_staged"] - ms["pipelined_staged"]) /
                               max(1e-9, min(ms["attn_only"], ms["swap_only_staged"]))}
    t, kvb, fl, rows, threads = oracle_sample(batch, args.cpu_seconds)
    cpu = {"value": fl / t / 1e12, "unit": unit, "cores": threads, "kind": "oracle",
           "sample": f"float64 oracle on {len(rows)} whole sequence(s) of one layer of the batch, "
                     f"{t:.1f}s; attention only (the oracle has no transfer to overlap)"}
    h2d_bytes = st.swap_bytes + sum(v.numel() * v.element_size() for v in st.hostin.values())
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms["pipelined_staged"], "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config("swap_pipeline", args, world, batch),
            "pool_gb": st.pool.numel() * 2 / 1e9,
            "roofline": roof, "pipeline": pipe, "cpu_baseline": cpu,
            "e2e": {"value": st.flops * world / (e2e_ms * 1e-3) / 1e12, "unit": unit,
                    "h2d_bytes_per_step": h2d_bytes,
                    "d2h_bytes_per_step": st.out.numel() * st.out.element_size(), "ms_per_step": e2e_ms},
            "gpu_launches": Lr * 4 * K, "device_status": flags, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def run_native_layout(args):
    """Block-first against layer-first pools (see LayoutStep)."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    peaks, peak_src = load_peaks()
    metric, unit, hib = metric_for("layout")
    batch = workload_batch("layout", args)
    st = LayoutStep(batch, dev, args.layers)
    h2d = h2d_peak_gbs(dev)
    K, Wm = args.steps, args.warmup

    def timed(fn, reps):
        for _ in range(Wm):
            fn()
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(dist, e0.elapsed_time(e1), dev) / reps

    ms = {"attn_layer_first": timed(lambda: st.attention("layer_first"), K)}
    for _ in range(Wm):
        st.attention("block_first")
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(K):
            st.attention("block_first")
        e1.record()
        torch.cuda.synchronize()
    ms["attn_block_first"] = max_over_ranks(dist, e0.elapsed_time(e1), dev) / K
    swap_reps = max(3, K // 100)
    for lay in ("layer_first", "block_first"):
        ms[f"swap_gather_{lay}"] = timed(lambda: st.swap_gather(lay), swap_reps)
        ms[f"swap_memcpy_{lay}"] = timed(lambda: st.swap_memcpy(lay), swap_reps)
    flags = st.pkg.device_status()
    e2e_ms = ms["attn_block_first"]
    if rank != 0:
        return
    gbs = {k: st.bytes_attn / (v * 1e-3) / 1e9 for k, v in ms.items() if k.startswith("attn")}
    value = gbs["attn_block_first"] * world
    roof = {"bound": "hbm", "achieved": gbs["attn_block_first"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs["attn_block_first"] / peaks["hbm_gbs"], "traffic": None,
            "algorithmic_bytes": st.bytes_attn,
            "kernel": f"pa_forward on one layer of a block-first {st.L}-layer pool (block stride "
                      f"{st.L * 2 * st.plane_bytes // 1024} KiB)", "peak_source": f"hbm_gbs of {peak_src}"}
    mb = st.memcpy_blocks
    seg = {"layer_first": st.plane_bytes, "block_first": st.L * 2 * st.plane_bytes}
    swap = {"blocks": st.hn, "bytes": st.swap_bytes, "h2d_peak_gbs": h2d,
            "gather_kernel_gbs": {lay: st.swap_bytes / (ms[f"swap_gather_{lay}"] * 1e-3) / 1e9
                                  for lay in ("layer_first", "block_first")},
            "memcpy_per_segment": {lay: {"segment_bytes": seg[lay],
                                         "copies": mb * (st.L * 2 if lay == "layer_first" else 1),
                                         "gbs": mb * st.L * 2 * st.plane_bytes / (ms[f"swap_memcpy_{lay}"] * 1e-3) / 1e9}
                                   for lay in ("layer_first", "block_first")},
            "note": f"memcpy rows move the first {mb} blocks, one cudaMemcpyAsync per contiguous segment"}
    t, kvb, fl, rows, threads = oracle_sample(batch, args.cpu_seconds)
    cpu = {"value": kvb / t / 1e9, "unit": unit, "cores": threads, "kind": "oracle",
           "sample": f"float64 oracle on {len(rows)} whole sequence(s) of the decode batch, {t:.1f}s"}
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms["attn_block_first"], "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config("layout", args, world, batch),
            "pool_gb": st.lf.numel() * 2 / 1e9,
            "roofline": roof,
            "layouts": {"attn_gbs": gbs, "block_first_over_layer_first": gbs["attn_block_first"] / gbs["attn_layer_first"],
                        "ms": {k: round(v, 4) for k, v in ms.items()}, "swap_in": swap},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                    "note": "device-resident pools; the swap-in rows above are the host transfers"},
            "gpu_launches": 2 * K, "device_status": flags, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode13b", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=8,
                    help="kvmove / swap_pipeline: layers resident on the GPU")
    ap.add_argument("--headline-only", action="store_true",
                    help="decode13b: leave out the mixed-prefill and long-prefill objects of the line")
    ap.add_argument("--seqs", type=int, default=None,
                    help="number of sequences or sessions (defaults 64 / 64 / 8 / 64; smaller for profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "kvmove":
        run_native_kvmove(args)
    elif args.workload == "swap_pipeline":
        run_native_swap(args)
    elif args.workload == "layout":
        run_native_layout(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
