#!/usr/bin/env python
"""Benchmark of the DFlash drafting step on GB300: one JSON line on stdout.

A step is one drafting cycle at a fixed context: the tapped hidden states of
the R = gamma + 1 newest verified positions are fused (dflash_ctx_fuse) and
injected into every layer's KV cache (dflash_kv_inject), the drafter drafts
one block over the N-row context (dflash_draft_block) and the block is
verified against synthetic target logits (dflash_verify_accept). The context
length is restored before every step, so every step sees exactly N rows.

Metric: drafted tokens/s (B * gamma per step) and the step time; value is the
device-timed throughput with inputs resident in HBM, e2e the same through
host buffers (pinned H2D of the step's inputs, D2H of its outputs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

DEFAULT_WORKLOAD = "qwen3_8b_L5_N2048_B1"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of graph replay")
    p.add_argument("--cpu-steps", type=int, default=2, help="oracle steps timed for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-next-rows", action="store_true",
                   help="skip the timing of the drafting variants (sampling, per-sequence gamma, unmasking)")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the other workloads, the prefill and the draft-verify loop")
    p.add_argument("--mode", choices=["step", "prefill", "loop"], default="step",
                   help="step: the drafting cycle (default, full JSON line); prefill: context fusion + "
                        "injection of a long prefill only; loop: the draft-verify loop workload only")
    p.add_argument("--prefill-rows", type=int, default=0,
                   help="--mode prefill: tokens of the prefill (default: the workload's context)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time, on every rank (replicas finish when the last does)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job drafted tokens/s: every rank drafts its own replica's batch."""
    return world * tokens_per_step * steps / (ms * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


class DraftCycle:
    """Device state of one drafting cycle for a workload (one replica)."""

    def __init__(self, dfl, wl: synth.Workload, device: str):
        self.dfl, self.wl, self.dev = dfl, wl, device
        R, B = wl.rows, wl.batch
        # capacity in whole 128-key pages, so that the paged variant covers the same positions
        self.cfg = dfl.config_from_workload(wl, ctx_capacity=(wl.capacity() + 127) // 128 * 128)
        self.W = synth.weights(wl, device)
        self.w = dfl.Weights(self.cfg, self.W, device)
        prefix = synth.ctx_lengths(wl) - R          # context before the step's injection
        if (prefix < 0).any():
            raise ValueError("context shorter than one block")
        self.prefix = prefix
        self.ws = dfl.Workspace(self.cfg, max(int(prefix.max()) * B, B * R, 16), device)
        dt = synth.torch_dtype(wl.dtype)
        shape = (wl.n_layers, self.cfg.max_batch, wl.n_kv_heads, self.cfg.ctx_capacity, wl.head_dim)
        self.k_cache = torch.zeros(shape, dtype=dt, device=device)
        self.v_cache = torch.zeros(shape, dtype=dt, device=device)
        self.ctx_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # prefill of the prefix context (set-up, not timed)
        tmax = int(prefix.max())
        taps = synth.taps(wl, B * tmax, "prefill", device).view(B, tmax, -1)
        h = torch.empty((B, tmax, wl.d_model), dtype=dt, device=device)
        for b in range(B):
            dfl.dflash_ctx_fuse(self.cfg, self.w, taps[b, : int(prefix[b])], h[b], self.ws)
        del taps
        dfl.dflash_kv_inject(self.cfg, self.w, h, torch.as_tensor(prefix, device=device),
                             self.ctx_len, self.k_cache, self.v_cache, self.status, self.ws)
        del h
        self.ctx0 = self.ctx_len.clone()
        # per-step inputs (anchors, then the tapped states 256 bytes in) and
        # outputs (drafts, acceptance lengths, committed tokens), each packed
        # in one device buffer, so that an end-to-end step moves each
        # direction with one copy
        taps = synth.taps(wl, B * R, "step", device)
        a_bytes = (4 * B + 255) // 256 * 256
        self.io_in = torch.zeros(a_bytes + taps.numel() * taps.element_size(), dtype=torch.uint8, device=device)
        self.anchor = self.io_in[: 4 * B].view(torch.int32)
        self.anchor.copy_(torch.as_tensor(synth.anchors(wl), device=device))
        self.step_taps = self.io_in[a_bytes:].view(taps.dtype).view(taps.shape)
        self.step_taps.copy_(taps)
        del taps
        self.h_new = torch.empty((B, R, wl.d_model), dtype=dt, device=device)
        self.n_new = torch.full((B,), R, dtype=torch.int32, device=device)
        self.target = synth.target_logits(wl, "step", device, torch.float32)
        self.io_out = torch.zeros(B * wl.gamma + B + B * R, dtype=torch.int32, device=device)
        self.draft = self.io_out[: B * wl.gamma].view(B, wl.gamma)
        self.tau = self.io_out[B * wl.gamma: B * wl.gamma + B]
        self.committed = self.io_out[B * wl.gamma + B:].view(B, R)
        self.next_anchor = torch.empty(B, dtype=torch.int32, device=device)
        self.max_ctx = int(synth.ctx_lengths(wl).max())
        # The library's trace counts an attention launch's K/V bytes (and
        # flops) as if every sequence had the longest context: it knows only
        # the host hint max_ctx, not the per-sequence lengths on the device.
        # Each sequence reads its own ctx_b + R keys, so for a ragged batch
        # the records are rescaled to sum_b (ctx_b + R) keys; the query and
        # output bytes, 2 B R Hq Dh elements, are not part of the rescaling.
        self.attn_key_ratio = attention_key_ratio(synth.ctx_lengths(wl), R, self.max_ctx)
        self.attn_qo_bytes = 2.0 * B * R * wl.n_q_heads * wl.head_dim * (2 if wl.dtype == "bf16" else 4)
        torch.cuda.synchronize()

    def algorithmic(self, kind: int, b: float, fl: float):
        """(bytes, flops) of one traced launch, attention counted per sequence."""
        if kind != self.dfl.K_ATTN or b <= 0.0:
            return b, fl
        return (b - self.attn_qo_bytes) * self.attn_key_ratio + self.attn_qo_bytes, fl * self.attn_key_ratio

    def step_inject(self, trace=None):
        """Fusion and injection of the step's new rows."""
        d, wl = self.dfl, self.wl
        self.ctx_len.copy_(self.ctx0)
        d.dflash_ctx_fuse(self.cfg, self.w, self.step_taps, self.h_new.view(-1, wl.d_model), self.ws,
                          trace=trace)
        d.dflash_kv_inject(self.cfg, self.w, self.h_new, self.n_new, self.ctx_len, self.k_cache,
                           self.v_cache, self.status, self.ws, trace=trace)

    def step_draft(self, trace=None):
        """Fusion and injection of the step's new rows, then the drafting pass."""
        d = self.dfl
        self.step_inject(trace)
        d.dflash_draft_block(self.cfg, self.w, self.anchor, self.ctx_len, self.max_ctx, self.k_cache,
                             self.v_cache, self.draft, self.status, self.ws, trace=trace)

    def step_verify(self, trace=None):
        self.dfl.dflash_verify_accept(self.cfg, self.target, self.draft, self.tau, self.committed,
                                      self.next_anchor, self.ws, trace=trace)

    def step(self, trace=None):
        self.step_draft(trace)
        self.step_verify(trace)

    # the cycle with the drafting variants built beyond the greedy one-pass draft
    def _variant_buffers(self):
        if not hasattr(self, "v_logits"):
            B, wl = self.wl.batch, self.wl
            self.v_logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device=self.dev)
            self.v_ids = torch.empty((B, wl.rows), dtype=torch.int32, device=self.dev)
            self.v_gamma = torch.full((B,), wl.gamma // 2, dtype=torch.int32, device=self.dev)

    def step_sample(self, trace=None, temperature=1.0, seed=12345):
        """Sampled drafts (temperature T) and rejection-acceptance verification."""
        d = self.dfl
        self._variant_buffers()
        self.step_inject(trace)
        d.dflash_draft_block_sample(self.cfg, self.w, self.anchor, self.ctx_len, self.max_ctx, self.k_cache,
                                    self.v_cache, temperature, seed, self.draft, self.v_logits, self.status,
                                    self.ws, trace=trace)
        d.dflash_verify_sample(self.cfg, self.target, self.v_logits, self.draft, temperature, seed, self.tau,
                               self.committed, self.next_anchor, self.ws, trace=trace)

    def step_dyn(self, trace=None):
        """Per-sequence block size gamma/2 (drafting and verification)."""
        d = self.dfl
        self._variant_buffers()
        self.step_inject(trace)
        d.dflash_draft_block_dyn(self.cfg, self.w, self.anchor, self.ctx_len, self.v_gamma, self.max_ctx,
                                 self.k_cache, self.v_cache, self.draft, self.status, self.ws, trace=trace)
        d.dflash_verify_accept_dyn(self.cfg, self.target, self.draft, self.v_gamma, self.tau, self.committed,
                                   self.next_anchor, self.ws, trace=trace)

    def _paged_state(self):
        """Page pools holding the same prefix as the contiguous cache, pages
        placed in a scrambled order (built once, outside any timing)."""
        if hasattr(self, "pages"):
            return
        d, wl, dev = self.dfl, self.wl, self.dev
        B, page = wl.batch, d.PAGE_KEYS
        pps = self.cfg.ctx_capacity // page
        n_pages = B * pps + 3
        table = np.random.default_rng(5).permutation(n_pages)[: B * pps].reshape(B, pps).astype(np.int32)
        shape = (wl.n_layers, n_pages, wl.n_kv_heads, page, wl.head_dim)
        dt = synth.torch_dtype(wl.dtype)
        self.k_pool = torch.zeros(shape, dtype=dt, device=dev)
        self.v_pool = torch.zeros(shape, dtype=dt, device=dev)
        self.pages = d.KvPages(self.k_pool, self.v_pool, torch.as_tensor(table, device=dev))
        tmax = int(self.prefix.max())
        taps = synth.taps(wl, B * tmax, "prefill", dev).view(B, tmax, -1)
        h = torch.empty((B, tmax, wl.d_model), dtype=dt, device=dev)
        for b in range(B):
            d.dflash_ctx_fuse(self.cfg, self.w, taps[b, : int(self.prefix[b])], h[b], self.ws)
        self.ctx_len_p = torch.zeros(B, dtype=torch.int32, device=dev)
        d.dflash_kv_inject_paged(self.cfg, self.w, h, torch.as_tensor(self.prefix, device=dev), self.ctx_len_p,
                                 self.pages, self.status, self.ws)
        self.ctx0_p = self.ctx_len_p.clone()
        torch.cuda.synchronize()

    def step_paged(self, trace=None):
        """The greedy cycle over a paged KV cache."""
        d, wl = self.dfl, self.wl
        self._paged_state()
        self.ctx_len_p.copy_(self.ctx0_p)
        d.dflash_ctx_fuse(self.cfg, self.w, self.step_taps, self.h_new.view(-1, wl.d_model), self.ws,
                          trace=trace)
        d.dflash_kv_inject_paged(self.cfg, self.w, self.h_new, self.n_new, self.ctx_len_p, self.pages,
                                 self.status, self.ws, trace=trace)
        d.dflash_draft_block_paged(self.cfg, self.w, self.anchor, self.ctx_len_p, self.max_ctx, self.pages,
                                   self.draft, self.status, self.ws, trace=trace)
        self.step_verify(trace)

    def step_unmask(self, trace=None, n_steps=4):
        """Multi-step confidence unmasking (n_steps passes), greedy verification."""
        d = self.dfl
        self._variant_buffers()
        self.step_inject(trace)
        d.dflash_draft_block_iter(self.cfg, self.w, self.anchor, self.ctx_len, self.max_ctx, self.k_cache,
                                  self.v_cache, n_steps, self.v_ids, self.draft, self.v_logits, self.status,
                                  self.ws, trace=trace)
        self.step_verify(trace)

    def launches_per_step(self) -> int:
        rec = self.dfl.TraceRecorder(256)
        self.step(trace=rec.struct)
        torch.cuda.synchronize()
        return rec.struct.count


def attention_key_ratio(ctx_lengths, rows: int, max_ctx_hint: int) -> float:
    """Keys the attention launches read, sum_b (ctx_b + rows), over the keys
    the library's trace counts, B (max_ctx_hint + rows)."""
    keys = np.asarray(ctx_lengths, dtype=np.float64) + rows
    return float(keys.sum() / (keys.size * (max_ctx_hint + rows)))


def time_steps(fn, steps: int, stream) -> float:
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def measure_variant(cyc: DraftCycle, fn, steps: int, tokens: int, peak_gbs: float) -> dict:
    """One drafting-variant cycle (fusion + injection + its drafting and
    verification) replayed as a graph: us per step, drafted tokens/s, and its
    algorithmic bytes (from one traced run) against the measured HBM peak."""
    fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(3):
        g.replay()
    ms = time_steps(g.replay, steps, torch.cuda.current_stream())
    rec = cyc.dfl.TraceRecorder(4096)
    rec.reset()
    fn(trace=rec.struct)
    torch.cuda.synchronize()
    b = sum(cyc.algorithmic(r[0], r[1], r[2])[0] for r in rec.records())
    us = 1000.0 * ms / steps
    gbs = b / (us * 1e-6) / 1e9
    return {"us_per_step": round(us, 2), "drafted_tok_s": round(tokens / (us * 1e-6), 1),
            "algorithmic_gb_per_step": round(b / 1e9, 3), "achieved_gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peak_gbs, 4), "steps": steps}


def kernel_roofline(cyc: DraftCycle, peak_gbs: float, step_ms: float, reps: int = 5):
    """Per-kind algorithmic bytes / time over traced steps.

    A traced step launches its kernels one at a time between CUDA events, so
    each kind's event time is its serialised time; inside the graph-replayed
    step, programmatic dependent launch overlaps each kernel's start with its
    predecessor's tail and the sum is shorter. Each kind's time within the
    step is its share of the serialised sum times the measured step time
    (step_ms), so that the kinds add up to the step; both are reported."""
    dfl = cyc.dfl
    rec = dfl.TraceRecorder(512)
    agg = {}
    for _ in range(reps):
        rec.reset()
        cyc.step(trace=rec.struct)
        for kind, b, fl, ms in rec.records():
            b, fl = cyc.algorithmic(kind, b, fl)
            a = agg.setdefault(kind, [0.0, 0.0, 0.0, 0])
            a[0] += b
            a[1] += fl
            a[2] += ms
            a[3] += 1
    names = {dfl.K_GEMM: "gemm_tc", dfl.K_ATTN: "attention", dfl.K_NORM: "row_kernels",
             dfl.K_ARGMAX: "argmax", dfl.K_VERIFY: "verify"}
    serial = sum(a[2] for a in agg.values()) / reps
    scale = min(1.0, step_ms / serial) if serial > 0 else 1.0
    out = {}
    for kind, (b, fl, ms, n) in agg.items():
        ms_in = ms / reps * scale          # this kind's time within one graph-replayed step
        gbs = b / reps / (ms_in * 1e-3) / 1e9 if ms_in > 0 else 0.0
        out[names.get(kind, str(kind))] = {
            "launches_per_step": n // reps, "ms_per_step": ms_in, "serialised_ms_per_step": ms / reps,
            "bytes_per_launch": b / n, "achieved_gbs": gbs, "frac_of_hbm": gbs / peak_gbs,
            "tflops": fl / reps / (ms_in * 1e-3) / 1e12 if ms_in > 0 else 0.0}
    return out


def long_context_attention(dfl, dev, peak_gbs: float, reps: int = 10) -> dict:
    """The split-KV attention kernel alone over a 32K-key context: one layer of
    the Qwen3-8B-shaped drafter, launches timed one by one with CUDA events."""
    wl = synth.WORKLOADS["qwen3_8b_L1_N32768_B1"]
    cyc = DraftCycle(dfl, wl, dev)
    for _ in range(3):
        cyc.step()
    # per launch: the attention kernel carries the K/V bytes; a merge kernel
    # (when the splits exceed a cluster) carries time but no algorithmic bytes
    rec = dfl.TraceRecorder(512)
    att_ms = merge_ms = att_bytes = 0.0
    for _ in range(reps):
        rec.reset()
        cyc.step(trace=rec.struct)
        for kind, b, _, ms in rec.records():
            if kind == dfl.K_ATTN:
                if b > 0:
                    att_ms += ms
                    att_bytes += b
                else:
                    merge_ms += ms
    att_us = 1e3 * att_ms / (reps * wl.n_layers)
    merge_us = 1e3 * merge_ms / (reps * wl.n_layers)
    per_layer = att_bytes / (reps * wl.n_layers)
    gbs = per_layer / (att_us * 1e-6) / 1e9
    gbs_all = per_layer / ((att_us + merge_us) * 1e-6) / 1e9
    # the same launches as they run inside a step: the layer's attention call
    # (kernel + merge, programmatic dependent launch between them) captured
    # n_graph times in a CUDA graph and replayed
    q = torch.randn((wl.rows, wl.n_q_heads * wl.head_dim), device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)

    def att():
        dfl.dflash_attention(cyc.cfg, q, cyc.ctx_len, cyc.max_ctx, 0, cyc.k_cache, cyc.v_cache, o,
                             cyc.status, cyc.ws)

    n_graph = 20
    att()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n_graph):
            att()
    g.replay()
    ms_g = time_steps(g.replay, reps, torch.cuda.current_stream()) / reps
    graph_us = 1e3 * ms_g / n_graph
    out = {"workload": wl.name, "bytes_per_layer": per_layer,
           "attention_us": round(att_us, 2), "merge_us": round(merge_us, 2),
           "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak_gbs, 4),
           "frac_of_hbm_with_merge": round(gbs_all / peak_gbs, 4),
           "in_graph_us_with_merge": round(graph_us, 2),
           "in_graph_frac_of_hbm_with_merge": round(per_layer / (graph_us * 1e-6) / 1e9 / peak_gbs, 4),
           "what": "tcgen05 split-KV attention of one layer over 32768 context + 17 block keys; "
                   "attention_us / merge_us: launches timed one by one with CUDA events (each time "
                   "includes its launch); in_graph: the layer's attention call (kernel + merge) "
                   "replayed back to back from a CUDA graph, as inside the step"}
    del g
    del cyc
    torch.cuda.empty_cache()
    return out


def prefill_row(dfl, wl: synth.Workload, W: dict, dev, T: int, tf_peak: float, reps: int) -> dict:
    """Context fusion + injection of a T-token prefill of one sequence (the
    context feature is computed once per position and cached, then reused by
    every drafting step): tokens along the GEMM's A rows, 128 x 256 tcgen05
    tiles, tensor-bound. Each call is timed on its own with CUDA events on the
    launching stream (fusion: the W_c GEMM and the norm pass; injection: the
    K|V GEMM of all layers and the length update); the GEMM launches alone are
    timed from one traced run."""
    R = wl.rows
    cfg = dfl.config_from_workload(wl, max_batch=1, ctx_capacity=(T + R + 127) // 128 * 128)
    w = dfl.Weights(cfg, W, dev)
    ws = dfl.Workspace(cfg, T, dev)
    dt = synth.torch_dtype(wl.dtype)
    taps = synth.taps(wl, T, f"prefill{T}", dev)
    h = torch.empty((1, T, wl.d_model), dtype=dt, device=dev)
    shape = (wl.n_layers, 1, wl.n_kv_heads, cfg.ctx_capacity, wl.head_dim)
    k_cache = torch.zeros(shape, dtype=dt, device=dev)
    v_cache = torch.zeros(shape, dtype=dt, device=dev)
    ctx_len = torch.zeros(1, dtype=torch.int32, device=dev)
    n_new = torch.full((1,), T, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def fuse(trace=None):
        dfl.dflash_ctx_fuse(cfg, w, taps, h[0], ws, trace=trace)

    def inject(trace=None):
        ctx_len.zero_()
        dfl.dflash_kv_inject(cfg, w, h, n_new, ctx_len, k_cache, v_cache, status, ws, trace=trace)

    for _ in range(2):
        fuse()
        inject()
    torch.cuda.synchronize()
    fuse_ms = time_steps(fuse, reps, stream) / reps
    inject_ms = time_steps(inject, reps, stream) / reps
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"prefill: device status {st}: {dfl.status_string(st)}")
    rec = dfl.TraceRecorder(16)
    gemm = {}
    for name, fn in (("fuse", fuse), ("inject", inject)):
        ms = fl = 0.0
        for _ in range(reps):
            rec.reset()
            fn(trace=rec.struct)
            for kind, _, f, t in rec.records():
                if kind == dfl.K_GEMM:
                    ms += t
                    fl += f
        gemm[name] = (ms / reps, fl / reps)
    K = wl.n_taps * wl.d_target
    fpl = 2 * wl.n_kv_heads * wl.head_dim
    flops = 2.0 * T * wl.d_model * K + 2.0 * T * wl.n_layers * fpl * wl.d_model
    tot_ms = fuse_ms + inject_ms
    g_ms = gemm["fuse"][0] + gemm["inject"][0]
    g_fl = gemm["fuse"][1] + gemm["inject"][1]
    out = {"tokens": T, "layers": wl.n_layers, "fuse_us": round(fuse_ms * 1e3, 1),
           "inject_us": round(inject_ms * 1e3, 1), "us": round(tot_ms * 1e3, 1),
           "gflop": round(flops / 1e9, 1), "tflops": round(flops / (tot_ms * 1e-3) / 1e12, 1),
           "frac_of_bf16_peak": round(flops / (tot_ms * 1e-3) / 1e12 / tf_peak, 4),
           "gemm_fuse_us": round(gemm["fuse"][0] * 1e3, 1), "gemm_inject_us": round(gemm["inject"][0] * 1e3, 1),
           "gemm_tflops": round(g_fl / (g_ms * 1e-3) / 1e12, 1) if g_ms > 0 else None,
           "gemm_frac_of_bf16_peak": round(g_fl / (g_ms * 1e-3) / 1e12 / tf_peak, 4) if g_ms > 0 else None,
           "floor_us": round(flops / (tf_peak * 1e12) * 1e6, 1),
           "what": f"context fusion (W_c over {wl.n_taps} taps) + K/V injection of all {wl.n_layers} layers "
                   f"for a {T}-token prefill; calls timed with CUDA events; peak = measured bf16 burst"}
    del taps, h, k_cache, v_cache, ws
    torch.cuda.empty_cache()
    return out


class LoopRun:
    """The full draft-verify loop: every cycle drafts a block over each
    sequence's context, the synthetic target verifies it (greedy
    accept), and the tapped states of the tau accepted positions are fused
    and injected, so the context grows by tau; the next anchor comes from
    verification. Nothing goes through the host between cycles: the whole
    loop is one CUDA graph.

    The target's logits are synthetic (synth.loop_target_logits): per cycle a
    resident N(0,1) noise tensor, in which the token the target picks for each
    row gets the row max + 1 before verification and its old value back after
    it (a few small torch kernels per cycle, inside the timed region). The
    target agrees with a drafted token with probability 0.8, decided by a
    hash of the token itself, so E[tau] = 1 + sum_k 0.8^k = 4.89."""

    def __init__(self, dfl, wl: synth.Workload, dev):
        self.dfl, self.wl, self.dev = dfl, wl, dev
        B, R, V, D = wl.batch, wl.rows, wl.vocab, wl.d_model
        self.cfg = dfl.config_from_workload(wl)
        self.W = synth.weights(wl, dev)
        self.w = dfl.Weights(self.cfg, self.W, dev)
        self.ws = dfl.Workspace(self.cfg, max(wl.ctx * B, B * R, 16), dev)
        dt = synth.torch_dtype(wl.dtype)
        shape = (wl.n_layers, B, wl.n_kv_heads, self.cfg.ctx_capacity, wl.head_dim)
        self.k_cache = torch.zeros(shape, dtype=dt, device=dev)
        self.v_cache = torch.zeros(shape, dtype=dt, device=dev)
        self.ctx_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # prefill of every sequence's context (set-up, not timed)
        taps = synth.taps(wl, B * wl.ctx, "prefill", dev).view(B, wl.ctx, -1)
        h = torch.empty((B, wl.ctx, D), dtype=dt, device=dev)
        for b in range(B):
            dfl.dflash_ctx_fuse(self.cfg, self.w, taps[b], h[b], self.ws)
        dfl.dflash_kv_inject(self.cfg, self.w, h, torch.full((B,), wl.ctx, dtype=torch.int32, device=dev),
                             self.ctx_len, self.k_cache, self.v_cache, self.status, self.ws)
        del taps, h
        self.ctx0 = self.ctx_len.clone()
        # per-cycle inputs: tapped states of the block's positions, the
        # target's noise and row maxima, the agreement keys
        self.taps = [synth.taps(wl, B * R, f"loop{c}", dev) for c in range(wl.cycles)]
        self.noise = [synth.normal((B, R, V), wl.seed, f"loop_noise/{c}", dev) for c in range(wl.cycles)]
        self.top = [n.max(dim=-1, keepdim=True).values + 1.0 for n in self.noise]
        plans = [synth.loop_plan(wl, c) for c in range(wl.cycles)]
        self.key16 = torch.as_tensor(np.stack([p[0] for p in plans]), device=dev)
        self.offset = torch.as_tensor(np.stack([p[1] for p in plans]), device=dev)
        self.anchor0 = torch.as_tensor(synth.anchors(wl), device=dev)
        self.anchor = self.anchor0.clone()
        self.draft = torch.empty((B, wl.gamma), dtype=torch.int32, device=dev)
        self.tau = torch.empty(B, dtype=torch.int32, device=dev)
        self.committed = torch.empty((B, R), dtype=torch.int32, device=dev)
        self.next_anchor = torch.empty(B, dtype=torch.int32, device=dev)
        self.h_new = torch.empty((B, R, D), dtype=dt, device=dev)
        self.taus = torch.zeros((wl.cycles, B), dtype=torch.int32, device=dev)
        torch.cuda.synchronize()

    def cycle(self, c: int):
        d, wl, cfg = self.dfl, self.wl, self.cfg
        hint = wl.ctx + c * wl.rows          # ctx_len[b] <= ctx + c * R before cycle c
        d.dflash_draft_block(cfg, self.w, self.anchor, self.ctx_len, hint, self.k_cache, self.v_cache,
                             self.draft, self.status, self.ws)
        idx = synth.loop_intended(wl, self.key16[c], self.offset[c], self.draft).unsqueeze(-1)
        logits = self.noise[c]
        saved = logits.gather(-1, idx)
        logits.scatter_(-1, idx, self.top[c])
        d.dflash_verify_accept(cfg, logits, self.draft, self.tau, self.committed, self.next_anchor, self.ws)
        logits.scatter_(-1, idx, saved)
        d.dflash_ctx_fuse(cfg, self.w, self.taps[c], self.h_new.view(-1, wl.d_model), self.ws)
        d.dflash_kv_inject(cfg, self.w, self.h_new, self.tau, self.ctx_len, self.k_cache, self.v_cache,
                           self.status, self.ws)
        self.anchor.copy_(self.next_anchor)
        self.taus[c].copy_(self.tau)

    def run(self):
        self.ctx_len.copy_(self.ctx0)
        self.anchor.copy_(self.anchor0)
        for c in range(self.wl.cycles):
            self.cycle(c)


def measure_loop(dfl, wl: synth.Workload, dev, reps: int, peak_gbs: float) -> dict:
    lr = LoopRun(dfl, wl, dev)
    lr.run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lr.run()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lr.run()
    g.replay()
    torch.cuda.synchronize()
    ms = time_steps(g.replay, reps, torch.cuda.current_stream()) / reps
    st = int(lr.status.item())
    if st != 0:
        raise RuntimeError(f"loop: device status {st}: {dfl.status_string(st)}")
    taus = lr.taus.cpu().numpy()
    committed = int(taus.sum())
    B, C = wl.batch, wl.cycles
    out = {"workload": wl.name, "cycles": C, "batch": B, "loop_ms": round(ms, 2),
           "us_per_cycle": round(1e3 * ms / C, 1), "mean_tau": round(float(taus.mean()), 4),
           "committed_tokens": committed, "committed_tok_s": round(committed / (ms * 1e-3), 1),
           "drafted_tok_s": round(C * B * wl.gamma / (ms * 1e-3), 1),
           "final_context": lr.ctx_len.cpu().tolist(), "replays": reps,
           "what": "draft -> greedy verify -> fusion + injection of the tau accepted positions, every "
                   "cycle on the device, the whole loop one CUDA graph; synthetic target agreeing with a "
                   "drafted token with probability 0.8 (E[tau] = 4.89); its per-cycle logit edits (a few "
                   "small torch kernels) are inside the timed region"}
    del g, lr
    torch.cuda.empty_cache()
    return out


def measure_workload(dfl, wl: synth.Workload, dev, steps: int, peak_gbs: float) -> dict:
    """One drafting cycle of another workload, graph-replayed like the headline."""
    cyc = DraftCycle(dfl, wl, dev)
    for _ in range(3):
        cyc.step()
    r = measure_variant(cyc, cyc.step, steps, wl.batch * wl.gamma, peak_gbs)
    kern = kernel_roofline(cyc, peak_gbs, r["us_per_step"] * 1e-3, reps=2)
    r["gemm_frac_of_hbm"] = round(kern.get("gemm_tc", {}).get("frac_of_hbm", 0.0), 4)
    r["attention_frac_of_hbm"] = round(kern.get("attention", {}).get("frac_of_hbm", 0.0), 4)
    r["gemm_tflops"] = round(kern.get("gemm_tc", {}).get("tflops", 0.0), 1)
    r["workload"] = wl.name
    st = int(cyc.status.item())
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status {st}: {dfl.status_string(st)}")
    del cyc
    torch.cuda.empty_cache()
    return r


def oracle_step_ms(wl_name: str, steps: int, threads: int | None) -> float:
    """ms per drafting cycle of the oracle on the host for a small workload, in a
    child process whose BLAS runs on `threads` threads (None: all cores)."""
    code = ("import sys, time, json; sys.path.insert(0, %r); import synth, bench\n"
            "wl = synth.WORKLOADS[%r]; oc = bench.OracleCycle(wl, synth.weights(wl, 'cpu'), 'cpu')\n"
            "oc.step(); t0 = time.perf_counter()\n"
            "for _ in range(%d): oc.step()\n"
            "print(json.dumps((time.perf_counter() - t0) * 1e3 / %d))") % (ROOT, wl_name, steps, steps)
    env = dict(os.environ)
    if threads is not None:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k] = str(threads)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
    if out.returncode != 0:
        return float("nan")
    return float(out.stdout.strip().splitlines()[-1])


class OracleCycle:
    """The CPU oracle running the same drafting cycle (float64 numpy)."""

    def __init__(self, wl: synth.Workload, W: dict, device: str):
        from oracle import dflash_ref as ref
        self.ref, self.wl = ref, wl
        self.oc = ref.Cfg(wl.n_layers, wl.d_target, wl.n_taps, wl.d_model, wl.n_q_heads,
                          wl.n_kv_heads, wl.head_dim, wl.d_ffn, wl.vocab, wl.gamma,
                          wl.mask_token_id, wl.rms_eps, wl.rope_theta)
        # weights as float64 once (set-up); the embedding stays a CPU tensor (gathered per use)
        self.W = {k: (v.cpu() if k == "embed" else ref.f64(v)) for k, v in W.items()}
        R, B = wl.rows, wl.batch
        prefix = synth.ctx_lengths(wl) - R
        tmax = int(prefix.max())
        taps = synth.taps(wl, B * tmax, "prefill", device).view(B, tmax, -1)
        self.k0, self.v0 = [], []
        for b in range(B):
            h = ref.ctx_fuse(self.oc, self.W["w_c"], self.W["g_c"], taps[b, : int(prefix[b])].float().cpu())
            kv = [ref.ctx_kv(self.oc, self.W["w_qkv"][l], h, 0) for l in range(wl.n_layers)]
            self.k0.append([k for k, _ in kv])
            self.v0.append([v for _, v in kv])
        self.prefix = prefix
        self.step_taps = synth.taps(wl, B * R, "step", device).float().cpu().view(B, R, -1)
        self.anchor = synth.anchors(wl)
        self.target = synth.target_logits(wl, "step", device, torch.float32).cpu().numpy()

    def step(self):
        ref, wl, W = self.ref, self.wl, self.W
        out = []
        for b in range(wl.batch):
            n0 = int(self.prefix[b])
            h = ref.ctx_fuse(self.oc, W["w_c"], W["g_c"], self.step_taps[b])
            ks, vs = [], []
            for l in range(wl.n_layers):
                k, v = ref.ctx_kv(self.oc, W["w_qkv"][l], h, n0)
                ks.append(np.concatenate([self.k0[b][l], k], axis=1))
                vs.append(np.concatenate([self.v0[b][l], v], axis=1))
            d = ref.draft_block(self.oc, W, int(self.anchor[b]), ks, vs, n0 + wl.rows)
            out.append(ref.verify_accept(self.target[b], d["draft"]))
        return out


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(wl, W, device, steps: int, unit_tokens: int):
    t0 = time.perf_counter()
    oc = OracleCycle(wl, W, device)
    setup_s = time.perf_counter() - t0
    oc.step()                               # untimed first pass
    t0 = time.perf_counter()
    for _ in range(steps):
        oc.step()
    dt = (time.perf_counter() - t0) / steps
    return {"value": unit_tokens / dt, "unit": "drafted tokens/s", "cores": oracle_threads(),
            "kind": "oracle", "s_per_step": dt,
            "sample": f"{steps} full drafting cycles of the same workload (fusion + injection of "
                      f"{wl.rows} rows, {wl.n_layers}-layer draft over the context, verify), "
                      f"float64 numpy on the host; weight conversion and prefix prefill "
                      f"({setup_s:.1f} s) excluded"}


METRIC = "draft-block step µs & drafted tokens/s (Qwen3-8B-shape drafter), % HBM roofline"


def traffic_from_profile(kernel_file: str, profile: str):
    """DRAM bytes per launch recorded by an ncu capture of the current source, else None."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, "block_diffusion_drafter_gb300", "csrc", kernel_file), "rb").read()
        sha = hashlib.sha256(src).hexdigest()[:16]
        rec = {}
        for line in open(os.path.join(ROOT, "profiles", profile)):
            if ":" in line and line.strip().startswith(("source_sha256", "traffic_bytes_per_launch")):
                k, v = line.strip().lstrip("-* ").split(":", 1)
                rec[k.strip()] = v.strip().strip("`")
        if rec.get("source_sha256") == sha:
            return float(rec["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


def run_gpu(args):
    rank, local, world = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    import block_diffusion_drafter_gb300 as dfl
    dfl.load()
    wl = synth.WORKLOADS[args.workload]
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    cyc = DraftCycle(dfl, wl, dev)
    tokens = wl.batch * wl.gamma
    for _ in range(max(args.warmup, 3)):
        cyc.step()
    torch.cuda.synchronize()
    graph, graph_note = None, "cuda graph replay of the whole step"
    if not args.no_graph:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                cyc.step()
            torch.cuda.current_stream().wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cyc.step()
            graph = g
        except Exception as e:  # capture unsupported: fall back to eager launches
            graph, graph_note = None, f"eager launches (graph capture failed: {type(e).__name__})"
    else:
        graph_note = "eager launches"
    fn = graph.replay if graph is not None else cyc.step
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        fn()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    t_end = time.time() + 0.6                  # bring clocks to steady state under load
    while time.time() < t_end:
        fn()
    if world > 1:
        torch.distributed.barrier()
    ms = time_steps(fn, args.steps, stream)
    clocks = sampler.stop()
    st = int(cyc.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {dfl.status_string(st)}")
    ms = max_over_ranks(ms, world, dev)
    value = job_throughput(world, tokens, args.steps, ms)

    # end to end through host buffers: inputs H2D from pinned memory, results D2H
    h_in = cyc.io_in.cpu().pin_memory()          # anchors + tapped states
    h_target = cyc.target.cpu().pin_memory()
    o_out = torch.empty_like(cyc.io_out, device="cpu").pin_memory()   # drafts, tau, committed

    def e2e_body():
        # the step's target logits are needed only by verification: their H2D
        # runs on a second stream while fusion, injection and drafting run. It
        # is ordered after the small input copy, which the step waits for:
        # both share the host-to-device copy engine, and queued behind the
        # 10 MB of logits the input copy would hold the step back ~35 us
        cur = torch.cuda.current_stream()
        cyc.io_in.copy_(h_in, non_blocking=True)
        copy_stream.wait_stream(cur)
        with torch.cuda.stream(copy_stream):
            cyc.target.copy_(h_target, non_blocking=True)
        cyc.step_draft()
        cur.wait_stream(copy_stream)
        cyc.step_verify()
        o_out.copy_(cyc.io_out, non_blocking=True)

    copy_stream = torch.cuda.Stream()
    e2e_step = e2e_body
    if graph is not None:   # the same copies and launches, captured once and replayed
        try:
            e2e_body()
            torch.cuda.synchronize()
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_body()
            e2e_step = g_e2e.replay
        except Exception:
            e2e_step = e2e_body

    for _ in range(3):
        e2e_step()
    if world > 1:
        torch.distributed.barrier()
    ms_e2e = max_over_ranks(time_steps(e2e_step, args.steps, stream), world, dev)
    h2d = h_in.numel() + h_target.numel() * 4
    d2h = o_out.numel() * 4

    launches = cyc.launches_per_step()
    kern = kernel_roofline(cyc, hbm, ms / args.steps)
    g = kern.get("gemm_tc", {})
    traffic = traffic_from_profile("gemm.cu", f"gemm_tc_{args.workload}.md")
    roof = {"kernel": "gemm_tc (every projection launch of a step: QKV, O, gate|up, down, LM head, "
                      "fusion, injection)",
            "bound": "hbm", "achieved": round(g.get("achieved_gbs", 0.0), 1), "peak": hbm,
            "unit": "GB/s", "frac": round(g.get("frac_of_hbm", 0.0), 4),
            "traffic": traffic, "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    step_bytes = sum(v["bytes_per_launch"] * v["launches_per_step"] for v in kern.values())
    next_rows = None
    if rank == 0 and not args.no_next_rows:
        B, gam = wl.batch, wl.gamma
        next_rows = {
            "sampling_T1": dict(measure_variant(cyc, cyc.step_sample, min(args.steps, 50), B * gam, hbm),
                                what="sampled drafts at T=1 + rejection-acceptance verification"),
            "per_sequence_gamma_half": dict(measure_variant(cyc, cyc.step_dyn, min(args.steps, 50),
                                                            B * (gam // 2), hbm),
                                            what=f"block size {gam // 2} of {gam} per sequence"),
            "unmask_4_passes": dict(measure_variant(cyc, cyc.step_unmask, min(args.steps, 20), B * gam, hbm),
                                    what="multi-step confidence unmasking, 4 passes"),
            "paged_kv": dict(measure_variant(cyc, cyc.step_paged, min(args.steps, 50), B * gam, hbm),
                             what="greedy cycle over a paged KV cache (128-key pages, scrambled)"),
        }
        if wl.dtype == "bf16":
            next_rows["attention_context_32k"] = long_context_attention(dfl, dev, hbm)
    extra = None
    if rank == 0 and not args.no_extra and wl.dtype == "bf16":
        extra = {}
        for T, reps in ((wl.ctx, 10), (32768, 3)):
            extra[f"prefill_{T}"] = prefill_row(dfl, wl, cyc.W, dev, T, tf_burst, reps)
        lwl = synth.WORKLOADS["qwen3_8b_L8_loop_B4"]
        extra["loop_" + lwl.name] = measure_loop(dfl, lwl, dev, 3, hbm)
        for name in ("tiny_f32_L1_N128", "qwen3_8b_L5_N32768_B1", "qwen3_8b_L5_ragged_B16"):
            if name != wl.name:
                extra[name] = measure_workload(dfl, synth.WORKLOADS[name], dev, min(args.steps, 20), hbm)
        # the tiny workload's oracle cycle on the host, one thread and all cores
        if "tiny_f32_L1_N128" in extra:
            extra["tiny_f32_L1_N128"]["oracle_ms_per_step_1_thread"] = round(
                oracle_step_ms("tiny_f32_L1_N128", 20, 1), 3)
            extra["tiny_f32_L1_N128"]["oracle_ms_per_step_all_cores"] = round(
                oracle_step_ms("tiny_f32_L1_N128", 20, None), 3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(wl, cyc.W, dev, args.cpu_steps, tokens)
        except MemoryError:
            cpu = {"value": None, "kind": "oracle", "sample": "host out of memory"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "drafted tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "us_per_step": round(1000 * ms / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1/fan_in) weights, N(0,1) taps and target logits)",
            "config": {"workload": wl.name, "layers": wl.n_layers, "batch_per_gpu": wl.batch,
                       "context": wl.ctx, "gamma": wl.gamma, "inject_rows_per_step": wl.rows,
                       "vocab": wl.vocab, "launch": graph_note,
                       "l2": "inputs larger than L2 (weights streamed per step: "
                             f"{step_bytes / 1e9:.2f} GB)", "parallelism": f"replicas x{world}"},
            "clocks": clocks,
            "e2e": {"value": round(job_throughput(world, tokens, args.steps, ms_e2e), 1),
                    "unit": "drafted tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "roofline": roof,
            "step_roofline": {"algorithmic_bytes": step_bytes, "achieved_gbs": round(step_bytes / (ms / args.steps * 1e-3) / 1e9, 1),
                              "frac": round(step_bytes / (ms / args.steps * 1e-3) / 1e9 / hbm, 4)},
            "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                        for k, v in kern.items()},
            "cpu_baseline": cpu,
            "next_rows": next_rows,
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = synth.weights(wl, dev)
    oc = OracleCycle(wl, W, dev)
    del W
    tokens = wl.batch * wl.gamma
    t0 = time.perf_counter()
    for _ in range(max(1, args.warmup)):
        oc.step()
        if time.perf_counter() - t0 > 60:
            break
    t1 = time.perf_counter()
    oc.step()
    one = time.perf_counter() - t1
    steps = max(1, min(args.steps, int(120.0 / max(one, 1e-3))))
    t1 = time.perf_counter()
    for _ in range(steps):
        oc.step()
    dt = (time.perf_counter() - t1) / steps
    value = tokens / dt
    sample = (f"{steps} of {args.steps} requested full drafting cycles timed (each "
              f"{dt:.2f} s), float64 numpy oracle on the host")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "drafted tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": wl.name},
        "cpu_baseline": {"value": round(value, 3), "unit": "drafted tokens/s", "kind": "oracle",
                         "cores": oracle_threads(), "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "drafted tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_mode(args):
    """--mode prefill / loop: one measurement alone (profiling captures)."""
    dev = "cuda:0"
    torch.cuda.set_device(dev)
    import block_diffusion_drafter_gb300 as dfl
    dfl.load()
    wl = synth.WORKLOADS[args.workload]
    hbm, tf_burst, _, _ = measured_peaks()
    if args.mode == "prefill":
        T = args.prefill_rows or wl.ctx
        out = prefill_row(dfl, wl, synth.weights(wl, dev), dev, T, tf_burst, max(args.steps, 1))
    else:
        lwl = wl if wl.cycles > 0 else synth.WORKLOADS["qwen3_8b_L8_loop_B4"]
        out = measure_loop(dfl, lwl, dev, max(args.steps, 1), hbm)
    print(json.dumps({"mode": args.mode, "workload": wl.name, **out}), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.mode != "step":
        run_mode(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
