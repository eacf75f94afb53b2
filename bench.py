#!/usr/bin/env python3
"""Benchmark of the varlen attention hot path on GB300 (one process per GPU).

A step is one pass of every hot-path operation over one synthetic batch
(config 2: 32768 packed tokens, lognormal document lengths with median 1024
and sigma 1.2 clipped to [64, 16384], 32 query / 4 key-value heads, d = 128,
bf16 inputs, float32 accumulation):

  1. nsp_attn_fwd    -- schedule + varlen causal attention forward (out, lse)
  2. nsp_attn_bwd    -- dq, dk, dv from out, lse, dout
  3. ring legs       -- the stream split into 8 shards of 4096 tokens; the
                        float32 partial of every non-empty causal (q-shard,
                        kv-shard) block in one nsp_attn_fwd_blocks call, then
                        one nsp_lse_merge_batch over every shard
  4. nsp_seq2head_permute -- q seq->head (8 groups) and back (head->seq)

``value`` = useful attention TFLOP/s of the whole step: (4 d fwd + 10 d bwd
+ 4 d ring partials) x Hq x allowed (causal, same-document) pairs, divided
by the step time; masked work is never counted.  Per-leg times, TFLOP/s and
GB/s and the roofline of the dominant kernel are reported beside it.

Timing: W warm-up steps; the C-ABI calls of each leg are then recorded once
as a CUDA graph and replayed (the library allocates nothing and its calls are
stream-ordered, so a leg's kernels launch back to back); K steps, each
preceded (outside its timed region) by an L2 flush (a 256 MiB write, larger
than the 129 MB L2), each timed with CUDA events on the launching stream;
barrier + synchronize on both sides; max over ranks.  ``gpu_launches`` is
the library kernels one step records times K.  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from variable_length_sequence_gb300.workloads import CONFIGS, make_workload, shard_bounds  # noqa: E402

METRIC = "varlen attn fwd+bwd useful TFLOP/s & % bf16 peak; merge/permute GB/s % HBM"
CONFIG_ID = 2                      # the bench workload; --config 3/4/5 time other configs
# legs timed per config: config 3 is the ring-style chunked forward plus the
# permutation; configs 2, 4 and 5 are forward + backward (config 2 also runs
# the ring legs and the permutation on its own 32768-token stream)
CONFIG_LEGS = {2: ("fwd", "bwd", "ring_partials", "merge", "permute"),
               3: ("ring_partials", "merge", "permute"),
               4: ("fwd", "bwd"),
               5: ("fwd", "bwd")}
RING_SHARDS = 8
PERMUTE_GROUPS = 8
DS_CACHE = True                    # backward dS cache (--no-ds-cache turns it off)
DS_CACHE_MAX = 32 << 30            # largest dS cache the bench allocates, bytes
E2E_RUNS = 3                       # end-to-end runs (median reported)
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a scalar over ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- peaks / clocks

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []           # (arrival time, csv line)
        self.t = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The main timed region, in time.perf_counter() seconds: only samples
        that arrive inside it (plus one sampling interval) are reported by
        stop()."""
        self.window = (t0, t1 + 0.06)

    def summary(self, t0: float, t1: float) -> dict:
        """Median SM clock, max clock and throttle reasons of the samples that
        arrived inside [t0, t1] (plus one sampling interval)."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        for t, ln in list(self.lines):
            if not (t0 <= t <= t1 + 0.06):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        if self.window is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return self.summary(*self.window)


# ----------------------------------------------------------------------------- ncu traffic

KERNEL_SOURCES = {"attn_fwd_tc_kernel": "attn_fwd_tc.cu", "attn_bwd_dkdv_tc_kernel": "attn_bwd_tc.cu",
                  "attn_bwd_dq_tc_kernel": "attn_bwd_tc.cu",
                  "attn_bwd_dkdv_tc_kernel+attn_bwd_dq_tc_kernel": "attn_bwd_tc.cu",
                  "attn_bwd_dq_cached_kernel": "attn_bwd_tc.cu",
                  "attn_bwd_dkdv_tc_kernel+attn_bwd_dq_cached_kernel": "attn_bwd_tc.cu",
                  "lse_merge_kernel": "merge.cu", "permute_vec_kernel": "permute.cu"}


def source_sha(kernel: str) -> str:
    """First 12 hex digits of the sha256 of the kernel's source file and of
    the headers every kernel includes (a profile taken on other sources is
    stale)."""
    import hashlib
    csrc = os.path.join(ROOT, "variable_length_sequence_gb300", "csrc")
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES[kernel], "tc_ptx.cuh", "nsp_internal.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic() -> dict:
    """DRAM bytes per launch from the committed ncu summaries: every line
    'traffic: KERNEL WORKLOAD LEG BYTES SHA' in profiles/*.md.  Kept only when
    SHA is the current source_sha(KERNEL): counters of an older kernel are not
    reported."""
    out = {}
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return out
    for f in sorted(os.listdir(d)):
        if not f.endswith(".md"):
            continue
        with open(os.path.join(d, f)) as fh:
            for ln in fh:
                ln = ln.strip().strip("`")
                if not ln.startswith("traffic:"):
                    continue
                parts = ln.split()
                if len(parts) != 6 or parts[1] not in KERNEL_SOURCES:
                    continue
                kern, wl, leg, nbytes, sha = parts[1], parts[2], parts[3], float(parts[4]), parts[5]
                if sha == source_sha(kern):
                    out[(kern, wl, leg)] = nbytes
    return out


# ----------------------------------------------------------------------------- workload

def allowed_pairs_blocks(cu: np.ndarray, bounds):
    """Non-empty causal (q-shard, kv-shard) pairs and their allowed pair counts
    (a host-side count from cu_seqlens; no attention arithmetic)."""
    cu = np.asarray(cu, np.int64)
    pairs = []
    for qs, (qa, qb) in enumerate(bounds):
        for ks, (ka, kb) in enumerate(bounds[:qs + 1]):
            n = 0
            for b in range(len(cu) - 1):
                s, e = int(cu[b]), int(cu[b + 1])
                lo_q, hi_q = max(s, qa), min(e, qb)
                if hi_q <= lo_q:
                    continue
                # queries t in [lo_q, hi_q) see keys [max(s, ka), min(t + 1, kb))
                ts = np.arange(lo_q, hi_q, dtype=np.int64)
                cnt = np.clip(np.minimum(ts + 1, kb) - max(s, ka), 0, None)
                n += int(cnt.sum())
            if n > 0:
                pairs.append((qs, ks, n))
    return pairs


class Problem:
    """Device-resident inputs, outputs and workspaces of one step."""

    def __init__(self, nsp, w, device, legs=CONFIG_LEGS[CONFIG_ID]):
        self.nsp = nsp
        self.LEGS = tuple(legs)
        self.w = w
        cfg = w.cfg
        self.T, self.Hq, self.Hkv, self.d = w.T, cfg.Hq, cfg.Hkv, cfg.d
        self.scale = self.d ** -0.5
        dev = device
        self.q = w.q.to(dev)
        self.k = w.k.to(dev)
        self.v = w.v.to(dev)
        self.dout = w.dout.to(dev) if w.dout is not None else None
        self.cu = torch.from_numpy(w.cu_seqlens).to(dev)
        T, Hq, Hkv, d = self.T, self.Hq, self.Hkv, self.d
        bf = torch.bfloat16
        self.out = torch.empty((T, Hq, d), dtype=bf, device=dev)
        self.lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        has_bwd = "bwd" in self.LEGS
        self.dq = torch.empty_like(self.q) if has_bwd else None
        self.dk = torch.empty_like(self.k) if has_bwd else None
        self.dv = torch.empty_like(self.v) if has_bwd else None
        self.ws_f = torch.empty(nsp.nsp_attn_fwd_workspace_size(T, T, Hq, Hkv, d),
                                dtype=torch.uint8, device=dev)
        # the backward's dS cache: every visible tile pair's dS kept in HBM, so
        # that dQ takes one product per pair instead of recomputing S and dP
        # (when it fits DS_CACHE_MAX; config 4's 256K-token document needs TBs)
        self.ds_cache_bytes = 0
        if has_bwd and DS_CACHE:
            need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, Hq, True)
            if 0 < need <= DS_CACHE_MAX:
                self.ds_cache_bytes = need
        self.ws_b = (nsp.bwd_workspace(T, Hq, Hkv, d, dev, ds_cache_bytes=self.ds_cache_bytes)
                     if has_bwd else torch.empty(16, dtype=torch.uint8, device=dev))
        # ring legs
        self.bounds = shard_bounds(T, RING_SHARDS)
        self.ring_pairs = (allowed_pairs_blocks(w.cu_seqlens, self.bounds)
                           if "ring_partials" in self.LEGS else [])
        n = T // RING_SHARDS
        self.part_o = {(qs, ks): torch.empty((n, Hq, d), dtype=torch.float32, device=dev)
                       for qs, ks, _ in self.ring_pairs}
        self.part_l = {(qs, ks): torch.empty((Hq, n), dtype=torch.float32, device=dev)
                       for qs, ks, _ in self.ring_pairs}
        self.ws_r = torch.empty(nsp.nsp_attn_fwd_workspace_size(n, n, Hq, Hkv, d),
                                dtype=torch.uint8, device=dev)
        ring = bool(self.ring_pairs)
        self.acc_o = torch.empty((T, Hq, d), dtype=torch.float32, device=dev) if ring else None
        self.acc_l = [torch.empty((Hq, n), dtype=torch.float32, device=dev)
                      for _ in range(RING_SHARDS)] if ring else None
        self.merged_o = torch.empty((T, Hq, d), dtype=bf, device=dev) if ring else None
        self.merged_l = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        # permutation
        perm = "permute" in self.LEGS
        self.perm = torch.empty((PERMUTE_GROUPS, T, Hq // PERMUTE_GROUPS, d), dtype=bf,
                                device=dev) if perm else None
        self.unperm = torch.empty_like(self.q) if perm else None
        # work accounting
        self.pairs = nsp.nsp_attn_pairs(w.cu_seqlens, True)
        self.fwd_flop = 4.0 * d * Hq * self.pairs if "fwd" in self.LEGS else 0.0
        self.bwd_flop = 10.0 * d * Hq * self.pairs if has_bwd else 0.0
        self.ring_flop = 4.0 * d * Hq * sum(c for _, _, c in self.ring_pairs)
        nb = lambda t: t.numel() * t.element_size()
        self.merge_bytes = 0
        for qs in range(RING_SHARDS):
            parts = [(a, b) for a, b, _ in self.ring_pairs if a == qs]
            self.merge_bytes += sum(nb(self.part_o[p]) + nb(self.part_l[p]) for p in parts)
        if ring:
            self.merge_bytes += nb(self.merged_o) + nb(self.merged_l)
        self.permute_bytes = 2 * (nb(self.q) + nb(self.perm)) if perm else 0  # read + write, both ways

    # individual legs -------------------------------------------------------------
    def fwd(self, stream):
        self.nsp.nsp_attn_fwd(self.q, self.k, self.v, self.cu, len(self.w.lengths), 0, self.T, 0,
                              self.T, self.Hq, self.Hkv, self.d, self.scale, True, self.out,
                              self.lse, self.ws_f, stream)

    def bwd(self, stream):
        self.nsp.nsp_attn_bwd(self.q, self.k, self.v, self.out, self.dout, self.lse, self.cu,
                              len(self.w.lengths), self.T, self.Hq, self.Hkv, self.d,
                              self.scale, True, self.dq, self.dk, self.dv, self.ws_b, stream)

    def ring_partials(self, stream):
        """Every non-empty causal (q-shard, kv-shard) block's float32 partial,
        all in one batched call (nsp_attn_fwd_blocks)."""
        n = self.T // RING_SHARDS
        if not hasattr(self, "_ring_blocks"):
            self._ring_blocks = [(self.bounds[qs][0], n, self.bounds[ks][0], n,
                                  self.part_o[(qs, ks)], self.part_l[(qs, ks)])
                                 for qs, ks, _ in self.ring_pairs]
            self._ws_blocks = torch.empty(self.nsp.nsp_attn_fwd_blocks_workspace_size(
                self._ring_blocks, self.Hq, self.Hkv, self.d), dtype=torch.uint8,
                device=self.q.device)
        self.nsp.nsp_attn_fwd_blocks(self.q, self.k, self.v, self.cu, len(self.w.lengths), self.T,
                                     self._ring_blocks, self.Hq, self.Hkv, self.d, self.scale, True,
                                     False, self._ws_blocks, stream)

    def merge(self, stream):
        """Every shard's partials merged in one launch (nsp_lse_merge_batch)."""
        n = self.T // RING_SHARDS
        segments, outs, lses = [], [], []
        for qs in range(RING_SHARDS):
            keys = [(a, b) for a, b, _ in self.ring_pairs if a == qs]
            qa = self.bounds[qs][0]
            segments.append(([self.part_o[p] for p in keys], [self.part_l[p] for p in keys]))
            outs.append(self.merged_o[qa:qa + n])
            lses.append(self.merged_l_view(qs))
        self.nsp.nsp_lse_merge_batch(segments, outs, lses, stream)

    def ring_accumulate(self, stream):
        """The ring legs with the merge fused into the attention epilogue, one
        batched call per ring step: step s meets query shard i with key shard
        i - s (the non-empty causal blocks); step 0 (the diagonal blocks)
        writes each shard's running float32 out and lse, the later steps merge
        into them in place."""
        n = self.T // RING_SHARDS
        if not hasattr(self, "_acc_steps"):
            pairs = {(qs, ks) for qs, ks, _ in self.ring_pairs}
            self._acc_steps = []
            for st in range(RING_SHARDS):
                bl = [(self.bounds[qs][0], n, self.bounds[qs - st][0], n,
                       self.acc_o[self.bounds[qs][0]:self.bounds[qs][0] + n], self.acc_l[qs])
                      for qs in range(st, RING_SHARDS) if (qs, qs - st) in pairs]
                if bl:
                    ws = torch.empty(self.nsp.nsp_attn_fwd_blocks_workspace_size(
                        bl, self.Hq, self.Hkv, self.d), dtype=torch.uint8, device=self.q.device)
                    self._acc_steps.append((st > 0, bl, ws))
        for acc, bl, ws in self._acc_steps:
            self.nsp.nsp_attn_fwd_blocks(self.q, self.k, self.v, self.cu, len(self.w.lengths),
                                         self.T, bl, self.Hq, self.Hkv, self.d, self.scale, True,
                                         acc, ws, stream)

    def ring_bwd(self, stream):
        """The ring backward: every causal (q-shard, kv-shard) block's dq/dk/dv
        added into whole-stream float32 accumulators (zeroed first) in one
        nsp_attn_bwd_blocks call, with the forward's out and lse."""
        n = self.T // RING_SHARDS
        if not hasattr(self, "_rb"):
            dev = self.q.device
            ranges = [(self.bounds[qs][0], n, self.bounds[ks][0], n) for qs, ks, _ in self.ring_pairs]
            self._rb = {
                "dq": torch.zeros((self.T, self.Hq, self.d), dtype=torch.float32, device=dev),
                "dk": torch.zeros((self.T, self.Hkv, self.d), dtype=torch.float32, device=dev),
                "dv": torch.zeros((self.T, self.Hkv, self.d), dtype=torch.float32, device=dev),
                "ranges": ranges}
            # the same dS cache as the whole-stream backward, when it fits
            nb = self.nsp.nsp_attn_bwd_blocks_workspace_size(self.T, ranges, self.Hq, self.Hkv,
                                                            self.d)
            cache = self.nsp.nsp_attn_bwd_blocks_ds_cache_size(self.w.cu_seqlens, ranges,
                                                              self.Hq) if DS_CACHE else 0
            if cache > DS_CACHE_MAX:
                cache = 0
            self._rb["ds_cache_bytes"] = cache
            if cache:
                nb = (nb + 1023) // 1024 * 1024 + cache
            self._rb["ws"] = torch.empty(nb, dtype=torch.uint8, device=dev)
        rb = self._rb
        for t in (rb["dq"], rb["dk"], rb["dv"]):
            t.zero_()
        self.nsp.nsp_attn_bwd_blocks(self.q, self.k, self.v, self.out, self.dout, self.lse, self.cu,
                                     len(self.w.lengths), self.T, rb["ranges"], self.Hq, self.Hkv,
                                     self.d, self.scale, True, rb["dq"], rb["dk"], rb["dv"],
                                     rb["ws"], stream)

    def fwd_headgroups(self, stream):
        """The forward on q in the all-to-all's receive layout [P][T][Hq/P][d]
        (the permute leg's output), out in the same layout: the permutations
        around an Ulysses attention folded into the attention kernel."""
        if not hasattr(self, "_hg_out"):
            self._hg_out = torch.empty_like(self.perm)
            self._hg_lse = torch.empty_like(self.lse)
        self.nsp.nsp_attn_fwd_headgroups(self.perm, self.k, self.v, self.cu, len(self.w.lengths),
                                         self.T, self.Hq, self.Hkv, self.d, PERMUTE_GROUPS,
                                         self.scale, True, self._hg_out, self._hg_lse, self.ws_f,
                                         stream)

    def bwd_headgroups(self, stream):
        """The backward in the same receive layout (q, out, dout, dq grouped;
        k, v, dk, dv packed), on the grouped forward's out and lse."""
        if not hasattr(self, "_hg_dout"):
            self._hg_dout = torch.empty_like(self.perm)
            self.nsp.nsp_seq2head_permute(self.dout, self._hg_dout, self.T, self.Hq, self.d,
                                          PERMUTE_GROUPS, False, stream)
            self._hg_dq = torch.empty_like(self.perm)
            self._hg_dk = torch.empty_like(self.k)
            self._hg_dv = torch.empty_like(self.v)
        self.nsp.nsp_attn_bwd_headgroups(self.perm, self.k, self.v, self._hg_out, self._hg_dout,
                                         self._hg_lse, self.cu, len(self.w.lengths), self.T,
                                         self.Hq, self.Hkv, self.d, PERMUTE_GROUPS, self.scale,
                                         True, self._hg_dq, self._hg_dk, self._hg_dv, self.ws_b,
                                         stream)

    def fwd_mha(self, stream):
        """The forward with the pages' own head layout, multi-head attention:
        as many key/value heads as query heads (the paired-tile tensor-core
        path), on the same documents and q."""
        if not hasattr(self, "_mha_k"):
            g = torch.Generator(device=self.q.device)
            g.manual_seed(77)
            shape = (self.T, self.Hq, self.d)
            self._mha_k = torch.randn(shape, generator=g, device=self.q.device).to(torch.bfloat16)
            self._mha_v = torch.randn(shape, generator=g, device=self.q.device).to(torch.bfloat16)
            self._mha_o = torch.empty_like(self.q)
            self._mha_l = torch.empty_like(self.lse)
        self.nsp.nsp_attn_fwd(self.q, self._mha_k, self._mha_v, self.cu, len(self.w.lengths), 0,
                              self.T, 0, self.T, self.Hq, self.Hq, self.d, self.scale, True,
                              self._mha_o, self._mha_l, self.ws_f, stream)

    def _d64(self):
        """Head dimension 64 inputs on the same documents and heads (q, k, v,
        dOut drawn on the device), their outputs and workspaces."""
        if not hasattr(self, "_d64_t"):
            g = torch.Generator(device=self.q.device)
            g.manual_seed(64)
            dev, T, Hq, Hkv = self.q.device, self.T, self.Hq, self.Hkv
            draw = lambda h: torch.randn((T, h, 64), generator=g, device=dev).to(torch.bfloat16)
            t = {"q": draw(Hq), "k": draw(Hkv), "v": draw(Hkv), "dout": draw(Hq)}
            t["out"] = torch.empty_like(t["q"])
            t["lse"] = torch.empty_like(self.lse)
            t["dq"], t["dk"], t["dv"] = (torch.empty_like(t[n]) for n in ("q", "k", "v"))
            t["ws_f"] = torch.empty(self.nsp.nsp_attn_fwd_workspace_size(T, T, Hq, Hkv, 64),
                                    dtype=torch.uint8, device=dev)
            t["ws_b"] = self.nsp.bwd_workspace(T, Hq, Hkv, 64, dev,
                                               ds_cache_bytes=self.ds_cache_bytes)
            self._d64_t = t
        return self._d64_t

    def fwd_d64(self, stream):
        """The forward at head dimension 64 (tensor cores), same documents."""
        t = self._d64()
        self.nsp.nsp_attn_fwd(t["q"], t["k"], t["v"], self.cu, len(self.w.lengths), 0, self.T, 0,
                              self.T, self.Hq, self.Hkv, 64, 64 ** -0.5, True, t["out"], t["lse"],
                              t["ws_f"], stream)

    def bwd_d64(self, stream):
        """The backward at head dimension 64 (after fwd_d64 has run once)."""
        t = self._d64()
        self.nsp.nsp_attn_bwd(t["q"], t["k"], t["v"], t["out"], t["dout"], t["lse"], self.cu,
                              len(self.w.lengths), self.T, self.Hq, self.Hkv, 64, 64 ** -0.5, True,
                              t["dq"], t["dk"], t["dv"], t["ws_b"], stream)

    def merged_l_view(self, qs):
        # [Hq, T] is not sliceable per shard contiguously; merge into a per-shard buffer
        if not hasattr(self, "_ml"):
            n = self.T // RING_SHARDS
            self._ml = [torch.empty((self.Hq, n), dtype=torch.float32, device=self.q.device)
                        for _ in range(RING_SHARDS)]
        return self._ml[qs]

    def permute(self, stream):
        self.nsp.nsp_seq2head_permute(self.q, self.perm, self.T, self.Hq, self.d,
                                      PERMUTE_GROUPS, False, stream)
        self.nsp.nsp_seq2head_permute(self.perm, self.unperm, self.T, self.Hq, self.d,
                                      PERMUTE_GROUPS, True, stream)

    def step(self, stream, events=None):
        for i, leg in enumerate(self.LEGS):
            if events is not None:
                events[i][0].record(stream)
            if self.graphs is not None:
                with torch.cuda.stream(stream):      # replay on the caller's stream
                    self.graphs[leg].replay()
            else:
                getattr(self, leg)(stream)
            if events is not None:
                events[i][1].record(stream)

    graphs = None
    launches_per_step = None

    def capture(self, stream, legs=None):
        """Record each leg's C-ABI calls once as a CUDA graph (the kernels of a
        leg then launch back to back on replay).  Returns the number of
        library kernels one step launches."""
        self.graphs = {}
        n0 = self.nsp.nsp_kernel_launches()
        tc0, cc0 = self.nsp.nsp_path_launches(True), self.nsp.nsp_path_launches(False)
        side = torch.cuda.Stream(stream.device)
        side.wait_stream(stream)
        for leg in legs or self.LEGS:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                getattr(self, leg)(side)
            self.graphs[leg] = g
        stream.wait_stream(side)
        torch.cuda.synchronize()
        self.launches_per_step = self.nsp.nsp_kernel_launches() - n0
        # attention kernels of one step on each path: a CUDA-core launch here
        # would mean the tensor-core path was not taken
        self.path_per_step = {"tensor_core": self.nsp.nsp_path_launches(True) - tc0,
                              "cuda_core": self.nsp.nsp_path_launches(False) - cc0}
        return self.launches_per_step


# ----------------------------------------------------------------------------- our arm

def time_steps(prob, stream, flush, K: int, warmup: int, settle: int = 2):
    """W warm-up steps, capture of each leg as a CUDA graph, `settle` replays,
    then K timed steps, each preceded by an L2 flush outside its timed
    region, with CUDA events on the launching stream around the step and
    around each leg.  Returns (step_ms [K], leg_ms [K, legs], launches per
    step, (t0, t1) of the timed region in time.perf_counter() seconds)."""
    for _ in range(warmup):
        flush.zero_()
        prob.step(stream)
    torch.cuda.synchronize()
    launches_per_step = prob.capture(stream)  # legs replayed as CUDA graphs from here on
    for _ in range(settle):
        flush.zero_()
        prob.step(stream)
    torch.cuda.synchronize()
    nlegs = len(prob.LEGS)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    leg_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nlegs)] for _ in range(K)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()                       # L2 flush, outside the timed region
        step_ev[i][0].record(stream)
        prob.step(stream, leg_ev[i])
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    step_ms = [x.elapsed_time(y) for x, y in step_ev]
    leg_ms = np.array([[x.elapsed_time(y) for x, y in legs] for legs in leg_ev])
    return step_ms, leg_ms, launches_per_step, (t0, t1)


def leg_records(prob, legs: dict, peaks: dict) -> dict:
    """Time, achieved rate and fraction of the measured peak of each leg."""
    out = {}
    for k, flop in (("fwd", prob.fwd_flop), ("bwd", prob.bwd_flop),
                    ("ring_partials", prob.ring_flop)):
        if k in legs:
            out[k] = {"ms": legs[k], "tflops": flop / legs[k] / 1e9}
            out[k]["frac_bf16"] = out[k]["tflops"] / peaks["bf16_tflops"]
    if "ring_partials" in legs:
        out["ring_partials"]["pairs"] = len(prob.ring_pairs)
    for k, nbytes in (("merge", prob.merge_bytes), ("permute", prob.permute_bytes)):
        if k in legs:
            out[k] = {"ms": legs[k], "gbs": nbytes / legs[k] / 1e6,
                      "frac_hbm": nbytes / legs[k] / 1e6 / peaks["hbm_gbs"]}
    if "fwd" in legs and "bwd" in legs:
        fb = (prob.fwd_flop + prob.bwd_flop) / (legs["fwd"] + legs["bwd"]) / 1e9
        out["fwd+bwd"] = {"ms": legs["fwd"] + legs["bwd"], "tflops": fb,
                          "frac_bf16": fb / peaks["bf16_tflops"]}
    return out


def roof_entry(kernel, cid, leg, bound, achieved, peak, unit, work, work_unit, launches,
               traffic_map, peak_kind="burst"):
    wl = CONFIGS[cid].name
    tr = traffic_map.get((kernel, wl, leg))
    return {"kernel": kernel, "workload": wl, "leg": leg, "bound": bound,
            "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "peak_kind": peak_kind, "algorithmic_per_launch": work / max(1, launches),
            "algorithmic_unit": work_unit, "launches_per_step": launches,
            "traffic": tr, "traffic_unit": "DRAM bytes per launch (ncu)" if tr else None}


def sub_config(nsp, cid, device, stream, flush, peaks, clocks, K, warmup, traffic_map):
    """One other config's legs, timed like the step (own clocks); inputs drawn
    on the device (seeded) to keep the default run short."""
    from variable_length_sequence_gb300.workloads import make_workload_device
    w = make_workload_device(cid, device)
    prob = Problem(nsp, w, device, CONFIG_LEGS[cid])
    step_ms, leg_ms, lps, (t0, t1) = time_steps(prob, stream, flush, K, warmup, settle=1)
    legs = dict(zip(prob.LEGS, leg_ms.mean(0).tolist()))
    rec = {"workload": CONFIGS[cid].name, "tokens": prob.T, "docs": len(w.lengths),
           "steps": K, "warmup": warmup, "ms_per_step": float(np.mean(step_ms)),
           "legs": leg_records(prob, legs, peaks), "clocks": clocks.summary(t0, t1),
           "gpu_launches_per_step": lps,
           "attention_launches_per_step": prob.path_per_step,
           "bwd_ds_cache": ds_cache_record(prob),
           "data": "synthetic (seeded lengths; Q/K/V/dOut N(0,1) drawn on the GPU, bf16)"}
    roofs = []
    if "fwd" in legs:
        roofs.append(roof_entry("attn_fwd_tc_kernel", cid, "fwd", "tensor",
                                rec["legs"]["fwd"]["tflops"], peaks["bf16_tflops"], "TFLOP/s",
                                prob.fwd_flop, "FLOP", 1, traffic_map))
    if "bwd" in legs:
        roofs.append(roof_entry(bwd_kernels(prob), cid, "bwd",
                                "tensor", rec["legs"]["bwd"]["tflops"], peaks["bf16_tflops"],
                                "TFLOP/s", prob.bwd_flop, "FLOP", 1, traffic_map))
    if "ring_partials" in legs:
        roofs.append(roof_entry("attn_fwd_tc_kernel", cid, "ring_partials", "tensor",
                                rec["legs"]["ring_partials"]["tflops"], peaks["bf16_tflops"],
                                "TFLOP/s", prob.ring_flop, "FLOP", 1, traffic_map))
    for k, kern in (("merge", "lse_merge_kernel"), ("permute", "permute_vec_kernel")):
        if k in legs:
            nb = prob.merge_bytes if k == "merge" else prob.permute_bytes
            roofs.append(roof_entry(kern, cid, k, "hbm", rec["legs"][k]["gbs"], peaks["hbm_gbs"],
                                    "GB/s", nb, "bytes", 1 if k == "merge" else 2, traffic_map))
    if cid == 5:
        # short documents are HBM-bound by their arithmetic intensity: the
        # compulsory bytes of each call against the copy rate
        cost = nsp.nsp_attn_cost(w.cu_seqlens, prob.Hq, prob.Hkv, prob.d)
        for k, nb in (("fwd", cost["fwd_bytes"]), ("bwd", cost["bwd_bytes"])):
            gbs = nb / legs[k] / 1e6
            rec["legs"][k]["compulsory_gb"] = nb / 1e9
            rec["legs"][k]["gbs_compulsory"] = gbs
            rec["legs"][k]["frac_hbm"] = gbs / peaks["hbm_gbs"]
        roofs = [roof_entry("attn_fwd_tc_kernel", cid, "fwd", "hbm",
                            rec["legs"]["fwd"]["gbs_compulsory"], peaks["hbm_gbs"], "GB/s",
                            cost["fwd_bytes"], "compulsory bytes", 1, traffic_map),
                 roof_entry(bwd_kernels(prob), cid, "bwd", "hbm",
                            rec["legs"]["bwd"]["gbs_compulsory"], peaks["hbm_gbs"], "GB/s",
                            cost["bwd_bytes"], "compulsory bytes", 1, traffic_map)]
    if cid == 3 and not getattr(sub_config, "skip_extra", False):
        reps = 5
        ta = time.perf_counter()
        ms = _time_leg(prob.ring_accumulate, stream, flush, reps)
        tb = time.perf_counter()
        tf = prob.ring_flop / ms / 1e9
        rec["legs"]["ring_accumulate"] = {"ms": ms, "tflops": tf,
                                          "frac_bf16": tf / peaks["bf16_tflops"],
                                          "blocks": len(prob.ring_pairs),
                                          "clocks": clocks.summary(ta, tb)}
    launches = lps * K
    del prob, w
    torch.cuda.empty_cache()
    return rec, roofs, launches


def run_ours(args, world, rank, local):
    from variable_length_sequence_gb300 import build as nsp_build
    from variable_length_sequence_gb300 import nsp

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    if rank == 0 or not os.path.exists(nsp.LIB_PATH):
        nsp_build.build()
    barrier(world)
    nsp.load()

    cid = args.config
    w = make_workload(cid)
    prob = Problem(nsp, w, device, CONFIG_LEGS[cid])
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    clocks.start()                          # nvidia-smi takes a while to start sampling
    K = args.steps
    barrier(world)
    step_ms, leg_ms, launches_per_step, (wall0, wall1) = time_steps(prob, stream, flush, K,
                                                                    args.warmup)
    barrier(world)
    wall = wall1 - wall0
    clocks.mark(wall0, wall1)
    # graph replays do not pass through the library's host launch counter:
    # the kernels of one step were counted while the graphs were recorded
    launches = launches_per_step * K

    total_ms = reduce_max(sum(step_ms), world, device)
    ms_per_step = total_ms / K
    useful = prob.fwd_flop + prob.bwd_flop + prob.ring_flop
    value = reduce_sum(useful * K, world, device) / (total_ms * 1e-3) / 1e12

    peaks = measured_peaks()
    legs = dict(zip(prob.LEGS, leg_ms.mean(0).tolist()))
    leg_stats = leg_records(prob, legs, peaks)
    traffic_map = profiled_traffic()

    # Roofline of the kernel with the largest share of the step's GPU time
    # (ncu launch list of this step: attn_fwd_tc_kernel, the main forward plus
    # the ring partials): useful FLOP of all its launches in a step / their
    # CUDA-event time on the launching stream (each call's time includes its
    # small tile-schedule kernel).  Every other kernel follows in "kernels".
    roofs = []
    if "fwd" in legs and "ring_partials" in legs:
        ach = (prob.fwd_flop + prob.ring_flop) / (legs["fwd"] + legs["ring_partials"]) / 1e9
        roof = roof_entry("attn_fwd_tc_kernel", cid, "fwd + ring_partials", "tensor", ach,
                          peaks["bf16_tflops"], "TFLOP/s", prob.fwd_flop + prob.ring_flop, "FLOP",
                          2, traffic_map)
        # one main forward launch and one batched launch of all ring blocks:
        # DRAM bytes per launch = the mean of the two profiled launches
        wl = CONFIGS[cid].name
        tr = [traffic_map.get(("attn_fwd_tc_kernel", wl, k)) for k in ("fwd", "ring_partials")]
        roof["traffic"] = sum(tr) / 2 if None not in tr else None
        roof["traffic_unit"] = "DRAM bytes per launch (ncu), mean of the 2 launches" \
            if roof["traffic"] else None
    else:
        k0 = "fwd" if "fwd" in legs else "ring_partials"
        roof = roof_entry("attn_fwd_tc_kernel", cid, k0, "tensor", leg_stats[k0]["tflops"],
                          peaks["bf16_tflops"], "TFLOP/s",
                          prob.fwd_flop if k0 == "fwd" else prob.ring_flop, "FLOP", 1, traffic_map)
    roof["peak_source"] = peaks["source"] + " (burst)"
    if "fwd" in legs:
        roofs.append(roof_entry("attn_fwd_tc_kernel", cid, "fwd", "tensor",
                                leg_stats["fwd"]["tflops"], peaks["bf16_tflops"], "TFLOP/s",
                                prob.fwd_flop, "FLOP", 1, traffic_map))
    if "ring_partials" in legs:
        roofs.append(roof_entry("attn_fwd_tc_kernel", cid, "ring_partials", "tensor",
                                leg_stats["ring_partials"]["tflops"], peaks["bf16_tflops"],
                                "TFLOP/s", prob.ring_flop, "FLOP", 1, traffic_map))
    if "bwd" in legs:
        roofs.append(roof_entry(bwd_kernels(prob), cid, "bwd",
                                "tensor", leg_stats["bwd"]["tflops"], peaks["bf16_tflops"],
                                "TFLOP/s", prob.bwd_flop, "FLOP", 1, traffic_map))
    for k, kern in (("merge", "lse_merge_kernel"), ("permute", "permute_vec_kernel")):
        if k in legs:
            nb = prob.merge_bytes if k == "merge" else prob.permute_bytes
            roofs.append(roof_entry(kern, cid, k, "hbm", leg_stats[k]["gbs"], peaks["hbm_gbs"],
                                    "GB/s", nb, "bytes", 1 if k == "merge" else 2, traffic_map))

    prob_path = prob.path_per_step
    ds_rec = ds_cache_record(prob)
    e2e = None
    if "bwd" in legs and not args.no_e2e:
        e2e = run_e2e(args, prob, nsp, w, device, stream, world)

    extra = None
    if prob.ring_pairs and not args.no_extra:
        extra = time_extra_legs(prob, stream, flush, K, peaks)
        extra["ring_accumulate"]["partials_plus_merge_ms"] = legs["ring_partials"] + legs["merge"]

    # the other configs' legs (rank 0's GPU; replicas only), each with its clocks
    configs = {}
    if cid == CONFIG_ID and not args.no_configs:
        del prob
        torch.cuda.empty_cache()
        for c, k_sub in ((3, 30), (4, 3), (5, 200)):
            rec, rr, n = sub_config(nsp, c, device, stream, flush, peaks, clocks, k_sub, 3,
                                    traffic_map)
            configs[str(c)] = rec
            roofs.extend(rr)
    targets = None
    if configs:
        fb = {"2": leg_stats["fwd+bwd"]["frac_bf16"]}
        fb.update({c: configs[c]["legs"]["fwd+bwd"]["frac_bf16"] for c in ("4", "5")})
        targets = {
            "attention fwd+bwd frac_bf16 (target >= 0.55 on configs 2-4)": fb,
            "config 3 ring forward frac_bf16 (it defines no backward)": {
                k: configs["3"]["legs"][k]["frac_bf16"]
                for k in ("ring_partials", "ring_accumulate") if k in configs["3"]["legs"]},
            "merge frac_hbm (target >= 0.75)": {"2": leg_stats["merge"]["frac_hbm"],
                                                "3": configs["3"]["legs"]["merge"]["frac_hbm"]},
            "permute frac_hbm (target >= 0.75)": {
                "2": leg_stats["permute"]["frac_hbm"],
                "3": configs["3"]["legs"]["permute"]["frac_hbm"]},
            "config 5 compulsory-bytes frac_hbm (HBM-bound; no target)": {
                k: configs["5"]["legs"][k]["frac_hbm"] for k in ("fwd", "bwd")}}
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and cid == CONFIG_ID:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        roof["kernels"] = roofs
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; lengths, Q/K/V/dOut N(0,1) rounded to bf16)",
            "config": {"workload": CONFIGS[cid].name, "tokens": int(w.T),
                       "docs": len(w.lengths), "heads_q": CONFIGS[cid].Hq,
                       "heads_kv": CONFIGS[cid].Hkv, "head_dim": CONFIGS[cid].d, "causal": True,
                       "ring_shards": RING_SHARDS, "permute_groups": PERMUTE_GROUPS,
                       "step": " + ".join(CONFIG_LEGS[cid]),
                       "l2": "flushed (256 MiB write) before every timed step",
                       "bwd_ds_cache": ds_rec,
                       "parallelism": f"replicas x{world}"},
            "useful_flop_per_step": useful,
            "legs": leg_stats,
            "extra_legs": extra,
            "configs": configs or None,
            "targets": targets,
            "roofline": roof,
            "attention_launches_per_step": prob_path,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": clk,
            "wall_s": wall,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def bwd_kernels(prob) -> str:
    """The backward's two tensor-core kernels (dQ from the dS cache when the
    step gives it one)."""
    dq = "attn_bwd_dq_cached_kernel" if prob.ds_cache_bytes else "attn_bwd_dq_tc_kernel"
    return "attn_bwd_dkdv_tc_kernel+" + dq


def ds_cache_record(prob):
    """The backward's dS cache as the step used it (bytes; whether the
    device-side check found room for every tile pair)."""
    if prob.dq is None:
        return None
    used = prob.nsp.nsp_bwd_ds_cache_used(prob.ws_b) if prob.ds_cache_bytes else False
    return {"bytes": int(prob.ds_cache_bytes), "used": bool(used)}


def _time_leg(fn, stream, flush, reps):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(stream.device)
    fn(stream)                              # warm (lazy buffers)
    torch.cuda.synchronize()
    side.wait_stream(stream)
    with torch.cuda.graph(g, stream=side):
        fn(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i in range(reps):
        flush.zero_()
        ev[i][0].record(stream)
        with torch.cuda.stream(stream):
            g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in ev)


def time_extra_legs(prob, stream, flush, K, peaks):
    """Entry points outside the step, timed alone the same way (graph replay,
    L2 flushed before each timed call, CUDA events on the stream):
    fwd_headgroups / bwd_headgroups, forward and backward on the all-to-all's
    receive layout; fwd_mha, the forward with multi-head attention (as many
    key/value heads as query heads); fwd_d64 / bwd_d64, head dimension 64;
    ring_accumulate, the ring legs with the merge fused into attention, and
    ring_bwd, the ring backward in one batched call (its three float32
    accumulators are zeroed inside the timed region, by PyTorch)."""
    reps = max(3, min(K, 50))
    extra = {}
    if prob.perm is not None and prob.fwd_flop > 0:
        ms = _time_leg(prob.fwd_headgroups, stream, flush, reps)
        tf = prob.fwd_flop / ms / 1e9
        extra["fwd_headgroups"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                                   "layout": f"q, out [{PERMUTE_GROUPS}][T][Hq/{PERMUTE_GROUPS}][d]"}
        if prob.bwd_flop > 0:
            ms = _time_leg(prob.bwd_headgroups, stream, flush, reps)
            tf = prob.bwd_flop / ms / 1e9
            extra["bwd_headgroups"] = {"ms": ms, "tflops": tf,
                                       "frac_bf16": tf / peaks["bf16_tflops"],
                                       "layout": "q, out, dout, dq grouped; k, v, dk, dv packed"}
    if prob.fwd_flop > 0:
        ms = _time_leg(prob.fwd_mha, stream, flush, reps)
        tf = prob.fwd_flop / ms / 1e9
        extra["fwd_mha"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                            "heads": f"{prob.Hq} query / {prob.Hq} key-value (multi-head)"}
    if prob.fwd_flop > 0:
        # head dimension 64: half the FLOPs of the same pairs
        ms = _time_leg(prob.fwd_d64, stream, flush, reps)
        flop = prob.fwd_flop * 64 / prob.d
        tf = flop / ms / 1e9
        extra["fwd_d64"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                            "head_dim": 64}
        if prob.bwd_flop > 0:
            ms = _time_leg(prob.bwd_d64, stream, flush, reps)
            flop = prob.bwd_flop * 64 / prob.d
            tf = flop / ms / 1e9
            extra["bwd_d64"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                                "head_dim": 64, "ds_cache": prob.ds_cache_bytes > 0}
    ms = _time_leg(prob.ring_accumulate, stream, flush, reps)
    tf = prob.ring_flop / ms / 1e9
    extra["ring_accumulate"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                                "blocks": len(prob.ring_pairs),
                                "out": "float32 out + lse per shard"}
    if prob.dout is not None:
        ms = _time_leg(prob.ring_bwd, stream, flush, reps)
        flop = prob.ring_flop * 10.0 / 4.0
        tf = flop / ms / 1e9
        extra["ring_bwd"] = {"ms": ms, "tflops": tf, "frac_bf16": tf / peaks["bf16_tflops"],
                             "blocks": len(prob.ring_pairs),
                             "out": "float32 dq, dk, dv accumulated over the blocks",
                             "ds_cache_bytes": int(prob._rb["ds_cache_bytes"]),
                             "ds_cache_used": prob.nsp.nsp_bwd_ds_cache_used(prob._rb["ws"])}
    return extra


def run_e2e(args, prob, nsp, w, device, stream, world):
    """Same step through the public API with host buffers: every step copies
    its inputs (q, k, v, dOut, cu_seqlens) in from pinned host memory and its
    results (out, lse, dq, dk, dv) back out, inside the timed region.  The
    steps are pipelined the way a training loop would run them: two sets of
    device buffers, a copy-in stream, the compute stream and a copy-out
    stream, so the copies of neighbouring steps overlap a step's compute.
    The time is from the first copy-in to the last copy-out."""
    prob2 = Problem(nsp, w, device, prob.LEGS)
    prob2.step(stream)                      # warm (lazy buffers), then record its graphs
    torch.cuda.synchronize()
    prob2.capture(stream)
    probs = (prob, prob2)
    host_in = {n: getattr(w, n).pin_memory() for n in ("q", "k", "v", "dout")}
    host_cu = torch.from_numpy(w.cu_seqlens).pin_memory()
    outs = {n: torch.empty(getattr(prob, n).shape, dtype=getattr(prob, n).dtype).pin_memory()
            for n in ("out", "lse", "dq", "dk", "dv")}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + host_cu.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    K = max(2, min(args.steps, 30))       # the pipeline fills and drains once per run
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def one_run() -> float:
        in_ready = [ev() for _ in range(K)]
        comp_done = [ev() for _ in range(K)]
        out_done = [ev() for _ in range(K)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(K):
            p = probs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])       # step i - 2 has read these inputs
                for n, t in host_in.items():
                    getattr(p, n).copy_(t, non_blocking=True)
                p.cu.copy_(host_cu, non_blocking=True)
                in_ready[i].record(s_in)
            stream.wait_event(in_ready[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])          # its results have been copied out
            p.step(stream)
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                for n, t in outs.items():
                    t.copy_(getattr(p, n), non_blocking=True)
                out_done[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        return reduce_max(t0.elapsed_time(t1), world, device)

    # The pinned host <-> device copy rate of the GPU machine is bimodal (H2D
    # about 210 or 40-75 GB/s, D2H about 190 or 75 GB/s, switching between
    # back-to-back copies of the same buffers with no kernel in between), so
    # one run lands on either mode: three runs, the median reported.
    runs = sorted(one_run() for _ in range(E2E_RUNS))
    total_ms = runs[len(runs) // 2]
    useful = prob.fwd_flop + prob.bwd_flop + prob.ring_flop
    val = reduce_sum(useful * K, world, device) / (total_ms * 1e-3) / 1e12
    return {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": K, "ms_per_step": total_ms / K,
            "runs_ms_per_step": [r / K for r in runs], "reported": f"median of {E2E_RUNS} runs",
            "pipelined": "copy-in / compute / copy-out streams, two device buffer sets"}


# ----------------------------------------------------------------------------- CPU oracle

def cpu_sample_rows(cu, n, seed):
    rng = np.random.default_rng(seed)
    T = int(cu[-1])
    return np.sort(rng.choice(T, size=min(n, T), replace=False))


def cpu_oracle_rate(w, seconds: float, seed: int = 0):
    """Time the fp64 oracle forward on growing random row samples of the
    workload (all heads) until about `seconds` of CPU work; return
    (useful TFLOP/s, rows, elapsed)."""
    import oracle
    q, k, v = (w.f64(n) for n in ("q", "k", "v"))
    cu = np.asarray(w.cu_seqlens, np.int64)
    d, Hq = w.cfg.d, w.cfg.Hq
    n = 16
    done_flop, done_s, done_rows = 0.0, 0.0, 0
    while done_s < seconds:
        rows = cpu_sample_rows(cu, n, seed + n)
        doc = np.searchsorted(cu, rows, side="right") - 1
        pairs = float((rows - cu[doc] + 1).sum())
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(q, k, v, cu, d ** -0.5, True, rows)
        dt = time.perf_counter() - t0
        done_flop += 4.0 * d * Hq * pairs
        done_s += dt
        done_rows += len(rows)
        n *= 2
    return done_flop / done_s / 1e12, done_rows, done_s


def cpu_baseline(w, seconds: float):
    rate, rows, el = cpu_oracle_rate(w, seconds)
    return {"value": rate, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 numpy oracle forward on {rows} random query rows of "
                      f"{w.cfg.name} (all {w.cfg.Hq} heads), {el:.1f} s; "
                      "useful FLOP = 4 d Hq x allowed pairs of those rows"}


def run_reference(args, world, rank, local):
    """Reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    w = make_workload(CONFIG_ID, with_dout=False)
    K, W = args.steps, args.warmup
    per_step = max(1.0, min(20.0, 150.0 / max(1, K + W)))
    for i in range(W):
        cpu_oracle_rate(w, per_step, seed=1000 + i)
    rates, wall = [], 0.0
    for i in range(K):
        r, rows, el = cpu_oracle_rate(w, per_step, seed=i)
        rates.append(r)
        wall += el
    value = statistics.mean(rates)
    cpu = {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"each step: fp64 oracle forward on random query rows of "
                     f"{CONFIGS[CONFIG_ID].name} (all heads) for ~{per_step:.0f} s"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": wall / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": {"workload": CONFIGS[CONFIG_ID].name},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the legs timed outside the step (ring accumulate / backward)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the sub-records of configs 3, 4 and 5")
    ap.add_argument("--config", type=int, choices=sorted(CONFIG_LEGS), default=CONFIG_ID,
                    help="workload (default: config 2, the bench workload)")
    ap.add_argument("--no-ds-cache", action="store_true",
                    help="backward without the dS cache (dQ recomputes S and dP)")
    args = ap.parse_args()
    global DS_CACHE
    DS_CACHE = not args.no_ds_cache
    if args.warmup < 3 and args.impl == "ours":
        print("bench: --warmup raised to 3 (minimum)", file=sys.stderr)
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
