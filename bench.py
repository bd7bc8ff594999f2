#!/usr/bin/env python
"""Throughput of the block-causal attention hot path on one GB300 (or N replicas).

One step = one pass of the whole path over one request of the two-reference
edit workload (B=1, 32 heads x 128, [t96][ref 4096][t32][ref 4096][t64]
[target 4096], S=12480): schedule prep + block-causal prefill, prefix cache
append, then one cached step (prefix decode of the 4096 target queries over
8384 cached + 4096 own keys).

metric: TFLOP/s counting only visible (q, k) pairs (4 * 128 * 32 flops each)
of prefill + decode, divided by the time of the whole step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--cache bf16|fp8-v|fp8-kv]

--cache fp8-v / fp8-kv runs the same step with the prefix cache in FP8 E4M3 (V, or
K and V, quantised by the append and expanded by each decode) and adds the PSNR of
the decode output against a bf16 cache.

Under torchrun each rank runs its own independent request (weak scaling, no
data-path collective); the per-step times are max-reduced over ranks.
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

METRIC = "block-causal attn TFLOP/s (visible pairs) prefill+prefix-decode; % of BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "edit_2ref_1024_s12480"
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


ATTN_SOURCES = ["prefix_kv_gb300/csrc/attn_fwd.cu", "prefix_kv_gb300/csrc/ptx.cuh",
                "prefix_kv_gb300/csrc/common.cuh"]
ATTN_PROFILE = "profiles/attn_fwd_edit_2ref_s12480.md"


def profiled_traffic():
    """DRAM bytes per prefill launch from the committed ncu summary, or None when the
    attention sources changed since that capture (their sha256 no longer matches)."""
    import hashlib
    try:
        h = hashlib.sha256()
        for f in ATTN_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        fields = {}
        with open(os.path.join(ROOT, ATTN_PROFILE)) as fh:
            for line in fh:
                if ":" in line and not line.startswith(("#", " ", "|", "*")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != h.hexdigest():
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}

    def bins(self, width: int = 60):
        """SM clock samples counted in `width`-MHz bins, keyed by the bin's lower edge."""
        out = {}
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            try:
                mhz = float(parts[1])
            except (IndexError, ValueError):
                continue
            lo = int(mhz // width * width)
            out[f"{lo}-{lo + width}"] = out.get(f"{lo}-{lo + width}", 0) + 1
        return dict(sorted(out.items()))


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(total_ms: float, seg_ms, dist, device):
    """The slowest rank's total and per-segment times (every rank gets them);
    unchanged when there is no process group."""
    if dist is None:
        return total_ms, list(seg_ms)
    t = torch.tensor([total_ms] + list(seg_ms), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t[0].item(), t[1:].tolist()


def whole_job_tflops(world: int, steps: int, step_flops: float, total_ms: float) -> float:
    """Weak scaling: every rank runs its own step, so the job does world x steps
    steps in the slowest rank's time."""
    return world * steps * step_flops / (total_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- inputs

def prefill_grids(num_heads, max_q, batch, sms):
    """Grids one prefill attention call launches: tile pairs (head in group x pair x
    sequence x head group) and, for a grid of at most four waves past two whole ones
    whose last wave is partly filled, a second grid of key-split single tiles."""
    per_group = num_heads
    for d in range(8, 3, -1):
        if num_heads > d and num_heads % d == 0:
            per_group = d
            break
    groups = num_heads // per_group
    if batch * groups > 65535:
        per_group, groups = num_heads, 1
    pairs = (-(-max_q // 128) + 1) // 2
    total = per_group * pairs * batch * groups
    tail = total % sms
    return 1 + int(0 < tail and total - tail >= 2 * sms and total <= 4 * sms)


def decode_grids(num_heads, max_q, batch, sms, max_prefix=None):
    """Grids one decode call launches: tile pairs (head x pair x sequence) fill
    whole waves of the SMs.  With a workspace (``max_prefix`` given), a last,
    partly filled wave worth balancing becomes two more grids: its pieces of equal
    key ranges (one range per SM, at least 8 key tiles per range, fewer pairs than
    ranges, and a range plus 16 key tiles shorter than the wave's cost otherwise)
    and their merge.  Otherwise a last wave at most half full becomes a second grid
    of key-split single tiles (two CTAs per pair), each about 0.6 of a pair."""
    pairs = (-(-max_q // 128) + 1) // 2
    items = num_heads * pairs * batch
    tail = items % sms
    if max_prefix is not None and tail > 0:
        nkv = -(-max_prefix // 128) + -(-max_q // 128)
        ranges = min(sms, 256, tail * nkv // 8)
        otherwise = 0.6 * nkv if 2 * tail <= sms else nkv
        if ranges > tail and tail * nkv / ranges + 16 < otherwise:
            return int(items > tail) + 2
    split_from = items - tail if 0 < tail and 2 * tail <= sms else items
    return int(split_from > 0) + int(items > split_from)


class Problem:
    """The workload's tensors, resident on the device (plus pinned host copies for e2e)."""

    def __init__(self, dev, with_host=True, cache="bf16", prologue=False, piecewise=False,
                 separate_append=False,
                 paged=False, workload=WORKLOAD):
        from prefix_kv_gb300 import flops
        from prefix_kv_gb300 import workloads as W
        wl = W.by_name(workload)
        self.wl = wl
        q, k, v = W.make_qkv(wl)
        tr = torch.from_numpy(wl.target_rows())
        self.H = wl.num_heads
        # packed totals, per-sequence maxima, and the first sequence (the CPU sample's)
        self.batch = wl.batch
        self.decode = wl.decode
        self.S, self.max_s = wl.total, max(wl.seq_lens)
        self.N = sum(wl.target_lens()) if wl.decode else 0
        self.P = sum(wl.prefix_lens()) if wl.decode else 0
        self.max_n, self.max_p = max(wl.target_lens()), max(wl.prefix_lens())
        self.S0, self.N0, self.P0 = wl.seq_lens[0], wl.target_lens()[0], wl.prefix_lens()[0]
        self.scale = 1.0 / math.sqrt(128)
        self.host = {
            "q": q, "k": k, "v": v,
            "q_tgt": q[tr].contiguous(), "k_tgt": k[tr].contiguous(), "v_tgt": v[tr].contiguous(),
            "block_id": torch.from_numpy(wl.block_id()),
            "cu": torch.from_numpy(wl.cu_seqlens()),
            "cu_pre": torch.from_numpy(wl.cu_prefix()),
            "cu_tgt": torch.from_numpy(wl.cu_target()),
        }
        if with_host:
            self.pinned = {n: t.pin_memory() for n, t in self.host.items()}
        self.dev = {n: t.to(dev) for n, t in self.host.items()}
        d = self.dev
        self.out = torch.empty_like(d["q"])
        self.lse = torch.empty((self.H, self.S), dtype=torch.float32, device=dev)
        self.dout = torch.empty_like(d["q_tgt"])
        self.dlse = torch.empty((self.H, self.N), dtype=torch.float32, device=dev)
        import prefix_kv_gb300 as bca
        self.cache = cache
        self.fp8_mode = {"bf16": None, "fp8-v": "v", "fp8-kv": "kv"}[cache]
        kdt = torch.uint8 if self.fp8_mode == "kv" else torch.bfloat16
        vdt = torch.bfloat16 if self.fp8_mode is None else torch.uint8
        self.cache_k = torch.empty((1, self.H, self.P, 128), dtype=kdt, device=dev)
        self.cache_v = torch.empty((1, self.H, self.P, 128), dtype=vdt, device=dev)
        # the decode's balanced tail: its partial rows (FP8: after the expanded layers)
        self.tail_bytes = bca.prefix_decode_workspace_bytes(self.batch, self.H, self.max_n,
                                                            self.max_p) if wl.decode else 0
        self.tail_ws = (torch.empty(self.tail_bytes, dtype=torch.uint8, device=dev)
                        if self.tail_bytes else None)
        if self.fp8_mode is not None:
            self.scale_k = torch.empty((1, self.H, self.P), dtype=torch.float32, device=dev)
            self.scale_v = torch.empty_like(self.scale_k)
            self.dec_ws = torch.empty(
                bca.prefix_decode_fp8_workspace_bytes(self.fp8_mode, self.H, self.P) +
                self.tail_bytes, dtype=torch.uint8, device=dev)
        self.ws = torch.empty(bca.prefill_workspace_bytes(self.batch, self.S, self.max_s),
                              dtype=torch.uint8,
                              device=dev)
        self.status = bca.new_status(dev)
        cu = wl.cu_seqlens()
        self.pairs_prefill = flops.prefill_visible_pairs(wl.block_id(), cu, cu)
        self.pairs_decode = (flops.decode_visible_pairs(wl.cu_target(), wl.cu_prefix())
                             if wl.decode else 0)
        self.flops_prefill = flops.attention_flops(self.pairs_prefill, self.H)
        self.flops_decode = flops.attention_flops(self.pairs_decode, self.H)
        rows = self.P * self.H
        if self.fp8_mode is None:
            self.append_bytes = 2 * 2 * rows * 128 * 2           # K and V, read + write
        elif self.fp8_mode == "v":                               # K copied, V quantised
            self.append_bytes = rows * (2 * 256 + 256 + 128 + 4)
        else:                                                    # K and V quantised
            self.append_bytes = rows * 2 * (256 + 128 + 4)
        # kernel launches per step: schedule prep, prefill, append, [expansions], decode
        # (prefill and decode: one grid of tile pairs and, for a short last wave, one of
        # key-split tiles)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.sms = sms
        pre_grids = prefill_grids(self.H, self.max_s, self.batch, sms)
        self.launches = (2 + pre_grids + {None: 0, "v": 1, "kv": 2}[self.fp8_mode] +
                         decode_grids(self.H, self.max_n, self.batch, sms,
                                      self.max_p if self.tail_bytes else None) if wl.decode
                         else 1 + pre_grids)   # prefill only: schedule prep + attention
        # optional Q/K prologue (RMS norm + three-axis RoPE; the prefill-side call also
        # appends): coordinates and rotation table once per layout, outside the step
        self.prologue = prologue
        # paged cache: the prefix's 128-token pages in a shuffled order of a larger pool
        self.paged = paged
        if paged:
            if self.fp8_mode is not None or prologue:
                raise SystemExit("--paged combines with the bf16 cache and no prologue")
            need = [(p_ + 127) // 128 for p_ in wl.prefix_lens()]
            n_pages = sum(need)
            pool_pages = n_pages + n_pages // 2
            perm = np.random.default_rng(11).permutation(pool_pages)[:n_pages].astype(np.int32)
            table = np.full((self.batch, max(need)), -1, dtype=np.int32)
            at = 0
            for b_, n_ in enumerate(need):
                table[b_, :n_] = perm[at:at + n_]
                at += n_
            self.page_table = torch.from_numpy(table).to(dev)
            self.cache_k = torch.empty((1, self.H, pool_pages * 128, 128), dtype=torch.bfloat16,
                                       device=dev)
            self.cache_v = torch.empty_like(self.cache_k)
        # the piecewise baseline: one prefill call per segment (two kernels + a copy each)
        self.piecewise = piecewise
        if piecewise:
            self.bid_host = wl.block_id()
            self.cu_host = wl.cu_seqlens()
            self.pw_ws = torch.empty(bca.prefill_piecewise_workspace_bytes(
                self.bid_host, self.cu_host, self.H), dtype=torch.uint8, device=dev)
            # one schedule prep and one attention call per run of equal ids
            piece_lens = []
            for a, e in zip(self.cu_host[:-1], self.cu_host[1:]):
                if e > a:
                    cuts = np.flatnonzero(np.diff(self.bid_host[a:e])) + 1
                    piece_lens += np.diff(np.concatenate([[0], cuts, [e - a]])).tolist()
            self.launches += (sum(1 + prefill_grids(self.H, int(n), 1, sms) for n in piece_lens)
                              - 1 - pre_grids)
        # the bf16 contiguous cache is written by the prefill launch itself
        # (bca_prefill_append) unless the two separate calls are asked for
        self.fused = (self.decode and self.fp8_mode is None and not piecewise
                      and not prologue and not separate_append)
        if self.fused:
            self.launches -= 1
        # named segments of the step, between consecutive CUDA events
        self.segments = (["prologue", "prefill", "target_prologue", "decode"] if prologue
                         else ["prefill", "append", "decode"])
        if prologue and not self.decode:
            raise SystemExit("--prologue needs a workload with a decode step")
        if prologue:
            if piecewise:
                raise SystemExit("--prologue runs the single-launch prefill; drop --piecewise")
            if self.fp8_mode is not None:
                raise SystemExit("--prologue appends a bf16 cache; combine it with --cache bf16")
            d = self.dev
            gw = torch.from_numpy(wl.grid_widths()).to(dev)
            pos3 = bca.rope_positions(d["block_id"], d["cu"], gw, status=self.status)
            self.table = bca.rope_table(pos3)
            self.table_tgt = self.table[torch.from_numpy(wl.target_rows()).to(dev)].contiguous()
            self.q_rot = torch.empty_like(d["q"])
            self.k_rot = torch.empty_like(d["k"])
            self.qt_rot = torch.empty_like(d["q_tgt"])
            self.kt_rot = torch.empty_like(d["k_tgt"])
            g = torch.Generator("cpu")
            g.manual_seed(5)
            self.gamma_q = (1 + 0.1 * torch.randn(128, generator=g)).to(dev)
            self.gamma_k = (1 + 0.1 * torch.randn(128, generator=g)).to(dev)
            self.launches += 1            # the target-side prologue (the append is fused)
            rows = self.S * self.H
            self.prologue_bytes = (rows * 4 * 256 + self.P * self.H * 3 * 256 + self.S * 512
                                   + self.N * self.H * 4 * 256 + self.N * 512)

    def step(self, d, events=None):
        """The whole path through the binding; `events` = 4 CUDA events to split it."""
        import prefix_kv_gb300 as bca
        if self.prologue:
            return self.step_prologue(d, events)
        if events:
            events[0].record()
        if self.piecewise:
            bca.prefill_piecewise(d["q"], d["k"], d["v"], d["block_id"], self.bid_host,
                                  self.cu_host, self.scale, out=self.out, lse=self.lse,
                                  workspace=self.pw_ws, status=self.status)
        elif self.fused:
            bca.prefill_append(d["q"], d["k"], d["v"], d["block_id"], d["cu"], d["cu"],
                               self.max_s, self.max_s, d["cu_pre"], self.cache_k, self.cache_v,
                               0, self.scale, out=self.out, lse=self.lse, workspace=self.ws,
                               page_table=self.page_table if self.paged else None,
                               status=self.status)
        else:
            bca.prefill(d["q"], d["k"], d["v"], d["block_id"], d["cu"], d["cu"], self.max_s,
                        self.max_s, self.scale, out=self.out, lse=self.lse, workspace=self.ws,
                        status=self.status)
        if events:
            events[1].record()
        if not self.decode:            # prefill-only workload: no cache, no cached step
            if events:
                events[2].record()
                events[3].record()
            return
        if self.fused:
            pass                       # written by the prefill launch
        elif self.paged:
            bca.prefix_cache_append_paged(d["k"], d["v"], d["cu"], d["cu_pre"], self.page_table,
                                          self.cache_k, self.cache_v, 0, status=self.status)
        elif self.fp8_mode is None:
            bca.prefix_cache_append(d["k"], d["v"], d["cu"], d["cu_pre"], self.cache_k,
                                    self.cache_v, 0, status=self.status)
        else:
            bca.prefix_cache_append_fp8(d["k"], d["v"], d["cu"], d["cu_pre"], self.cache_k,
                                        self.cache_v, self.scale_k, self.scale_v, 0,
                                        mode=self.fp8_mode, status=self.status)
        if events:
            events[2].record()
        if self.paged:
            bca.prefix_decode_paged(d["q_tgt"], self.cache_k, self.cache_v, 0, d["cu_pre"],
                                    self.page_table, d["k_tgt"], d["v_tgt"], d["cu_tgt"],
                                    self.max_n, self.max_p, self.scale, out=self.dout, lse=self.dlse,
                                    status=self.status, workspace=self.tail_ws)
        elif self.fp8_mode is None:
            bca.prefix_decode(d["q_tgt"], self.cache_k, self.cache_v, 0, d["cu_pre"], d["k_tgt"],
                              d["v_tgt"], d["cu_tgt"], self.max_n, self.max_p, self.scale, out=self.dout,
                              lse=self.dlse, status=self.status, workspace=self.tail_ws)
        else:
            bca.prefix_decode_fp8(d["q_tgt"], self.cache_k, self.cache_v, self.scale_k,
                                  self.scale_v, 0, d["cu_pre"], d["k_tgt"], d["v_tgt"],
                                  d["cu_tgt"], self.max_n, self.max_p, self.scale, mode=self.fp8_mode,
                                  out=self.dout, lse=self.dlse, workspace=self.dec_ws,
                                  status=self.status)
        if events:
            events[3].record()


def time_standalone_append(prob: "Problem", flush, n: int = 10) -> float:
    """Median ms of bca_prefix_cache_append on the step's inputs.  L2 is emptied before each
    launch by reading a buffer larger than it: a read leaves clean lines, where a write
    would leave dirty ones whose write-back competes with the copy being timed."""
    import prefix_kv_gb300 as bca
    d = prob.dev
    ts = []
    for i in range(n + 2):
        flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if prob.paged:
            bca.prefix_cache_append_paged(d["k"], d["v"], d["cu"], d["cu_pre"], prob.page_table,
                                          prob.cache_k, prob.cache_v, 0, status=prob.status)
        else:
            bca.prefix_cache_append(d["k"], d["v"], d["cu"], d["cu_pre"], prob.cache_k,
                                    prob.cache_v, 0, status=prob.status)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def fp8_decode_psnr(prob: "Problem", dev) -> float:
    """PSNR (dB, peak = max |reference|) of the decode output over the FP8 cache
    against the same decode over a bf16 cache of the same prefix."""
    import prefix_kv_gb300 as bca
    d = prob.dev
    ck = torch.empty((1, prob.H, prob.P, 128), dtype=torch.bfloat16, device=dev)
    cv = torch.empty_like(ck)
    bca.prefix_cache_append(d["k"], d["v"], d["cu"], d["cu_pre"], ck, cv, 0, status=prob.status)
    ref, _ = bca.prefix_decode(d["q_tgt"], ck, cv, 0, d["cu_pre"], d["k_tgt"], d["v_tgt"],
                               d["cu_tgt"], prob.max_n, prob.max_p, prob.scale,
                               status=prob.status)
    prob.step(d)
    torch.cuda.synchronize()
    ref = ref.float()
    mse = (prob.dout.float() - ref).pow(2).mean().item()
    peak = ref.abs().max().item()
    del ck, cv
    return round(10 * math.log10(peak * peak / mse), 2) if mse > 0 else float("inf")


def _prologue_step(self, d, events=None):
    """The step with the Q/K prologue: norm + RoPE + append, prefill on the rotated
    Q/K; norm + RoPE of the target rows, decode over the cache.  Events split it
    into (prologue + prefill, prologue, decode) at the same four marks."""
    import prefix_kv_gb300 as bca
    if events:
        events[0].record()
    bca.qk_norm_rope_append(d["q"], d["k"], self.table, d["cu"], v=d["v"], cu_prefix=d["cu_pre"],
                            cache_k=self.cache_k, cache_v=self.cache_v, layer=0,
                            gamma_q=self.gamma_q, gamma_k=self.gamma_k, q_out=self.q_rot,
                            k_out=self.k_rot, status=self.status)
    if events:
        events[1].record()
    bca.prefill(self.q_rot, self.k_rot, d["v"], d["block_id"], d["cu"], d["cu"], self.max_s,
                self.max_s,
                self.scale, out=self.out, lse=self.lse, workspace=self.ws, status=self.status)
    if events:
        events[2].record()
    bca.qk_norm_rope_append(d["q_tgt"], d["k_tgt"], self.table_tgt, d["cu_tgt"],
                            gamma_q=self.gamma_q, gamma_k=self.gamma_k, q_out=self.qt_rot,
                            k_out=self.kt_rot, status=self.status)
    if events:
        events[3].record()
    bca.prefix_decode(self.qt_rot, self.cache_k, self.cache_v, 0, d["cu_pre"], self.kt_rot,
                      d["v_tgt"], d["cu_tgt"], self.max_n, self.max_p, self.scale, out=self.dout,
                      lse=self.dlse, status=self.status, workspace=self.tail_ws)
    if events:
        events[4].record()


Problem.step_prologue = _prologue_step


# ----------------------------------------------------------------------------- oracle timing

def oracle_sample(prob: "Problem", step_idx: int, target_s: float = 3.0):
    """Time the CPU oracle on a bounded sample of the workload; returns (flops, seconds, desc)."""
    import oracle
    wl, h = prob.wl, step_idx % prob.H
    host = prob.host
    cu = wl.cu_seqlens()
    S = prob.S0                        # rows of the first sequence
    # prefill: blocks of query rows of one head, until about target_s / 2
    from prefix_kv_gb300 import flops
    e_rows = flops.row_ends(wl.block_id()[:S], S)
    t0 = time.perf_counter()
    rows_done, pairs, n = 0, 0, 512
    start = (step_idx * 1543) % S
    while time.perf_counter() - t0 < target_s / 2 and rows_done < S:
        r0 = (start + rows_done) % S
        rows = np.arange(r0, min(S, r0 + n))
        oracle.prefill(host["q"], host["k"], host["v"], wl.block_id(), cu, cu, prob.scale,
                       rows=rows, heads=np.array([h]))
        pairs += int(e_rows[rows].sum())
        rows_done += len(rows)
    t_prefill = time.perf_counter() - t0
    # decode: query rows of the same head
    drows_done, dpairs = 0, 0
    n_dec = prob.N0 if wl.decode else 0
    if "k_pre" not in host and n_dec:
        pr = torch.from_numpy(wl.prefix_rows())
        host = dict(host, k_pre=host["k"][pr].contiguous(), v_pre=host["v"][pr].contiguous())
    t1 = time.perf_counter()
    while time.perf_counter() - t1 < target_s / 2 and drows_done < n_dec:
        rows = np.arange(drows_done, min(n_dec, drows_done + n))
        oracle.prefix_decode(host["q_tgt"], host["k_pre"], host["v_pre"], wl.cu_prefix(),
                             host["k_tgt"], host["v_tgt"], wl.cu_target(), prob.scale,
                             rows=rows, heads=np.array([h]))
        dpairs += len(rows) * (prob.P0 + prob.N0)
        drows_done += len(rows)
    t_decode = time.perf_counter() - t1
    fl = 4.0 * 128 * (pairs + dpairs)
    desc = (f"head {h}: {rows_done} prefill rows + {drows_done} decode rows of {wl.name} "
            f"(float64 NumPy oracle with explicit mask)")
    return fl, t_prefill + t_decode, desc


class HostProblem:
    """The workload's host tensors only (the CPU legs never touch a GPU)."""

    def __init__(self, workload):
        from prefix_kv_gb300 import workloads as W
        wl = W.by_name(workload)
        q, k, v = W.make_qkv(wl)
        tr = torch.from_numpy(wl.target_rows())
        pr = torch.from_numpy(wl.prefix_rows())
        self.wl, self.H, self.S0 = wl, wl.num_heads, wl.seq_lens[0]
        self.N0, self.P0 = wl.target_lens()[0], wl.prefix_lens()[0]
        self.scale = 1.0 / math.sqrt(128)
        self.host = {"q": q, "k": k, "v": v, "q_tgt": q[tr].contiguous(),
                     "k_tgt": k[tr].contiguous(), "v_tgt": v[tr].contiguous(),
                     "k_pre": k[pr].contiguous(), "v_pre": v[pr].contiguous()}


def host_problem(workload):
    return HostProblem(workload)


def oracle_one_thread(workload, seconds):
    """The same oracle sample on one host thread: bench.py runs itself with the BLAS and
    OpenMP thread counts set to 1 (they cannot change once NumPy is loaded)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                            str(seconds), "--workload", workload], env=env,
                           capture_output=True, text=True, timeout=30 * seconds + 120)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": round(d["flops"] / d["seconds"] / 1e12, 6), "unit": UNIT,
                "cores": d["threads"], "seconds": round(d["seconds"], 2),
                "sample": d["sample"]}
    except (subprocess.SubprocessError, ValueError, KeyError, IndexError) as e:
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [i.get("num_threads") for i in info if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    # without threadpoolctl: the thread-count variables BLAS and OpenMP honour, if set
    limits = [int(os.environ[v]) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                                           "MKL_NUM_THREADS")
              if os.environ.get(v, "").isdigit() and int(os.environ[v]) > 0]
    return min(limits) if limits else (os.cpu_count() or 1)


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustained-seconds", type=float, default=3.0,
                    help="length of the sustained leg (steps back to back, L2 not flushed, "
                         "clocks sampled throughout); 0 skips it")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="another config's workload (tiny_mixed_s40, t2i_1024_s4352, "
                         "cfg_edit_4ref_varlen, neo_mixed_32seq); the default is the headline")
    ap.add_argument("--paged", action="store_true",
                    help="prefix cache in 128-token pages of a shuffled page table")
    ap.add_argument("--piecewise", action="store_true",
                    help="baseline: prefill as one attention call per segment")
    ap.add_argument("--prologue", action="store_true",
                    help="add the fused Q/K RMS norm + three-axis RoPE (+ cache append) "
                         "before prefill and decode")
    ap.add_argument("--cache", default="bf16", choices=["bf16", "fp8-v", "fp8-kv"],
                    help="prefix cache format: bf16, or E4M3 with V / K and V quantised")
    ap.add_argument("--separate-append", action="store_true",
                    help="time the cache append as its own launch instead of fused into the "
                         "prefill (bf16 contiguous cache)")
    ap.add_argument("--oracle-sample", type=float, default=None, metavar="SECONDS",
                    help="internal: time one oracle sample on the host, print it as JSON "
                         "and exit (how the one-thread CPU baseline is taken)")
    args = ap.parse_args()

    if args.oracle_sample is not None:
        fl, secs, desc = oracle_sample(host_problem(args.workload), 0, target_s=args.oracle_sample)
        print(json.dumps({"flops": fl, "seconds": secs, "threads": cpu_threads(),
                          "sample": desc}), flush=True)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    peaks = load_peaks()

    if args.impl == "reference":
        return run_reference(args, rank, world, peaks)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if dist is not None:
        dist.barrier()
        build()

    import prefix_kv_gb300 as bca
    prob = Problem(dev, with_host=not args.no_e2e, cache=args.cache, prologue=args.prologue,
                   piecewise=args.piecewise, paged=args.paged, workload=args.workload,
                   separate_append=args.separate_append)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(max(3, args.warmup)):
        prob.step(prob.dev)
    torch.cuda.synchronize()
    code = bca.read_status(prob.status)
    if code != 0:
        raise SystemExit(f"device status {code} after warm-up")

    nseg = len(prob.segments)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)]
           for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()          # L2 flush between timed steps (outside the events)
            prob.step(prob.dev, evs[i])
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    code = bca.read_status(prob.status)
    if code != 0:
        raise SystemExit(f"device status {code} after timed steps")

    seg_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(nseg)]
    tot_ms = sum(e[0].elapsed_time(e[nseg]) for e in evs)
    tot_ms, seg_ms = max_over_ranks(tot_ms, seg_ms, dist, dev)
    seg = dict(zip(prob.segments, seg_ms))
    s_pre, s_dec = seg["prefill"], seg["decode"]
    K = args.steps
    step_flops = prob.flops_prefill + prob.flops_decode
    value = whole_job_tflops(world, K, step_flops, tot_ms)
    pre_tf = prob.flops_prefill / (s_pre / K * 1e-3) / 1e12
    dec_tf = prob.flops_decode / (s_dec / K * 1e-3) / 1e12 if prob.decode else 0.0
    if prob.prologue:
        s_app = seg["prologue"] + seg["target_prologue"]
        app_gbs = prob.prologue_bytes / (s_app / K * 1e-3) / 1e9
    elif prob.fused:
        # the step writes the cache inside the prefill launch; the standalone append
        # kernel is timed on its own (L2 flushed before each launch) for its HBM row
        s_app = K * time_standalone_append(prob, flush)
        app_gbs = prob.append_bytes / (s_app / K * 1e-3) / 1e9
    else:
        s_app = seg["append"]
        app_gbs = prob.append_bytes / (s_app / K * 1e-3) / 1e9 if prob.decode else 0.0

    # ---- sustained: seconds of back-to-back steps, as a model's layers run them -----
    # The timed region above is tens of milliseconds, short enough to finish before
    # the power limit pulls the clocks down.  Here the same step runs back to back
    # (no L2 flush) for a few seconds, timed by one pair of events, with the SM
    # clock sampled every 100 ms; the figure is set against the sustained GEMM peak.
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(10, int(args.sustained_seconds * 1e3 / max(tot_ms / K, 1e-3)))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as sus_clocks:
            ev0.record()
            for _ in range(n_sus):
                prob.step(prob.dev)
            ev1.record()
            torch.cuda.synchronize()
        code = bca.read_status(prob.status)
        if code != 0:
            raise SystemExit(f"device status {code} after the sustained leg")
        sus_ms, _ = max_over_ranks(ev0.elapsed_time(ev1), [], dist, dev)
        sus_tf = whole_job_tflops(world, n_sus, step_flops, sus_ms)
        sustained = {"value": round(sus_tf, 2), "unit": UNIT, "steps": n_sus,
                     "seconds": round(sus_ms / 1e3, 3), "ms_per_step": round(sus_ms / n_sus, 4),
                     "peak": peaks["bf16_sustained"],
                     "frac_of_sustained_peak": round(sus_tf / world / peaks["bf16_sustained"], 4),
                     "frac_of_burst_peak": round(sus_tf / world / peaks["bf16"], 4),
                     "l2": "not flushed (steps back to back)",
                     "clocks": sus_clocks.summary(), "clock_bins_mhz": sus_clocks.bins()}

    # ---- FP8 cache: PSNR of the decode output against a bf16 cache (untimed) ---------
    psnr = None
    if prob.fp8_mode is not None:
        psnr = fp8_decode_psnr(prob, dev)

    # ---- e2e through the public API with host buffers -------------------------------
    # Every step uploads its inputs from pinned host memory and downloads its
    # results.  As a serving loop would, the upload of step i+1 and the download
    # of step i run on copy streams under step i's kernels (inputs and outputs
    # double-buffered on the device); the events bracket all of it.
    e2e = None
    if not args.no_e2e:
        dbuf = [{n: torch.empty_like(t) for n, t in prob.dev.items()} for _ in range(2)]
        out_names = ("out", "lse", "dout", "dlse")
        obuf = [{n: torch.empty_like(getattr(prob, n)) for n in out_names} for _ in range(2)]
        hbuf = [{n: torch.empty(getattr(prob, n).shape, dtype=getattr(prob, n).dtype).pin_memory()
                 for n in out_names} for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in prob.pinned.values())
        d2h = sum(t.numel() * t.element_size() for t in hbuf[0].values())
        keep = {n: getattr(prob, n) for n in out_names}
        cur = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_run(n):
            ready = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            sent = [torch.cuda.Event() for _ in range(n)]
            s_in.wait_stream(cur)
            s_out.wait_stream(cur)
            for i in range(n):
                bi = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(done[i - 2])       # buffer bi's last reader finished
                    for name, t in prob.pinned.items():
                        dbuf[bi][name].copy_(t, non_blocking=True)
                    ready[i].record(s_in)
                cur.wait_event(ready[i])
                if i >= 2:
                    cur.wait_event(sent[i - 2])            # buffer bi's results were downloaded
                for name in out_names:
                    setattr(prob, name, obuf[bi][name])
                prob.step(dbuf[bi])
                done[i].record(cur)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[i])
                    for name in out_names:
                        hbuf[bi][name].copy_(obuf[bi][name], non_blocking=True)
                    sent[i].record(s_out)
            cur.wait_stream(s_out)
            cur.wait_stream(s_in)

        e2e_run(2)
        torch.cuda.synchronize()
        n_e2e = max(3, K // 2)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record()
        e2e_run(n_e2e)
        ev1.record()
        torch.cuda.synchronize()
        for name, t in keep.items():
            setattr(prob, name, t)
        e_ms, _ = max_over_ranks(ev0.elapsed_time(ev1), [], dist, dev)
        e2e = {"value": round(whole_job_tflops(world, n_e2e, step_flops, e_ms), 2),
               "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e_ms / n_e2e, 4), "steps": n_e2e,
               "copies": "upload of step i+1 and download of step i on copy streams under "
                         "step i's kernels, device buffers doubled"}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only) -------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, secs, desc = oracle_sample(prob, 0, target_s=args.cpu_seconds)
        cpu = {"value": round(fl / secs / 1e12, 6), "unit": UNIT, "cores": cpu_threads(),
               "kind": "oracle", "sample": desc, "seconds": round(secs, 2),
               "one_thread": oracle_one_thread(prob.wl.name, args.cpu_seconds / 2)}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    roofline = {"bound": "tensor", "kernel": "bca_prefill (block-causal attention forward)",
                "achieved": round(pre_tf, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(pre_tf / peaks["bf16"], 4),
                "peak_source": f"{peaks['source']} bf16 dense burst",
                "frac_of_sustained": round(pre_tf / peaks["bf16_sustained"], 4),
                "traffic": None if prob.piecewise else profiled_traffic(),
                "traffic_source": ATTN_PROFILE,
                "algorithmic": f"{prob.flops_prefill:.4e} flop per launch "
                               f"({prob.pairs_prefill} visible pairs/head x 32 heads x 512)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(tot_ms / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": prob.wl.name, "batch": prob.batch,
                   "seq_len": prob.wl.seq_lens if prob.batch > 1 else prob.S,
                   "num_heads": prob.H, "head_dim": 128,
                   "prefix_len": (prob.wl.prefix_lens() if prob.batch > 1 else prob.P)
                   if prob.decode else 0,
                   "target_len": (prob.wl.target_lens() if prob.batch > 1 else prob.N)
                   if prob.decode else 0,
                   "step": ("Q/K RMS norm + 3-axis RoPE + cache append, schedule prep + "
                            "prefill, target Q/K norm + RoPE, prefix decode") if prob.prologue
                           else ("piecewise prefill (schedule prep + attention + lse copy per "
                                 "segment) + cache append + prefix decode") if prob.piecewise
                           else ("schedule prep + prefill with the cache append in the same "
                                 "launch + prefix decode") if prob.fused
                           else "schedule prep + prefill + cache append + prefix decode",
                   "prefix_cache_pages": ("128-token pages, shuffled page table" if prob.paged
                                          else "contiguous"),
                   "prefix_cache": {"bf16": "bf16", "fp8-v": "V in FP8 E4M3 (per token-head "
                                    "fp32 scale), K bf16", "fp8-kv": "K and V in FP8 E4M3 "
                                    "(per token-head fp32 scales)"}[args.cache],
                   "l2": "flushed (256 MiB write) between timed steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_bf16_peak": round(100 * value / peaks["bf16"], 2),
        "breakdown": {"prefill_ms": round(s_pre / K, 4), "prefill_tflops": round(pre_tf, 2),
                      ("prologue_ms" if prob.prologue else "append_ms"): round(s_app / K, 4),
                      ("prologue_gbs" if prob.prologue else "append_gbs"): round(app_gbs, 1),
                      ("prologue_frac_of_hbm" if prob.prologue else "append_frac_of_hbm"):
                          round(app_gbs / peaks["hbm"], 4),
                      "decode_ms": round(s_dec / K, 4), "decode_tflops": round(dec_tf, 2),
                      "decode_frac": round(dec_tf / peaks["bf16"], 4),
                      **({"append_in_step": "inside the prefill launch (bca_prefill_append); "
                                            "append_* time the standalone kernel on the same "
                                            "inputs, median of 10 launches, L2 emptied by a "
                                            "256 MiB read before each"}
                         if prob.fused else {})},
        "fp8_decode_psnr_db_vs_bf16_cache": psnr,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "sustained": sustained,
        "gpu_launches": prob.launches * K,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args, rank, world, peaks):
    """The oracle as it stands on the host cores, each step a bounded sample."""
    if rank != 0:
        return
    hp = host_problem(args.workload)   # this leg never touches a GPU
    wl = hp.wl
    for i in range(args.warmup):
        oracle_sample(hp, i, target_s=1.0)
    fl_tot, s_tot, desc = 0.0, 0.0, ""
    for i in range(args.steps):
        fl, secs, desc = oracle_sample(hp, args.warmup + i, target_s=2.0)
        fl_tot += fl
        s_tot += secs
    value = fl_tot / s_tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * s_tot / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "seq_len": wl.seq_lens,
                   "num_heads": hp.H, "head_dim": 128, "prefix_len": wl.prefix_lens(),
                   "target_len": wl.target_lens(),
                   "step": "bounded sample of prefill + prefix decode rows (oracle)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cpu_threads(),
                         "kind": "oracle", "sample": "each step: " + desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
