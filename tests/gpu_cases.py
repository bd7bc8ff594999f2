"""Shared helpers for the GPU parity tests: running the CUDA path through the
binding and comparing it with the CPU oracle at the stated tolerances.

Tolerances (bf16 output, fp32 LSE): max |out - ref| <= 2e-2, mean |out - ref|
<= 2e-3, |lse - ref| <= 1e-3 * max(1, |ref|).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W

OUT_MAX, OUT_MEAN, LSE_REL = 2e-2, 2e-3, 1e-3
SCALE = 1.0 / math.sqrt(128)
DEV = "cuda"


def assert_close(out, lse, ref_out, ref_lse, rows=None, heads=None, what=""):
    o = out.float().cpu().numpy() if isinstance(out, torch.Tensor) else out
    l = lse.float().cpu().numpy() if isinstance(lse, torch.Tensor) else lse
    if rows is not None:
        o, l = o[rows], l[:, rows]
    if heads is not None:
        o, l = o[:, heads], l[heads]
    assert o.shape == ref_out.shape and l.shape == ref_lse.shape
    assert np.isfinite(o).all() and np.isfinite(l).all(), what
    err = np.abs(o - ref_out)
    rel = np.abs(l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))
    assert err.max() <= OUT_MAX, f"{what}: out max err {err.max():.3e}"
    assert err.mean() <= OUT_MEAN, f"{what}: out mean err {err.mean():.3e}"
    assert rel.max() <= LSE_REL, f"{what}: lse rel err {rel.max():.3e}"
    return float(err.max()), float(err.mean()), float(rel.max())


class PrefillCase:
    """Packed varlen prefill inputs on the CPU (bf16) and their device copies."""

    def __init__(self, q, k, v, block_id, cu_q, cu_k):
        self.q, self.k, self.v = q, k, v
        self.block_id = np.asarray(block_id, dtype=np.int32)
        self.cu_q = np.asarray(cu_q, dtype=np.int32)
        self.cu_k = np.asarray(cu_k, dtype=np.int32)
        self.max_q = int(np.diff(self.cu_q).max()) if len(self.cu_q) > 1 else 0
        self.max_k = int(np.diff(self.cu_k).max()) if len(self.cu_k) > 1 else 0

    @classmethod
    def from_workload(cls, wl):
        q, k, v = W.make_qkv(wl)
        cu = wl.cu_seqlens()
        return cls(q, k, v, wl.block_id(), cu, cu)

    def run(self, status=None, out=None):
        d = lambda t: t.to(DEV)
        ti = lambda a: torch.from_numpy(a).to(DEV)
        return bca.prefill(d(self.q), d(self.k), d(self.v), ti(self.block_id), ti(self.cu_q),
                           ti(self.cu_k), self.max_q, self.max_k, SCALE, status=status, out=out)

    def reference(self, rows=None, heads=None):
        return oracle.prefill(self.q, self.k, self.v, self.block_id, self.cu_q, self.cu_k, SCALE,
                              rows=rows, heads=heads)


def ragged_case(seed, kv_lens, q_lens=None, heads=3, **layout_kw):
    """Random block-causal layouts per sequence; q_len <= kv_len uses bottom-right rows."""
    rng = np.random.default_rng(seed)
    q_lens = kv_lens if q_lens is None else q_lens
    bids = []
    for L in kv_lens:
        segs = W.random_layout(rng, L, **layout_kw)
        bids.append(np.concatenate([np.full(s.length, s.block, np.int32) for s in segs])
                    if L > 0 else np.zeros(0, np.int32))
    cu_k = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = W.randn_bf16((int(cu_q[-1]), heads, 128), seed * 3 + 1)
    k = W.randn_bf16((int(cu_k[-1]), heads, 128), seed * 3 + 2)
    v = W.randn_bf16((int(cu_k[-1]), heads, 128), seed * 3 + 3)
    return PrefillCase(q, k, v, np.concatenate(bids), cu_q, cu_k)


def tile_boundary_rows(cu, extra=0, seed=0):
    """Every query row of the first/last 128-row tile of each sequence, the rows
    around each tile edge, plus `extra` seeded random rows."""
    rows = set()
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        rows.update(range(a, min(e, a + 128)))
        rows.update(range(max(a, e - 128), e))
        for t in range(a + 128, e, 128):
            rows.update((t - 1, t))
    rng = np.random.default_rng(seed)
    if extra and cu[-1] > 0:
        rows.update(rng.integers(0, int(cu[-1]), size=extra).tolist())
    return np.array(sorted(rows), dtype=np.int64)


class DecodeCase:
    """Prefix decode inputs: packed prefix K/V laid into a [L, H, cap, 128] cache."""

    def __init__(self, q_tgt, k_tgt, v_tgt, k_pre, v_pre, cu_q, cu_pre, layers=1, layer=0,
                 capacity=None, cache_fill=0.0):
        self.q_tgt, self.k_tgt, self.v_tgt = q_tgt, k_tgt, v_tgt
        self.k_pre, self.v_pre = k_pre, v_pre
        self.cu_q = np.asarray(cu_q, dtype=np.int32)
        self.cu_pre = np.asarray(cu_pre, dtype=np.int32)
        self.layers, self.layer = layers, layer
        H = q_tgt.shape[1]
        cap = int(self.cu_pre[-1]) + 64 if capacity is None else capacity
        self.capacity = cap
        # test plumbing: lay the packed prefix into the cache layout with torch indexing
        ck = torch.full((layers, H, cap, 128), cache_fill, dtype=torch.bfloat16)
        cv = torch.full((layers, H, cap, 128), cache_fill, dtype=torch.bfloat16)
        n = int(self.cu_pre[-1])
        ck[layer, :, :n] = k_pre.permute(1, 0, 2)
        cv[layer, :, :n] = v_pre.permute(1, 0, 2)
        self.cache_k, self.cache_v = ck, cv
        self.max_q = int(np.diff(self.cu_q).max())
        self.max_pre = int(np.diff(self.cu_pre).max())

    @classmethod
    def from_workload(cls, wl, **kw):
        q, k, v = W.make_qkv(wl)
        tr, pr = wl.target_rows(), wl.prefix_rows()
        return cls(q[tr].contiguous(), k[tr].contiguous(), v[tr].contiguous(),
                   k[pr].contiguous(), v[pr].contiguous(), wl.cu_target(), wl.cu_prefix(), **kw)

    def run(self, status=None, balanced_tail=True, workspace=None, max_pre=None, out=None,
            lse=None):
        d = lambda t: t.to(DEV)
        ti = lambda a: torch.from_numpy(a).to(DEV)
        return bca.prefix_decode(d(self.q_tgt), d(self.cache_k), d(self.cache_v), self.layer,
                                 ti(self.cu_pre), d(self.k_tgt), d(self.v_tgt), ti(self.cu_q),
                                 self.max_q, self.max_pre if max_pre is None else max_pre, SCALE,
                                 status=status, balanced_tail=balanced_tail, workspace=workspace,
                                 out=out, lse=lse)

    def reference(self, rows=None, heads=None):
        return oracle.prefix_decode(self.q_tgt, self.k_pre, self.v_pre, self.cu_pre, self.k_tgt,
                                    self.v_tgt, self.cu_q, SCALE, rows=rows, heads=heads)
