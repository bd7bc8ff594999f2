"""Seeded synthetic workloads shaped like the single-stream diffusion sequences
described on the Qwen-Image 2.1 pages ("One stream for text, reference images,
and the target"; "Block-causal attention is the cache-enabling boundary") and
the NEO-Unify mixed-mask prefill table ("NEO-Unify 多模态 Prefill 的注意力").

This module only lays out sequences (segment lengths and image-block ids) and
draws seeded random tensors.  It holds none of the attention arithmetic, so the
CPU oracle and the CUDA path can both be fed from it without sharing any of the
method's code.

Tensor recipe: ``torch.Generator('cpu')`` seeded with ``1000 + index``; q, k, v
drawn in that order as fp32 N(0, 1) of shape ``[total, H, 128]``; for the
workloads marked ``rms_norm`` every (token, head) 128-vector of q and k is
divided by ``sqrt(mean(x^2) + 1e-6)`` in fp32; everything is then rounded to
bf16.  Layout draws (only the NEO-style mix has any) use
``numpy.random.default_rng(0)``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

HEAD_DIM = 128
TEXT = -1


@dataclass(frozen=True)
class Segment:
    """A run of positions: text (block id -1) or one image block (id >= 0)."""
    length: int
    block: int = TEXT

    @property
    def is_image(self) -> bool:
        return self.block >= 0


@dataclass
class Workload:
    name: str
    num_heads: int
    seqs: List[List[Segment]]
    rms_norm: bool = False
    decode: bool = True          # last segment of every sequence is the target
    seed: int = 1000
    description: str = ""
    head_dim: int = HEAD_DIM

    # ---- layout -----------------------------------------------------------
    @property
    def seq_lens(self) -> List[int]:
        return [sum(s.length for s in segs) for segs in self.seqs]

    @property
    def batch(self) -> int:
        return len(self.seqs)

    @property
    def total(self) -> int:
        return sum(self.seq_lens)

    def block_id(self) -> np.ndarray:
        out = []
        for segs in self.seqs:
            for s in segs:
                out.append(np.full(s.length, s.block, dtype=np.int32))
        return np.concatenate(out) if out else np.zeros(0, np.int32)

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int32)

    # decode split: prefix = everything before the final (target) segment
    def target_lens(self) -> List[int]:
        return [segs[-1].length for segs in self.seqs]

    def prefix_lens(self) -> List[int]:
        return [L - n for L, n in zip(self.seq_lens, self.target_lens())]

    def cu_target(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.target_lens())]).astype(np.int32)

    def cu_prefix(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.prefix_lens())]).astype(np.int32)

    def target_rows(self) -> np.ndarray:
        """Packed row indices (into the prefill tensors) of every target token."""
        cu = self.cu_seqlens()
        rows = [np.arange(cu[b + 1] - n, cu[b + 1]) for b, n in enumerate(self.target_lens())]
        return np.concatenate(rows).astype(np.int64)

    def grid_widths(self) -> np.ndarray:
        """Width in latent tokens of every image block, int32 ``[batch, n_ids]``
        (0 where a sequence has no such id): square images (4x4, 64x64, 128x128)
        use the side; other spans the largest divisor of their length not above
        its square root."""
        n_ids = 1 + max([s.block for segs in self.seqs for s in segs] + [0])
        out = np.zeros((self.batch, n_ids), dtype=np.int32)
        for b, segs in enumerate(self.seqs):
            for s in segs:
                if s.is_image:
                    out[b, s.block] = image_width(s.length)
        return out

    def prefix_rows(self) -> np.ndarray:
        cu = self.cu_seqlens()
        rows = [np.arange(cu[b], cu[b] + p) for b, p in enumerate(self.prefix_lens())]
        return np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)


def image_width(n: int) -> int:
    """Largest divisor of ``n`` not above sqrt(n) (the side of a square image)."""
    best = 1
    d = 1
    while d * d <= n:
        if n % d == 0:
            best = d
        d += 1
    return best


# ---- tensors -----------------------------------------------------------------

def _rms(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6)


def make_qkv(wl: Workload, seed: Optional[int] = None):
    """q, k, v as bf16 CPU tensors ``[total, H, head_dim]``."""
    g = torch.Generator("cpu")
    g.manual_seed(wl.seed if seed is None else seed)
    shape = (wl.total, wl.num_heads, wl.head_dim)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if wl.rms_norm:
        q, k = _rms(q), _rms(k)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def randn_bf16(shape, seed: int) -> torch.Tensor:
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


# ---- the five workloads --------------------------------------------------------

def tiny_mixed() -> Workload:
    """[text 5][ref image 4x4, block 0][text 3][target 4x4, block 1], 2 heads."""
    return Workload(
        name="tiny_mixed_s40", num_heads=2,
        seqs=[[Segment(5), Segment(16, 0), Segment(3), Segment(16, 1)]],
        seed=1000, description="B=1 H=2 S=40 [t5][img16 id0][t3][img16 id1]")


def t2i_1024() -> Workload:
    """Text-to-image 1024x1024: [text 256][target 64x64 latents, block 0]."""
    return Workload(
        name="t2i_1024_s4352", num_heads=32,
        seqs=[[Segment(256), Segment(4096, 0)]], rms_norm=True,
        seed=1001, description="B=1 H=32 S=4352 [t256][img4096 id0]")


def edit_two_ref() -> Workload:
    """Two-reference edit 1024x1024: [t96][A][t32][B][t64][target], S=12480."""
    return Workload(
        name="edit_2ref_1024_s12480", num_heads=32,
        seqs=[[Segment(96), Segment(4096, 0), Segment(32), Segment(4096, 1),
               Segment(64), Segment(4096, 2)]], rms_norm=True,
        seed=1002, description="B=1 H=32 S=12480; decode Q=4096 over P=8384 + 4096")


def cfg_large_edit() -> Workload:
    """CFG pair of varlen sequences with four 64x64 references and a 128x128 target.

    cond:   [t512][ref0][t24][ref1][t24][ref2][t24][ref3][target 16384, id 4] = 33352
    uncond: [t64][ref0][ref1][ref2][ref3][target 16384, id 4]                = 32832
    (adjacent references keep distinct ids 0..3)
    """
    cond = [Segment(512)]
    for r in range(4):
        if r:
            cond.append(Segment(24))
        cond.append(Segment(4096, r))
    cond.append(Segment(16384, 4))
    uncond = [Segment(64)] + [Segment(4096, r) for r in range(4)] + [Segment(16384, 4)]
    return Workload(name="cfg_edit_4ref_varlen", num_heads=32, seqs=[cond, uncond],
                    seed=1003, description="B=2 H=32 S=33352+32832; decode Q=16384 each")


def neo_mixed(n_seqs: int = 32, lo: int = 2048, hi: int = 8192,
              image_total: int = 536, seed_layout: int = 0) -> Workload:
    """NEO-Unify style packed varlen prefill: text causal, 1-3 image spans per sequence.

    Span counts ~ U{1..3} and lengths ~ U{8..256} are drawn, then shrunk
    proportionally (floor 8) until the batch holds ``image_total`` image tokens
    (within 5%).  Spans are placed at uniform non-overlapping positions with at
    least one text token between two spans; ids are 0.. in order per sequence.
    """
    rng = np.random.default_rng(seed_layout)
    lens = rng.integers(lo, hi + 1, size=n_seqs)
    counts = rng.integers(1, 4, size=n_seqs)
    raw = [rng.integers(8, 257, size=c) for c in counts]
    allraw = np.concatenate(raw).astype(np.float64)

    def shrink(f):
        return [np.maximum(8, np.round(r * f)).astype(np.int64) for r in raw]
    lo_f, hi_f = 0.0, 1.0
    for _ in range(60):
        mid = 0.5 * (lo_f + hi_f)
        if sum(int(s.sum()) for s in shrink(mid)) > image_total:
            hi_f = mid
        else:
            lo_f = mid
    spans = shrink(lo_f)
    tot = sum(int(s.sum()) for s in spans)
    assert abs(tot - image_total) <= 0.05 * image_total, tot
    del allraw

    seqs = []
    for L, sp in zip(lens, spans):
        n = len(sp)
        free = int(L) - int(sp.sum()) - (n - 1)
        gaps = np.sort(rng.integers(0, free + 1, size=n))
        segs: List[Segment] = []
        pos = 0
        for i in range(n):
            start = int(gaps[i]) + int(sp[:i].sum()) + i
            if start > pos:
                segs.append(Segment(start - pos))
            segs.append(Segment(int(sp[i]), i))
            pos = start + int(sp[i])
        if pos < L:
            segs.append(Segment(int(L) - pos))
        seqs.append(segs)
    return Workload(name="neo_mixed_32seq", num_heads=32, seqs=seqs, decode=False,
                    seed=1004, description=f"B={n_seqs} H=32 L~U[{lo},{hi}] image={tot}")


def all_workloads() -> List[Workload]:
    return [tiny_mixed(), t2i_1024(), edit_two_ref(), cfg_large_edit(), neo_mixed()]


def by_name(name: str) -> Workload:
    for w in all_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


def random_layout(rng: np.random.Generator, length: int, max_spans: int = 3,
                  min_span: int = 1, max_span: int = 64, adjacent_ok: bool = True) -> List[Segment]:
    """A random sequence layout for ragged parity cases (seeded by the caller)."""
    segs: List[Segment] = []
    pos, bid = 0, 0
    while pos < length:
        rem = length - pos
        if bid < max_spans and rng.random() < 0.5:
            n = int(min(rem, rng.integers(min_span, max_span + 1)))
            segs.append(Segment(n, bid))
            bid += 1
            if not adjacent_ok and pos + n < length:
                segs.append(Segment(1))
                n += 1
        else:
            n = int(min(rem, rng.integers(1, max_span + 1)))
            segs.append(Segment(n))
        pos += n
    return segs
