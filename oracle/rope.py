"""CPU oracle for the Q/K prologue of the attention path: per-head RMS
normalisation, three-axis rotary position embedding and the prefix cache
append of the rotated keys (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the CUDA path never does.  Everything is float64 NumPy,
written as the plain definition: no tables shared with the GPU path, no fusion.

Sources ("Qwen-Image 2.1: Block-Causal Attention, Prefix KV Cache, and Turbo",
flozi.net):
  * the paragraph on the 32 attention heads of width 128: Q and K are
    RMS-normalised per head before RoPE;
  * "Three-axis RoPE preserves image geometry": the 128 dimensions of a head
    are split (16, 56, 56) across the frame, height and width axes with RoPE
    base 10000; text positions advance one shared coordinate on all three
    axes; inside an image block the frame coordinate stays at the position the
    preceding text reached while height and width form a grid centred on zero;
    RoPE changes Q and K, not V, and keeps the cache width at 128;
  * "Timestep-zero conditioning makes the prefix invariant": the cache holds
    the post-RoPE prefix keys (and the values).

Readings where the page is silent (each is listed in the design notes):
  * Coordinates: a running coordinate c starts at 0 in every sequence.  A text
    token takes (c, c, c) and advances c by one.  An image block of Hg x Wg
    tokens, stored row-major (token i at row i // Wg, column i % Wg), takes
    frame c and (row - Hg // 2, column - Wg // 2), then advances c by one.
  * Rotation: the RoFormer rotation of interleaved pairs.  Axis a covers d_a
    consecutive dimensions from offset o_a (0, 16, 72); its pair k (dimensions
    o_a + 2k, o_a + 2k + 1) turns by the angle p_a * 10000^(-2k / d_a):
    (x, y) -> (x cos t - y sin t, x sin t + y cos t).
  * RMS normalisation: y = x / sqrt(mean(x^2) + 1e-6) * gamma over the 128
    values of one (token, head) row, gamma a per-dimension weight (1 if none).
"""
from __future__ import annotations

import numpy as np

AXES = (16, 56, 56)            # frame, height, width
AXIS_OFFSET = (0, 16, 72)
BASE = 10000.0
EPS = 1e-6
HEAD_DIM = 128


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def rope_positions(block_id, cu_seqlens, grid_w) -> np.ndarray:
    """(frame, height, width) coordinates of every packed token, int64 [total, 3].

    ``grid_w[b][i]`` is the width in tokens of image block ``i`` of sequence b;
    the block's length must be a multiple of it (the height is the quotient).
    """
    bid = np.asarray(block_id, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    gw = np.asarray(grid_w, dtype=np.int64)
    pos = np.zeros((len(bid), 3), dtype=np.int64)
    for b in range(len(cu) - 1):
        c = 0
        t = int(cu[b])
        end = int(cu[b + 1])
        while t < end:
            if bid[t] < 0:                      # text: one shared coordinate
                pos[t] = (c, c, c)
                c += 1
                t += 1
                continue
            run_end = t
            while run_end < end and bid[run_end] == bid[t]:
                run_end += 1
            n = run_end - t
            wg = int(gw[b, bid[t]])
            if wg <= 0 or n % wg != 0:
                raise ValueError(f"image block {bid[t]} of sequence {b}: {n} tokens, width {wg}")
            hg = n // wg
            i = np.arange(n)
            pos[t:run_end, 0] = c
            pos[t:run_end, 1] = i // wg - hg // 2
            pos[t:run_end, 2] = i % wg - wg // 2
            c += 1
            t = run_end
    return pos


def rope_angles(pos3) -> np.ndarray:
    """Rotation angle of each of the 64 dimension pairs, float64 [total, 64]."""
    pos = np.asarray(pos3, dtype=np.float64)
    cols = []
    for a, d in enumerate(AXES):
        k = np.arange(d // 2, dtype=np.float64)
        inv_freq = BASE ** (-2.0 * k / d)
        cols.append(pos[:, a:a + 1] * inv_freq[None, :])
    return np.concatenate(cols, axis=1)


def rotate(x, pos3) -> np.ndarray:
    """Apply the three-axis rotation to rows [total, H, 128] (float64 result)."""
    x = _as_f64(x)
    th = rope_angles(pos3)[:, None, :]            # [total, 1, 64]
    c, s = np.cos(th), np.sin(th)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def rms_norm(x, gamma=None, eps: float = EPS) -> np.ndarray:
    """Per-row RMS normalisation over the last axis, times ``gamma`` (float64)."""
    x = _as_f64(x)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x / r
    if gamma is not None:
        y = y * _as_f64(gamma)
    return y


def qk_norm_rope(q, k, gamma_q, gamma_k, pos3, eps: float = EPS):
    """RMS-normalise Q and K per head, then rotate both (float64 results)."""
    return rotate(rms_norm(q, gamma_q, eps), pos3), rotate(rms_norm(k, gamma_k, eps), pos3)


def qk_norm_rope_append(q, k, v, gamma_q, gamma_k, pos3, cu_seqlens, cu_prefix, layer: int,
                        cache_k: np.ndarray, cache_v: np.ndarray, eps: float = EPS):
    """The fused prologue: returns (q_out, k_out) and writes the rotated prefix keys
    and the prefix values of every sequence into ``cache_{k,v}[layer]``
    (``[L][H][cap][128]`` float64 arrays, updated in place)."""
    q_out, k_out = qk_norm_rope(q, k, gamma_q, gamma_k, pos3, eps)
    vf = _as_f64(v)
    ck = np.asarray(cu_seqlens, dtype=np.int64)
    cp = np.asarray(cu_prefix, dtype=np.int64)
    for b in range(len(ck) - 1):
        n = cp[b + 1] - cp[b]
        for t in range(n):
            src = ck[b] + t
            cache_k[layer, :, cp[b] + t, :] = k_out[src]
            cache_v[layer, :, cp[b] + t, :] = vf[src]
    return q_out, k_out
