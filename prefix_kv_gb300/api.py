"""Python binding of the C ABI (``include/bca.h``), for torch CUDA tensors.

Argument marshalling only: shapes and dtypes are checked, outputs and the
workspace are allocated with torch when not given, raw pointers and the
current CUDA stream are handed to the library.  Every step of the computation
runs in the library's kernels; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
from typing import Optional, Tuple

import torch

from . import _native

HEAD_DIM = 128


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype, dim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {tuple(t.shape)}")


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the ``status_dev`` arguments."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device status code (0 = ok)."""
    return int(_native.load().bca_read_device_status(_ptr(status), _stream(stream)))


def check_status(status: torch.Tensor, where: str = "device", stream=None) -> None:
    _native.check(read_status(status, stream), where)


def prefill_workspace_bytes(batch: int, total_q: int, max_seqlen_q: int) -> int:
    return int(_native.load().bca_prefill_workspace_bytes(batch, total_q, max_seqlen_q))


def schedule_prep(block_id, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, status=None,
                  stream=None, total_q: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-row visible-key ends e(r) and per-tile records ``[B, tiles, 4]``.

    ``total_q`` (the length of the returned ``row_end``) defaults to the last query
    offset; the keys are all of ``block_id``."""
    _need(block_id, "block_id", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    batch = cu_seqlens_q.numel() - 1
    if total_q is None:
        total_q = int(cu_seqlens_q[-1].item()) if batch > 0 else 0
    tiles_per_seq = (max_seqlen_q + 127) // 128
    dev = block_id.device
    row_end = torch.zeros(total_q, dtype=torch.int32, device=dev)
    tiles = torch.zeros((batch, tiles_per_seq, 4), dtype=torch.int32, device=dev)
    code = _native.load().bca_schedule_prep(_ptr(block_id), _ptr(cu_seqlens_q),
                                            _ptr(cu_seqlens_k), batch, total_q,
                                            block_id.numel(), max_seqlen_q, _ptr(row_end),
                                            _ptr(tiles), _ptr(status), _stream(stream))
    _native.check(code, "bca_schedule_prep")
    return row_end, tiles


def prefill(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
            max_seqlen_k: int, softmax_scale: Optional[float] = None, out=None, lse=None,
            workspace=None, status=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-causal attention forward; returns ``(out [total_q, H, 128] bf16, lse [H, total_q] f32)``."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3)
    _need(block_id, "block_id", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    total_q, H, D = q.shape
    total_k = k.shape[0]
    if k.shape != (total_k, H, D) or v.shape != k.shape or block_id.numel() != total_k:
        raise ValueError("k, v, block_id shapes do not match")
    batch = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    ws_bytes = prefill_workspace_bytes(batch, total_q, max_seqlen_q)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    code = _native.load().bca_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(block_id), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        batch, H, D, total_q, total_k, max_seqlen_q, max_seqlen_k, float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _native.check(code, "bca_prefill")
    return out, lse


def prefill_append(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                   max_seqlen_k: int, cu_prefix, cache_k, cache_v, layer: int,
                   softmax_scale: Optional[float] = None, out=None, lse=None, workspace=None,
                   page_table=None, status=None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """``prefill`` with ``prefix_cache_append`` fused in: returns ``(out, lse)`` and writes the
    first ``cu_prefix[b+1]-cu_prefix[b]`` keys/values of every sequence into cache tokens
    ``cu_prefix[b]..`` of ``layer`` (cache ``[L, H, capacity, 128]`` bf16), or, with
    ``page_table [batch, max_pages]``, through it (as ``prefix_cache_append_paged``)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3)
    _need(block_id, "block_id", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    _need(cache_k, "cache_k", torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.bfloat16, 4)
    total_q, H, D = q.shape
    total_k = k.shape[0]
    if k.shape != (total_k, H, D) or v.shape != k.shape or block_id.numel() != total_k:
        raise ValueError("k, v, block_id shapes do not match")
    L, Hc, cap, Dc = cache_k.shape
    if cache_v.shape != cache_k.shape or Hc != H or Dc != D:
        raise ValueError("cache shape does not match q/k/v")
    if not 0 <= layer < L:
        raise ValueError(f"layer {layer} outside [0, {L})")
    batch = cu_seqlens_q.numel() - 1
    if cu_prefix.numel() != batch + 1 or cu_seqlens_k.numel() != batch + 1:
        raise ValueError("cu_prefix / cu_seqlens_k must have batch + 1 entries")
    if page_table is not None:
        _, _, n_pages, _ = _paged_shapes(cache_k, cache_v, page_table)
        if page_table.shape[0] != batch:
            raise ValueError("page_table needs one row per sequence")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    ws_bytes = prefill_workspace_bytes(batch, total_q, max_seqlen_q)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    lib = _native.load()
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(block_id), _ptr(cu_seqlens_q),
            _ptr(cu_seqlens_k), batch, H, D, total_q, total_k, max_seqlen_q, max_seqlen_k,
            float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(cu_prefix))
    if page_table is None:
        code = lib.bca_prefill_append(*args, _ptr(cache_k), _ptr(cache_v), layer, L, cap,
                                      _ptr(status), _stream(stream))
        _native.check(code, "bca_prefill_append")
    else:
        code = lib.bca_prefill_append_paged(*args, _ptr(page_table), page_table.shape[1],
                                            _ptr(cache_k), _ptr(cache_v), layer, L, n_pages,
                                            _ptr(status), _stream(stream))
        _native.check(code, "bca_prefill_append_paged")
    return out, lse


def prefix_decode_workspace_bytes(batch: int, num_heads: int, max_seqlen_q: int, max_prefix: int,
                                  head_dim: int = 128) -> int:
    """Bytes of the decode workspace that enables the balanced tail (0: none needed)."""
    return int(_native.load().bca_prefix_decode_workspace_bytes(batch, num_heads, head_dim,
                                                                max_seqlen_q, max_prefix))


def _tail_workspace(workspace, balanced_tail: bool, batch: int, H: int, max_seqlen_q: int,
                    max_prefix: int, D: int, device, extra: int = 0):
    """The caller's workspace, or one allocated here: ``extra`` bytes for the FP8
    decodes' bf16 layers, then the balanced tail's slots when ``balanced_tail``."""
    if workspace is not None:
        return workspace
    tail = prefix_decode_workspace_bytes(batch, H, max_seqlen_q, max_prefix, D) \
        if balanced_tail else 0
    if extra + tail == 0:
        return None
    return torch.empty(extra + tail, dtype=torch.uint8, device=device)


def prefix_decode(q_tgt, cache_k, cache_v, layer: int, cu_prefix, k_tgt, v_tgt, cu_seqlens_q,
                  max_seqlen_q: int, max_prefix: int, softmax_scale: Optional[float] = None,
                  out=None, lse=None, status=None, stream=None, workspace=None,
                  balanced_tail: bool = True):
    """Target queries over [cached prefix; own K/V], no mask.  Cache ``[L, H, cap, 128]``.

    ``workspace``: a device uint8 tensor of ``prefix_decode_workspace_bytes`` bytes for
    the balanced tail, allocated here when omitted; ``balanced_tail=False`` (and no
    workspace) runs the key-split tail instead."""
    for name, t in (("q_tgt", q_tgt), ("k_tgt", k_tgt), ("v_tgt", v_tgt)):
        _need(t, name, torch.bfloat16, 3)
    _need(cache_k, "cache_k", torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.bfloat16, 4)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    total_q, H, D = q_tgt.shape
    L, Hc, cap, Dc = cache_k.shape
    if (Hc, Dc) != (H, D) or cache_v.shape != cache_k.shape:
        raise ValueError("cache shape does not match q_tgt")
    if k_tgt.shape != q_tgt.shape or v_tgt.shape != q_tgt.shape:
        raise ValueError("k_tgt / v_tgt shapes do not match q_tgt")
    batch = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q_tgt)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q_tgt.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    workspace = _tail_workspace(workspace, balanced_tail, batch, H, max_seqlen_q, max_prefix, D,
                                q_tgt.device)
    code = _native.load().bca_prefix_decode(
        _ptr(q_tgt), _ptr(cache_k), _ptr(cache_v), layer, L, cap, _ptr(cu_prefix), _ptr(k_tgt),
        _ptr(v_tgt), _ptr(cu_seqlens_q), batch, H, D, total_q, max_seqlen_q, max_prefix,
        float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_decode")
    return out, lse


def prefix_cache_append(k, v, cu_seqlens_k, cu_prefix, cache_k, cache_v, layer: int,
                        status=None, stream=None) -> None:
    """Clone each sequence's prefix K/V into ``cache_{k,v}[layer]`` (``[L, H, cap, 128]``)."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    _need(cache_k, "cache_k", torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.bfloat16, 4)
    total_k, H, D = k.shape
    L, Hc, cap, Dc = cache_k.shape
    if (Hc, Dc) != (H, D) or cache_v.shape != cache_k.shape or v.shape != k.shape:
        raise ValueError("shapes do not match")
    batch = cu_seqlens_k.numel() - 1
    code = _native.load().bca_prefix_cache_append(
        _ptr(k), _ptr(v), _ptr(cu_seqlens_k), _ptr(cu_prefix), batch, H, D, total_k,
        _ptr(cache_k), _ptr(cache_v), layer, L, cap, _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_cache_append")


FP8_MODES = {"v": 1, "kv": 2}


def prefix_cache_append_fp8(k, v, cu_seqlens_k, cu_prefix, cache_k, cache_v, scale_k, scale_v,
                            layer: int, mode: str = "v", status=None, stream=None) -> None:
    """Quantising append into an FP8 E4M3 cache.

    mode "v": cache_k bf16 ``[L, H, cap, 128]``, cache_v uint8 codes, scale_v fp32
    ``[L, H, cap]`` (scale_k may be None).  mode "kv": cache_k and cache_v uint8
    codes, scale_k and scale_v fp32.
    """
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    m = FP8_MODES[mode]
    _need(cache_k, "cache_k", torch.uint8 if mode == "kv" else torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.uint8, 4)
    _need(scale_v, "scale_v", torch.float32, 3)
    if mode == "kv":
        _need(scale_k, "scale_k", torch.float32, 3)
    total_k, H, D = k.shape
    L, Hc, cap, Dc = cache_v.shape
    if (Hc, Dc) != (H, D) or tuple(cache_k.shape) != tuple(cache_v.shape) or \
            tuple(scale_v.shape) != (L, H, cap):
        raise ValueError("cache shapes do not match")
    if mode == "kv" and tuple(scale_k.shape) != (L, H, cap):
        raise ValueError("scale_k shape does not match the cache")
    batch = cu_seqlens_k.numel() - 1
    code = _native.load().bca_prefix_cache_append_fp8(
        _ptr(k), _ptr(v), _ptr(cu_seqlens_k), _ptr(cu_prefix), batch, H, D, total_k, m,
        _ptr(cache_k), _ptr(cache_v), _ptr(scale_k), _ptr(scale_v), layer, L, cap, _ptr(status),
        _stream(stream))
    _native.check(code, "bca_prefix_cache_append_fp8")


def prefix_decode_fp8_workspace_bytes(mode: str, num_heads: int, capacity: int,
                                      head_dim: int = 128) -> int:
    return int(_native.load().bca_prefix_decode_fp8_workspace_bytes(FP8_MODES[mode], num_heads,
                                                                    head_dim, capacity))


def prefix_cache_dequant_fp8(codes, scales, cu_prefix, layer: int, out=None, status=None,
                             stream=None):
    """bf16 ``[H, cap, 128]`` expansion of rows ``cu_prefix[0]..cu_prefix[-1]`` of one
    layer of an E4M3 cache (codes uint8 ``[L, H, cap, 128]``, scales fp32 ``[L, H, cap]``)."""
    _need(codes, "codes", torch.uint8, 4)
    _need(scales, "scales", torch.float32, 3)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    L, H, cap, D = codes.shape
    if tuple(scales.shape) != (L, H, cap):
        raise ValueError("scales shape does not match the codes")
    if out is None:
        out = torch.empty((H, cap, D), dtype=torch.bfloat16, device=codes.device)
    _need(out, "out", torch.bfloat16, 3)
    if tuple(out.shape) != (H, cap, D):
        raise ValueError("out must be [H, cap, 128]")
    code = _native.load().bca_prefix_cache_dequant_fp8(
        _ptr(codes), _ptr(scales), _ptr(cu_prefix), cu_prefix.numel() - 1, H, D, layer, L, cap,
        _ptr(out), _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_cache_dequant_fp8")
    return out


def prefix_decode_fp8(q_tgt, cache_k, cache_v, scale_k, scale_v, layer: int, cu_prefix, k_tgt,
                      v_tgt, cu_seqlens_q, max_seqlen_q: int, max_prefix: int,
                      softmax_scale: Optional[float] = None, mode: str = "v", out=None, lse=None,
                      workspace=None, status=None, stream=None, balanced_tail: bool = True):
    """``prefix_decode`` over an FP8 E4M3 cache written by ``prefix_cache_append_fp8``
    in the same ``mode`` (cache and scale layouts as there).  ``workspace``: a
    device uint8 tensor of ``prefix_decode_fp8_workspace_bytes`` bytes, plus
    ``prefix_decode_workspace_bytes`` for the balanced tail (allocated here when
    omitted)."""
    for name, t in (("q_tgt", q_tgt), ("k_tgt", k_tgt), ("v_tgt", v_tgt)):
        _need(t, name, torch.bfloat16, 3)
    m = FP8_MODES[mode]
    _need(cache_k, "cache_k", torch.uint8 if mode == "kv" else torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.uint8, 4)
    _need(scale_v, "scale_v", torch.float32, 3)
    if mode == "kv":
        _need(scale_k, "scale_k", torch.float32, 3)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    total_q, H, D = q_tgt.shape
    L, Hc, cap, Dc = cache_v.shape
    if (Hc, Dc) != (H, D) or tuple(cache_k.shape) != tuple(cache_v.shape) or \
            tuple(scale_v.shape) != (L, H, cap) or \
            (mode == "kv" and tuple(scale_k.shape) != (L, H, cap)):
        raise ValueError("cache shapes do not match q_tgt")
    if k_tgt.shape != q_tgt.shape or v_tgt.shape != q_tgt.shape:
        raise ValueError("k_tgt / v_tgt shapes do not match q_tgt")
    batch = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q_tgt)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q_tgt.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    workspace = _tail_workspace(workspace, balanced_tail, batch, H, max_seqlen_q, max_prefix, D,
                                q_tgt.device, prefix_decode_fp8_workspace_bytes(mode, H, cap, D))
    code = _native.load().bca_prefix_decode_fp8(
        _ptr(q_tgt), _ptr(cache_k), _ptr(cache_v), m, _ptr(scale_k) if mode == "kv" else None,
        _ptr(scale_v), layer, L, cap, _ptr(cu_prefix), _ptr(k_tgt), _ptr(v_tgt),
        _ptr(cu_seqlens_q), batch, H, D, total_q, max_seqlen_q, max_prefix,
        float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_decode_fp8")
    return out, lse


def rope_positions(block_id, cu_seqlens, grid_w, status=None, stream=None):
    """(frame, height, width) RoPE coordinates, int32 ``[total, 3]``.

    ``grid_w``: int32 ``[batch, n_ids]`` width in tokens of image block ``i`` of
    sequence ``b`` (entries of absent ids are not read)."""
    _need(block_id, "block_id", torch.int32, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(grid_w, "grid_w", torch.int32, 2)
    total = block_id.numel()
    batch = cu_seqlens.numel() - 1
    if grid_w.shape[0] != batch:
        raise ValueError("grid_w must have one row per sequence")
    pos3 = torch.empty((total, 3), dtype=torch.int32, device=block_id.device)
    code = _native.load().bca_rope_positions(_ptr(block_id), _ptr(cu_seqlens), batch, total,
                                             _ptr(grid_w), grid_w.shape[1], _ptr(pos3),
                                             _ptr(status), _stream(stream))
    _native.check(code, "bca_rope_positions")
    return pos3


def rope_table(pos3, stream=None):
    """fp32 ``[total, 64, 2]`` (cos, sin) of every token's 64 dimension pairs."""
    _need(pos3, "pos3", torch.int32, 2)
    total = pos3.shape[0]
    table = torch.empty((total, 64, 2), dtype=torch.float32, device=pos3.device)
    code = _native.load().bca_rope_table(_ptr(pos3), total, _ptr(table), _stream(stream))
    _native.check(code, "bca_rope_table")
    return table


def qk_norm_rope_append(q, k, table, cu_seqlens, v=None, cu_prefix=None, cache_k=None,
                        cache_v=None, layer: int = 0, gamma_q=None, gamma_k=None,
                        eps: float = 1e-6, q_out=None, k_out=None, status=None, stream=None):
    """RMS-normalise and rotate Q and K (``[total, H, 128]`` bf16); with ``cu_prefix``
    also write the rotated prefix keys and the values into ``cache_{k,v}[layer]``.
    Returns ``(q_out, k_out)``; pass ``q_out=q, k_out=k`` to work in place."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(table, "table", torch.float32, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    total, H, D = q.shape
    if k.shape != q.shape or tuple(table.shape) != (total, 64, 2):
        raise ValueError("q, k and table shapes do not match")
    for name, g in (("gamma_q", gamma_q), ("gamma_k", gamma_k)):
        if g is not None:
            _need(g, name, torch.float32, 1)
    L, cap = 1, 0
    if cu_prefix is not None:
        _need(cu_prefix, "cu_prefix", torch.int32, 1)
        _need(v, "v", torch.bfloat16, 3)
        _need(cache_k, "cache_k", torch.bfloat16, 4)
        _need(cache_v, "cache_v", torch.bfloat16, 4)
        L, Hc, cap, Dc = cache_k.shape
        if (Hc, Dc) != (H, D) or cache_v.shape != cache_k.shape or v.shape != q.shape:
            raise ValueError("cache / v shapes do not match q")
    if q_out is None:
        q_out = torch.empty_like(q)
    if k_out is None:
        k_out = torch.empty_like(k)
    batch = cu_seqlens.numel() - 1
    code = _native.load().bca_qk_norm_rope_append(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _ptr(table), _ptr(cu_seqlens),
        _ptr(cu_prefix), batch, H, D, total, float(eps), _ptr(q_out), _ptr(k_out),
        _ptr(cache_k), _ptr(cache_v), layer, L, cap, _ptr(status), _stream(stream))
    _native.check(code, "bca_qk_norm_rope_append")
    return q_out, k_out


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def prefill_piecewise_workspace_bytes(block_id_host, cu_seqlens_host, num_heads: int) -> int:
    bid, cu = _host_i32(block_id_host), _host_i32(cu_seqlens_host)
    return int(_native.load().bca_prefill_piecewise_workspace_bytes(
        bid.ctypes.data, cu.ctypes.data, len(cu) - 1, num_heads))


def prefill_piecewise(q, k, v, block_id, block_id_host, cu_seqlens_host,
                      softmax_scale: Optional[float] = None, out=None, lse=None, workspace=None,
                      status=None, stream=None):
    """Block-causal prefill as one attention call per segment (the piecewise baseline);
    same results as ``prefill`` for square sequences.  ``block_id_host`` and
    ``cu_seqlens_host`` are host copies (NumPy or CPU tensors) of the ids and offsets."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3)
    _need(block_id, "block_id", torch.int32, 1)
    bid, cu = _host_i32(block_id_host), _host_i32(cu_seqlens_host)
    total, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or bid.shape[0] != total:
        raise ValueError("shapes do not match")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        workspace = torch.empty(prefill_piecewise_workspace_bytes(bid, cu, H), dtype=torch.uint8,
                                device=q.device)
    code = _native.load().bca_prefill_piecewise(
        _ptr(q), _ptr(k), _ptr(v), _ptr(block_id), bid.ctypes.data, cu.ctypes.data, len(cu) - 1,
        H, D, total, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel(), _ptr(status), _stream(stream))
    _native.check(code, "bca_prefill_piecewise")
    return out, lse


# ---- paged prefix cache ---------------------------------------------------------------

PAGE_TOKENS = 128


class PagePool:
    """Host-side page pool (``bca_pool_*``): page ids with references, a hash index
    of published full pages, and reuse of idle cached pages.  The K/V data live in
    cache tensors ``[L, H, num_pages * 128, 128]``."""

    def __init__(self, num_pages: int):
        self._lib = _native.load()
        self.num_pages = num_pages
        self._h = self._lib.bca_pool_create(num_pages)
        if not self._h:
            raise ValueError("num_pages must be positive")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.bca_pool_destroy(h)

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), dtype=np.int32)
        _native.check(self._lib.bca_pool_alloc(self._h, n, out.ctypes.data), "bca_pool_alloc")
        return out[:n]

    def match(self, hashes) -> np.ndarray:
        hs = np.ascontiguousarray(np.asarray(hashes, dtype=np.uint64))
        out = np.zeros(max(len(hs), 1), dtype=np.int32)
        n = self._lib.bca_pool_match(self._h, hs.ctypes.data, len(hs), out.ctypes.data)
        return out[:n]

    def publish(self, page: int, h: int) -> None:
        _native.check(self._lib.bca_pool_publish(self._h, int(page), int(h)), "bca_pool_publish")

    def release(self, pages) -> None:
        p = np.ascontiguousarray(np.asarray(pages, dtype=np.int32))
        _native.check(self._lib.bca_pool_release(self._h, p.ctypes.data, len(p)),
                      "bca_pool_release")

    def stats(self) -> Tuple[int, int, int]:
        """(free pages, idle cached pages, referenced pages)."""
        a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._lib.bca_pool_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        return a.value, b.value, c.value

    def refs(self, page: int) -> int:
        return int(self._lib.bca_pool_refs(self._h, int(page)))


def _paged_shapes(cache_k, cache_v, page_table):
    _need(cache_k, "cache_k", torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    L, H, cap, D = cache_k.shape
    if cache_v.shape != cache_k.shape or cap % PAGE_TOKENS:
        raise ValueError("paged cache must be [L, H, num_pages * 128, 128]")
    return L, H, cap // PAGE_TOKENS, D


def prefix_cache_append_paged(k, v, cu_seqlens_k, cu_prefix, page_table, cache_k, cache_v,
                              layer: int, status=None, stream=None) -> None:
    """``prefix_cache_append`` into a paged cache through ``page_table [batch, max_pages]``."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    L, H, n_pages, D = _paged_shapes(cache_k, cache_v, page_table)
    total_k = k.shape[0]
    batch = cu_seqlens_k.numel() - 1
    code = _native.load().bca_prefix_cache_append_paged(
        _ptr(k), _ptr(v), _ptr(cu_seqlens_k), _ptr(cu_prefix), _ptr(page_table),
        page_table.shape[1], batch, H, D, total_k, _ptr(cache_k), _ptr(cache_v), layer, L,
        n_pages, _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_cache_append_paged")


def prefix_decode_paged(q_tgt, cache_k, cache_v, layer: int, cu_prefix, page_table, k_tgt, v_tgt,
                        cu_seqlens_q, max_seqlen_q: int, max_prefix: int,
                        softmax_scale: Optional[float] = None, out=None, lse=None, status=None,
                        stream=None, workspace=None, balanced_tail: bool = True):
    """``prefix_decode`` with the prefix read through ``page_table`` (``workspace`` and
    ``balanced_tail`` as there)."""
    for name, t in (("q_tgt", q_tgt), ("k_tgt", k_tgt), ("v_tgt", v_tgt)):
        _need(t, name, torch.bfloat16, 3)
    _need(cu_prefix, "cu_prefix", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    L, H, n_pages, D = _paged_shapes(cache_k, cache_v, page_table)
    total_q = q_tgt.shape[0]
    batch = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q_tgt)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q_tgt.device)
    workspace = _tail_workspace(workspace, balanced_tail, batch, H, max_seqlen_q, max_prefix, D,
                                q_tgt.device)
    code = _native.load().bca_prefix_decode_paged(
        _ptr(q_tgt), _ptr(cache_k), _ptr(cache_v), layer, L, n_pages, _ptr(cu_prefix),
        _ptr(page_table), page_table.shape[1], _ptr(k_tgt), _ptr(v_tgt), _ptr(cu_seqlens_q),
        batch, H, D, total_q, max_seqlen_q, max_prefix, float(softmax_scale), _ptr(out),
        _ptr(lse), _ptr(workspace), 0 if workspace is None else workspace.numel(), _ptr(status),
        _stream(stream))
    _native.check(code, "bca_prefix_decode_paged")
    return out, lse


def pool_copy_rows(cache_k, cache_v, layer: int, src_page: int, dst_page: int, n_rows: int,
                   stream=None) -> None:
    """Copy rows ``[0, n_rows)`` of one page to another (all heads, K and V, one layer)."""
    _need(cache_k, "cache_k", torch.bfloat16, 4)
    L, H, cap, D = cache_k.shape
    code = _native.load().bca_pool_copy_rows(_ptr(cache_k), _ptr(cache_v), layer, L, H,
                                             cap // PAGE_TOKENS, src_page, dst_page, n_rows,
                                             _stream(stream))
    _native.check(code, "bca_pool_copy_rows")


def prefix_cache_append_fp8_paged(k, v, cu_seqlens_k, cu_prefix, page_table, cache_k, cache_v,
                                  scale_k, scale_v, layer: int, mode: str = "v", status=None,
                                  stream=None) -> None:
    """``prefix_cache_append_fp8`` into a paged cache (``[L, H, num_pages * 128, 128]``
    codes, ``[L, H, num_pages * 128]`` scales) through ``page_table``."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(page_table, "page_table", torch.int32, 2)
    m = FP8_MODES[mode]
    _need(cache_k, "cache_k", torch.uint8 if mode == "kv" else torch.bfloat16, 4)
    _need(cache_v, "cache_v", torch.uint8, 4)
    _need(scale_v, "scale_v", torch.float32, 3)
    if mode == "kv":
        _need(scale_k, "scale_k", torch.float32, 3)
    L, H, cap, D = cache_v.shape
    if cap % PAGE_TOKENS or tuple(cache_k.shape) != tuple(cache_v.shape) or \
            tuple(scale_v.shape) != (L, H, cap):
        raise ValueError("paged FP8 cache shapes do not match")
    batch = cu_seqlens_k.numel() - 1
    code = _native.load().bca_prefix_cache_append_fp8_paged(
        _ptr(k), _ptr(v), _ptr(cu_seqlens_k), _ptr(cu_prefix), _ptr(page_table),
        page_table.shape[1], batch, H, D, k.shape[0], m, _ptr(cache_k), _ptr(cache_v),
        _ptr(scale_k) if mode == "kv" else None, _ptr(scale_v), layer, L, cap // PAGE_TOKENS,
        _ptr(status), _stream(stream))
    _native.check(code, "bca_prefix_cache_append_fp8_paged")


def prefix_decode_fp8_paged(q_tgt, cache_k, cache_v, scale_k, scale_v, layer: int, cu_prefix,
                            page_table, prefix_rows: int, k_tgt, v_tgt, cu_seqlens_q,
                            max_seqlen_q: int, max_prefix: int,
                            softmax_scale: Optional[float] = None, mode: str = "v", out=None,
                            lse=None, workspace=None, status=None, stream=None,
                            balanced_tail: bool = True):
    """Decode over a paged FP8 cache: gather (+ dequantise) the prefixes into a
    workspace packed by ``cu_prefix`` (``prefix_rows >= cu_prefix[-1]``), then
    the contiguous decode (its balanced tail in the workspace's remaining bytes)."""
    for name, t in (("q_tgt", q_tgt), ("k_tgt", k_tgt), ("v_tgt", v_tgt)):
        _need(t, name, torch.bfloat16, 3)
    m = FP8_MODES[mode]
    _need(cache_v, "cache_v", torch.uint8, 4)
    _need(page_table, "page_table", torch.int32, 2)
    L, H, cap, D = cache_v.shape
    total_q = q_tgt.shape[0]
    batch = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q_tgt)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q_tgt.device)
    lib = _native.load()
    workspace = _tail_workspace(workspace, balanced_tail, batch, H, max_seqlen_q, max_prefix, D,
                                q_tgt.device,
                                lib.bca_prefix_decode_fp8_paged_workspace_bytes(H, D, prefix_rows))
    code = lib.bca_prefix_decode_fp8_paged(
        _ptr(q_tgt), _ptr(cache_k), _ptr(cache_v), m, _ptr(scale_k) if mode == "kv" else None,
        _ptr(scale_v), layer, L, cap // PAGE_TOKENS, _ptr(cu_prefix), _ptr(page_table),
        page_table.shape[1], prefix_rows, _ptr(k_tgt), _ptr(v_tgt), _ptr(cu_seqlens_q), batch, H,
        D, total_q, max_seqlen_q, max_prefix, float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), 0 if workspace is None else workspace.numel(), _ptr(status),
        _stream(stream))
    _native.check(code, "bca_prefix_decode_fp8_paged")
    return out, lse
