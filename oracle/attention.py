"""CPU oracle for block-causal attention with a prefix K/V cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this module.  The
product path (the CUDA library and its Python binding) never calls it.

Everything here is the plain definition of what the path computes, written out
in float64 NumPy with an explicit boolean visibility mask.  There is no tiling,
no online softmax and no reordering beyond what the definition states.

Sources (page title, section):
  * Qwen-Image 2.1 deployment notes (10100.com), "Block-Causal mask":
    ``visible = (query_position >= key_position) or same_image_block``; text is
    causal, each image block is internally bidirectional and sees everything
    before it, but nothing after it.
  * Same page, piecewise-attention paragraph: when Q is shorter than K/V the
    causal mask is bottom-right aligned, ``ones(q_len, kv_len).tril(kv_len - q_len)``.
  * "Qwen-Image 2.1: Block-Causal Attention, Prefix KV Cache, and Turbo"
    (flozi.net), "Block-causal attention is the cache-enabling boundary":
    block id -1 for text, a unique non-negative id per image (adjacent
    references keep distinct ids).
  * Same page, "Timestep-zero conditioning makes the prefix invariant":
    cached steps run only the target queries over [cached prefix K/V, target
    K/V] with no mask; the cache stores a clone of the post-RoPE prefix slices.
  * Same page, "The prefix cache is a compute-for-memory trade": the cache holds
    K and V per layer and head, 128 values per token.

Readings where the pages are silent (each is listed in the design notes):
  * ``same_image_block`` means both ids are >= 0 and equal; text never matches
    text.  The rule is evaluated literally, even for ids that are not one
    contiguous run.
  * Bottom-right alignment for block-causal rows: query i of a sequence with
    q_len queries and kv_len keys sits at key position ``kv_len - q_len + i``
    and takes that position's block id.
  * LSE is the natural log of the sum of exp over the *scaled* visible scores,
    laid out ``[H, total_q]``.
  * Cache layout ``[layer][head][token][head_dim]``; sequence b's prefix lands
    at cache tokens ``cu_prefix[b] .. cu_prefix[b+1]`` and is the first
    ``cu_prefix[b+1] - cu_prefix[b]`` keys of that sequence.
"""
from __future__ import annotations

import numpy as np

ROW_CHUNK = 1024


def _f64(x) -> np.ndarray:
    """Accept NumPy arrays or (CPU) torch tensors of any float dtype."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if hasattr(x, "float"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# the mask
# ---------------------------------------------------------------------------

def query_positions(q_len: int, kv_len: int, rows=None) -> np.ndarray:
    """Key-axis position of each query: bottom-right alignment."""
    i = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    return (kv_len - q_len) + i


def visibility(block_id_seq, q_len: int | None = None, rows=None) -> np.ndarray:
    """Boolean mask ``[rows, kv_len]`` of one sequence.

    ``M[i, j] = (p_i >= j) or (bid[p_i] >= 0 and bid[p_i] == bid[j])``
    with ``p_i = kv_len - q_len + i``.
    """
    bid = _i64(block_id_seq)
    kv_len = bid.shape[0]
    if q_len is None:
        q_len = kv_len
    p = query_positions(q_len, kv_len, rows)
    j = np.arange(kv_len)
    bq = bid[p]
    causal = p[:, None] >= j[None, :]
    same_block = (bq[:, None] >= 0) & (bq[:, None] == bid[None, :])
    return causal | same_block


# ---------------------------------------------------------------------------
# attention over an explicit mask
# ---------------------------------------------------------------------------

def _logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """ln sum_j exp(s_ij), stable; rows with no visible key give -inf."""
    m = np.max(s, axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    return m_safe + np.log(np.sum(np.exp(s - m_safe[:, None]), axis=1))


def masked_attention(q, k, v, mask, scale: float):
    """softmax(scale * q k^T, masked) v for one head.

    q [n, D], k and v [L, D], mask [n, L] -> (out [n, D], lse [n]).
    """
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    lse = _logsumexp_rows(s)
    p = np.exp(s - lse[:, None])
    return p @ v, lse


def prefill(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, softmax_scale: float,
            rows=None, heads=None):
    """Block-causal attention over packed varlen sequences.

    q ``[total_q, H, D]``; k, v ``[total_k, H, D]``; block_id ``[total_k]``;
    cu_seqlens ``[B+1]``.  ``rows`` (packed query indices) and ``heads`` select a
    sample; by default every row and head is computed.

    Returns ``out [n_rows, n_heads, D]`` and ``lse [n_heads, n_rows]`` (float64).
    """
    bid = _i64(block_id)
    cq, ck = _i64(cu_seqlens_q), _i64(cu_seqlens_k)
    H, D = q.shape[1], q.shape[2]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = np.arange(H) if heads is None else np.asarray(heads, dtype=np.int64)
    out = np.zeros((rows.shape[0], heads.shape[0], D))
    lse = np.zeros((heads.shape[0], rows.shape[0]))
    seq_of_row = np.searchsorted(cq, rows, side="right") - 1
    for b in np.unique(seq_of_row):
        sel = np.nonzero(seq_of_row == b)[0]
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        local = rows[sel] - q0
        for hi, h in enumerate(heads):
            kh, vh = _f64(k[k0:k1, h]), _f64(v[k0:k1, h])   # float64 per (sequence, head)
            for c in range(0, sel.shape[0], ROW_CHUNK):
                part = sel[c:c + ROW_CHUNK]
                mask = visibility(bid[k0:k1], q1 - q0, local[c:c + ROW_CHUNK])
                o, l = masked_attention(_f64(q[rows[part], h]), kh, vh, mask, softmax_scale)
                out[part, hi] = o
                lse[hi, part] = l
    return out, lse


def piece_mask(is_text: bool, q_len: int, kv_len: int) -> np.ndarray:
    """Mask of one piece: a text piece is causal over itself, bottom-right aligned
    (``ones(q_len, kv_len).tril(kv_len - q_len)``); an image piece sees every key."""
    if is_text:
        return np.tril(np.ones((q_len, kv_len), dtype=bool), kv_len - q_len)
    return np.ones((q_len, kv_len), dtype=bool)


def prefill_piecewise(q, k, v, block_id, cu_seqlens, softmax_scale: float):
    """Block-causal prefill as separate exact attention calls, one per segment.

    Qwen-Image 2.1 deployment notes, piecewise-attention paragraph, and flozi
    "Two exact attention paths": the default diffusers processor runs one
    attention call for every text or image segment of the prefix and one for
    the target.  The queries of segment [a, e) of a sequence starting at s
    attend over keys [s, e): a text segment with its causal triangle
    (bottom-right aligned), an image segment (the target included) with no
    mask.  Square sequences only (every query has its own key).  Returns
    ``out [total, H, D]`` and ``lse [H, total]`` (float64).
    """
    bid = _i64(block_id)
    cu = _i64(cu_seqlens)
    total, H, D = q.shape
    out = np.zeros((total, H, D))
    lse = np.zeros((H, total))
    for b in range(len(cu) - 1):
        s, end = cu[b], cu[b + 1]
        a = s
        while a < end:
            e = a + 1
            while e < end and bid[e] == bid[a]:
                e += 1
            mask = piece_mask(bid[a] < 0, e - a, e - s)
            for h in range(H):
                o, l = masked_attention(_f64(q[a:e, h]), _f64(k[s:e, h]), _f64(v[s:e, h]), mask,
                                        softmax_scale)
                out[a:e, h] = o
                lse[h, a:e] = l
            a = e
    return out, lse


def prefix_decode(q_tgt, k_prefix, v_prefix, cu_prefix, k_tgt, v_tgt, cu_seqlens_q,
                  softmax_scale: float, rows=None, heads=None):
    """Cached-step attention: target queries over [prefix K/V; target K/V], no mask.

    q_tgt, k_tgt, v_tgt ``[total_q, H, D]`` packed by ``cu_seqlens_q``;
    k_prefix, v_prefix ``[total_prefix, H, D]`` packed by ``cu_prefix``.
    Returns ``out [n_rows, n_heads, D]`` and ``lse [n_heads, n_rows]``.
    """
    cq, cp = _i64(cu_seqlens_q), _i64(cu_prefix)
    H, D = q_tgt.shape[1], q_tgt.shape[2]
    rows = np.arange(q_tgt.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = np.arange(H) if heads is None else np.asarray(heads, dtype=np.int64)
    out = np.zeros((rows.shape[0], heads.shape[0], D))
    lse = np.zeros((heads.shape[0], rows.shape[0]))
    seq_of_row = np.searchsorted(cq, rows, side="right") - 1
    for b in np.unique(seq_of_row):
        sel = np.nonzero(seq_of_row == b)[0]
        for hi, h in enumerate(heads):
            kk = np.concatenate([_f64(k_prefix[cp[b]:cp[b + 1], h]), _f64(k_tgt[cq[b]:cq[b + 1], h])])
            vv = np.concatenate([_f64(v_prefix[cp[b]:cp[b + 1], h]), _f64(v_tgt[cq[b]:cq[b + 1], h])])
            for c in range(0, sel.shape[0], ROW_CHUNK):
                part = sel[c:c + ROW_CHUNK]
                mask = np.ones((part.shape[0], kk.shape[0]), dtype=bool)
                o, l = masked_attention(_f64(q_tgt[rows[part], h]), kk, vv, mask, softmax_scale)
                out[part, hi] = o
                lse[hi, part] = l
    return out, lse


# ---------------------------------------------------------------------------
# the prefix cache
# ---------------------------------------------------------------------------

def cache_append(k, v, cu_seqlens_k, cu_prefix, cache_k, cache_v, layer: int):
    """Clone each sequence's prefix K/V into the ``[layer][head][token][D]`` cache.

    Sequence b's first ``cu_prefix[b+1] - cu_prefix[b]`` keys go to cache tokens
    ``cu_prefix[b] ..``.  ``cache_k``/``cache_v`` are NumPy arrays updated in
    place and returned.
    """
    ck, cp = _i64(cu_seqlens_k), _i64(cu_prefix)
    kk, vv = np.asarray(k), np.asarray(v)
    for b in range(ck.shape[0] - 1):
        n = cp[b + 1] - cp[b]
        for t in range(n):
            for h in range(kk.shape[1]):
                cache_k[layer, h, cp[b] + t, :] = kk[ck[b] + t, h, :]
                cache_v[layer, h, cp[b] + t, :] = vv[ck[b] + t, h, :]
    return cache_k, cache_v


def visible_pairs(block_id, cu_seqlens_q, cu_seqlens_k) -> int:
    """Number of visible (query, key) pairs per head, counted from the mask."""
    bid, cq, ck = _i64(block_id), _i64(cu_seqlens_q), _i64(cu_seqlens_k)
    total = 0
    for b in range(cq.shape[0] - 1):
        q_len, (k0, k1) = cq[b + 1] - cq[b], (ck[b], ck[b + 1])
        for c in range(0, q_len, ROW_CHUNK):
            r = np.arange(c, min(q_len, c + ROW_CHUNK))
            total += int(visibility(bid[k0:k1], q_len, r).sum())
    return total
