"""Work counts for the throughput metric (host side, NumPy).

Only visible (query, key) pairs are counted: a prefill row r sees the key
prefix [0, e(r)) (e = p+1 for text, the end of the image run for an image
token), a decode row sees all P + N keys of its sequence.  Each visible pair
costs 2*D flops in Q K^T and 2*D in P V, so FLOPs = 4 * D * H * pairs.
"""
from __future__ import annotations

import numpy as np


def row_ends(block_id_seq, q_len: int) -> np.ndarray:
    """e(r) for the q_len query rows of one sequence (bottom-right aligned)."""
    kb = np.asarray(block_id_seq, dtype=np.int64)
    L = kb.shape[0]
    end = np.arange(1, L + 1, dtype=np.int64)              # text: p + 1
    img = kb >= 0
    if img.any():
        # exclusive end of each image run, propagated backwards over the run
        change = np.ones(L, dtype=bool)
        change[:-1] = kb[1:] != kb[:-1]
        run_end = np.where(change, np.arange(1, L + 1), L + 1)
        run_end = np.minimum.accumulate(run_end[::-1])[::-1]
        end = np.where(img, run_end, end)
    return end[L - q_len:]


def prefill_visible_pairs(block_id, cu_seqlens_q, cu_seqlens_k) -> int:
    """Sum over query rows of e(r), per head."""
    bid = np.asarray(block_id, dtype=np.int64)
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    total = 0
    for b in range(len(cq) - 1):
        n = int(cq[b + 1] - cq[b])
        if n > 0:
            total += int(row_ends(bid[ck[b]:ck[b + 1]], n).sum())
    return total


def decode_visible_pairs(cu_seqlens_q, cu_prefix) -> int:
    cq = np.diff(np.asarray(cu_seqlens_q, dtype=np.int64))
    cp = np.diff(np.asarray(cu_prefix, dtype=np.int64))
    return int((cq * (cp + cq)).sum())


def attention_flops(pairs: int, num_heads: int, head_dim: int = 128) -> float:
    return 4.0 * head_dim * num_heads * pairs
