"""CPU oracle for the paged prefix cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the CUDA path never does.

Source: SenseNova-U1 / Prism-Infer inference notes (the Prism-Infer section on
prefix KV reuse): the KV cache lives in a pool of pages; requests with a common
prefix share its pages; a shared tail page is copied for its common rows only.
Reading (listed in the design notes): a page holds 128 consecutive prefix
tokens of one sequence for every head of one layer, i.e. one layer's pool is a
cache of capacity num_pages * 128 tokens, ``pool[layer][head][page * 128 + slot]``;
sequence b's prefix token t lives in page ``page_table[b][t // 128]`` at slot
``t % 128``.  The prefix of sequence b is its first ``cu_prefix[b+1] -
cu_prefix[b]`` keys and values (as in the contiguous cache).
"""
from __future__ import annotations

import numpy as np

from .attention import prefix_decode

PAGE_TOKENS = 128


def page_slot(page_table, b: int, t: int) -> int:
    """Cache token (page * 128 + slot) of prefix token t of sequence b."""
    return int(page_table[b][t // PAGE_TOKENS]) * PAGE_TOKENS + t % PAGE_TOKENS


def paged_append(k, v, cu_seqlens_k, cu_prefix, page_table, layer: int, pool_k, pool_v):
    """Write every sequence's prefix keys/values into its pages (in place)."""
    kf = k.detach().cpu().float().numpy() if hasattr(k, "detach") else np.asarray(k)
    vf = v.detach().cpu().float().numpy() if hasattr(v, "detach") else np.asarray(v)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    cp = np.asarray(cu_prefix, dtype=np.int64)
    for b in range(len(ck) - 1):
        for t in range(int(cp[b + 1] - cp[b])):
            c = page_slot(page_table, b, t)
            pool_k[layer, :, c] = kf[ck[b] + t]
            pool_v[layer, :, c] = vf[ck[b] + t]


def paged_gather(pool, cu_prefix, page_table, layer: int) -> np.ndarray:
    """The packed prefixes ``[sum P_b, H, D]`` read back through the page table."""
    cp = np.asarray(cu_prefix, dtype=np.int64)
    rows = []
    for b in range(len(cp) - 1):
        for t in range(int(cp[b + 1] - cp[b])):
            rows.append(pool[layer, :, page_slot(page_table, b, t)])
    H, D = pool.shape[1], pool.shape[3]
    return np.stack(rows) if rows else np.zeros((0, H, D))


def paged_prefix_decode(q_tgt, pool_k, pool_v, cu_prefix, page_table, layer: int, k_tgt, v_tgt,
                        cu_seqlens_q, softmax_scale: float, rows=None, heads=None):
    """Cached-step attention with the prefix read through the page table."""
    kp = paged_gather(pool_k, cu_prefix, page_table, layer)
    vp = paged_gather(pool_v, cu_prefix, page_table, layer)
    return prefix_decode(q_tgt, kp, vp, cu_prefix, k_tgt, v_tgt, cu_seqlens_q, softmax_scale,
                         rows=rows, heads=heads)
