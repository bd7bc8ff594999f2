"""The bench's visible-pair count agrees with the oracle's explicit mask."""
import numpy as np
import pytest

import oracle
from prefix_kv_gb300 import flops
from prefix_kv_gb300 import workloads as W


def test_tiny_counts():
    wl = W.tiny_mixed()
    cu = wl.cu_seqlens()
    assert flops.prefill_visible_pairs(wl.block_id(), cu, cu) == 1060
    assert flops.decode_visible_pairs(wl.cu_target(), wl.cu_prefix()) == 640


@pytest.mark.parametrize("seed", range(6))
def test_random_layouts_match_oracle(seed):
    rng = np.random.default_rng(seed)
    kv = rng.integers(1, 300, size=3)
    ql = [int(rng.integers(1, L + 1)) for L in kv]
    bids = [np.concatenate([np.full(s.length, s.block) for s in W.random_layout(rng, int(L))])
            for L in kv]
    bid = np.concatenate(bids)
    ck = np.concatenate([[0], np.cumsum(kv)])
    cq = np.concatenate([[0], np.cumsum(ql)])
    assert flops.prefill_visible_pairs(bid, cq, ck) == oracle.visible_pairs(bid, cq, ck)


def test_edit_two_ref_count():
    wl = W.edit_two_ref()
    cu = wl.cu_seqlens()
    n = flops.prefill_visible_pairs(wl.block_id(), cu, cu)
    assert n == oracle.visible_pairs(wl.block_id(), cu, cu) == 103_041_120
    assert flops.decode_visible_pairs(wl.cu_target(), wl.cu_prefix()) == 4096 * 12480
