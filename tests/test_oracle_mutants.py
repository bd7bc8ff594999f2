"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Every mutant is applied with ``monkeypatch`` to the oracle module only for the
duration of one test; the real oracle is never modified.
"""
import numpy as np
import pytest

import oracle.attention as orc
from oracle_pins import ALL_PINS

_real_visibility = orc.visibility
_real_masked_attention = orc.masked_attention
_real_lse = orc._logsumexp_rows
_real_decode = orc.prefix_decode
_real_cache_append = orc.cache_append


def _vis_variant(causal_op="ge", text_matches_text=False, image_clause=True):
    def vis(block_id_seq, q_len=None, rows=None):
        bid = np.asarray(block_id_seq, dtype=np.int64)
        L = bid.shape[0]
        q_len = L if q_len is None else q_len
        p = orc.query_positions(q_len, L, rows)
        j = np.arange(L)
        bq = bid[p]
        causal = (p[:, None] >= j[None]) if causal_op == "ge" else (p[:, None] > j[None])
        same = bq[:, None] == bid[None, :]
        if not text_matches_text:
            same &= bq[:, None] >= 0
        return causal | same if image_clause else causal
    return vis


_real_piece_mask = orc.piece_mask

MUTANTS = {
    "piecewise_text_top_left": ("piece_mask",
                                lambda is_text, q_len, kv_len:
                                np.tril(np.ones((q_len, kv_len), dtype=bool))
                                if is_text else _real_piece_mask(is_text, q_len, kv_len)),
    "top_left_alignment": ("query_positions",
                           lambda q_len, kv_len, rows=None:
                           np.arange(q_len) if rows is None else np.asarray(rows)),
    "strict_causal": ("visibility", _vis_variant(causal_op="gt")),
    "text_matches_text": ("visibility", _vis_variant(text_matches_text=True)),
    "no_image_clause": ("visibility", _vis_variant(image_clause=False)),
    "transposed_mask": ("visibility",
                        lambda b, q_len=None, rows=None:
                        _real_visibility(b, q_len, rows).T
                        if (q_len is None or q_len == len(b)) and rows is None
                        else _real_visibility(b, q_len, rows)),
    "lse_log2": ("_logsumexp_rows", lambda s: _real_lse(s) / np.log(2.0)),
    "no_max_subtraction": ("_logsumexp_rows",
                           lambda s: np.log(np.sum(np.exp(s), axis=1))),
    "scale_dropped": ("masked_attention",
                      lambda q, k, v, m, scale: _real_masked_attention(q, k, v, m, 1.0)),
    "value_transposed_rows": ("masked_attention",
                              lambda q, k, v, m, scale:
                              _real_masked_attention(q, k, v[::-1], m, scale)),
    "decode_drops_target_keys": ("prefix_decode",
                                 lambda qt, kp, vp, cp, kt, vt, cq, sc, rows=None, heads=None:
                                 _decode_prefix_only(qt, kp, vp, cp, cq, sc)),
    "append_off_by_one": ("cache_append",
                          lambda k, v, ck, cp, cK, cV, layer:
                          _real_cache_append(k[1:], v[1:], ck, cp, cK, cV, layer)),
}


def _decode_prefix_only(qt, kp, vp, cp, cq, sc):
    qt = np.asarray(qt, dtype=np.float64)
    H, D = qt.shape[1], qt.shape[2]
    out = np.zeros_like(qt)
    lse = np.zeros((H, qt.shape[0]))
    for b in range(len(cq) - 1):
        for h in range(H):
            q = qt[cq[b]:cq[b + 1], h]
            k, v = np.asarray(kp)[cp[b]:cp[b + 1], h], np.asarray(vp)[cp[b]:cp[b + 1], h]
            o, l = _real_masked_attention(q, k, v, np.ones((q.shape[0], k.shape[0]), bool), sc)
            out[cq[b]:cq[b + 1], h] = o
            lse[h, cq[b]:cq[b + 1]] = l
    return out, lse


def _failing_pins():
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(orc, attr, fn)
    failed = _failing_pins()
    assert failed, f"mutant {name} passed every pin"


def test_real_oracle_passes_every_pin():
    assert _failing_pins() == []
