"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` takes the oracle module and raises ``AssertionError`` when the
oracle disagrees with a fact that does not come from the oracle itself: a
fixture typed from the pages' worked examples, a closed form, a library routine
for a special case the method reduces to, an invariant the pages state, or a
brute-force enumeration using a different formulation of the rule.

``test_oracle_pins.py`` runs every pin on the real oracle; the mutant tests run
them on deliberately broken copies to show each plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

from conftest import load_golden

D = 128
SCALE = 1.0 / math.sqrt(D)


def _rng_arrays(seed, *shapes):
    r = np.random.default_rng(seed)
    return [r.standard_normal(s) for s in shapes]


def _prefix_form_mask(bid, q_len):
    """Visibility as the key prefix [0, e(p)): e = p+1 for text, the end of the
    image run containing p for an image token (valid when every id >= 0 forms a
    single contiguous run).  Written from the page's remark that an image block
    [a, b) sees everything before it plus its own block."""
    L = len(bid)
    end = np.zeros(L, dtype=np.int64)
    j = L - 1
    while j >= 0:
        if bid[j] < 0:
            end[j] = j + 1
            j -= 1
            continue
        k = j
        while k - 1 >= 0 and bid[k - 1] == bid[j]:
            k -= 1
        end[k:j + 1] = j + 1
        j = k - 1
    m = np.zeros((q_len, L), dtype=bool)
    for i in range(q_len):
        p = L - q_len + i
        m[i, :end[p]] = True
    return m


def _segments_mask(lengths_ids):
    """Mask from the segment description (one row band per segment)."""
    L = sum(n for n, _ in lengths_ids)
    m = np.zeros((L, L), dtype=bool)
    a = 0
    for n, bid in lengths_ids:
        for r in range(a, a + n):
            if bid < 0:
                m[r, :r + 1] = True          # causal text
            else:
                m[r, :a + n] = True          # everything before + own block
        a += n
    return m


def _torch64(x):
    return torch.from_numpy(np.ascontiguousarray(x))


# ---------------------------------------------------------------------------
# the mask
# ---------------------------------------------------------------------------

def pin_worked_example_mask(orc):
    rows = load_golden("mask_t0t1_refA_t2_targetB.txt")
    bid = np.array(rows[0])
    expect = np.array(rows[1:], dtype=bool)
    got = orc.visibility(bid)
    assert got.shape == expect.shape and (got == expect).all(), got.astype(int)


def pin_bottom_right(orc):
    rows = load_golden("bottom_right_q3_kv8.txt")
    q_len, kv_len = rows[0]
    expect = np.array(rows[1:], dtype=bool)
    # the closed form printed on the page
    assert (expect == np.tril(np.ones((q_len, kv_len)), kv_len - q_len).astype(bool)).all()
    got = orc.visibility(np.full(kv_len, -1), q_len)
    assert (got == expect).all(), got.astype(int)
    # top-left alignment (tril(0)) would cut almost the whole prefix
    assert not (got == np.tril(np.ones((q_len, kv_len))).astype(bool)).all()


def pin_tiny_layout(orc):
    """[t5][ref 16, id 0][t3][target 16, id 1]: pair count and the page's bullets."""
    bid = np.array([-1] * 5 + [0] * 16 + [-1] * 3 + [1] * 16)
    m = orc.visibility(bid)
    # 1+..+5 text, 16 ref rows x 21, 22+23+24 text, 16 target rows x 40
    assert int(m.sum()) == 15 + 16 * 21 + (22 + 23 + 24) + 16 * 40 == 1060
    ref, t2, tgt = slice(5, 21), slice(21, 24), slice(24, 40)
    assert not m[ref, t2].any() and not m[ref, tgt].any()   # ref cannot read later text / target
    assert m[t2, ref].all()                                  # later text reads the reference
    assert m[tgt].all()                                      # target reads everything
    assert m[ref, ref].all()                                 # bidirectional inside the block
    assert (m == _segments_mask([(5, -1), (16, 0), (3, -1), (16, 1)])).all()


def pin_adjacent_references(orc):
    """Adjacent references keep distinct ids; the earlier must not read the later."""
    bid = np.array([-1, -1, 0, 0, 0, 1, 1, 1, -1])
    m = orc.visibility(bid)
    assert not m[2:5, 5:8].any()
    assert m[5:8, 2:8].all()
    merged = np.array([-1, -1, 0, 0, 0, 0, 0, 0, -1])
    assert orc.visibility(merged)[2:5, 5:8].all()


def _valid_layouts(n, max_id=3):
    """All id strings of length n over {-1, 0..max_id-1} where every id >= 0 is
    one contiguous run (the pages' unique-id-per-image layout)."""
    for ids in itertools.product(range(-1, max_id), repeat=n):
        ok = True
        for b in range(max_id):
            pos = [i for i, x in enumerate(ids) if x == b]
            if pos and pos[-1] - pos[0] + 1 != len(pos):
                ok = False
                break
        if ok:
            yield np.array(ids)


def pin_brute_force_small(orc):
    """Every valid layout up to length 6, every q_len: rule == prefix form."""
    count = 0
    for n in range(1, 7):
        for bid in _valid_layouts(n):
            for q_len in range(1, n + 1):
                got = orc.visibility(bid, q_len)
                assert (got == _prefix_form_mask(bid, q_len)).all(), (bid, q_len)
                count += 1
    assert count > 1000


# ---------------------------------------------------------------------------
# attention values
# ---------------------------------------------------------------------------

def pin_zero_query_closed_form(orc):
    """q = 0: every visible score is 0, so lse = ln(#visible) and out = mean of visible v."""
    bid = np.array([-1] * 3 + [0] * 4 + [-1] * 2 + [1] * 5 + [2] * 3 + [-1])
    L, H = len(bid), 2
    (k, v) = _rng_arrays(1, (L, H, D), (L, H, D))
    q = np.zeros((L, H, D))
    cu = np.array([0, L])
    out, lse = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    m = _prefix_form_mask(bid, L)
    for h in range(H):
        for i in range(L):
            cnt = m[i].sum()
            assert abs(lse[h, i] - math.log(cnt)) < 1e-12
            assert np.allclose(out[i, h], v[m[i], h].mean(axis=0), atol=1e-12)


def pin_causal_text_equals_sdpa(orc):
    """All-text prefill is plain causal attention (torch SDPA, float64)."""
    L, H = 37, 3
    q, k, v = _rng_arrays(2, (L, H, D), (L, H, D), (L, H, D))
    cu = np.array([0, L])
    out, lse = orc.prefill(q, k, v, np.full(L, -1), cu, cu, SCALE)
    tq, tk, tv = (_torch64(x).permute(1, 0, 2) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=SCALE)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    s = torch.einsum("hid,hjd->hij", tq, tk) * SCALE
    s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), -math.inf)
    assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def pin_single_block_equals_full(orc):
    """One image block spanning the sequence is unmasked attention."""
    L, H = 29, 2
    q, k, v = _rng_arrays(3, (L, H, D), (L, H, D), (L, H, D))
    cu = np.array([0, L])
    out, lse = orc.prefill(q, k, v, np.zeros(L, dtype=np.int64), cu, cu, SCALE)
    tq, tk, tv = (_torch64(x).permute(1, 0, 2) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, scale=SCALE)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    s = torch.einsum("hid,hjd->hij", tq, tk) * SCALE
    assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def pin_decode_equals_full(orc):
    """Decode is unmasked attention over [prefix; target] (two sequences)."""
    H = 2
    P, N = [7, 19], [5, 11]
    kp, vp = _rng_arrays(4, (sum(P), H, D), (sum(P), H, D))
    qt, kt, vt = _rng_arrays(5, (sum(N), H, D), (sum(N), H, D), (sum(N), H, D))
    cp, cq = np.array([0, 7, 26]), np.array([0, 5, 16])
    out, lse = orc.prefix_decode(qt, kp, vp, cp, kt, vt, cq, SCALE)
    for b in range(2):
        kk = np.concatenate([kp[cp[b]:cp[b + 1]], kt[cq[b]:cq[b + 1]]])
        vv = np.concatenate([vp[cp[b]:cp[b + 1]], vt[cq[b]:cq[b + 1]]])
        tq, tk, tv = (_torch64(x).permute(1, 0, 2)
                      for x in (qt[cq[b]:cq[b + 1]], kk, vv))
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=SCALE)
        assert np.allclose(out[cq[b]:cq[b + 1]], ref.permute(1, 0, 2).numpy(), atol=1e-12)
        s = torch.einsum("hid,hjd->hij", tq, tk) * SCALE
        assert np.allclose(lse[:, cq[b]:cq[b + 1]], torch.logsumexp(s, -1).numpy(), atol=1e-12)


def pin_large_scores_stable(orc):
    """Scores of magnitude ~1e3 (beyond exp overflow) stay finite and match a stable library logsumexp."""
    L, H = 16, 1
    q, k, v = _rng_arrays(6, (L, H, D), (L, H, D), (L, H, D))
    q *= 400.0
    bid = np.array([-1] * 4 + [0] * 8 + [-1] * 4)
    cu = np.array([0, L])
    out, lse = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    m = torch.from_numpy(_prefix_form_mask(bid, L))
    s = torch.einsum("id,jd->ij", _torch64(q[:, 0]), _torch64(k[:, 0])) * SCALE
    s = s.masked_fill(~m, -math.inf)
    assert np.allclose(lse[0], torch.logsumexp(s, -1).numpy(), rtol=1e-13)
    ref = torch.softmax(s, -1) @ _torch64(v[:, 0])
    assert np.allclose(out[:, 0], ref.numpy(), atol=1e-12)


def pin_constant_values(orc):
    """v constant per head -> out equals that constant (weights sum to one)."""
    bid = np.array([-1] * 2 + [0] * 6 + [-1] + [1] * 6)
    L, H = len(bid), 2
    q, k = _rng_arrays(7, (L, H, D), (L, H, D))
    c = np.stack([np.full(D, 0.25), np.linspace(-1, 1, D)])
    v = np.broadcast_to(c[None], (L, H, D)).copy()
    cu = np.array([0, L])
    out, _ = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    assert np.allclose(out, v, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants the pages state
# ---------------------------------------------------------------------------

def _tiny_inputs(seed):
    bid = np.array([-1] * 5 + [0] * 16 + [-1] * 3 + [1] * 16)
    L, H = len(bid), 2
    q, k, v = _rng_arrays(seed, (L, H, D), (L, H, D), (L, H, D))
    return bid, q, k, v


def pin_prefix_independent_of_target(orc):
    """The prefix cannot read the target: replacing the target's q/k/v leaves
    every prefix row bit-identical."""
    bid, q, k, v = _tiny_inputs(8)
    cu = np.array([0, 40])
    out1, lse1 = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    (r,) = _rng_arrays(9, (16, 2, D))
    q2[24:] += r
    k2[24:] -= 3 * r
    v2[24:] = r
    out2, lse2 = orc.prefill(q2, k2, v2, bid, cu, cu, SCALE)
    assert (out1[:24] == out2[:24]).all() and (lse1[:, :24] == lse2[:, :24]).all()
    assert not np.allclose(out1[24:], out2[24:])


def pin_cached_equals_uncached(orc):
    """Target rows of the full prefill equal prefix decode over [prefix; target]."""
    bid, q, k, v = _tiny_inputs(10)
    cu = np.array([0, 40])
    out, lse = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    dout, dlse = orc.prefix_decode(q[24:], k[:24], v[:24], np.array([0, 24]),
                                   k[24:], v[24:], np.array([0, 16]), SCALE)
    assert np.allclose(out[24:], dout, atol=1e-12) and np.allclose(lse[:, 24:], dlse, atol=1e-12)


def pin_short_q_rows_match_square(orc):
    """Bottom-right alignment: prefill with only the last q_len queries equals
    those rows of the square prefill, for block-causal layouts too."""
    bid, q, k, v = _tiny_inputs(11)
    cu = np.array([0, 40])
    out, lse = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    for q_len in (1, 3, 17, 22):
        o2, l2 = orc.prefill(q[40 - q_len:], k, v, bid, np.array([0, q_len]), cu, SCALE)
        assert np.allclose(o2, out[40 - q_len:], atol=1e-12)
        assert np.allclose(l2, lse[:, 40 - q_len:], atol=1e-12)


def pin_varlen_matches_separate(orc):
    """Packing sequences back to back changes nothing (ids compared per sequence)."""
    b1 = np.array([-1, -1, 0, 0, 0, -1, 1, 1])
    b2 = np.array([0, 0, -1, -1, 1, 1, 1])
    H = 2
    q, k, v = _rng_arrays(12, (15, H, D), (15, H, D), (15, H, D))
    cu = np.array([0, 8, 15])
    out, lse = orc.prefill(q, k, v, np.concatenate([b1, b2]), cu, cu, SCALE)
    o1, l1 = orc.prefill(q[:8], k[:8], v[:8], b1, np.array([0, 8]), np.array([0, 8]), SCALE)
    o2, l2 = orc.prefill(q[8:], k[8:], v[8:], b2, np.array([0, 7]), np.array([0, 7]), SCALE)
    assert np.allclose(out, np.concatenate([o1, o2]), atol=1e-12)
    assert np.allclose(lse, np.concatenate([l1, l2], axis=1), atol=1e-12)


def pin_row_sampling(orc):
    """Sampled rows/heads equal the same entries of the full computation."""
    bid, q, k, v = _tiny_inputs(13)
    cu = np.array([0, 40])
    out, lse = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    rows, heads = np.array([39, 0, 21, 5]), np.array([1])
    o, l = orc.prefill(q, k, v, bid, cu, cu, SCALE, rows=rows, heads=heads)
    assert np.allclose(o[:, 0], out[rows, 1], atol=0) and np.allclose(l[0], lse[1, rows], atol=0)


def pin_cache_append_layout(orc):
    """Append copies prefix token t of sequence b, head h, to cache[layer, h, cu_prefix[b]+t]."""
    H, Dd, layers, cap = 3, 4, 2, 10
    cu_k = np.array([0, 5, 12])
    cu_p = np.array([0, 3, 7])       # prefixes of 3 and 4 tokens
    tok = np.arange(12)[:, None, None]
    hh = np.arange(H)[None, :, None]
    dd = np.arange(Dd)[None, None, :]
    k = (1000 * tok + 10 * hh + dd).astype(np.int32)
    v = -k
    ck = np.full((layers, H, cap, Dd), -7, dtype=np.int32)
    cv = ck.copy()
    orc.cache_append(k, v, cu_k, cu_p, ck, cv, layer=1)
    # sequence 0 tokens 0..2 -> cache 0..2 ; sequence 1 tokens 5..8 -> cache 3..6
    for h in range(H):
        for c, src in zip(range(7), [0, 1, 2, 5, 6, 7, 8]):
            assert (ck[1, h, c] == 1000 * src + 10 * h + np.arange(Dd)).all()
            assert (cv[1, h, c] == -(1000 * src + 10 * h + np.arange(Dd))).all()
    assert (ck[0] == -7).all() and (ck[1, :, 7:] == -7).all()


def pin_piecewise_equals_block_causal(orc):
    """The pages call both prefill paths exact: per-segment attention calls (text
    causal over itself, images over everything before and themselves) equal the
    one block-causal masked attention, on every valid layout up to length 6 and
    on the tiny layout."""
    H = 1
    for n in range(1, 7):
        for bid in _valid_layouts(n):
            q, k, v = _rng_arrays(100 + n, (n, H, D), (n, H, D), (n, H, D))
            cu = np.array([0, n])
            o1, l1 = orc.prefill(q, k, v, bid, cu, cu, SCALE)
            o2, l2 = orc.prefill_piecewise(q, k, v, bid, cu, SCALE)
            assert np.allclose(o1, o2, rtol=0, atol=1e-12), bid
            assert np.allclose(l1, l2, rtol=0, atol=1e-12), bid
    bid, q, k, v = _tiny_inputs(13)
    cu = np.array([0, 40])
    o1, l1 = orc.prefill(q, k, v, bid, cu, cu, SCALE)
    o2, l2 = orc.prefill_piecewise(q, k, v, bid, cu, SCALE)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


ALL_PINS = [
    pin_worked_example_mask, pin_bottom_right, pin_tiny_layout, pin_adjacent_references,
    pin_brute_force_small, pin_zero_query_closed_form, pin_causal_text_equals_sdpa,
    pin_single_block_equals_full, pin_decode_equals_full, pin_large_scores_stable,
    pin_constant_values, pin_prefix_independent_of_target, pin_cached_equals_uncached,
    pin_short_q_rows_match_square, pin_varlen_matches_separate, pin_row_sampling,
    pin_cache_append_layout, pin_piecewise_equals_block_causal,
]
