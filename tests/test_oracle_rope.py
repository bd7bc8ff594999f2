"""Pins of the Q/K prologue oracle (RMS normalisation, three-axis RoPE, cache
append) against what the page and the mathematics fix, and planted mistakes
that each fail at least one pin.

Page: "Qwen-Image 2.1: Block-Causal Attention, Prefix KV Cache, and Turbo"
(flozi.net), "Three-axis RoPE preserves image geometry" and the paragraph on the
32 heads of width 128 (Q/K RMS-normalised per head before RoPE).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle.rope as rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_positions_t2_img2x3_t1_img1x2.txt")


def _read_golden():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    bid = np.array(rows[0], dtype=np.int64)
    gw = np.array(rows[1], dtype=np.int64)
    pos = np.array(rows[2:], dtype=np.int64)
    return bid, gw, pos


def _layout(segments):
    """segments: list of ('t', n) or ('i', id, rows, cols) -> block ids and widths."""
    bid, widths = [], {}
    for s in segments:
        if s[0] == "t":
            bid += [-1] * s[1]
        else:
            bid += [s[1]] * (s[2] * s[3])
            widths[s[1]] = s[3]
    gw = np.zeros((1, max(widths) + 1 if widths else 1), dtype=np.int64)
    for i, w in widths.items():
        gw[0, i] = w
    return np.array(bid, dtype=np.int64), gw


# ------------------------------------------------------------------------------- pins

def pin_positions_golden():
    bid, gw, pos = _read_golden()
    got = rope.rope_positions(bid, [0, len(bid)], gw[None, :])
    assert np.array_equal(got, pos)


def pin_positions_text_only():
    bid = -np.ones(9, dtype=np.int64)
    got = rope.rope_positions(bid, [0, 4, 9], np.zeros((2, 1), np.int64))
    exp = np.concatenate([np.arange(4), np.arange(5)])
    assert np.array_equal(got, np.stack([exp] * 3, axis=1))


def pin_moving_a_block_changes_only_its_frame():
    # the page: moving a reference block later changes its frame coordinate but
    # not its internal height/width grid
    a_bid, a_gw = _layout([("t", 2), ("i", 0, 3, 4), ("t", 4)])
    b_bid, b_gw = _layout([("t", 5), ("i", 0, 3, 4), ("t", 1)])
    pa = rope.rope_positions(a_bid, [0, len(a_bid)], a_gw)
    pb = rope.rope_positions(b_bid, [0, len(b_bid)], b_gw)
    ia, ib = a_bid == 0, b_bid == 0
    assert np.array_equal(pa[ia, 1:], pb[ib, 1:])
    assert np.all(pb[ib, 0] - pa[ia, 0] == 3)


def pin_grid_centred_on_zero():
    for rows, cols in ((5, 7), (4, 6), (1, 3)):
        bid, gw = _layout([("t", 3), ("i", 0, rows, cols)])
        p = rope.rope_positions(bid, [0, len(bid)], gw)[bid == 0]
        h, w = np.unique(p[:, 1]), np.unique(p[:, 2])
        assert len(h) == rows and len(w) == cols
        assert h.min() == -(rows // 2) and w.min() == -(cols // 2)   # zero inside the grid
        assert h.max() - h.min() == rows - 1 and w.max() - w.min() == cols - 1
        if rows % 2:
            assert h.sum() == 0
        if cols % 2:
            assert w.sum() == 0


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_rotation_identity_at_zero():
    x = _rand((5, 2, 128), 1)
    assert np.array_equal(rope.rotate(x, np.zeros((5, 3), np.int64)), x)


def pin_rotation_complex_form():
    # (x_2k + i x_2k+1) * exp(i t): the rotation as complex multiplication
    x = _rand((6, 3, 128), 2)
    pos = np.array([[0, 0, 0], [5, -3, 2], [17, 4, -9], [1, 1, 1], [300, 31, -32], [2, 0, 0]])
    th = rope.rope_angles(pos)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * th)[:, None, :]
    out = rope.rotate(x, pos)
    assert np.allclose(out[..., 0::2], z.real, rtol=0, atol=1e-12)
    assert np.allclose(out[..., 1::2], z.imag, rtol=0, atol=1e-12)


def pin_angles_hand_values():
    # frame pair 0 at frame 1: angle 1; height pair 1 (dims 18, 19) at height 1:
    # 10000^(-2/56); width pair 27 (dims 126, 127) at width 3: 3 * 10000^(-54/56);
    # frame pair 7 (dims 14, 15) at frame 2: 2 * 10000^(-14/16)
    th = rope.rope_angles(np.array([[1, 1, 3], [2, 0, 0]]))
    assert th.shape == (2, 64)
    assert th[0, 0] == 1.0
    assert math.isclose(th[0, 8 + 1], 10000.0 ** (-2.0 / 56.0), rel_tol=1e-15)
    assert math.isclose(th[0, 36 + 27], 3.0 * 10000.0 ** (-54.0 / 56.0), rel_tol=1e-15)
    assert math.isclose(th[1, 7], 2.0 * 10000.0 ** (-14.0 / 16.0), rel_tol=1e-15)
    assert th[1, 8] == 0.0 and th[1, 36] == 0.0


def pin_rotation_direction_hand_value():
    # e_0 at frame 1 (angle 1 on pair 0) turns towards +e_1: (cos 1, sin 1)
    x = np.zeros((1, 1, 128))
    x[0, 0, 0] = 1.0
    out = rope.rotate(x, np.array([[1, 0, 0]]))
    assert math.isclose(out[0, 0, 0], math.cos(1.0)) and math.isclose(out[0, 0, 1], math.sin(1.0))
    assert np.all(out[0, 0, 2:] == 0)


def pin_rotation_preserves_pair_norms():
    x = _rand((7, 2, 128), 3)
    pos = np.random.default_rng(4).integers(-64, 4000, size=(7, 3))
    out = rope.rotate(x, pos)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = out[..., 0::2] ** 2 + out[..., 1::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-12, atol=0)


def pin_relative_position():
    # <R(p) a, R(p') b> depends only on p - p', axis by axis
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    p, pp = np.array([[3, -2, 7]]), np.array([[11, 5, -4]])
    base = np.sum(rope.rotate(a, p) * rope.rotate(b, pp))
    for shift in ([5, 0, 0], [0, -9, 0], [0, 0, 13], [100, 7, -6]):
        s = np.array([shift])
        assert math.isclose(np.sum(rope.rotate(a, p + s) * rope.rotate(b, pp + s)), base,
                            rel_tol=1e-9, abs_tol=1e-9)


def pin_rms_norm_matches_torch():
    x = _rand((4, 3, 128), 6) * np.array([1e-3, 1.0, 50.0])[None, :, None]
    g = _rand((128,), 7)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(g), eps=1e-6)
    assert np.allclose(rope.rms_norm(x, g), ref.numpy(), rtol=1e-13, atol=0)


def pin_rms_norm_properties():
    x = _rand((5, 2, 128), 8) * 7.0
    y = rope.rms_norm(x)
    assert np.allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-6)
    assert np.allclose(rope.rms_norm(3.0 * x), y, rtol=1e-6)
    assert np.all(rope.rms_norm(np.zeros((1, 1, 128))) == 0)


def pin_norm_before_rope_hand_value():
    # q = e_1, gamma = 2 on dimension 0 and 1 elsewhere, frame coordinate 1:
    # normalise first -> sqrt(128) e_1 (gamma_1 = 1), rotate pair 0 by angle 1 ->
    # (-sqrt(128) sin 1, sqrt(128) cos 1).  Rotating first would put the weight 2
    # on the rotated dimension 0.
    q = np.zeros((1, 1, 128))
    q[0, 0, 1] = 1.0
    g = np.ones(128)
    g[0] = 2.0
    qo, _ = rope.qk_norm_rope(q, q, g, g, np.array([[1, 0, 0]]))
    r = math.sqrt(128.0) / math.sqrt(1.0 + 128e-6)
    assert math.isclose(qo[0, 0, 0], -r * math.sin(1.0), rel_tol=1e-12)
    assert math.isclose(qo[0, 0, 1], r * math.cos(1.0), rel_tol=1e-12)


def pin_append_layout():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((9, 2, 128))
    k = rng.standard_normal((9, 2, 128))
    v = rng.standard_normal((9, 2, 128))
    pos = rng.integers(0, 50, size=(9, 3))
    cu, cp = [0, 4, 9], [0, 3, 5]                       # prefixes of 3 and 2 tokens
    ck = np.full((2, 2, 8, 128), -7.0)
    cv = np.full((2, 2, 8, 128), -7.0)
    _, ko = rope.qk_norm_rope_append(q, k, v, None, None, pos, cu, cp, 1, ck, cv)
    assert np.array_equal(ck[1, :, 0:3], ko[0:3].transpose(1, 0, 2))
    assert np.array_equal(ck[1, :, 3:5], ko[4:6].transpose(1, 0, 2))
    assert np.array_equal(cv[1, :, 0:3], v[0:3].transpose(1, 0, 2))
    assert np.array_equal(cv[1, :, 3:5], v[4:6].transpose(1, 0, 2))
    assert np.all(ck[0] == -7) and np.all(ck[1, :, 5:] == -7) and np.all(cv[1, :, 5:] == -7)


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------- mutants

_real_angles = rope.rope_angles
_real_rotate = rope.rotate
_real_norm = rope.rms_norm
_real_positions = rope.rope_positions


def _angles_variant(axes=rope.AXES, base=rope.BASE, per_axis_d=True):
    def ang(pos3):
        pos = np.asarray(pos3, dtype=np.float64)
        order = {(16, 56, 56): (0, 1, 2), (56, 56, 16): (1, 2, 0)}[tuple(axes)]
        cols = []
        for d, a in zip(axes, order):
            k = np.arange(d // 2, dtype=np.float64)
            dd = d if per_axis_d else 128
            cols.append(pos[:, a:a + 1] * (base ** (-2.0 * k / dd))[None, :])
        return np.concatenate(cols, axis=1)
    return ang


def _rotate_half(x, pos3):
    x = np.asarray(x, dtype=np.float64)
    th = _real_angles(pos3)[:, None, :]
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., :64], x[..., 64:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _positions_variant(frame_minus_one=False, no_advance=False, uncentred=False, frame_only=False):
    def positions(block_id, cu_seqlens, grid_w):
        p = _real_positions(block_id, cu_seqlens, grid_w).copy()
        bid = np.asarray(block_id)
        img = bid >= 0
        if frame_minus_one:
            p[img, 0] -= 1
        if uncentred:
            for i in np.unique(bid[img]):
                m = bid == i
                p[m, 1] -= p[m, 1].min()
                p[m, 2] -= p[m, 2].min()
        if frame_only:
            p[~img, 1:] = 0
        if no_advance:       # the image does not advance the running coordinate
            cu = np.asarray(cu_seqlens)
            for b in range(len(cu) - 1):
                seen = 0
                for t in range(cu[b], cu[b + 1]):
                    if bid[t] >= 0 and (t == cu[b] or bid[t - 1] != bid[t]):
                        seen += 1
                    if bid[t] < 0:
                        p[t] -= seen
        return p
    return positions


MUTANTS = {
    "axes_reordered": ("rope_angles", _angles_variant(axes=(56, 56, 16))),
    "base_1000": ("rope_angles", _angles_variant(base=1000.0)),
    "one_ladder_over_128": ("rope_angles", _angles_variant(per_axis_d=False)),
    "rotate_half_pairs": ("rotate", _rotate_half),
    "sin_sign_flipped": ("rotate", lambda x, pos3: _real_rotate(x, -np.asarray(pos3))),
    "norm_after_rope": ("qk_norm_rope",
                        lambda q, k, gq, gk, pos3, eps=rope.EPS:
                        (_real_norm(_real_rotate(q, pos3), gq, eps),
                         _real_norm(_real_rotate(k, pos3), gk, eps))),
    "eps_1e-5": ("rms_norm", lambda x, gamma=None, eps=rope.EPS: _real_norm(x, gamma, 1e-5)),
    "image_frame_minus_one": ("rope_positions", _positions_variant(frame_minus_one=True)),
    "image_does_not_advance": ("rope_positions", _positions_variant(no_advance=True)),
    "grid_not_centred": ("rope_positions", _positions_variant(uncentred=True)),
    "text_frame_axis_only": ("rope_positions", _positions_variant(frame_only=True)),
    "append_v_rotated": ("qk_norm_rope_append", None),
}


def _append_v_rotated(q, k, v, gq, gk, pos3, cu, cp, layer, ck, cv, eps=rope.EPS):
    qo, ko = rope.qk_norm_rope(q, k, gq, gk, pos3, eps)
    vr = _real_rotate(v, pos3)
    cu, cp = np.asarray(cu), np.asarray(cp)
    for b in range(len(cu) - 1):
        for t in range(cp[b + 1] - cp[b]):
            ck[layer, :, cp[b] + t] = ko[cu[b] + t]
            cv[layer, :, cp[b] + t] = vr[cu[b] + t]
    return qo, ko


MUTANTS["append_v_rotated"] = ("qk_norm_rope_append", _append_v_rotated)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(rope, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
