"""Pins of the paged prefix cache oracle: hand-worked page addresses, round
trips through a permuted page table, shared pages, and paged decode equal to
the contiguous decode; planted addressing mistakes each fail a pin."""
import numpy as np
import pytest

import oracle.attention as orc
import oracle.paged as pg

D = 128


def pin_hand_worked_addresses():
    # sequence 0: prefix of 300 tokens in pages 3, 0, 5; sequence 1: 5 tokens in page 1
    pt = [[3, 0, 5], [1, -1, -1]]
    assert pg.page_slot(pt, 0, 0) == 384
    assert pg.page_slot(pt, 0, 127) == 511
    assert pg.page_slot(pt, 0, 128) == 0
    assert pg.page_slot(pt, 0, 299) == 5 * 128 + 43
    assert pg.page_slot(pt, 1, 4) == 132


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_round_trip_permuted_pages():
    H, L = 2, 2
    pre = [300, 5, 129]
    cp = np.concatenate([[0], np.cumsum(pre)])
    kl = [310, 5, 200]
    ck = np.concatenate([[0], np.cumsum(kl)])
    k, v = _rand(1, int(ck[-1]), H, D), _rand(2, int(ck[-1]), H, D)
    n_pages = [3, 1, 2]
    perm = np.random.default_rng(3).permutation(8)
    pt, at = np.full((3, 3), -1), 0
    for b, n in enumerate(n_pages):
        pt[b, :n] = perm[at:at + n]
        at += n
    pool_k = np.full((L, H, 8 * 128, D), 9.0)
    pool_v = np.full((L, H, 8 * 128, D), 9.0)
    pg.paged_append(k, v, ck, cp, pt, 1, pool_k, pool_v)
    gk = pg.paged_gather(pool_k, cp, pt, 1)
    gv = pg.paged_gather(pool_v, cp, pt, 1)
    exp_k = np.concatenate([k[ck[b]:ck[b] + pre[b]] for b in range(3)])
    exp_v = np.concatenate([v[ck[b]:ck[b] + pre[b]] for b in range(3)])
    assert np.array_equal(gk, exp_k) and np.array_equal(gv, exp_v)
    # pages nobody references, and the other layer, are untouched
    used = set(perm[:6].tolist())
    for page in range(8):
        if page not in used:
            assert np.all(pool_k[1, :, page * 128:(page + 1) * 128] == 9.0)
    assert np.all(pool_k[0] == 9.0)


def pin_shared_pages_read_the_same_rows():
    H = 1
    k, v = _rand(4, 256, H, D), _rand(5, 256, H, D)
    pt = [[2, 0], [2, 0]]                      # two sequences sharing both pages
    pool_k = np.zeros((1, H, 3 * 128, D))
    pool_v = np.zeros((1, H, 3 * 128, D))
    pg.paged_append(k, v, [0, 256], [0, 256], pt[:1], 0, pool_k, pool_v)
    g = pg.paged_gather(pool_k, [0, 256, 256 + 200], pt, 0)
    assert np.array_equal(g[256:], k[:200])


def pin_paged_decode_equals_contiguous():
    H = 2
    pre, tgt = [200, 70], [64, 30]
    cp = np.concatenate([[0], np.cumsum(pre)])
    cq = np.concatenate([[0], np.cumsum(tgt)])
    kp, vp = _rand(6, cp[-1], H, D), _rand(7, cp[-1], H, D)
    qt, kt, vt = _rand(8, cq[-1], H, D), _rand(9, cq[-1], H, D), _rand(10, cq[-1], H, D)
    pt = [[4, 1], [2, -1]]
    pool_k = np.zeros((1, H, 5 * 128, D))
    pool_v = np.zeros((1, H, 5 * 128, D))
    pg.paged_append(kp, vp, cp, cp, pt, 0, pool_k, pool_v)
    o1, l1 = pg.paged_prefix_decode(qt, pool_k, pool_v, cp, pt, 0, kt, vt, cq, 0.088)
    o2, l2 = orc.prefix_decode(qt, kp, vp, cp, kt, vt, cq, 0.088)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


MUTANTS = {
    "slot_and_page_swapped": lambda pt, b, t: int(pt[b][t % 128]) * 128 + t // 128
    if t % 128 < len(pt[b]) else -1,
    "next_page": lambda pt, b, t: int(pt[b][min(t // 128 + 1, len(pt[b]) - 1)]) * 128 + t % 128,
    "slot_ignored": lambda pt, b, t: int(pt[b][t // 128]) * 128,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    monkeypatch.setattr(pg, "page_slot", MUTANTS[name])
    failed = 0
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, IndexError):
            failed += 1
    assert failed, name
