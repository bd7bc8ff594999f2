"""The host page pool of the paged prefix cache (no GPU): allocation, the hash
index, references, and the page rules of the Prism-Infer notes (publish only
after the write, copied tail pages without the old hash, idle pages lent out
but referenced pages never reclaimed, capacity by physical page)."""
import random
import threading

import numpy as np
import pytest

import prefix_kv_gb300 as bca


def test_alloc_release_and_capacity():
    pool = bca.PagePool(6)
    a = pool.alloc(4)
    assert sorted(a.tolist()) == sorted(set(a.tolist())) and pool.stats() == (2, 0, 4)
    with pytest.raises(RuntimeError, match="status 5 "):
        pool.alloc(3)
    assert pool.stats() == (2, 0, 4)                 # a failed alloc takes nothing
    pool.release(a[:2])
    assert pool.stats() == (4, 0, 2)


def test_publish_match_and_idle_cache():
    pool = bca.PagePool(8)
    pages = pool.alloc(3)
    for p, h in zip(pages, (11, 12, 13)):
        pool.publish(p, h)
    assert pool.match([11, 12, 99, 13]).tolist() == pages[:2].tolist()   # stops at a miss
    assert pool.refs(pages[0]) == 2
    pool.release(pages)                              # the writer's references
    pool.release(pages[:2])                          # the matcher's
    assert pool.stats() == (5, 3, 0)                 # all three cached, idle
    again = pool.match([11, 12, 13])
    assert again.tolist() == pages.tolist() and pool.stats() == (5, 0, 3)


def test_publish_needs_an_owner_and_a_new_hash():
    pool = bca.PagePool(4)
    p, q = pool.alloc(2)
    pool.publish(p, 1)
    with pytest.raises(RuntimeError):
        pool.publish(p, 2)                           # already published
    with pytest.raises(RuntimeError):
        pool.publish(q, 1)                           # hash taken
    pool.release([q])
    with pytest.raises(RuntimeError):
        pool.publish(q, 3)                           # nobody references it
    assert pool.match([3]).size == 0


def test_copied_tail_page_has_no_hash():
    # rule 2: a request sharing only part of a tail page gets a fresh page for the
    # common rows; that page is unpublished and the old hash still finds the old page
    pool = bca.PagePool(4)
    (old,) = pool.alloc(1)
    pool.publish(old, 77)
    (tail,) = pool.alloc(1)
    assert tail != old
    assert pool.match([77]).tolist() == [old]
    pool.release([tail])
    assert pool.stats()[0] >= 2                      # the copy went back to the free list


def test_idle_pages_are_lent_but_referenced_pages_are_not():
    pool = bca.PagePool(4)
    pages = pool.alloc(4)
    for i, p in enumerate(pages):
        pool.publish(p, 100 + i)
    pool.release(pages[:3])                          # 3 idle cached, 1 still referenced
    assert pool.stats() == (0, 3, 1)
    got = pool.alloc(2)                              # least recently released first
    assert got.tolist() == pages[:2].tolist()
    assert pool.match([100]).size == 0               # evicted pages left the index
    with pytest.raises(RuntimeError, match="status 5 "):
        pool.alloc(2)                                # only one idle page is left
    assert pool.match([103]).tolist() == [pages[3]]  # the referenced page stayed


def test_shared_pages_count_once():
    pool = bca.PagePool(4)
    (p,) = pool.alloc(1)
    pool.publish(p, 5)
    pool.match([5])
    pool.match([5])
    assert pool.refs(p) == 3 and pool.stats() == (3, 0, 1)


def test_release_is_checked_before_anything_changes():
    pool = bca.PagePool(4)
    a = pool.alloc(2)
    with pytest.raises(RuntimeError):
        pool.release([a[0], 9])
    with pytest.raises(RuntimeError):
        pool.release([a[0], a[0]])                   # would drop below zero
    assert pool.refs(a[0]) == 1 and pool.stats() == (2, 0, 2)


def test_concurrent_use_keeps_pages_unique():
    pool = bca.PagePool(64)
    held, errors = [], []
    lock = threading.Lock()

    def worker(seed):
        rng = random.Random(seed)
        mine = []
        for _ in range(300):
            if mine and rng.random() < 0.5:
                pool.release([mine.pop()])
            else:
                try:
                    mine.extend(pool.alloc(1).tolist())
                except RuntimeError:
                    pass
        with lock:
            held.extend(mine)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert len(held) == len(set(held)) and pool.stats() == (64 - len(held), 0, len(held))


def test_random_operations_follow_a_model():
    """Random alloc / publish / match / release against a plain model of the rules."""
    rng = random.Random(7)
    n = 12
    pool = bca.PagePool(n)
    refs = {}                      # page -> references
    pub = {}                       # hash -> page
    page_hash = {}                 # page -> hash
    idle = []                      # published, unreferenced, oldest first
    next_hash = 1
    for _ in range(2000):
        op = rng.choice(["alloc", "alloc", "publish", "match", "release"])
        free = n - len(refs) - len(idle)
        if op == "alloc":
            k = rng.randint(1, 3)
            if k > free + len(idle):
                with pytest.raises(RuntimeError):
                    pool.alloc(k)
                continue
            got = pool.alloc(k).tolist()
            take_idle = max(0, k - free)
            expect_idle = idle[:take_idle]
            assert set(expect_idle) <= set(got)
            for p in expect_idle:
                idle.remove(p)
                del pub[page_hash.pop(p)]
            for p in got:
                assert p not in refs
                refs[p] = 1
        elif op == "publish" and refs:
            p = rng.choice(sorted(refs))
            if p in page_hash:
                with pytest.raises(RuntimeError):
                    pool.publish(p, next_hash)
            else:
                pool.publish(p, next_hash)
                pub[next_hash] = p
                page_hash[p] = next_hash
                next_hash += 1
        elif op == "match" and pub:
            hs = [rng.choice(sorted(pub)) for _ in range(rng.randint(1, 3))]
            got = pool.match(hs).tolist()
            assert got == [pub[h] for h in hs]
            for p in got:
                if p in idle:
                    idle.remove(p)
                refs[p] = refs.get(p, 0) + 1
        elif op == "release" and refs:
            p = rng.choice(sorted(refs))
            pool.release([p])
            refs[p] -= 1
            if refs[p] == 0:
                del refs[p]
                if p in page_hash:
                    idle.append(p)
        free = n - len(refs) - len(idle)
        assert pool.stats() == (free, len(idle), len(refs))
        for p, r in refs.items():
            assert pool.refs(p) == r
