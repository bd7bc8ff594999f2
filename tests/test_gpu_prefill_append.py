"""bca_prefill_append (the prefill with the prefix cache append fused in) against the two
separate calls: its attention output must be bit-identical to bca_prefill's and its cache
rows bit-identical to the oracle's append (and to bca_prefix_cache_append's), with every
cache row it must not touch left as it was."""
import numpy as np
import pytest
import torch

import oracle
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV, ragged_case

pytestmark = pytest.mark.gpu


def _status():
    return bca.new_status(DEV)


def _expected_cache(k, v, cu_k, cu_p, layers, layer, cap):
    H = k.shape[1]
    ek = np.full((layers, H, cap, 128), -1, dtype=np.int16)
    ev = ek.copy()
    oracle.cache_append(k.view(torch.int16).numpy(), v.view(torch.int16).numpy(), cu_k, cu_p,
                        ek, ev, layer)
    return ek, ev


def _sentinel_cache(layers, H, cap):
    ck = torch.full((layers, H, cap, 128), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    return ck, ck.clone()


def _run_both(case, cu_p, layers, layer, cap, status=None):
    d = lambda x: x.to(DEV)
    ti = lambda x: torch.from_numpy(np.asarray(x, dtype=np.int32)).to(DEV)
    args = (d(case.q), d(case.k), d(case.v), ti(case.block_id), ti(case.cu_q), ti(case.cu_k),
            case.max_q, case.max_k)
    out1, lse1 = bca.prefill(*args)
    ck, cv = _sentinel_cache(layers, case.q.shape[1], cap)
    out2, lse2 = bca.prefill_append(*args, ti(cu_p), ck, cv, layer, status=status)
    return out1, lse1, out2, lse2, ck, cv


@pytest.mark.parametrize("seed,kv,ql,pre,heads", [
    (91, [300, 5, 129, 1000], None, [299, 0, 128, 777], 3),   # ragged, empty, whole tiles
    (92, [640, 200], [640, 33], [640, 199], 16),               # bottom-right rows, 2 head groups
    (93, [12, 129, 256], None, [12, 1, 255], 20),              # 4 head groups of 5
])
def test_prefill_append_matches_separate_calls(seed, kv, ql, pre, heads):
    case = ragged_case(seed, kv, ql, heads=heads)
    # the prefixes start at cache token 5: rows before them must stay untouched
    cu_p = np.concatenate([[5], 5 + np.cumsum(pre)]).astype(np.int32)
    layers, layer = 2, 1
    cap = int(cu_p[-1]) + 9
    st = _status()
    out1, lse1, out2, lse2, ck, cv = _run_both(case, cu_p, layers, layer, cap, status=st)
    assert bca.read_status(st) == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    ek, ev = _expected_cache(case.k, case.v, case.cu_k, cu_p, layers, layer, cap)
    assert np.array_equal(ck.view(torch.int16).cpu().numpy(), ek)
    assert np.array_equal(cv.view(torch.int16).cpu().numpy(), ev)
    # and the standalone append writes the same rows
    sk, sv = _sentinel_cache(layers, heads, cap)
    bca.prefix_cache_append(case.k.to(DEV), case.v.to(DEV), torch.from_numpy(case.cu_k).to(DEV),
                            torch.from_numpy(cu_p).to(DEV), sk, sv, layer)
    assert torch.equal(sk.view(torch.int16), ck.view(torch.int16))
    assert torch.equal(sv.view(torch.int16), cv.view(torch.int16))


@pytest.mark.parametrize("pre,cap,code", [
    ([100, 30], 200, 8),     # the first prefix is longer than its 90 keys: BCA_ERR_SEQLENS
    ([80, 30], 100, 5),      # 110 prefix rows in a 100-token cache: BCA_ERR_CAPACITY
])
def test_prefill_append_rejects_without_writing(pre, cap, code):
    case = ragged_case(94, [90, 300], heads=2)
    cu_p = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    st = _status()
    out1, lse1, out2, lse2, ck, cv = _run_both(case, cu_p, 1, 0, cap, status=st)
    assert bca.read_status(st) == code
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)   # attention still computed
    assert (ck.view(torch.int16) == -1).all() and (cv.view(torch.int16) == -1).all()


def test_prefill_append_block_id_error_skips_that_sequence():
    case = ragged_case(95, [200, 260], heads=2)
    bid = case.block_id.copy()
    bid[10:20] = 7
    bid[30:40] = 7                   # id 7 split into two runs in sequence 0
    case.block_id = bid
    cu_p = np.array([0, 150, 410], dtype=np.int32)
    st = _status()
    d = lambda x: x.to(DEV)
    ti = lambda x: torch.from_numpy(np.asarray(x, dtype=np.int32)).to(DEV)
    ck, cv = _sentinel_cache(1, 2, 410)
    bca.prefill_append(d(case.q), d(case.k), d(case.v), ti(bid), ti(case.cu_q), ti(case.cu_k),
                       case.max_q, case.max_k, ti(cu_p), ck, cv, 0, status=st)
    assert bca.read_status(st) == 3                      # BCA_ERR_BLOCK_ID
    assert (ck[0, :, :150].view(torch.int16) == -1).all()
    ek, ev = _expected_cache(case.k, case.v, case.cu_k, cu_p, 1, 0, 410)
    assert np.array_equal(ck[0, :, 150:].view(torch.int16).cpu().numpy(), ek[0, :, 150:])
    assert np.array_equal(cv[0, :, 150:].view(torch.int16).cpu().numpy(), ev[0, :, 150:])


def test_prefill_append_full_size_edit():
    wl = W.edit_two_ref()
    q, k, v = W.make_qkv(wl)
    cu = torch.from_numpy(wl.cu_seqlens()).to(DEV)
    bid = torch.from_numpy(wl.block_id()).to(DEV)
    cu_p = torch.from_numpy(wl.cu_prefix()).to(DEV)
    P, S = wl.prefix_lens()[0], wl.seq_lens[0]
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out1, lse1 = bca.prefill(qd, kd, vd, bid, cu, cu, S, S)
    ck = torch.zeros((2, 32, P, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    st = _status()
    out2, lse2 = bca.prefill_append(qd, kd, vd, bid, cu, cu, S, S, cu_p, ck, cv, 1, status=st)
    assert bca.read_status(st) == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    assert torch.equal(ck[1], kd[:P].permute(1, 0, 2))
    assert torch.equal(cv[1], vd[:P].permute(1, 0, 2))
    assert (ck[0] == 0).all() and (cv[0] == 0).all()


def _page_table(pre, pool, seed):
    """Shuffled distinct pages of a pool, ceil(P_b / 128) per sequence, rows padded with -1."""
    need = [(p + 127) // 128 for p in pre]
    perm = np.random.default_rng(seed).permutation(pool)
    rows, at = [], 0
    width = max(need + [1])
    for n in need:
        rows.append(list(perm[at:at + n]) + [-1] * (width - n))
        at += n
    return torch.tensor(rows, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("seed,kv,pre,heads", [
    (96, [300, 5, 129, 1000], [299, 0, 128, 777], 3),
    (97, [640, 200], [640, 199], 16),
])
def test_prefill_append_paged_matches_standalone(seed, kv, pre, heads):
    case = ragged_case(seed, kv, heads=heads)
    cu_p = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    pool = sum((p + 127) // 128 for p in pre) + 3
    pt = _page_table(pre, pool, seed)
    d = lambda x: x.to(DEV)
    ti = lambda x: torch.from_numpy(np.asarray(x, dtype=np.int32)).to(DEV)
    args = (d(case.q), d(case.k), d(case.v), ti(case.block_id), ti(case.cu_q), ti(case.cu_k),
            case.max_q, case.max_k)
    out1, lse1 = bca.prefill(*args)
    ck, cv = _sentinel_cache(2, heads, pool * 128)
    st = _status()
    out2, lse2 = bca.prefill_append(*args, ti(cu_p), ck, cv, 1, page_table=pt, status=st)
    assert bca.read_status(st) == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    sk, sv = _sentinel_cache(2, heads, pool * 128)
    bca.prefix_cache_append_paged(d(case.k), d(case.v), ti(case.cu_k), ti(cu_p), pt, sk, sv, 1)
    assert torch.equal(sk.view(torch.int16), ck.view(torch.int16))
    assert torch.equal(sv.view(torch.int16), cv.view(torch.int16))


def test_prefill_append_paged_rejects_bad_page():
    case = ragged_case(98, [300, 200], heads=2)
    cu_p = np.array([0, 250, 450], dtype=np.int32)
    pt = _page_table([250, 200], 6, 98)
    pt[1, 1] = 6                                   # outside the 6-page pool
    d = lambda x: x.to(DEV)
    ti = lambda x: torch.from_numpy(np.asarray(x, dtype=np.int32)).to(DEV)
    ck, cv = _sentinel_cache(1, 2, 6 * 128)
    st = _status()
    bca.prefill_append(d(case.q), d(case.k), d(case.v), ti(case.block_id), ti(case.cu_q),
                       ti(case.cu_k), case.max_q, case.max_k, ti(cu_p), ck, cv, 0,
                       page_table=pt, status=st)
    assert bca.read_status(st) == 5                # BCA_ERR_CAPACITY
    assert (ck.view(torch.int16) == -1).all() and (cv.view(torch.int16) == -1).all()


@pytest.mark.parametrize("paged", [False, True], ids=["contiguous", "paged"])
def test_prefill_append_key_split_tail_keeps_the_appending_pair(paged):
    """A pair grid of 8 x 16 x 4 = 512 CTAs (under four waves of 152): its 56 cheapest
    pairs (the first tile pair of every sequence and head, and the second of most)
    become key-split single-tile items.  Sequence 1 has 200 rows: its only pair, which
    appends its prefix to the cache, lies among them and stays a pair CTA (its second
    pairs, past its end, are split items with no rows); both calls match the oracle
    and the cache is bit-exact (against the oracle's append, or the standalone paged
    append through the same page table)."""
    from gpu_cases import assert_close, tile_boundary_rows
    case = ragged_case(95, [4096, 200], heads=16)
    pre = [3000, 150]
    cu_p = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    d = lambda x: x.to(DEV)
    ti = lambda x: torch.from_numpy(np.asarray(x, dtype=np.int32)).to(DEV)
    args = (d(case.q), d(case.k), d(case.v), ti(case.block_id), ti(case.cu_q), ti(case.cu_k),
            case.max_q, case.max_k)
    st = _status()
    out1, lse1 = bca.prefill(*args, status=st)
    if paged:
        pool = sum((p + 127) // 128 for p in pre) + 5
        pt = _page_table(pre, pool, 95)
        ck, cv = _sentinel_cache(1, 16, pool * 128)
        out2, lse2 = bca.prefill_append(*args, ti(cu_p), ck, cv, 0, page_table=pt, status=st)
    else:
        cap = int(cu_p[-1]) + 64
        ck, cv = _sentinel_cache(1, 16, cap)
        out2, lse2 = bca.prefill_append(*args, ti(cu_p), ck, cv, 0, status=st)
    assert bca.read_status(st) == 0
    rows = np.unique(np.concatenate([tile_boundary_rows(case.cu_q, extra=200, seed=3),
                                     np.arange(4096, 4296)]))   # every row of sequence 1
    heads = np.array([2, 9, 15])
    ref = case.reference(rows=rows, heads=heads)
    assert_close(out1, lse1, *ref, rows=rows, heads=heads, what="prefill")
    assert_close(out2, lse2, *ref, rows=rows, heads=heads, what="prefill_append")
    if paged:
        sk, sv = _sentinel_cache(1, 16, pool * 128)
        bca.prefix_cache_append_paged(d(case.k), d(case.v), ti(case.cu_k), ti(cu_p), pt, sk, sv, 0)
        assert torch.equal(sk.view(torch.int16), ck.view(torch.int16))
        assert torch.equal(sv.view(torch.int16), cv.view(torch.int16))
    else:
        ek, ev = _expected_cache(case.k, case.v, case.cu_k, cu_p, 1, 0, cap)
        assert np.array_equal(ck.view(torch.int16).cpu().numpy(), ek)
        assert np.array_equal(cv.view(torch.int16).cpu().numpy(), ev)
