"""The paged prefix cache on the GPU: append through a page table (bit-exact
against the oracle), decode through it (against the oracle, and bit-identical
to the contiguous decode when the tiles hold the same rows), the tail-row copy,
bad page ids, and two requests sharing pages through the host pool."""
import math

import numpy as np
import pytest
import torch

import oracle.paged as pg
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV, SCALE, DecodeCase, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()


def _ti(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(DEV)


def _page_table(pre, n_pages, seed):
    need = [math.ceil(p / 128) for p in pre]
    perm = np.random.default_rng(seed).permutation(n_pages)
    width = max(need + [1])
    pt = np.full((len(pre), width), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[at:at + n]
        at += n
    return pt, set(perm[:at].tolist())


def _case(seed, pre, tgt, H=3):
    kp = W.randn_bf16((sum(pre), H, 128), seed)
    vp = W.randn_bf16((sum(pre), H, 128), seed + 1)
    qt = W.randn_bf16((sum(tgt), H, 128), seed + 2)
    kt = W.randn_bf16((sum(tgt), H, 128), seed + 3)
    vt = W.randn_bf16((sum(tgt), H, 128), seed + 4)
    return kp, vp, qt, kt, vt, np.concatenate([[0], np.cumsum(pre)]), np.concatenate([[0], np.cumsum(tgt)])


@pytest.mark.parametrize("seed,pre,tgt", [(91, [300, 0, 129, 5], [16, 200, 1, 256]), (92, [1000], [130])])
def test_paged_append_and_decode(seed, pre, tgt):
    H, L, layer, n_pages = 3, 2, 1, 16
    kp, vp, qt, kt, vt, cp, cq = _case(seed, pre, tgt, H)
    pt, used = _page_table(pre, n_pages, seed)
    ck = torch.full((L, H, n_pages * 128, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    cv = torch.full_like(ck, float("nan"))
    st = bca.new_status(DEV)
    # the prefix rows are the first keys of each "sequence" (here: the prefix alone)
    bca.prefix_cache_append_paged(kp.to(DEV), vp.to(DEV), _ti(cp), _ti(cp), _ti(pt), ck, cv, layer,
                                  status=st)
    assert bca.read_status(st) == 0
    exp_k = np.full(tuple(ck.shape), np.nan, np.float32)
    exp_v = np.full(tuple(cv.shape), np.nan, np.float32)
    pg.paged_append(kp, vp, cp, cp, pt, layer, exp_k, exp_v)
    assert np.array_equal(ck.float().cpu().numpy(), exp_k, equal_nan=True)
    assert np.array_equal(cv.float().cpu().numpy(), exp_v, equal_nan=True)
    out, lse = bca.prefix_decode_paged(qt.to(DEV), ck, cv, layer, _ti(cp), _ti(pt), kt.to(DEV),
                                       vt.to(DEV), _ti(cq), int(max(tgt)), int(max(pre)), SCALE,
                                       status=st)
    assert bca.read_status(st) == 0
    ref = pg.paged_prefix_decode(qt, exp_k.astype(np.float64), exp_v.astype(np.float64), cp, pt,
                                 layer, kt, vt, cq, SCALE)
    assert_close(out, lse, *ref, what=f"paged decode {seed}")


def test_paged_decode_equals_contiguous_on_edit():
    case = DecodeCase.from_workload(W.edit_two_ref())
    H, P = case.q_tgt.shape[1], int(case.cu_pre[-1])
    n_pages = math.ceil(P / 128) + 3
    pt, _ = _page_table([P], n_pages, 5)
    ck = torch.zeros((1, H, n_pages * 128, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    bca.prefix_cache_append_paged(case.k_pre.to(DEV), case.v_pre.to(DEV), _ti(case.cu_pre),
                                  _ti(case.cu_pre), _ti(pt), ck, cv, 0)
    d = lambda t: t.to(DEV)
    out_p, lse_p = bca.prefix_decode_paged(d(case.q_tgt), ck, cv, 0, _ti(case.cu_pre), _ti(pt),
                                           d(case.k_tgt), d(case.v_tgt), _ti(case.cu_q),
                                           case.max_q, case.max_pre, SCALE)
    out_c, lse_c = case.run()
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse_p, lse_c)


def test_bad_page_ids_are_rejected():
    H, n_pages = 2, 4
    kp, vp, qt, kt, vt, cp, cq = _case(93, [200], [64], H)
    ck = torch.zeros((1, H, n_pages * 128, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    for pt in ([[1, 4]], [[-1, 0]], [[2]]):          # out of the pool; negative; too few pages
        st = bca.new_status(DEV)
        bca.prefix_cache_append_paged(kp.to(DEV), vp.to(DEV), _ti(cp), _ti(cp), _ti(pt), ck, cv, 0,
                                      status=st)
        assert bca.read_status(st) == 5 and bool((ck == 0).all())
        st = bca.new_status(DEV)
        bca.prefix_decode_paged(qt.to(DEV), ck, cv, 0, _ti(cp), _ti(pt), kt.to(DEV), vt.to(DEV),
                                _ti(cq), 64, 200, SCALE, status=st)
        assert bca.read_status(st) == 5


def test_copy_rows():
    H, L, n_pages = 2, 2, 5
    ck = W.randn_bf16((L, H, n_pages * 128, 128), 7).to(DEV)
    cv = W.randn_bf16((L, H, n_pages * 128, 128), 8).to(DEV)
    k0, v0 = ck.clone(), cv.clone()
    bca.pool_copy_rows(ck, cv, 1, 3, 1, 77)
    torch.cuda.synchronize()
    exp_k, exp_v = k0.clone(), v0.clone()
    exp_k[1, :, 128:128 + 77] = k0[1, :, 384:384 + 77]
    exp_v[1, :, 128:128 + 77] = v0[1, :, 384:384 + 77]
    assert torch.equal(ck, exp_k) and torch.equal(cv, exp_v)


def test_two_requests_share_pages_through_the_pool():
    """Request A writes a 300-token prefix into 3 pages and publishes the 2 full
    ones; request B has the same first 280 tokens: it matches the 2 full pages,
    copies the 24 common rows of A's tail page into a page of its own, appends
    its remaining rows there, and decodes as if its prefix were contiguous."""
    H, n_pages = 2, 8
    pool = bca.PagePool(n_pages)
    ck = torch.zeros((1, H, n_pages * 128, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    kA = W.randn_bf16((300, H, 128), 1)
    vA = W.randn_bf16((300, H, 128), 2)
    kB, vB = kA.clone(), vA.clone()
    kB[280:] = W.randn_bf16((20, H, 128), 3)
    vB[280:] = W.randn_bf16((20, H, 128), 4)
    pages_a = pool.alloc(3)
    bca.prefix_cache_append_paged(kA.to(DEV), vA.to(DEV), _ti([0, 300]), _ti([0, 300]),
                                  _ti([pages_a]), ck, cv, 0)
    torch.cuda.synchronize()                         # written: now publish the full pages
    pool.publish(pages_a[0], 1001)
    pool.publish(pages_a[1], 1002)
    hit = pool.match([1001, 1002, 1003])
    assert hit.tolist() == pages_a[:2].tolist()
    (tail,) = pool.alloc(1)
    bca.pool_copy_rows(ck, cv, 0, int(pages_a[2]), int(tail), 280 - 256)
    # B appends only its own rows 280..299: a "sequence" whose prefix is tokens
    # 0..299 but whose first 280 are already in place -- write the whole tail page
    pt_b = np.array([[hit[0], hit[1], tail]], np.int32)
    kb_tail = torch.cat([kA[256:280], kB[280:]])      # rows of B's third page
    vb_tail = torch.cat([vA[256:280], vB[280:]])
    bca.prefix_cache_append_paged(kb_tail.to(DEV), vb_tail.to(DEV), _ti([0, 44]), _ti([0, 44]),
                                  _ti([[tail]]), ck, cv, 0)
    qt = W.randn_bf16((64, H, 128), 5)
    kt = W.randn_bf16((64, H, 128), 6)
    vt = W.randn_bf16((64, H, 128), 7)
    out, lse = bca.prefix_decode_paged(qt.to(DEV), ck, cv, 0, _ti([0, 300]), _ti(pt_b),
                                       kt.to(DEV), vt.to(DEV), _ti([0, 64]), 64, 300, SCALE)
    import oracle
    ref = oracle.prefix_decode(qt, kB, vB, [0, 300], kt, vt, [0, 64], SCALE)
    assert_close(out, lse, *ref, what="shared pages")
    assert pool.refs(pages_a[0]) == 2 and pool.stats()[2] == 4


# ---------------------------------------------------------------- FP8 E4M3 pages

from oracle import fp8 as ofp8
import oracle as _oracle


@pytest.mark.parametrize("mode", ["v", "kv"])
def test_fp8_paged_append_and_decode(mode):
    H, n_pages = 3, 12
    pre, tgt = [300, 129, 5], [40, 200, 64]
    kp, vp, qt, kt, vt, cp, cq = _case(95, pre, tgt, H)
    pt, _ = _page_table(pre, n_pages, 6)
    cap = n_pages * 128
    kdt = torch.uint8 if mode == "kv" else torch.bfloat16
    fill_k = 0x7F if mode == "kv" else float("nan")
    ck = torch.full((1, H, cap, 128), fill_k, dtype=kdt, device=DEV)
    cv = torch.full((1, H, cap, 128), 0x7F, dtype=torch.uint8, device=DEV)
    sk = torch.full((1, H, cap), float("nan"), dtype=torch.float32, device=DEV)
    sv = torch.full_like(sk, float("nan"))
    st = bca.new_status(DEV)
    bca.prefix_cache_append_fp8_paged(kp.to(DEV), vp.to(DEV), _ti(cp), _ti(cp), _ti(pt), ck, cv,
                                      sk if mode == "kv" else None, sv, 0, mode=mode, status=st)
    assert bca.read_status(st) == 0
    # expected codes / scales: the oracle's quantisation, placed through the page table
    vc, vs = ofp8.quantize_rows(vp)
    kc, ks = ofp8.quantize_rows(kp)
    got_cv, got_sv = cv.cpu().numpy(), sv.cpu().numpy()
    got_ck, got_sk = ck.cpu(), sk.cpu().numpy()
    for b in range(len(pre)):
        for t in range(pre[b]):
            r, slot = int(cp[b]) + t, pg.page_slot(pt, b, t)
            assert np.array_equal(got_cv[0, :, slot], vc[r])
            assert np.array_equal(got_sv[0, :, slot].view(np.uint32), vs[r].view(np.uint32))
            if mode == "kv":
                assert np.array_equal(got_ck.numpy()[0, :, slot], kc[r])
                assert np.array_equal(got_sk[0, :, slot].view(np.uint32), ks[r].view(np.uint32))
            else:
                assert torch.equal(got_ck[0, :, slot].view(torch.int16), kp[r].view(torch.int16))
    rows = int(cp[-1])
    out, lse = bca.prefix_decode_fp8_paged(qt.to(DEV), ck, cv, sk if mode == "kv" else None, sv,
                                           0, _ti(cp), _ti(pt), rows, kt.to(DEV), vt.to(DEV),
                                           _ti(cq), max(tgt), max(pre), SCALE, mode=mode,
                                           status=st)
    assert bca.read_status(st) == 0
    vh = torch.from_numpy(ofp8.dequantize_rows(vc, vs)).to(torch.bfloat16)
    kh = torch.from_numpy(ofp8.dequantize_rows(kc, ks)).to(torch.bfloat16) if mode == "kv" else kp
    ref = _oracle.prefix_decode(qt, kh, vh, cp, kt, vt, cq, SCALE)
    assert_close(out, lse, *ref, what=f"fp8 paged {mode}")


def test_fp8_paged_decode_equals_contiguous():
    H, n_pages, mode = 2, 6, "kv"
    pre, tgt = [333, 50], [128, 77]
    kp, vp, qt, kt, vt, cp, cq = _case(96, pre, tgt, H)
    pt, _ = _page_table(pre, n_pages, 8)
    d = lambda t: t.to(DEV)
    # paged
    ck = torch.zeros((1, H, n_pages * 128, 128), dtype=torch.uint8, device=DEV)
    cv = torch.zeros_like(ck)
    sk = torch.zeros((1, H, n_pages * 128), dtype=torch.float32, device=DEV)
    sv = torch.zeros_like(sk)
    bca.prefix_cache_append_fp8_paged(d(kp), d(vp), _ti(cp), _ti(cp), _ti(pt), ck, cv, sk, sv, 0,
                                      mode=mode)
    out_p, lse_p = bca.prefix_decode_fp8_paged(d(qt), ck, cv, sk, sv, 0, _ti(cp), _ti(pt),
                                               int(cp[-1]), d(kt), d(vt), _ti(cq), max(tgt),
                                               max(pre), SCALE, mode=mode)
    # contiguous
    cap = int(cp[-1])
    ck2 = torch.zeros((1, H, cap, 128), dtype=torch.uint8, device=DEV)
    cv2 = torch.zeros_like(ck2)
    sk2 = torch.zeros((1, H, cap), dtype=torch.float32, device=DEV)
    sv2 = torch.zeros_like(sk2)
    bca.prefix_cache_append_fp8(d(kp), d(vp), _ti(cp), _ti(cp), ck2, cv2, sk2, sv2, 0, mode=mode)
    out_c, lse_c = bca.prefix_decode_fp8(d(qt), ck2, cv2, sk2, sv2, 0, _ti(cp), d(kt), d(vt),
                                         _ti(cq), max(tgt), max(pre), SCALE, mode=mode)
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse_p, lse_c)
