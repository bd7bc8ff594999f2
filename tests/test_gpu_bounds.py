"""The bounds-checked build (``libbca_gb300_debug.so``, compiled with
``-DBCA_BOUNDS_CHECK``) on small odd cases: every computed index, TMA coordinate
and store address in its kernels is tested against its buffer before use, and a
failed test reports ``BCA_ERR_BOUNDS`` (9) instead of touching memory.  It stands
in for a memory checker, which this GPU pool does not offer.

Each case runs through the debug library, must end with status 0, must match the
oracle at the parity tolerances, and must be bit-identical to the release
library's result (the checks change no arithmetic).  The shapes are the ragged
ones where partial tiles are written: sequence lengths 1, 127, 129 and 1537,
queries shorter than keys, a prefix that ends inside a tile, an empty prefix,
paged tables whose last page is partly used, and prefill and decode grids large
enough to run both the tile-pair grid and the key-split grid, or the decode's
balanced tail (its pieces and their merge).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.paged as opg
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import _native
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV, SCALE, DecodeCase, assert_close, ragged_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build_all()


def _ti(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(DEV)


def _both(fn):
    """fn(status) run through the release and the debug library; the debug run's
    status must be 0.  Returns (release result, debug result)."""
    st = bca.new_status(DEV)
    rel = fn(st)
    assert bca.read_status(st) == 0
    st = bca.new_status(DEV)
    with _native.using_debug():
        dbg = fn(st)
        code = bca.read_status(st)
    assert code == 0, f"bounds-checked build reported status {code}"
    return rel, dbg


def _same(a, b):
    """Bit-identical (NaN fills included)."""
    for x, y in zip(a, b):
        assert x.dtype == y.dtype and x.shape == y.shape
        assert torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8))


# ---------------------------------------------------------------- prefill + cache append

def test_bounds_prefill_append_ragged():
    """Lengths 1 / 127 / 129 / 1537 with q shorter than k in two sequences; the
    prefixes are empty, end inside a tile, fill exactly one tile, end inside a
    later tile.  Output, LSE and cache rows against the oracle; the cache rows
    past the prefixes keep their NaN fill."""
    kv = [1, 127, 129, 1537]
    ql = [1, 100, 129, 1500]
    pre = [0, 27, 128, 700]
    case = ragged_case(201, kv, ql)
    H = case.q.shape[1]
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cap = int(cp[-1]) + 64
    L, layer = 2, 1

    def run(st):
        ck = torch.full((L, H, cap, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        cv = torch.full_like(ck, float("nan"))
        out, lse = bca.prefill_append(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV),
                                      _ti(case.block_id), _ti(case.cu_q), _ti(case.cu_k),
                                      case.max_q, case.max_k, _ti(cp), ck, cv, layer, SCALE,
                                      status=st)
        return out, lse, ck, cv

    rel, dbg = _both(run)
    _same(rel, dbg)
    out, lse, ck, cv = dbg
    ref_out, ref_lse = case.reference()
    assert_close(out, lse, ref_out, ref_lse, what="debug prefill")
    for b in range(len(kv)):
        k0 = int(case.cu_k[b])
        rows = slice(int(cp[b]), int(cp[b + 1]))
        assert torch.equal(ck[layer, :, rows].cpu(), case.k[k0:k0 + pre[b]].permute(1, 0, 2))
        assert torch.equal(cv[layer, :, rows].cpu(), case.v[k0:k0 + pre[b]].permute(1, 0, 2))
    assert torch.isnan(ck[layer, :, int(cp[-1]):].float()).all()
    assert torch.isnan(ck[0].float()).all()


def test_bounds_prefill_paged_append_last_page_partial():
    """The fused append through a page table whose last page of each prefix is
    partly used (prefixes 300, 0, 129 and 5 tokens)."""
    kv = [400, 40, 129, 260]
    pre = [300, 0, 129, 5]
    case = ragged_case(202, kv)
    H = case.q.shape[1]
    n_pages = 12
    need = [math.ceil(p / 128) for p in pre]
    perm = np.random.default_rng(202).permutation(n_pages)
    pt = np.full((len(pre), max(need)), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[at:at + n]
        at += n
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)

    def run(st):
        ck = torch.full((1, H, n_pages * 128, 128), float("nan"), dtype=torch.bfloat16,
                        device=DEV)
        cv = torch.full_like(ck, float("nan"))
        out, lse = bca.prefill_append(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV),
                                      _ti(case.block_id), _ti(case.cu_q), _ti(case.cu_k),
                                      case.max_q, case.max_k, _ti(cp), ck, cv, 0, SCALE,
                                      page_table=_ti(pt), status=st)
        return out, lse, ck, cv

    rel, dbg = _both(run)
    _same(rel, dbg)
    out, lse, ck, cv = dbg
    ref_out, ref_lse = case.reference()
    assert_close(out, lse, ref_out, ref_lse, what="debug paged prefill")
    pool_k = np.full((1, H, n_pages * 128, 128), np.nan)
    pool_v = np.full((1, H, n_pages * 128, 128), np.nan)
    opg.paged_append(case.k, case.v, case.cu_k, cp, pt, 0, pool_k, pool_v)
    for got, exp in ((ck, pool_k), (cv, pool_v)):
        g = got.float().cpu().numpy()
        written = ~np.isnan(exp)
        assert np.array_equal(g[written], exp[written])
        assert np.isnan(g[~written]).all()


@pytest.mark.parametrize("kv,ql,pre", [([2300, 2400], [2300, 1900], [1000, 1700]),
                                       ([2300, 260], [2300, 200], [1000, 150])],
                         ids=["long", "short-second"])
def test_bounds_prefill_key_split_tail(kv, ql, pre):
    """A pair grid short enough for the key-split grid (32 heads, a sequence of 2300 and
    a bottom-right one: 576 pair CTAs, the 120 cheapest pairs split), with the cache
    append.  With a 200-row second sequence its only pair, which appends, is among the
    cheapest and stays a pair CTA, and the split items past its end have no rows.
    Sampled rows against the oracle, bit-identical to the release build."""
    case = ragged_case(203, kv, ql, heads=32, max_spans=6, max_span=700)
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cap = int(cp[-1]) + 64

    def run(st):
        ck = torch.full((1, 32, cap, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        cv = torch.full_like(ck, float("nan"))
        out, lse = bca.prefill_append(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV),
                                      _ti(case.block_id), _ti(case.cu_q), _ti(case.cu_k),
                                      case.max_q, case.max_k, _ti(cp), ck, cv, 0, SCALE,
                                      status=st)
        return out, lse, ck, cv

    rel, dbg = _both(run)
    _same(rel, dbg)
    rows = np.r_[0:130, 1020:1040, 2170:2300, 2300:2430, (4100 if ql[1] > 1800 else 2430):2300 + ql[1]]
    heads = np.array([1, 20, 31])
    ref_out, ref_lse = case.reference(rows=rows, heads=heads)
    assert_close(dbg[0], dbg[1], ref_out, ref_lse, rows=rows, heads=heads, what="debug split")


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("pre,tgt,H,balanced", [
    ([0, 27, 300], [1, 127, 129], 3, True),   # empty prefix, prefix ending mid-tile, 1-row target
    # 160 tile pairs: the pair grid, then 8 pairs of 76 key tiles as the balanced tail
    # (pieces and merge) or, without a workspace, as key-split tiles
    ([8384], [1200], 32, True),
    ([8384], [1200], 32, False),
])
def test_bounds_decode(pre, tgt, H, balanced):
    kp = W.randn_bf16((sum(pre), H, 128), 211)
    vp = W.randn_bf16((sum(pre), H, 128), 212)
    qt = W.randn_bf16((sum(tgt), H, 128), 213)
    kt = W.randn_bf16((sum(tgt), H, 128), 214)
    vt = W.randn_bf16((sum(tgt), H, 128), 215)
    cq = np.concatenate([[0], np.cumsum(tgt)])
    cp = np.concatenate([[0], np.cumsum(pre)])
    case = DecodeCase(qt, kt, vt, kp, vp, cq, cp, layers=2, layer=1, cache_fill=float("nan"))
    rel, dbg = _both(lambda st: case.run(status=st, balanced_tail=balanced))
    _same(rel, dbg)
    rows = None
    if sum(tgt) > 600:   # sampled rows: the tile edges and the last tile
        rows = np.r_[0:130, 255:258, 1000:1200]
    ref_out, ref_lse = case.reference(rows=rows)
    assert_close(dbg[0], dbg[1], ref_out, ref_lse, rows=rows, what="debug decode")


def test_bounds_decode_paged_last_page_partial():
    pre, tgt, H, n_pages = [300, 0, 129, 5], [16, 200, 1, 256], 3, 12
    kp = W.randn_bf16((sum(pre), H, 128), 221)
    vp = W.randn_bf16((sum(pre), H, 128), 222)
    qt = W.randn_bf16((sum(tgt), H, 128), 223)
    kt = W.randn_bf16((sum(tgt), H, 128), 224)
    vt = W.randn_bf16((sum(tgt), H, 128), 225)
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cq = np.concatenate([[0], np.cumsum(tgt)]).astype(np.int32)
    need = [math.ceil(p / 128) for p in pre]
    perm = np.random.default_rng(221).permutation(n_pages)
    pt = np.full((len(pre), max(need)), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[at:at + n]
        at += n

    def run(st):
        ck = torch.full((1, H, n_pages * 128, 128), float("nan"), dtype=torch.bfloat16,
                        device=DEV)
        cv = torch.full_like(ck, float("nan"))
        bca.prefix_cache_append_paged(kp.to(DEV), vp.to(DEV), _ti(cp), _ti(cp), _ti(pt), ck, cv,
                                      0, status=st)
        out, lse = bca.prefix_decode_paged(qt.to(DEV), ck, cv, 0, _ti(cp), _ti(pt), kt.to(DEV),
                                           vt.to(DEV), _ti(cq), max(tgt), max(pre), SCALE,
                                           status=st)
        return out, lse, ck

    rel, dbg = _both(run)
    _same(rel, dbg)
    ref_out, ref_lse = oracle.prefix_decode(qt, kp, vp, cp, kt, vt, cq, SCALE)
    assert_close(dbg[0], dbg[1], ref_out, ref_lse, what="debug paged decode")


# ---------------------------------------------------------------- FP8 cache and prologue

@pytest.mark.parametrize("mode", ["v", "kv"])
def test_bounds_fp8_append_and_decode(mode):
    pre, tgt, H = [27, 300, 0], [129, 1, 127], 3
    kp = W.randn_bf16((sum(pre), H, 128), 231)
    vp = W.randn_bf16((sum(pre), H, 128), 232)
    qt = W.randn_bf16((sum(tgt), H, 128), 233)
    kt = W.randn_bf16((sum(tgt), H, 128), 234)
    vt = W.randn_bf16((sum(tgt), H, 128), 235)
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cq = np.concatenate([[0], np.cumsum(tgt)]).astype(np.int32)
    cap, L = int(cp[-1]) + 40, 2

    def run(st):
        kdt = torch.uint8 if mode == "kv" else torch.bfloat16
        ck = torch.zeros((L, H, cap, 128), dtype=kdt, device=DEV)
        cv = torch.zeros((L, H, cap, 128), dtype=torch.uint8, device=DEV)
        sk = torch.zeros((L, H, cap), dtype=torch.float32, device=DEV) if mode == "kv" else None
        sv = torch.zeros((L, H, cap), dtype=torch.float32, device=DEV)
        bca.prefix_cache_append_fp8(kp.to(DEV), vp.to(DEV), _ti(cp), _ti(cp), ck, cv, sk, sv, 1,
                                    mode=mode, status=st)
        out, lse = bca.prefix_decode_fp8(qt.to(DEV), ck, cv, sk, sv, 1, _ti(cp), kt.to(DEV),
                                         vt.to(DEV), _ti(cq), max(tgt), max(pre), SCALE,
                                         mode=mode, status=st)
        return (out, lse, ck, cv, sv) + ((sk,) if sk is not None else ())

    rel, dbg = _both(run)
    _same(rel, dbg)


def test_bounds_rope_prologue():
    """Coordinates, table and the fused norm + RoPE + append on a ragged layout."""
    case = ragged_case(241, [129, 1, 300], heads=2)
    H = case.q.shape[1]
    cu = case.cu_k
    n_ids = int(case.block_id.max()) + 1 if (case.block_id >= 0).any() else 1
    grid_w = np.ones((len(cu) - 1, max(n_ids, 1)), np.int32)   # width 1: any block length fits
    pre = [100, 0, 129]
    cp = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cap = int(cp[-1]) + 8

    def run(st):
        pos3 = bca.rope_positions(_ti(case.block_id), _ti(cu), _ti(grid_w), status=st)
        table = bca.rope_table(pos3)
        ck = torch.zeros((1, H, cap, 128), dtype=torch.bfloat16, device=DEV)
        cv = torch.zeros_like(ck)
        qo, ko = bca.qk_norm_rope_append(case.q.to(DEV), case.k.to(DEV), table, _ti(cu),
                                         v=case.v.to(DEV), cu_prefix=_ti(cp), cache_k=ck,
                                         cache_v=cv, layer=0, status=st)
        return pos3, table, qo, ko, ck, cv

    rel, dbg = _both(run)
    _same(rel, dbg)


# ---------------------------------------------------------------- validations the checks led to

def test_rope_positions_rejects_tokens_past_total():
    """cu_seqlens whose second sequence runs 60 tokens past `total`: that sequence
    fails with BCA_ERR_SEQLENS and nothing is written behind pos3; the first
    sequence's text coordinates are written."""
    lib = _native.load()
    total = 100
    bid = torch.full((total + 64,), -1, dtype=torch.int32, device=DEV)
    cu = _ti([0, 60, 160])
    grid_w = torch.ones((2, 1), dtype=torch.int32, device=DEV)
    pos3 = torch.full(((total + 64) * 3,), -7, dtype=torch.int32, device=DEV)
    st = bca.new_status(DEV)
    code = lib.bca_rope_positions(bid.data_ptr(), cu.data_ptr(), 2, total, grid_w.data_ptr(), 1,
                                  pos3.data_ptr(), st.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert code == 0
    assert bca.read_status(st) == 8
    p = pos3.view(-1, 3).cpu()
    assert torch.equal(p[:60], torch.arange(60, dtype=torch.int32)[:, None].expand(60, 3))
    assert (p[60:] == -7).all()


@pytest.mark.parametrize("fp8", [False, True])
def test_append_rejects_source_rows_past_total_k(fp8):
    """A prefix whose source keys run past total_k: BCA_ERR_SEQLENS, and no cache
    row is written (by the bf16 and by the FP8 append)."""
    lib = _native.load()
    H, total_k, cap = 2, 200, 512
    k = W.randn_bf16((total_k + 128, H, 128), 251).to(DEV)
    v = W.randn_bf16((total_k + 128, H, 128), 252).to(DEV)
    cu_k = _ti([0, 100, 300])          # the second sequence ends 100 keys past total_k
    cu_p = _ti([0, 50, 200])           # and its 150-token prefix reaches 50 past it
    st = bca.new_status(DEV)
    s = torch.cuda.current_stream().cuda_stream
    if not fp8:
        ck = torch.full((1, H, cap, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        cv = torch.full_like(ck, float("nan"))
        code = lib.bca_prefix_cache_append(k.data_ptr(), v.data_ptr(), cu_k.data_ptr(),
                                           cu_p.data_ptr(), 2, H, 128, total_k, ck.data_ptr(),
                                           cv.data_ptr(), 0, 1, cap, st.data_ptr(), s)
        assert code == 0 and bca.read_status(st) == 8
        assert torch.isnan(ck.float()).all() and torch.isnan(cv.float()).all()
    else:
        ck = torch.full((1, H, cap, 128), 0x55, dtype=torch.uint8, device=DEV)
        cv = torch.full_like(ck, 0x55)
        sk = torch.full((1, H, cap), -1.0, dtype=torch.float32, device=DEV)
        sv = torch.full_like(sk, -1.0)
        code = lib.bca_prefix_cache_append_fp8(k.data_ptr(), v.data_ptr(), cu_k.data_ptr(),
                                               cu_p.data_ptr(), 2, H, 128, total_k, 2,
                                               ck.data_ptr(), cv.data_ptr(), sk.data_ptr(),
                                               sv.data_ptr(), 0, 1, cap, st.data_ptr(), s)
        assert code == 0 and bca.read_status(st) == 8
        assert (ck == 0x55).all() and (cv == 0x55).all()
        assert (sk == -1.0).all() and (sv == -1.0).all()
