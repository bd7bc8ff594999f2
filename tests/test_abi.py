"""The C-ABI library loads and exports every symbol the header declares; host-side
argument validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bca.h")


@pytest.fixture(scope="module")
def lib():
    from prefix_kv_gb300 import _native, build_native
    build_native.build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bca_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("bca_prefill", "bca_prefix_decode", "bca_prefix_cache_append",
              "bca_schedule_prep", "bca_prefill_workspace_bytes", "bca_status_string",
              "bca_read_device_status", "bca_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_header():
    from prefix_kv_gb300 import _native
    assert set(_native.SIGNATURES) == set(declared_functions())


def declared_arity():
    """Number of parameters of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(bca_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_header():
    from prefix_kv_gb300 import _native
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, (_, argtypes) in _native.SIGNATURES.items():
        assert len(argtypes) == arity[name], name


def test_status_strings(lib):
    assert lib.bca_status_string(0) == b"ok"
    for code in range(1, 10):
        assert lib.bca_status_string(code) not in (b"ok", b"unknown status")
    assert lib.bca_status_string(99) == b"unknown status"
    assert lib.bca_version() >= 100


def test_workspace_bytes(lib):
    # row ends (4 B per query row) + 16 B per (sequence, 128-row tile), each 256-B rounded
    assert lib.bca_prefill_workspace_bytes(1, 12480, 12480) == 49920 + 1792
    assert lib.bca_prefill_workspace_bytes(2, 66184, 33352) == 264960 + 8448
    assert lib.bca_prefill_workspace_bytes(-1, 1, 1) == 0


def _prefill(lib, **kw):
    a = dict(q=16, k=16, v=16, bid=16, cq=16, ck=16, batch=1, H=2, D=128, tq=8, tk=8, mq=8,
             mk=8, scale=0.1, out=16, lse=16, ws=16, wsb=1 << 20, status=None, stream=None)
    a.update(kw)
    return lib.bca_prefill(a["q"], a["k"], a["v"], a["bid"], a["cq"], a["ck"], a["batch"],
                           a["H"], a["D"], a["tq"], a["tk"], a["mq"], a["mk"], a["scale"],
                           a["out"], a["lse"], a["ws"], a["wsb"], a["status"], a["stream"])


def test_prefill_host_validation(lib):
    assert _prefill(lib, D=64) == 2                     # UNSUPPORTED head dim
    assert _prefill(lib, H=0) == 1
    assert _prefill(lib, scale=0.0) == 1
    assert _prefill(lib, scale=float("nan")) == 1
    assert _prefill(lib, mq=9, mk=8) == 1               # q longer than kv
    assert _prefill(lib, q=None) == 1
    assert _prefill(lib, q=24) == 1                     # misaligned
    assert _prefill(lib, ws=None) == 4                  # workspace missing
    assert _prefill(lib, wsb=8) == 4                    # workspace too small
    assert _prefill(lib, tq=0) == 0                     # nothing to do
    assert _prefill(lib, batch=0) == 0
    assert _prefill(lib, tk=0) == 8


def _prefill_append(lib, **kw):
    a = dict(q=16, k=16, v=16, bid=16, cq=16, ck=16, batch=1, H=2, D=128, tq=8, tk=8, mq=8,
             mk=8, scale=0.1, out=16, lse=16, ws=16, wsb=1 << 20, cp=16, cck=16, ccv=16,
             layer=0, L=1, cap=64, status=None, stream=None)
    a.update(kw)
    return lib.bca_prefill_append(a["q"], a["k"], a["v"], a["bid"], a["cq"], a["ck"], a["batch"],
                                  a["H"], a["D"], a["tq"], a["tk"], a["mq"], a["mk"], a["scale"],
                                  a["out"], a["lse"], a["ws"], a["wsb"], a["cp"], a["cck"],
                                  a["ccv"], a["layer"], a["L"], a["cap"], a["status"],
                                  a["stream"])


def test_prefill_append_host_validation(lib):
    assert _prefill_append(lib, D=64) == 2               # UNSUPPORTED head dim
    assert _prefill_append(lib, layer=1, L=1) == 1       # layer outside the cache
    assert _prefill_append(lib, layer=-1) == 1
    assert _prefill_append(lib, cap=-1) == 1
    assert _prefill_append(lib, cck=None) == 1           # cache missing
    assert _prefill_append(lib, cp=None) == 1
    assert _prefill_append(lib, ccv=24) == 1             # misaligned cache
    assert _prefill_append(lib, scale=0.0) == 1          # the prefill's own checks follow
    assert _prefill_append(lib, ws=None) == 4
    assert _prefill_append(lib, tq=0) == 0               # nothing to do


def test_prefill_append_paged_host_validation(lib):
    def call(**kw):
        a = dict(D=128, pt=16, mp=2, cck=16, ccv=16, layer=0, L=1, pages=4, cp=16)
        a.update(kw)
        return lib.bca_prefill_append_paged(16, 16, 16, 16, 16, 16, 1, 2, a["D"], 8, 8, 8, 8, 0.1,
                                            16, 16, 16, 1 << 20, a["cp"], a["pt"], a["mp"],
                                            a["cck"], a["ccv"], a["layer"], a["L"], a["pages"],
                                            None, None)
    assert call(D=64) == 2
    assert call(pages=0) == 1                  # empty pool
    assert call(pages=(1 << 24) + 1) == 1
    assert call(mp=-1) == 1
    assert call(pt=None) == 1
    assert call(layer=1) == 1
    assert call(ccv=24) == 1                   # misaligned cache


def test_decode_and_append_host_validation(lib):
    dec = lib.bca_prefix_decode
    #         q   ck  cv  layer L  cap  cup tk  tv  cq  B  H  D    tq mq mp scale out lse ws wsb st s
    args = [16, 16, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1, 16, 16, None, 0, None,
            None]

    def call(**kw):
        a = list(args)
        for name, val in kw.items():
            a[{"layer": 3, "ck": 1, "D": 12, "tq": 13, "scale": 16, "ws": 19, "wsb": 20}[name]] = val
        return dec(*a)

    assert call(D=96) == 2
    assert call(layer=1) == 1
    assert call(scale=-1.0) == 1
    assert call(tq=0) == 0
    assert call(ck=8) == 1
    assert call(ws=24, wsb=1 << 20) == 4            # a misaligned workspace
    wsb = lib.bca_prefix_decode_workspace_bytes
    #          B  H  D    mq    mp
    assert wsb(1, 2, 64, 1000, 1000) == 0            # head_dim other than 128
    assert wsb(0, 2, 128, 1000, 1000) == 0 and wsb(1, 2, 128, 0, 1000) == 0
    app = lib.bca_prefix_cache_append
    #          k   v  ck  cp  B  H  D    tk ck  cv  layer L cap st  s
    assert app(16, 16, 16, 16, 1, 2, 64, 8, 16, 16, 0, 1, 64, None, None) == 2
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 16, 16, 2, 2, 64, None, None) == 1
    assert app(16, 16, 16, 16, 1, 2, 128, 8, None, 16, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 0, 2, 128, 8, 16, 16, 0, 1, 64, None, None) == 0


def test_fp8_entry_points_host_validation(lib):
    app = lib.bca_prefix_cache_append_fp8
    #          k   v  ck  cp  B  H  D    tk mode ck  cv  sk  sv  layer L cap st  s
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 0, 16, 16, 16, 16, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 1, 2, 64, 8, 1, 16, 16, 16, 16, 0, 1, 64, None, None) == 2
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 1, 16, 16, 16, None, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 2, 16, 16, None, 16, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 1, 16, 16, 16, 18, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 0, 2, 128, 8, 1, 16, 16, 16, 16, 0, 1, 64, None, None) == 0
    deq = lib.bca_prefix_cache_dequant_fp8
    #          codes sc  cp  B  H  D    layer L cap out st  s
    assert deq(16, 16, 16, 1, 2, 64, 0, 1, 64, 16, None, None) == 2
    assert deq(16, 16, 16, 1, 2, 128, 1, 1, 64, 16, None, None) == 1
    assert deq(16, 16, 16, 1, 2, 128, 0, 1, 64, None, None, None) == 1
    assert deq(24, 16, 16, 1, 2, 128, 0, 1, 64, 16, None, None) == 1
    assert deq(16, 16, 16, 1, 2, 128, 0, 1, 0, 16, None, None) == 0
    wsb = lib.bca_prefix_decode_fp8_workspace_bytes
    assert wsb(1, 2, 128, 64) == 2 * 64 * 128 * 2
    assert wsb(2, 2, 128, 64) == 2 * 2 * 64 * 128 * 2
    assert wsb(0, 2, 128, 64) == 0 and wsb(1, 2, 64, 64) == 0
    dec = lib.bca_prefix_decode_fp8
    # q ck cv mode sk sv layer L cap cup tk tv cq B H D tq mq mp scale out lse ws wsb st s
    args = [16, 16, 16, 1, 16, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1, 16, 16,
            16, 1 << 20, None, None]
    bad_mode = list(args); bad_mode[3] = 0
    assert dec(*bad_mode) == 1
    no_ws = list(args); no_ws[22] = None
    assert dec(*no_ws) == 4
    small_ws = list(args); small_ws[23] = 100
    assert dec(*small_ws) == 4


def test_prologue_entry_points_host_validation(lib):
    pos = lib.bca_rope_positions
    #          bid cu  B  total gw  n_ids pos st  s
    assert pos(16, 16, 1, 8, 16, 5000, 16, None, None) == 2
    assert pos(16, 16, -1, 8, 16, 1, 16, None, None) == 1
    assert pos(16, 16, 1, 8, None, 1, 16, None, None) == 1
    assert pos(16, 16, 0, 8, 16, 1, 16, None, None) == 0
    tab = lib.bca_rope_table
    assert tab(16, -1, 16, None) == 1
    assert tab(16, 4, 24, None) == 1                  # table misaligned
    assert tab(16, 0, 16, None) == 0
    qk = lib.bca_qk_norm_rope_append
    # q k v gq gk table cu cp B H D total eps qo ko ck cv layer L cap st s
    base = [16, 16, 16, 16, 16, 16, 16, None, 1, 2, 128, 8, 1e-6, 16, 16, None, None, 0, 1, 0,
            None, None]
    d64 = list(base); d64[10] = 64
    assert qk(*d64) == 2
    neg_eps = list(base); neg_eps[12] = -1.0
    assert qk(*neg_eps) == 1
    nan_eps = list(base); nan_eps[12] = float("nan")
    assert qk(*nan_eps) == 1
    bad_gamma = list(base); bad_gamma[3] = 20
    assert qk(*bad_gamma) == 1
    app_no_v = list(base); app_no_v[7] = 16; app_no_v[2] = None; app_no_v[15] = 16
    app_no_v[16] = 16; app_no_v[19] = 64
    assert qk(*app_no_v) == 1
    empty = list(base); empty[11] = 0
    assert qk(*empty) == 0


def test_piecewise_host_validation(lib):
    bid = (ctypes.c_int32 * 8)(-1, -1, 0, 0, 0, -1, 1, 1)
    cu = (ctypes.c_int32 * 2)(0, 8)
    need = lib.bca_prefill_piecewise_workspace_bytes(bid, cu, 1, 2)
    assert need > 0
    assert lib.bca_prefill_piecewise_workspace_bytes(None, cu, 1, 2) == 0
    pw = lib.bca_prefill_piecewise
    # q k v bid bid_h cu_h B H D total scale out lse ws wsb st s
    args = [16, 16, 16, 16, bid, cu, 1, 2, 128, 8, 0.1, 16, 16, 16, need, None, None]
    d64 = list(args); d64[8] = 64
    assert pw(*d64) == 2
    short = list(args); short[9] = 9                    # cu_seqlens does not end at total
    assert pw(*short) == 8
    small = list(args); small[14] = need - 1
    assert pw(*small) == 4
    empty = list(args); empty[6] = 0
    assert pw(*empty) == 0


def test_paged_entry_points_host_validation(lib):
    app = lib.bca_prefix_cache_append_paged
    # k v ck cp pt maxp B H D tk ck cv layer L npages st s
    assert app(16, 16, 16, 16, 16, 2, 1, 2, 128, 8, 16, 16, 0, 1, 0, None, None) == 1
    assert app(16, 16, 16, 16, None, 2, 1, 2, 128, 8, 16, 16, 0, 1, 4, None, None) == 1
    assert app(16, 16, 16, 16, 16, 2, 1, 2, 64, 8, 16, 16, 0, 1, 4, None, None) == 2
    dec = lib.bca_prefix_decode_paged
    # q ck cv layer L npages cp pt maxp tk tv cq B H D tq mq mp scale out lse ws wsb st s
    args = [16, 16, 16, 0, 1, 4, 16, 16, 2, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1, 16, 16, None, 0,
            None, None]
    no_pages = list(args); no_pages[5] = 0
    assert dec(*no_pages) == 1
    no_table = list(args); no_table[7] = None
    assert dec(*no_table) == 1
    odd_ws = list(args); odd_ws[21] = 40; odd_ws[22] = 1 << 20
    assert dec(*odd_ws) == 4
    cp = lib.bca_pool_copy_rows
    # ck cv layer L H npages src dst rows s
    assert cp(16, 16, 0, 1, 2, 4, 1, 1, 10, None) == 0   # same page: nothing to do
    assert cp(16, 16, 0, 1, 2, 4, 1, 2, 129, None) == 1
    assert cp(16, 16, 0, 1, 2, 4, 4, 2, 10, None) == 1
    assert cp(16, 16, 0, 1, 2, 4, 1, 2, 0, None) == 0
    a8 = lib.bca_prefix_cache_append_fp8_paged
    # k v ck cp pt maxp B H D tk mode ck cv sk sv layer L npages st s
    assert a8(16, 16, 16, 16, 16, 2, 1, 2, 128, 8, 1, 16, 16, 16, 16, 0, 1, 0, None, None) == 1
    assert a8(16, 16, 16, 16, 16, 2, 1, 2, 128, 8, 3, 16, 16, 16, 16, 0, 1, 4, None, None) == 1
    d8 = lib.bca_prefix_decode_fp8_paged
    # q ck cv mode sk sv layer L npages cp pt maxp rows tk tv cq B H D tq mq mp scale out lse ws wsb st s
    args8 = [16, 16, 16, 1, 16, 16, 0, 1, 4, 16, 16, 2, 256, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1,
             16, 16, 16, 1 << 20, None, None]
    m0 = list(args8); m0[3] = 0
    assert d8(*m0) == 1
    small = list(args8); small[26] = 10
    assert d8(*small) == 4
    assert lib.bca_prefix_decode_fp8_paged_workspace_bytes(2, 128, 256) == 2 * 2 * 256 * 128 * 2
