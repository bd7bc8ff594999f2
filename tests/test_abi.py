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


def test_status_strings(lib):
    assert lib.bca_status_string(0) == b"ok"
    for code in range(1, 9):
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


def test_decode_and_append_host_validation(lib):
    dec = lib.bca_prefix_decode
    #         q   ck  cv  layer L  cap  cup tk  tv  cq  B  H  D    tq mq mp scale out lse st  s
    assert dec(16, 16, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 96, 8, 8, 8, 0.1, 16, 16, None, None) == 2
    assert dec(16, 16, 16, 1, 1, 64, 16, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1, 16, 16, None, None) == 1
    assert dec(16, 16, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 128, 8, 8, 8, -1.0, 16, 16, None, None) == 1
    assert dec(16, 16, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 128, 0, 8, 8, 0.1, 16, 16, None, None) == 0
    assert dec(16, 8, 16, 0, 1, 64, 16, 16, 16, 16, 1, 2, 128, 8, 8, 8, 0.1, 16, 16, None, None) == 1
    app = lib.bca_prefix_cache_append
    #          k   v  ck  cp  B  H  D    tk ck  cv  layer L cap st  s
    assert app(16, 16, 16, 16, 1, 2, 64, 8, 16, 16, 0, 1, 64, None, None) == 2
    assert app(16, 16, 16, 16, 1, 2, 128, 8, 16, 16, 2, 2, 64, None, None) == 1
    assert app(16, 16, 16, 16, 1, 2, 128, 8, None, 16, 0, 1, 64, None, None) == 1
    assert app(16, 16, 16, 16, 0, 2, 128, 8, 16, 16, 0, 1, 64, None, None) == 0
