"""ctypes view of ``libbca_gb300.so``: loading and C signatures only.

The library is built in-tree by ``prefix_kv_gb300.build_native`` (or
``__graft_entry__.build()``).  If it is missing, every call raises: there is no
fallback implementation.

``libbca_gb300_debug.so`` is the same library compiled with device-side bounds
checks (a failed check skips the access and reports ``BCA_ERR_BOUNDS``);
``using_debug()`` routes every binding call through it for a ``with`` block.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

_LIB_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib")
_LIB_PATH = os.path.join(_LIB_DIR, "libbca_gb300.so")
_DEBUG_PATH = os.path.join(_LIB_DIR, "libbca_gb300_debug.so")
_lock = threading.Lock()
_libs = {}
_lib = None          # the library the bindings call (release unless using_debug() is active)

c_i32, c_i64, c_f32, c_size, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                      ctypes.c_size_t, ctypes.c_void_p)

# name -> (restype, argtypes); mirrors include/bca.h
SIGNATURES = {
    "bca_status_string": (ctypes.c_char_p, [c_i32]),
    "bca_version": (c_i32, []),
    "bca_read_device_status": (c_i32, [c_vp, c_vp]),
    "bca_selftest_wait_timeout": (c_i32, [ctypes.c_uint64, c_vp, c_vp, c_vp]),
    "bca_schedule_prep": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp,
                                  c_vp]),
    "bca_prefill_workspace_bytes": (c_size, [c_i32, c_i32, c_i32]),
    "bca_prefill": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                            c_i32, c_i32, c_i32, c_f32, c_vp, c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_prefill_append": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32,
                                   c_i32, c_i32, c_i32, c_i32, c_f32, c_vp, c_vp, c_vp, c_size,
                                   c_vp, c_vp, c_vp, c_i32, c_i32, c_i64, c_vp, c_vp]),
    "bca_prefill_append_paged": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32,
                                         c_i32, c_i32, c_i32, c_i32, c_i32, c_f32, c_vp, c_vp,
                                         c_vp, c_size, c_vp, c_vp, c_i32, c_vp, c_vp, c_i32,
                                         c_i32, c_i32, c_vp, c_vp]),
    "bca_prefill_noalloc": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                    c_i32, c_i32, c_i32, c_f32, c_vp, c_vp, c_vp, c_vp]),
    "bca_prefix_decode": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp,
                                  c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_f32, c_vp,
                                  c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_prefix_decode_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "bca_prefix_decode_fp8": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_i32, c_i64,
                                      c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32,
                                      c_i32, c_f32, c_vp, c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_prefix_decode_fp8_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i64]),
    "bca_prefix_cache_dequant_fp8": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32,
                                             c_i64, c_vp, c_vp, c_vp]),
    "bca_prefill_piecewise_workspace_bytes": (c_size, [c_vp, c_vp, c_i32, c_i32]),
    "bca_prefill_piecewise": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32,
                                      c_i32, c_f32, c_vp, c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_prefix_cache_append_paged": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32,
                                              c_i32, c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp,
                                              c_vp]),
    "bca_prefix_decode_paged": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_i32,
                                        c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                        c_f32, c_vp, c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_prefix_cache_append_fp8_paged": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32,
                                                  c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp,
                                                  c_vp, c_i32, c_i32, c_i32, c_vp, c_vp]),
    "bca_prefix_decode_fp8_paged_workspace_bytes": (c_size, [c_i32, c_i32, c_i64]),
    "bca_prefix_decode_fp8_paged": (c_i32, [c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_i32,
                                            c_i32, c_vp, c_vp, c_i32, c_i64, c_vp, c_vp, c_vp,
                                            c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_f32, c_vp,
                                            c_vp, c_vp, c_size, c_vp, c_vp]),
    "bca_pool_copy_rows": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                   c_vp]),
    "bca_pool_create": (c_vp, [c_i32]),
    "bca_pool_destroy": (None, [c_vp]),
    "bca_pool_alloc": (c_i32, [c_vp, c_i32, c_vp]),
    "bca_pool_match": (c_i32, [c_vp, c_vp, c_i32, c_vp]),
    "bca_pool_publish": (c_i32, [c_vp, c_i32, ctypes.c_uint64]),
    "bca_pool_release": (c_i32, [c_vp, c_vp, c_i32]),
    "bca_pool_stats": (None, [c_vp, c_vp, c_vp, c_vp]),
    "bca_pool_refs": (c_i32, [c_vp, c_i32]),
    "bca_rope_positions": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp]),
    "bca_rope_table": (c_i32, [c_vp, c_i32, c_vp, c_vp]),
    "bca_qk_norm_rope_append": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                                        c_i32, c_i32, c_i32, c_f32, c_vp, c_vp, c_vp, c_vp, c_i32,
                                        c_i32, c_i64, c_vp, c_vp]),
    "bca_prefix_cache_append_fp8": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                            c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i64,
                                            c_vp, c_vp]),
    "bca_prefix_cache_append": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                        c_vp, c_vp, c_i32, c_i32, c_i64, c_vp, c_vp]),
}


def lib_path() -> str:
    return _LIB_PATH


def _open(path: str):
    with _lock:
        if path not in _libs:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _libs[path] = lib
        return _libs[path]


def load():
    """The library the bindings call: the release build (loaded once with its C
    signatures), or the bounds-checked build inside ``using_debug()``."""
    global _lib
    if _lib is None:
        _lib = _open(_LIB_PATH)
    return _lib


def load_debug():
    """The bounds-checked build, ``libbca_gb300_debug.so``."""
    return _open(_DEBUG_PATH)


@contextlib.contextmanager
def using_debug():
    """Route every binding call through the bounds-checked build (not thread-safe:
    meant for tests)."""
    global _lib
    prev = load()
    _lib = load_debug()
    try:
        yield _lib
    finally:
        _lib = prev


class BcaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().bca_status_string(code).decode()
        super().__init__(f"{where}: status {code} ({msg})")


def check(code: int, where: str) -> None:
    if code != 0:
        raise BcaError(code, where)
