"""ctypes view of ``libbca_gb300.so``: loading and C signatures only.

The library is built in-tree by ``prefix_kv_gb300.build_native`` (or
``__graft_entry__.build()``).  If it is missing, every call raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libbca_gb300.so")
_lock = threading.Lock()
_lib = None

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
                                  c_vp, c_vp, c_vp]),
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
                                        c_f32, c_vp, c_vp, c_vp, c_vp]),
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


def load():
    """Load the shared library (once) and attach the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {_LIB_PATH} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class BcaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().bca_status_string(code).decode()
        super().__init__(f"{where}: status {code} ({msg})")


def check(code: int, where: str) -> None:
    if code != 0:
        raise BcaError(code, where)
