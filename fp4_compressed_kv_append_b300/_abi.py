"""ctypes view of libcsa2.so: structs, prototypes and status handling.

Loading fails loudly when the library is missing: there is no other
implementation of these operations in this package.
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libcsa2.so")

# csa2_status
OK, ERR_ARG, ERR_ALIGN, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS, ERR_WORKSPACE = range(8)
F32, BF16 = 0, 1
FULL, REINDEX, REUSE = 0, 1, 2
LATENT_DIM, INDEXER_DIM, INDEXER_HEADS, MAX_TOPK, MAX_WINDOW = 512, 128, 4, 16384, 1024
STATIC_WS_BYTES = 24 << 20  # CSA2_STATIC_WS_BYTES


class CacheView(C.Structure):
    _fields_ = [("lat_codes", C.c_void_p), ("lat_scales", C.c_void_p), ("idx_codes", C.c_void_p),
                ("idx_scales", C.c_void_p), ("len", C.c_void_p), ("cap", C.c_int64), ("batch", C.c_int32)]


class LayerDesc(C.Structure):
    _fields_ = [("mode", C.c_int), ("cache", C.POINTER(CacheView)), ("own_idx_codes", C.c_void_p),
                ("own_idx_scales", C.c_void_p), ("q_idx", C.c_void_p), ("w_idx", C.c_void_p),
                ("pool", C.c_int32), ("q_idx2", C.c_void_p), ("w_idx2", C.c_void_p), ("q", C.c_void_p),
                ("swa", C.c_void_p), ("swa_codes", C.c_void_p), ("swa_scales", C.c_void_p), ("W", C.c_int32),
                ("out", C.c_void_p), ("idx_out", C.c_void_p)]


class StoreLayer(C.Structure):
    _fields_ = [("lat", C.c_void_p), ("ikey", C.c_void_p), ("ratio", C.c_int32), ("w0_lat", C.c_void_p),
                ("w1_lat", C.c_void_p), ("w0_idx", C.c_void_p), ("w1_idx", C.c_void_p),
                ("cache", C.POINTER(CacheView))]


class Csa2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


_lib = None

_PROTOS = {
    "kv_quant_append": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_void_p, C.POINTER(CacheView), C.c_void_p]),
    "indexer_score": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                                C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p]),
    "topk_select": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32,
                              C.c_void_p]),
    "sparse_latent_attn": (C.c_int, [C.c_void_p, C.c_int, C.c_int32, C.c_float, C.POINTER(CacheView), C.c_void_p,
                                     C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p,
                                     C.c_void_p]),
    "csa2_swa_quant": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_store_append": (C.c_int, [C.POINTER(StoreLayer), C.c_int32, C.c_int, C.c_int32, C.c_void_p]),
    "csa2_decode_step": (C.c_int, [C.POINTER(LayerDesc), C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int,
                                   C.c_void_p, C.c_size_t, C.c_void_p]),
    "csa2_decode_step_static": (C.c_int, [C.POINTER(LayerDesc), C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int,
                                          C.c_void_p]),
    "csa2_workspace_size": (C.c_size_t, [C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "csa2_sync_status": (C.c_int, [C.c_void_p]),
    "csa2_status_str": (C.c_char_p, [C.c_int]),
    "csa2_launch_count": (C.c_uint64, []),
    "csa2_set_scan_events": (C.c_int, [C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int32]),
    "csa2_selftest_wait_timeout": (C.c_int, [C.c_uint64, C.c_void_p]),
}


def lib() -> C.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcsa2.so not built ({LIB_PATH}); run "
                              "`python -m fp4_compressed_kv_append_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _PROTOS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().csa2_status_str(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != OK:
        raise Csa2Error(status, what)
