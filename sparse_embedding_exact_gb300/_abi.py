"""ctypes declarations of the C ABI in include/sparsecos.h.

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

SS_OK = 0
SS_ERR_INVALID_ARG = 1
SS_ERR_UNSORTED = 2
SS_ERR_OUT_OF_RANGE = 3
SS_ERR_OOM = 4
SS_ERR_CUDA = 5
SS_ERR_DEVICE_CHECK = 6
SS_ERR_TIMEOUT = 7
SS_ERR_LIMIT = 8
SS_VALIDATE = 0x1
SS_TOPK_MAX = 64
SS_VERIFY_STREAM = 0x4
SS_ALGO_POSTING_LISTS = 0x2
SS_ALGO_TILES = 0x8
SS_ALGO_TENSOR = 0x10
SS_MAX_CHUNK_ROWS = 65536
SS_VALUES_F32 = 0
SS_VALUES_BF16 = 1
SS_VALUES_F16 = 2
SS_EXPORT_HOT_MAX = 160
SS_DEVICE_OK = 0
SS_DEVICE_UNSORTED = 1
SS_DEVICE_OUT_OF_RANGE = 2
SS_DEVICE_CAPACITY = 3
SS_DEVICE_STALL = 4
SS_DEVICE_RANGE = 5


class ss_csr(ctypes.Structure):
    _fields_ = [
        ("indptr", ctypes.c_void_p),
        ("indices", ctypes.c_void_p),
        ("values", ctypes.c_void_p),
        ("n_rows", ctypes.c_int64),
        ("nnz", ctypes.c_int64),
        ("dim", ctypes.c_int64),
    ]


ss_chunk_consumer = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.POINTER(ctypes.c_float), ctypes.c_int64,
                                     ctypes.c_int64)

_P = ctypes.c_void_p
_CSR = ctypes.POINTER(ss_csr)
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32

# name -> (restype, argtypes); one entry per function declared in the header.
SIGNATURES = {
    "ss_create": (_I32, [ctypes.POINTER(_P), ctypes.c_int, _I64, _I32, _I32]),
    "ss_row_norms": (_I32, [_P, _CSR, _P, _P]),
    "ss_build_item_index": (_I32, [_P, _CSR, _I64, _I64, ctypes.POINTER(_P), _P]),
    "ss_build_batch": (_I32, [_P]),
    "ss_build_item_indexes": (_I32, [_P, _CSR, _I64, _I64, ctypes.POINTER(_P), ctypes.POINTER(_I32), _P]),
    "ss_score_chunk": (_I32, [_P, _CSR, _P, _P, _P, _P, _I64, _P]),
    "ss_score_all": (_I32, [_P, _CSR, _P, _CSR, _P, _P, _I64, _P]),
    "ss_topk_reset": (_I32, [_P, _I64, _I32, _P, _P, _P]),
    "ss_score_chunk_topk": (_I32, [_P, _CSR, _P, _P, _P, _I32, _P, _P, _P]),
    "ss_topk_all": (_I32, [_P, _CSR, _P, _CSR, _P, _I32, _P, _P, _P]),
    "ss_tile_checksum": (_I32, [_P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "ss_tile_checksum_host": (_I32, [_P, _I64, _I64, _I64, _P, _P]),
    "ss_stream_checksum": (_I32, [_P, _I64, _P, _P]),
    "ss_bulk_cosine_host": (_I32, [_P, _CSR, _CSR, _P, _I64, ss_chunk_consumer, _P, _I32, _I32]),
    "ss_set_device_limit": (_I32, [_P, _I64]),
    "ss_set_host_values": (_I32, [_P, _I32]),
    "ss_plan_host_pass": (_I32, [_P, _I64, _P, _I64, _I32, _I64, _I32, _I32, _P, _I64,
                                 ctypes.POINTER(_I64), _P, _I64, ctypes.POINTER(_I64)]),
    "ss_validate_csr": (_I32, [_P, _CSR, _P]),
    "ss_check_device": (_I32, [_P, _P]),
    "ss_invalidate": (_I32, [_P]),
    "ss_index_stats": (_I32, [_P, _P, ctypes.POINTER(ctypes.c_int64), _P]),
    "ss_index_export": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, ctypes.POINTER(_I64), _P]),
    "ss_lists_export": (_I32, [_P, ctypes.POINTER(_I64), _P, _P, _P, _P, _I64, ctypes.POINTER(_I64), _P]),
    "ss_cosine_chunk_noalloc": (_I32, [_CSR, _CSR, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "ss_kernel_launches": (ctypes.c_uint64, [_P]),
    "ss_inject_alloc_failure": (_I64, [_I64]),
    "ss_profile_scorer": (_I32, [_P, _I32]),
    "ss_scorer_time": (_I32, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64)]),
    "ss_destroy": (_I32, [_P]),
    "ss_status_string": (ctypes.c_char_p, [_I32]),
    "ss_last_error": (ctypes.c_char_p, [_P]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded CUDA library; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path) or not _build.up_to_date():
        if build_if_missing:
            _build.build()
        elif not os.path.exists(path):
            raise ImportError(
                f"the sparsecos CUDA library is not built ({path} is missing); "
                "run __graft_entry__.build() or python -m sparse_embedding_exact_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class SparseCosError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status
