"""CPU oracle for exact bulk cosine similarity over CSR sparse embeddings.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline / reference legs may import this package; the library under
``sparse_embedding_exact_gb300`` never does.  It shares no code with the CUDA
path.

The arithmetic lives in ``cosine_oracle.c`` (plain C, double precision, the
two-pointer merge of the post's section 3.1); this module compiles it with gcc
and calls it through ctypes.  Every function here is pinned by tests that do
not call it to compute their expected values: dense float64 brute force,
scipy.sparse products, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cosine_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_libs = {}
_lock = threading.Lock()

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def library_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one of its planted-mistake mutants) with gcc."""
    out = library_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-pthread", "-shared", "-fPIC", "-fno-fast-math",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        lib = _libs.get(mutant)
        if lib is None:
            lib = ctypes.CDLL(build(mutant))
            lib.oracle_row_norms.argtypes = [ctypes.c_int64, _i64p, _f32p, _f64p]
            lib.oracle_row_norms.restype = ctypes.c_int
            lib.oracle_check_csr.argtypes = [ctypes.c_int64, _i64p, _i32p, ctypes.c_int64]
            lib.oracle_check_csr.restype = ctypes.c_int64
            common = [_i64p, _i32p, _f32p, ctypes.c_int64, _i64p, _i32p, _f32p, ctypes.c_int64,
                      _i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            lib.oracle_cosine.argtypes = common + [_f64p, _f32p, ctypes.c_int]
            lib.oracle_cosine.restype = ctypes.c_int
            lib.oracle_dot.argtypes = common + [_f64p]
            lib.oracle_dot.restype = ctypes.c_int
            lib.oracle_mutant_id.restype = ctypes.c_int
            _libs[mutant] = lib
        return lib


def _ptr(a: Optional[np.ndarray], typ):
    if a is None:
        return ctypes.cast(None, typ)
    return a.ctypes.data_as(typ)


def _csr(m):
    indptr = np.ascontiguousarray(m.indptr, dtype=np.int64)
    indices = np.ascontiguousarray(m.indices, dtype=np.int32)
    values = np.ascontiguousarray(m.values, dtype=np.float32)
    return indptr, indices, values, int(indptr.shape[0] - 1)


def threads_available() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def row_norms(m, mutant: int = 0) -> np.ndarray:
    """float64 Euclidean norm of every row over its stored values (section 5.2)."""
    indptr, _, values, n = _csr(m)
    out = np.empty(n, np.float64)
    rc = _load(mutant).oracle_row_norms(n, _ptr(indptr, _i64p), _ptr(values, _f32p), _ptr(out, _f64p))
    if rc:
        raise ValueError("oracle_row_norms: bad argument")
    return out


def check_csr(m) -> int:
    """First row breaking the CSR rules (sorted unique indices in range), or -1."""
    indptr, indices, _, n = _csr(m)
    return int(_load().oracle_check_csr(n, _ptr(indptr, _i64p), _ptr(indices, _i32p), int(m.dim)))


def _args(Q, I, q_rows, i_begin, i_end):
    qp, qi, qv, n_q = _csr(Q)
    ip, ii, iv, n_i = _csr(I)
    if i_end is None:
        i_end = n_i
    if q_rows is not None:
        q_rows = np.ascontiguousarray(q_rows, dtype=np.int64)
        n_sel = int(q_rows.shape[0])
    else:
        n_sel = n_q
    keep = (qp, qi, qv, ip, ii, iv, q_rows)
    args = [_ptr(qp, _i64p), _ptr(qi, _i32p), _ptr(qv, _f32p), n_q,
            _ptr(ip, _i64p), _ptr(ii, _i32p), _ptr(iv, _f32p), n_i,
            _ptr(q_rows, _i64p), n_sel, int(i_begin), int(i_end)]
    return keep, args, n_sel, int(i_end) - int(i_begin)


def cosine(Q, I, q_rows=None, i_begin: int = 0, i_end: Optional[int] = None,
           f64: bool = False, threads: Optional[int] = None, mutant: int = 0) -> np.ndarray:
    """S[s, c] = cos(Q[q_rows[s]], I[i_begin + c]).

    Returns float32 (rounded once from double) unless f64 is set, in which case
    the double value before rounding is returned.
    """
    keep, args, n_sel, width = _args(Q, I, q_rows, i_begin, i_end)
    out = np.empty((n_sel, width), np.float64 if f64 else np.float32)
    o64 = out if f64 else None
    o32 = None if f64 else out
    rc = _load(mutant).oracle_cosine(*args, _ptr(o64, _f64p), _ptr(o32, _f32p),
                                     int(threads or threads_available()))
    del keep
    if rc:
        raise ValueError(f"oracle_cosine failed ({rc})")
    return out


def dot(Q, I, q_rows=None, i_begin: int = 0, i_end: Optional[int] = None,
        mutant: int = 0) -> np.ndarray:
    """Unnormalised sparse dot products in float64 (section 3.1)."""
    keep, args, n_sel, width = _args(Q, I, q_rows, i_begin, i_end)
    out = np.empty((n_sel, width), np.float64)
    rc = _load(mutant).oracle_dot(*args, _ptr(out, _f64p))
    del keep
    if rc:
        raise ValueError(f"oracle_dot failed ({rc})")
    return out


def mutant_id(mutant: int) -> int:
    return int(_load(mutant).oracle_mutant_id())
