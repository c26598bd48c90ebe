"""Exact bulk cosine similarity between CSR batches of sparse embeddings on GB300.

A thin Python layer over the C ABI of ``include/sparsecos.h``: it turns torch
tensors into pointers and sizes and calls the CUDA library.  Every step of the
computation runs in the library's kernels; this package has no fallback path
and raises if the library is missing.

    S[q, i] = (Q_q . I_i) / (|Q_q|_2 |I_i|_2)

The calls mirror the C ABI: ``row_norms``, ``build_item_index``,
``score_chunk``, ``score_all`` (the device-resident chunk loop),
``topk_all`` / ``score_chunk_topk`` (the k best items per query row instead
of the matrix) and ``bulk_cosine_host`` (host buffers in, result streamed
back chunk by chunk; ``set_device_limit`` bounds its device memory, with
item batches streamed and queries tiled, see ``plan_host_pass``; 16-bit
host values with ``host_values="bf16"`` or ``"f16"``).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np
import torch

from . import _abi
from ._abi import SparseCosError, SS_VALIDATE  # noqa: F401

DEFAULT_CHUNK_ROWS = 8192


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@dataclass
class DeviceCsr:
    """A CSR matrix in device memory (int64 indptr, int32 indices, float32 values)."""

    indptr: torch.Tensor
    indices: torch.Tensor
    values: torch.Tensor
    dim: int

    @property
    def n_rows(self) -> int:
        return int(self.indptr.shape[0] - 1)

    @property
    def nnz(self) -> int:
        return int(self.indices.shape[0])

    def abi(self) -> _abi.ss_csr:
        return _abi.ss_csr(self.indptr.data_ptr(), self.indices.data_ptr(), self.values.data_ptr(),
                           self.n_rows, self.nnz, int(self.dim))

    @staticmethod
    def from_host(batch, device="cuda") -> "DeviceCsr":
        """Copies a host CSR (anything with indptr/indices/values/dim arrays)."""
        def dev(a, dt):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(device)
        return DeviceCsr(dev(batch.indptr, np.int64), dev(batch.indices, np.int32),
                         dev(batch.values, np.float32), int(batch.dim))


_HOST_VALUES = {"f32": _abi.SS_VALUES_F32, "bf16": _abi.SS_VALUES_BF16, "f16": _abi.SS_VALUES_F16}


def _host_csr(batch, host_values="f32"):
    indptr = np.ascontiguousarray(batch.indptr, dtype=np.int64)
    indices = np.ascontiguousarray(batch.indices, dtype=np.int32)
    if host_values == "f32":
        values = np.ascontiguousarray(batch.values, dtype=np.float32)
    else:  # 2-byte bit patterns, passed through untouched
        v = np.asarray(batch.values)
        if v.dtype not in (np.uint16, np.int16, np.float16) or (host_values == "bf16" and v.dtype == np.float16):
            raise TypeError(f"host_values={host_values!r} wants 16-bit values (uint16 bit patterns"
                            f"{'' if host_values == 'bf16' else ' or float16'}), got {v.dtype}")
        values = np.ascontiguousarray(v).view(np.uint16)
    m = _abi.ss_csr(indptr.ctypes.data, indices.ctypes.data, values.ctypes.data,
                    int(indptr.shape[0] - 1), int(indices.shape[0]), int(batch.dim))
    return m, (indptr, indices, values)


class SparseCosine:
    """One library handle: a device, a dimension and a chunk size."""

    ALGORITHMS = ("auto", "hybrid", "posting", "tensor")

    def __init__(self, dim: int, chunk_rows: int = DEFAULT_CHUNK_ROWS, device: int = 0,
                 validate: bool = False, algorithm: str = "auto", verify_stream: bool = False):
        """algorithm: "hybrid" (item tiles: dense hot dimensions + per-tile
        inverted indexes in shared memory), "posting" (per query row, the
        chunk's posting lists of its dimensions, summed exactly in fixed
        point), "tensor" (up to 128 frequent dimensions as a split-fp16
        dense product on the tensor cores, the others summed exactly in
        fixed point), or "auto" (the default: per item matrix, posting lists
        when most item tiles of its first build overflow).
        verify_stream: bulk_cosine_host checks every chunk's checksum on the
        device against its host copy (and records them, see stream_checksums)."""
        self._lib = _abi.load()
        self.dim = int(dim)
        self.chunk_rows = int(chunk_rows)
        self.device = int(device)
        if algorithm not in self.ALGORITHMS:
            raise ValueError(f"algorithm must be one of {self.ALGORITHMS}")
        self.algorithm = algorithm
        flags = (SS_VALIDATE if validate else 0)
        if algorithm == "posting":
            flags |= _abi.SS_ALGO_POSTING_LISTS
        elif algorithm == "hybrid":
            flags |= _abi.SS_ALGO_TILES
        elif algorithm == "tensor":
            flags |= _abi.SS_ALGO_TENSOR
        if verify_stream:
            flags |= _abi.SS_VERIFY_STREAM
        h = ctypes.c_void_p()
        st = self._lib.ss_create(ctypes.byref(h), self.device, self.dim, self.chunk_rows, flags)
        if st != _abi.SS_OK:
            raise SparseCosError(st, f"ss_create: {self._lib.ss_status_string(st).decode()}")
        self._h = h

    # -- plumbing
    def _check(self, st: int, what: str):
        if st != _abi.SS_OK:
            msg = self._lib.ss_last_error(self._h).decode() if self._h else ""
            raise SparseCosError(st, f"{what}: {self._lib.ss_status_string(st).decode()}: {msg}")

    def close(self):
        if getattr(self, "_h", None):
            self._lib.ss_destroy(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- the calls
    def row_norms(self, m: DeviceCsr, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(m.n_rows, dtype=torch.float32, device=m.indptr.device)
        c = m.abi()
        self._check(self._lib.ss_row_norms(self._h, ctypes.byref(c), _ptr(out), _stream_ptr(stream)),
                    "ss_row_norms")
        return out

    def build_item_index(self, items: DeviceCsr, row_begin: int, row_end: int, stream=None):
        c = items.abi()
        idx = ctypes.c_void_p()
        self._check(self._lib.ss_build_item_index(self._h, ctypes.byref(c), int(row_begin),
                                                  int(row_end), ctypes.byref(idx),
                                                  _stream_ptr(stream)), "ss_build_item_index")
        return idx

    @property
    def build_batch(self) -> int:
        """How many chunks one ``build_item_indexes`` call can build."""
        return int(self._lib.ss_build_batch(self._h))

    def build_item_indexes(self, items: DeviceCsr, row_begin: int, row_end: int, stream=None):
        """Indexes of the chunks of ``chunk_rows`` items that split
        [row_begin, row_end) (at most ``build_batch`` of them), built in one
        launch; a list of (chunk_row_begin, chunk_row_end, index)."""
        c = items.abi()
        arr = (ctypes.c_void_p * max(1, self.build_batch))()
        n = ctypes.c_int32(0)
        self._check(self._lib.ss_build_item_indexes(self._h, ctypes.byref(c), int(row_begin),
                                                    int(row_end), arr, ctypes.byref(n),
                                                    _stream_ptr(stream)), "ss_build_item_indexes")
        out = []
        for k in range(n.value):
            b = int(row_begin) + k * self.chunk_rows
            out.append((b, min(b + self.chunk_rows, int(row_end)), ctypes.c_void_p(arr[k])))
        return out

    def score_chunk(self, queries: DeviceCsr, inv_q: torch.Tensor, index, inv_i_chunk: torch.Tensor,
                    out: torch.Tensor, ld_out: int, stream=None):
        c = queries.abi()
        self._check(self._lib.ss_score_chunk(self._h, ctypes.byref(c), _ptr(inv_q), index,
                                             _ptr(inv_i_chunk), _ptr(out), int(ld_out),
                                             _stream_ptr(stream)), "ss_score_chunk")

    def score_all(self, queries: DeviceCsr, inv_q: torch.Tensor, items: DeviceCsr,
                  inv_i: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((queries.n_rows, items.n_rows), dtype=torch.float32,
                              device=queries.indptr.device)
        cq, ci = queries.abi(), items.abi()
        self._check(self._lib.ss_score_all(self._h, ctypes.byref(cq), _ptr(inv_q), ctypes.byref(ci),
                                           _ptr(inv_i), _ptr(out), int(out.stride(0)),
                                           _stream_ptr(stream)), "ss_score_all")
        return out

    def topk_reset(self, n_q: int, k: int, device=None, stream=None):
        """A fresh running top-k for n_q query rows: (best_val float32, best_item
        int64) device tensors of shape (n_q, k), filled with -inf and -1."""
        dev = device if device is not None else torch.device("cuda", self.device)
        best_val = torch.empty((n_q, k), dtype=torch.float32, device=dev)
        best_item = torch.empty((n_q, k), dtype=torch.int64, device=dev)
        self._check(self._lib.ss_topk_reset(self._h, int(n_q), int(k), _ptr(best_val),
                                            _ptr(best_item), _stream_ptr(stream)), "ss_topk_reset")
        return best_val, best_item

    def score_chunk_topk(self, queries: DeviceCsr, inv_q: torch.Tensor, index,
                         inv_i_chunk: torch.Tensor, best_val: torch.Tensor,
                         best_item: torch.Tensor, stream=None):
        """Scores one chunk and merges its best items into (best_val, best_item)."""
        c = queries.abi()
        k = int(best_val.shape[1])
        self._check(self._lib.ss_score_chunk_topk(self._h, ctypes.byref(c), _ptr(inv_q), index,
                                                  _ptr(inv_i_chunk), k, _ptr(best_val),
                                                  _ptr(best_item), _stream_ptr(stream)),
                    "ss_score_chunk_topk")

    def topk_all(self, queries: DeviceCsr, inv_q: torch.Tensor, items: DeviceCsr,
                 inv_i: torch.Tensor, k: int, stream=None):
        """Per query row, the k items of largest cosine (larger first, ties to
        the smaller item): (values float32, items int64), shape (n_q, k)."""
        dev = queries.indptr.device
        best_val = torch.empty((queries.n_rows, k), dtype=torch.float32, device=dev)
        best_item = torch.empty((queries.n_rows, k), dtype=torch.int64, device=dev)
        cq, ci = queries.abi(), items.abi()
        self._check(self._lib.ss_topk_all(self._h, ctypes.byref(cq), _ptr(inv_q), ctypes.byref(ci),
                                          _ptr(inv_i), int(k), _ptr(best_val), _ptr(best_item),
                                          _stream_ptr(stream)), "ss_topk_all")
        return best_val, best_item

    def tile_checksum(self, tile: torch.Tensor, stream=None):
        """(bits_sum, value_sum) of a 2-D float32 device tile (rows contiguous):
        the sum of the values' bit patterns as unsigned 32-bit integers modulo
        2**64, and the sum of the values in double.  Synchronises."""
        assert tile.dtype == torch.float32 and tile.dim() == 2 and tile.stride(1) == 1
        sums = torch.zeros(2, dtype=torch.int64, device=tile.device)
        self._check(self._lib.ss_tile_checksum(self._h, _ptr(tile), int(tile.shape[0]),
                                               int(tile.shape[1]), int(tile.stride(0)),
                                               ctypes.c_void_p(sums.data_ptr()),
                                               ctypes.c_void_p(sums.data_ptr() + 8),
                                               _stream_ptr(stream)), "ss_tile_checksum")
        host = sums.cpu().numpy()
        return int(host[:1].view(np.uint64)[0]), float(host[1:].view(np.float64)[0])

    def stream_checksums(self):
        """Per chunk of the last verified bulk_cosine_host pass: (bits_sum, value_sum)."""
        out, c = [], 0
        b, v = ctypes.c_uint64(0), ctypes.c_double(0.0)
        while self._lib.ss_stream_checksum(self._h, c, ctypes.byref(b), ctypes.byref(v)) == _abi.SS_OK:
            out.append((int(b.value), float(v.value)))
            c += 1
        return out

    def bulk_cosine_host(self, queries, items, out: Optional[np.ndarray] = None,
                         consumer: Optional[Callable] = None, ring_depth: int = 3,
                         timeout_ms: int = 0, host_values: str = "f32"):
        """Host CSR in, result streamed back chunk by chunk.

        out: a float32 (n_q, n_i) host array (numpy or a CPU torch tensor,
        ideally page-locked) or None; consumer(chunk, item_begin, item_end,
        tile) receives each chunk as a (n_q, width) numpy view valid during
        the call.  host_values: "f32", or "bf16" / "f16" for 16-bit values
        (uint16 bit patterns, or float16 for "f16"), sent to the device at
        2 bytes a value and widened there exactly (ss_set_host_values).
        """
        if host_values not in _HOST_VALUES:
            raise ValueError(f"host_values must be one of {sorted(_HOST_VALUES)}")
        cq, keep_q = _host_csr(queries, host_values)
        ci, keep_i = _host_csr(items, host_values)
        self._check(self._lib.ss_set_host_values(self._h, _HOST_VALUES[host_values]), "ss_set_host_values")
        out_ptr, ld = ctypes.c_void_p(0), 0
        if out is not None:
            if isinstance(out, torch.Tensor):
                assert out.dtype == torch.float32 and out.device.type == "cpu" and out.stride(1) == 1
                out_ptr, ld = ctypes.c_void_p(out.data_ptr()), out.stride(0)
            else:
                assert out.dtype == np.float32 and out.strides[1] == 4
                out_ptr, ld = ctypes.c_void_p(out.ctypes.data), out.strides[0] // 4
        cb = _abi.ss_chunk_consumer(0)
        if consumer is not None:
            def _cb(user, chunk, b, e, tile, ld_t, n_q):
                try:
                    arr = np.ctypeslib.as_array(tile, shape=(int(n_q), int(ld_t)))[:, : e - b]
                    r = consumer(int(chunk), int(b), int(e), arr)
                    return 0 if r is None else int(r)
                except Exception:  # stop the pass; the error surfaces as a status
                    return 1
            cb = _abi.ss_chunk_consumer(_cb)
        st = self._lib.ss_bulk_cosine_host(self._h, ctypes.byref(cq), ctypes.byref(ci), out_ptr, ld,
                                           cb, None, int(ring_depth), int(timeout_ms))
        del keep_q, keep_i
        self._check(st, "ss_bulk_cosine_host")
        return out

    def set_device_limit(self, nbytes: int) -> None:
        """Caps the device bytes bulk_cosine_host holds for input copies, norms
        and output tiles (0: no cap); above it the pass streams item batches
        and tiles the queries (ss_plan_host_pass)."""
        self._check(self._lib.ss_set_device_limit(self._h, int(nbytes)), "ss_set_device_limit")

    def validate_csr(self, m: DeviceCsr, stream=None):
        c = m.abi()
        self._check(self._lib.ss_validate_csr(self._h, ctypes.byref(c), _stream_ptr(stream)),
                    "ss_validate_csr")

    def profile_scorer(self, on: bool = True) -> None:
        """Record CUDA events around each launch of the scoring kernel
        (not the call's other kernels) on the caller's stream."""
        self._check(self._lib.ss_profile_scorer(self._h, 1 if on else 0), "ss_profile_scorer")

    def scorer_time(self):
        """(total milliseconds, launches) of the scoring-kernel launches
        recorded since the last read; synchronises."""
        ms = ctypes.c_double()
        n = ctypes.c_int64()
        self._check(self._lib.ss_scorer_time(self._h, ctypes.byref(ms), ctypes.byref(n)), "ss_scorer_time")
        return ms.value, n.value

    def index_stats(self, index, stream=None) -> dict:
        """Diagnostics of the last built index (synchronises the stream).
        "algorithm" is 0 for item tiles, 1 for posting lists, 2 for the
        tensor path; for posting lists and the tensor path "ell_entries"
        holds the chunk's list entries."""
        out = (ctypes.c_int64 * 8)()
        self._check(self._lib.ss_index_stats(self._h, index, out, _stream_ptr(stream)),
                    "ss_index_stats")
        keys = ("algorithm", "items", "tiles", "hot_dims", "heavy_entries", "ell_width_max",
                "ell_entries", "tiles_without_image")
        return {k: int(out[j]) for j, k in enumerate(keys)}

    def index_export(self, index, stream=None) -> dict:
        """The chunk index read back as host arrays (posting lists or tensor
        path; synchronises): "hot" (dense dimensions, ascending),
        "hot_values" (items x len(hot)), and the lists of the other
        dimensions as a CSC of the chunk: "col_ptr" (dim + 1), "item" and
        "value" (items ascending inside each list)."""
        lib = self._lib
        n_hot = ctypes.c_int32(0)
        n = ctypes.c_int64(0)
        self._check(lib.ss_index_export(self._h, index, None, None, None, None, None, None, 0,
                                        ctypes.byref(n), _stream_ptr(stream)), "ss_index_export")
        stats = self.index_stats(index, stream)
        n_items = stats["items"]
        hot = np.zeros(_abi.SS_EXPORT_HOT_MAX, np.int32)
        hot_values = np.zeros((n_items, _abi.SS_EXPORT_HOT_MAX), np.float32)
        col_ptr = np.zeros(self.dim + 1, np.int32)
        item = np.zeros(max(1, n.value), np.int32)
        value = np.zeros(max(1, n.value), np.float32)
        self._check(lib.ss_index_export(self._h, index, ctypes.byref(n_hot), hot.ctypes.data,
                                        hot_values.ctypes.data, col_ptr.ctypes.data, item.ctypes.data,
                                        value.ctypes.data, int(item.shape[0]), ctypes.byref(n),
                                        _stream_ptr(stream)), "ss_index_export")
        H = n_hot.value
        return {"hot": hot[:H], "hot_values": hot_values[:, :H], "col_ptr": col_ptr,
                "item": item[: n.value], "value": value[: n.value]}

    def lists_export(self, stream=None) -> dict:
        """The queries' lists the tensor path's scoring calls walk, as host
        arrays (synchronises): "dims" (the dimensions some query holds
        outside the hot set, ascending), "col_ptr" (len(dims) + 1), "query"
        (ascending inside each list) and "value" (the query's value times
        its row's inverse norm)."""
        lib = self._lib
        nd, n = ctypes.c_int64(0), ctypes.c_int64(0)
        self._check(lib.ss_lists_export(self._h, ctypes.byref(nd), None, None, None, None, 0, ctypes.byref(n),
                                        _stream_ptr(stream)), "ss_lists_export")
        dims = np.zeros(self.dim + 1, np.int32)
        col_ptr = np.zeros(self.dim + 1, np.int32)
        query = np.zeros(max(1, n.value), np.int32)
        value = np.zeros(max(1, n.value), np.float32)
        self._check(lib.ss_lists_export(self._h, ctypes.byref(nd), dims.ctypes.data, col_ptr.ctypes.data,
                                        query.ctypes.data, value.ctypes.data, int(query.shape[0]), ctypes.byref(n),
                                        _stream_ptr(stream)), "ss_lists_export")
        k = nd.value
        return {"dims": dims[:k], "col_ptr": col_ptr[: k + 1], "query": query[: n.value], "value": value[: n.value]}

    def invalidate(self):
        """Forget the hot set and the prepared queries (after in-place edits)."""
        self._check(self._lib.ss_invalidate(self._h), "ss_invalidate")

    def kernel_launches(self) -> int:
        """Kernels this handle has queued so far (counted by the library)."""
        return int(self._lib.ss_kernel_launches(self._h))

    def check_device(self, stream=None):
        self._check(self._lib.ss_check_device(self._h, _stream_ptr(stream)), "ss_check_device")


def library_path() -> str:
    return _abi.library_path()


def plan_host_pass(q_indptr, i_indptr, chunk_rows: int, device_limit: int, direct_output: bool = False,
                   host_values: str = "f32"):
    """Query-tile and item-batch boundaries of a bulk_cosine_host pass under
    a device limit (host only: runs without a GPU)."""
    lib = _abi.load()
    qp = np.ascontiguousarray(q_indptr, dtype=np.int64)
    ip = np.ascontiguousarray(i_indptr, dtype=np.int64)
    vt = _HOST_VALUES[host_values]
    nq, ni = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib.ss_plan_host_pass(qp.ctypes.data, len(qp) - 1, ip.ctypes.data, len(ip) - 1, int(chunk_rows),
                               int(device_limit), int(bool(direct_output)), vt, None, 0, ctypes.byref(nq),
                               None, 0, ctypes.byref(ni))
    if st != _abi.SS_OK:
        raise _abi.SparseCosError(st, "ss_plan_host_pass: " + lib.ss_status_string(st).decode())
    qb = np.zeros(nq.value + 1, dtype=np.int64)
    ib = np.zeros(ni.value + 1, dtype=np.int64)
    st = lib.ss_plan_host_pass(qp.ctypes.data, len(qp) - 1, ip.ctypes.data, len(ip) - 1, int(chunk_rows),
                               int(device_limit), int(bool(direct_output)), vt, qb.ctypes.data, len(qb),
                               ctypes.byref(nq), ib.ctypes.data, len(ib), ctypes.byref(ni))
    if st != _abi.SS_OK:
        raise _abi.SparseCosError(st, "ss_plan_host_pass: " + lib.ss_status_string(st).decode())
    return qb, ib


def tile_checksum_host(tile: np.ndarray):
    """(bits_sum, value_sum) of a 2-D float32 host array (rows contiguous),
    computed by the library's host routine (the counterpart of
    SparseCosine.tile_checksum)."""
    assert tile.dtype == np.float32 and tile.ndim == 2
    empty = tile.size == 0
    assert empty or tile.strides[1] == 4
    ld = int(tile.shape[1]) if empty else int(tile.strides[0] // 4)
    b, v = ctypes.c_uint64(0), ctypes.c_double(0.0)
    st = _abi.load().ss_tile_checksum_host(ctypes.c_void_p(tile.ctypes.data), int(tile.shape[0]),
                                           int(tile.shape[1]), ld, ctypes.byref(b), ctypes.byref(v))
    if st != _abi.SS_OK:
        raise SparseCosError(st, "ss_tile_checksum_host: bad arguments")
    return int(b.value), float(v.value)
