"""ss_cosine_chunk_noalloc: the entry point for callers that cannot allocate
device memory (a host whose pool owns the GPU, a graph capture in progress, a
plug-in with a fixed budget).  It is called through the C ABI and must match
the CPU oracle and the handle-based entry points on two different chunks in a
row, since the static scratch it works in keeps the previous call's contents;
its device status word must report a chunk_nnz that is too small.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test by the time it gets here.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402

from workload import CONFIGS, generate_rows  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 2e-6


@pytest.fixture(scope="module")
def sec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_embedding_exact_gb300 as sec
    from sparse_embedding_exact_gb300 import build

    build.build()
    sec._abi.load()
    return sec


def _noalloc(sec, q, i, row_begin, row_end, chunk_nnz, out, status=None):
    lib = sec._abi.load()
    cq, ci = q.abi(), i.abi()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st_ptr = ctypes.c_void_p(0 if status is None else status.data_ptr())
    return lib.ss_cosine_chunk_noalloc(ctypes.byref(cq), ctypes.byref(ci), row_begin, row_end,
                                       chunk_nnz, ctypes.c_void_p(out.data_ptr()), out.stride(0),
                                       st_ptr, stream)


def test_noalloc_matches_handle_entry_points_twice(sec):
    cfg = CONFIGS["d1.2m_q5k_i200k"]
    Q, I = generate_rows(cfg, 0, 0, 300), generate_rows(cfg, 1, 0, 9000)
    q, i = sec.DeviceCsr.from_host(Q, "cuda"), sec.DeviceCsr.from_host(I, "cuda")
    with sec.SparseCosine(cfg.dim, chunk_rows=8192) as h:
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        for rb, re in ((0, 3000), (3000, 9000 - 808)):  # two different chunks, back to back
            width = re - rb
            ref = torch.empty((Q.n_rows, width), dtype=torch.float32, device="cuda")
            idx = h.build_item_index(i, rb, re)
            h.score_chunk(q, inv_q, idx, inv_i[rb:], ref, width)
            out = torch.full((Q.n_rows, width), float("nan"), dtype=torch.float32, device="cuda")
            status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            nnz = int(I.indptr[re] - I.indptr[rb])
            assert _noalloc(sec, q, i, rb, re, nnz, out, status) == sec._abi.SS_OK
            torch.cuda.synchronize()
            assert int(status.item()) == sec._abi.SS_DEVICE_OK
            got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy()
            assert np.isfinite(got).all()
            # against the CPU oracle (the definition), then against the handle path
            exact = oracle.cosine(Q, I, i_begin=rb, i_end=re)
            assert float(np.abs(got - exact).max()) <= TOL
            assert float(np.abs(got - want).max()) <= 2 * TOL


def test_noalloc_status_reports_a_short_chunk_nnz(sec):
    """chunk_nnz one below the chunk's nonzeros: the lists are cut short, and
    the status word the caller passed says so (SS_DEVICE_CAPACITY)."""
    cfg = CONFIGS["d65k_q1k_i10k"]
    Q, I = generate_rows(cfg, 0, 0, 64), generate_rows(cfg, 1, 0, 700)
    q, i = sec.DeviceCsr.from_host(Q, "cuda"), sec.DeviceCsr.from_host(I, "cuda")
    rb, re = 100, 700
    nnz = int(I.indptr[re] - I.indptr[rb])
    out = torch.empty((Q.n_rows, re - rb), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert _noalloc(sec, q, i, rb, re, nnz - 1, out, status) == sec._abi.SS_OK
    torch.cuda.synchronize()
    assert int(status.item()) == sec._abi.SS_DEVICE_CAPACITY
    # the exact count clears the word again and gives the oracle's cosines
    assert _noalloc(sec, q, i, rb, re, nnz, out, status) == sec._abi.SS_OK
    torch.cuda.synchronize()
    assert int(status.item()) == sec._abi.SS_DEVICE_OK
    exact = oracle.cosine(Q, I, i_begin=rb, i_end=re)
    assert float(np.abs(out.cpu().numpy().astype(np.float64) - exact).max()) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(sec):
    from workload.tiny import csr_from_rows

    big_dim = 8_000_000  # per-dimension counters alone need 64 MB > 32 MB
    X = csr_from_rows([([1, 5], [1.0, 2.0])] * 4, big_dim)
    x = sec.DeviceCsr.from_host(X, "cuda")
    out = torch.empty((4, 4), dtype=torch.float32, device="cuda")
    assert _noalloc(sec, x, x, 0, 4, int(X.nnz), out) == sec._abi.SS_ERR_LIMIT
    # a chunk_nnz larger than the matrix holds is an argument error
    assert _noalloc(sec, x, x, 0, 4, int(X.nnz) + 1, out) == sec._abi.SS_ERR_INVALID_ARG
