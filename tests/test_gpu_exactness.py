"""Exactness pins of the GPU path that a cosine tolerance alone would not see.

- The chunk index is integer and copy work: read back with ss_index_export,
  it must equal the chunk's CSC from scipy (``csr_matrix.tocsc()``) bit for
  bit, with the dense ("hot") dimensions given apart and equal to the
  chunk's own values; the tensor path's hot set must be the one its
  selection rule picks, recomputed here on the host.
- The split-fp16 tensor product against adversarial rows: values whose low
  fp16 part falls into fp16's subnormal range, 128 equal-magnitude hot
  dimensions whose signs cancel, and normalised values just inside and just
  outside the path's range guards.
- The full 5,000 x 200,000 matrix of the 1.2M-dimension workload, every
  entry against the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
sp = pytest.importorskip("scipy.sparse")

import oracle  # noqa: E402
from workload import CONFIGS, generate_rows, generate_side  # noqa: E402
from workload.tiny import csr_from_rows  # noqa: E402

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


def _dev(sec, batch):
    return sec.DeviceCsr.from_host(batch, "cuda")


def _scipy(batch, begin=0, end=None):
    end = batch.n_rows if end is None else end
    lo, hi = int(batch.indptr[begin]), int(batch.indptr[end])
    return sp.csr_matrix((batch.values[lo:hi], batch.indices[lo:hi], batch.indptr[begin:end + 1] - lo),
                         shape=(end - begin, batch.dim))


TENSOR_HOT_MAX = 160  # the tensor path's largest hot set (the header's SS_EXPORT_HOT_MAX)


def tensor_hot_set(I, k=TENSOR_HOT_MAX):
    """The tensor path's hot set, by its stated rule, on the host: the rows
    j * n / n_s (j < n_s, n_s = 32768 * n / nnz clamped to [16, n]) are
    sampled; a dimension qualifies when at least max(2, ceil(0.2% of n_s))
    sampled rows hold it; the k (160) with the most sampled rows are taken
    (counts of 1,023 or more count as equal), ties to the lower dimension,
    and none of a tie larger than 4,096 dimensions."""
    n, nnz = I.n_rows, I.nnz
    n_s = max(16, min(n, int(32768.0 * n / nnz)))
    rows = np.arange(n_s, dtype=np.int64) * n // n_s
    lens = I.indptr[rows + 1] - I.indptr[rows]
    flat = np.repeat(I.indptr[rows], lens) + (np.arange(lens.sum()) - np.repeat(np.cumsum(lens) - lens, lens))
    counts = np.bincount(I.indices[flat], minlength=I.dim)
    floor_c = min(1023, max(2, (n_s * 2 + 999) // 1000))
    cand = np.nonzero(counts >= floor_c)[0]
    cc = np.minimum(counts[cand], 1023)
    if cand.size <= k:
        return np.sort(cand)
    order = np.lexsort((cand, -cc))
    t = cc[order[k - 1]]
    above = cand[cc > t]
    ties = np.sort(cand[cc == t])
    if ties.size > 4096:
        return np.sort(above)
    return np.sort(np.concatenate([above, ties[: k - above.size]]))


# ------------------------------------------------------------------ index vs scipy
@pytest.mark.parametrize("algorithm", ["posting", "tensor"])
@pytest.mark.parametrize("name,n_i,rb,re", [
    ("d65k_q1k_i10k", 10_000, 8192, 10_000),        # the ragged last chunk
    ("d1.2m_q5k_i200k", 30_000, 3000, 3000 + 8192),  # a full chunk not aligned to 8,192
    ("d1.2m_q20k_i1m_heavy", 6000, 1000, 5000),      # heavy-tailed rows
    ("d500k_q50k_i500k_uniform", 3000, 0, 1500),     # ~500 nonzeros a row, no head
])
def test_index_is_the_chunks_csc(sec, algorithm, name, n_i, rb, re):
    cfg = CONFIGS[name]
    I = generate_rows(cfg, 1, 0, n_i)
    with sec.SparseCosine(cfg.dim, chunk_rows=8192, algorithm=algorithm) as h:
        idx = h.build_item_index(_dev(sec, I), rb, re)
        h.check_device()
        ex = h.index_export(idx)
    chunk = _scipy(I, rb, re)
    hot = ex["hot"]
    assert np.all(np.diff(hot) > 0) and (hot.size == 0 or (hot[0] >= 0 and hot[-1] < cfg.dim))
    if algorithm == "tensor":
        assert np.array_equal(hot, tensor_hot_set(I)), "hot set differs from its selection rule"
    # the dense part: each item's values of the hot dimensions, 0 where absent
    want_hot = chunk[:, hot].toarray().astype(np.float32)
    assert np.array_equal(ex["hot_values"].view(np.uint32), want_hot.view(np.uint32))
    # the lists: the chunk without its hot columns, as a CSC
    coo = chunk.tocoo()
    keep = ~np.isin(coo.col, hot)
    cold = sp.csr_matrix((coo.data[keep], (coo.row[keep], coo.col[keep])), shape=chunk.shape).tocsc()
    cold.sort_indices()
    assert np.array_equal(ex["col_ptr"].astype(np.int64), cold.indptr.astype(np.int64))
    assert np.array_equal(ex["item"], cold.indices.astype(np.int32))
    assert np.array_equal(ex["value"].view(np.uint32), cold.data.astype(np.float32).view(np.uint32))
    # hot + lists hold every stored entry of the chunk once
    assert ex["item"].size + int((want_hot != 0).sum()) == chunk.nnz - int((coo.data[~keep] == 0).sum())


@pytest.mark.parametrize("name,n_q", [("d1.2m_q5k_i200k", 5000), ("d65k_q1k_i10k", 1000),
                                      ("d1.2m_q20k_i1m_heavy", 3000)])
def test_query_lists_are_the_normalised_queries_csc_over_their_cold_dims(sec, name, n_q):
    """The tensor path sorts the queries' nonzeros outside the hot set by
    dimension, once per query matrix: its lists must be the CSC of the
    normalised queries restricted to exactly those dimensions, bit for bit
    (each value the float32 product of the stored value and its row's
    inverse norm), the same for every chunk of a build and for a second
    build scored with them."""
    cfg = CONFIGS[name]
    Q, I = generate_rows(cfg, 0, 0, n_q), generate_rows(cfg, 1, 0, 9000)
    with sec.SparseCosine(cfg.dim, chunk_rows=4500, algorithm="tensor") as h:
        q, i = _dev(sec, Q), _dev(sec, I)
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        exports = []
        views = h.build_item_indexes(i, 0, 9000)
        assert len(views) == 2
        hot = h.index_export(views[0][2])["hot"]
        for b, e, vw in views:
            out = torch.empty((n_q, e - b), dtype=torch.float32, device="cuda")
            h.score_chunk(q, inv_q, vw, inv_i[b:], out, e - b)
            h.check_device()
            exports.append(h.lists_export())
        idx = h.build_item_index(i, 0, 4500)  # a second build with the same queries
        out = torch.empty((n_q, 4500), dtype=torch.float32, device="cuda")
        h.score_chunk(q, inv_q, idx, inv_i, out, 4500)
        h.check_device()
        exports.append(h.lists_export())
        invq = inv_q.cpu().numpy()
    qs = _scipy(Q)
    rows = np.repeat(np.arange(n_q), np.diff(qs.indptr))
    norm = sp.csr_matrix((qs.data.astype(np.float32) * invq[rows], qs.indices, qs.indptr), shape=qs.shape)
    qcold = np.setdiff1d(np.unique(Q.indices), hot)  # the queries' cold dimensions
    csc = norm[:, qcold].tocsc()
    csc.sort_indices()
    for k, ex in enumerate(exports):
        assert np.array_equal(ex["dims"], qcold.astype(np.int32)), k
        assert np.array_equal(ex["col_ptr"].astype(np.int64), csc.indptr.astype(np.int64)), k
        assert np.array_equal(ex["query"], csc.indices.astype(np.int32)), k
        assert np.array_equal(ex["value"].view(np.uint32), csc.data.astype(np.float32).view(np.uint32)), k


def test_index_export_rejects_item_tiles(sec):
    from sparse_embedding_exact_gb300 import SparseCosError, _abi

    cfg = CONFIGS["d65k_q1k_i10k"]
    I = generate_rows(cfg, 1, 0, 2000)
    with sec.SparseCosine(cfg.dim, algorithm="hybrid") as h:
        idx = h.build_item_index(_dev(sec, I), 0, 2000)
        with pytest.raises(SparseCosError) as e:
            h.index_export(idx)
        assert e.value.status == _abi.SS_ERR_INVALID_ARG


# ------------------------------------------------------------------ split-fp16 product
def _tensor_scores(sec, Q, I, chunk_rows=8192, inv_scale=1.0):
    with sec.SparseCosine(Q.dim, chunk_rows=chunk_rows, algorithm="tensor") as h:
        q, i = _dev(sec, Q), _dev(sec, I)
        inv_q, inv_i = h.row_norms(q) * inv_scale, h.row_norms(i) * inv_scale
        idx = h.build_item_index(i, 0, min(chunk_rows, I.n_rows))
        st = h.index_stats(idx)
        S = h.score_all(q, inv_q, i, inv_i)
        h.check_device()
        return S.cpu().numpy(), st


def _head_rows(rng, n, hot_vals, d, cold_per_row=3):
    """Rows holding all 128 head dimensions (values given per row) plus a few
    random dimensions past the head."""
    rows = []
    for r in range(n):
        extra = np.sort(rng.choice(np.arange(128, d), size=cold_per_row, replace=False))
        idx = np.concatenate([np.arange(128), extra])
        val = np.concatenate([hot_vals[r], rng.lognormal(0, 1, cold_per_row)]).astype(np.float32)
        nz = val != 0
        rows.append((idx[nz], val[nz]))
    return rows


def test_split_with_subnormal_low_parts(sec):
    """Query rows: one dominant head value and 127 values near 3e-5, whose
    normalised fp16 high part is itself subnormal and whose low part lies
    far inside fp16's subnormal range (spacing 2^-24); item rows of many
    equal-sized head values make those tiny products the whole score."""
    rng = np.random.default_rng(31)
    d = 4096
    qh = np.zeros((48, 128))
    qh[:, 0] = 1.0
    qh[:, 1:] = 3e-5 * (1.0 + rng.random((48, 127)))
    qh[::3, 1:] *= -1.0
    qh[1::4, 0] = 0.0  # some query rows only the tiny values
    ih = np.abs(rng.normal(1.0, 0.05, (160, 128)))
    ih[:80, 0] = 0.0  # half the items lack the dominant dimension
    Q = csr_from_rows(_head_rows(rng, 48, qh, d), d)
    I = csr_from_rows(_head_rows(rng, 160, ih, d), d)
    got, st = _tensor_scores(sec, Q, I)
    assert st["algorithm"] == 2 and st["hot_dims"] >= 128  # the head (and any extra dim sampled twice)
    err = float(np.abs(got.astype(np.float64) - oracle.cosine(Q, I, f64=True)).max())
    print(f"split fp16, subnormal low parts: max |error| {err:.3e}")
    assert err <= TOL


def test_split_with_cancelling_equal_magnitudes(sec):
    """128 head dimensions of equal magnitude (within 1e-3) and random signs
    on both sides: the products cancel, so the float32 sums run through
    partial sums much larger than the result."""
    rng = np.random.default_rng(32)
    d = 2048
    def signs(n):
        return rng.choice([-1.0, 1.0], (n, 128)) * (1.0 + 1e-3 * rng.random((n, 128)))
    qh, ih = signs(64), signs(192)
    ih[0] = np.where(np.arange(128) % 2 == 0, 1.0, -1.0)  # alternating signs, exactly
    qh[0] = 1.0
    qh[1, :64], qh[1, 64:] = 1.0, -1.0  # a positive run, then a negative one
    Q = csr_from_rows(_head_rows(rng, 64, qh, d, cold_per_row=1), d)
    I = csr_from_rows(_head_rows(rng, 192, ih, d, cold_per_row=1), d)
    got, st = _tensor_scores(sec, Q, I)
    assert st["algorithm"] == 2 and st["hot_dims"] >= 128  # the head (and any extra dim sampled twice)
    err = float(np.abs(got.astype(np.float64) - oracle.cosine(Q, I, f64=True)).max())
    print(f"split fp16, cancelling equal magnitudes: max |error| {err:.3e}")
    assert err <= TOL


def test_range_guards_of_the_tensor_path(sec):
    """Inverse norms scaled by 1 + 2^-11 keep every normalised value within
    1 + 2^-10 and every row's squares within 1 + 2^-6: accepted, and the
    scores are the oracle's times (1 + 2^-11)^2.  Scaled by 1 + 2^-9, a row
    with one nonzero exceeds the value guard; scaled by 1.01, a row of many
    small values stays under the value guard but its squares exceed theirs:
    both are reported and the handle stays usable."""
    from sparse_embedding_exact_gb300 import SparseCosError, _abi

    cfg = CONFIGS["d65k_q1k_i10k"]
    Q, I = generate_rows(cfg, 0, 0, 40), generate_rows(cfg, 1, 0, 1500)
    s = 1.0 + 2.0 ** -11
    got, _ = _tensor_scores(sec, Q, I, inv_scale=s)
    assert float(np.abs(got - oracle.cosine(Q, I, f64=True) * s * s).max()) <= TOL

    single = csr_from_rows([([7], [3.0])] + [([1, 5, 9], [1.0, 2.0, 3.0])] * 3, 64)
    many = csr_from_rows([(list(range(0, 60)), [1.0] * 60)] * 4, 64)
    for X, scale in ((single, 1.0 + 2.0 ** -9), (many, 1.01)):
        with sec.SparseCosine(64, algorithm="tensor") as h:
            x = _dev(sec, X)
            inv = h.row_norms(x)
            h.score_all(x, inv * scale, x, inv * scale)
            with pytest.raises(SparseCosError) as e:
                h.check_device()
            assert e.value.status == _abi.SS_ERR_DEVICE_CHECK
            S = h.score_all(x, inv, x, inv).cpu().numpy()
            h.check_device()
        assert float(np.abs(S - oracle.cosine(X, X, f64=True)).max()) <= TOL


# ------------------------------------------------------------------ the full 1.2M-dimension matrix
def test_full_matrix_of_the_1_2m_workload(sec):
    """All 5,000 x 200,000 entries (25 chunks of 8,192 items, the launch
    shape the benchmark times) against the oracle, compared in item slabs."""
    cfg = CONFIGS["d1.2m_q5k_i200k"]
    Q, I = generate_side(cfg, 0), generate_side(cfg, 1)
    with sec.SparseCosine(cfg.dim, chunk_rows=8192) as h:
        q, i = _dev(sec, Q), _dev(sec, I)
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        S = h.score_all(q, inv_q, i, inv_i)
        h.check_device()
        algo = h.index_stats(h.build_item_index(i, 0, 8192))["algorithm"]
        worst = 0.0
        slab = 25_000
        for b in range(0, I.n_rows, slab):
            e = min(b + slab, I.n_rows)
            got = S[:, b:e].cpu().numpy().astype(np.float64)
            ref = oracle.cosine(Q, I, i_begin=b, i_end=e, f64=True)
            worst = max(worst, float(np.abs(got - ref).max()))
    print(f"full 5,000 x 200,000 matrix (algorithm {algo}): max |error| {worst:.3e}")
    assert worst <= TOL


def test_query_slices_of_the_1_2m_workload(sec):
    """24,000 queries: the queries' lists come in several slices of rows
    (one records launch each); sampled rows of every slice, the slices'
    first and last rows among them, match the oracle over a whole chunk,
    and the exported lists merge the slices into the queries' CSC."""
    from workload import sample_query_rows

    cfg = CONFIGS["d1.2m_q5k_i200k"].scaled(24_000, 8192)
    Q, I = generate_side(cfg, 0), generate_side(cfg, 1)
    with sec.SparseCosine(cfg.dim, chunk_rows=8192, algorithm="tensor") as h:
        q, i = _dev(sec, Q), _dev(sec, I)
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        S = h.score_all(q, inv_q, i, inv_i)
        h.check_device()
        ex = h.lists_export()
        hot = h.index_export(h.build_item_index(i, 0, 8192))["hot"]
        rows = np.unique(np.concatenate([sample_query_rows(Q.n_rows, 192), np.arange(0, Q.n_rows, 2560),
                                         np.arange(2559, Q.n_rows, 2560), [Q.n_rows - 1]])).astype(np.int64)
        got = S[torch.as_tensor(rows, device=S.device)].cpu().numpy().astype(np.float64)
        invq = inv_q.cpu().numpy()
    err = float(np.abs(got - oracle.cosine(Q, I, q_rows=rows, f64=True)).max())
    print(f"24,000 x 8,192 in query slices: max |error| {err:.3e}")
    assert err <= TOL
    qs = _scipy(Q)
    norm = sp.csr_matrix((qs.data.astype(np.float32) * invq[np.repeat(np.arange(Q.n_rows), np.diff(qs.indptr))],
                          qs.indices, qs.indptr), shape=qs.shape)
    qcold = np.setdiff1d(np.unique(Q.indices), hot)
    csc = norm[:, qcold].tocsc()
    csc.sort_indices()
    assert np.array_equal(ex["dims"], qcold.astype(np.int32))
    assert np.array_equal(ex["col_ptr"].astype(np.int64), csc.indptr.astype(np.int64))
    assert np.array_equal(ex["query"], csc.indices.astype(np.int32))
    assert np.array_equal(ex["value"].view(np.uint32), csc.data.astype(np.float32).view(np.uint32))


# ------------------------------------------------------------------ record overflow paths
def test_tensor_records_beyond_every_buffer(sec):
    """Queries far denser in the items' cold dimensions than the item sample
    suggests: buckets hold more records than the epilogue keeps in registers
    and in shared memory (it reads the rest from the bucket), and more than
    the buckets' room, sized from the sample (the scorer computes those
    blocks from the lists itself).  Every entry still matches the oracle."""
    rng = np.random.default_rng(41)
    d = 50_000
    items = [(np.sort(rng.choice(d, 40, replace=False)), rng.lognormal(0, 1, 40)) for _ in range(8192)]
    queries = [(np.sort(rng.choice(d, 400, replace=False)), rng.standard_normal(400)) for _ in range(2048)]
    I, Q = csr_from_rows(items, d), csr_from_rows(queries, d)
    with sec.SparseCosine(d, chunk_rows=8192, algorithm="tensor") as h:
        q, i = _dev(sec, Q), _dev(sec, I)
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        S = h.score_all(q, inv_q, i, inv_i)
        h.check_device()
        got = S.cpu().numpy().astype(np.float64)
    err = float(np.abs(got - oracle.cosine(Q, I, f64=True)).max())
    print(f"tensor path, records past every buffer: max |error| {err:.3e}")
    assert err <= TOL
