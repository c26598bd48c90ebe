"""The seeded input recipe: every workload's rows follow its stated laws,
and any row range regenerates to the same bytes on its own (rows come in
independently seeded blocks)."""
import numpy as np
import pytest

from workload import CONFIGS, generate_rows
from workload.generate import BLOCK_ROWS


def check_structure(m, cfg):
    lens = np.diff(m.indptr)
    assert m.indptr[0] == 0 and m.indptr[-1] == m.indices.size == m.values.size
    assert lens.min() >= cfg.nnz_lo and lens.max() <= cfg.nnz_hi
    assert m.indices.dtype == np.int32 and m.values.dtype == np.float32
    assert m.indices.min() >= 0 and m.indices.max() < cfg.dim
    # strictly increasing indices inside every row (distinct, sorted)
    step = np.diff(m.indices.astype(np.int64))
    row_start = np.zeros(m.indices.size, bool)
    row_start[m.indptr[:-1][lens > 0]] = True
    assert np.all(step[~row_start[1:]] > 0)
    assert np.isfinite(m.values).all()
    if cfg.value_law == "lognormal":
        assert m.values.min() > 0


@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("side", [0, 1])
def test_rows_follow_the_laws(name, side):
    cfg = CONFIGS[name]
    n = min(2000, cfg.n_rows(side))
    m = generate_rows(cfg, side, 0, n, workers=1)
    check_structure(m, cfg)
    lens = np.diff(m.indptr).astype(np.float64)
    if cfg.nnz_law == "poisson":
        # clipping at the bounds moves the mean by far less than 3 standard errors here
        assert abs(lens.mean() - cfg.nnz_center) < 4 * np.sqrt(cfg.nnz_center / n) + 0.05
    else:
        assert abs(np.log(np.median(lens)) - np.log(cfg.nnz_center)) < 0.15
    vals = m.values.astype(np.float64)
    if cfg.value_law == "lognormal":
        assert abs(np.log(vals).mean()) < 0.05 and abs(np.log(vals).std() - 1.0) < 0.05
    else:
        assert abs(vals.mean()) < 0.05 and abs(vals.std() - 1.0) < 0.05
    counts = np.bincount(m.indices, minlength=cfg.dim)
    if cfg.index_law == "zipf":
        # a skewed head: the first dimensions are far more frequent than the tail
        head, mid = counts[:10].mean(), counts[1000:2000].mean()
        assert head > 20 * max(mid, 1e-9)
        assert counts[0] >= counts[100] >= 0
    else:
        # uniform: the two halves of the dimension range are about as full
        half = cfg.dim // 2
        a, b = counts[:half].sum(), counts[half:].sum()
        assert abs(a - b) < 5 * np.sqrt(a + b)


def test_any_row_range_regenerates_alone():
    cfg = CONFIGS["d65k_q1k_i10k"].scaled(100, 40_000)
    whole = generate_rows(cfg, 1, BLOCK_ROWS - 300, BLOCK_ROWS + 300, workers=1)
    part = generate_rows(cfg, 1, BLOCK_ROWS - 10, BLOCK_ROWS + 5, workers=1)  # across a block edge
    ref = whole.rows(290, 305)
    assert np.array_equal(part.indptr, ref.indptr)
    assert np.array_equal(part.indices, ref.indices)
    assert np.array_equal(part.values.view(np.uint32), ref.values.view(np.uint32))
    again = generate_rows(cfg, 1, BLOCK_ROWS - 10, BLOCK_ROWS + 5, workers=1)
    assert np.array_equal(again.values.view(np.uint32), part.values.view(np.uint32))


def test_sides_and_seeds_differ():
    cfg = CONFIGS["d65k_q1k_i10k"]
    q = generate_rows(cfg, 0, 0, 50, workers=1)
    i = generate_rows(cfg, 1, 0, 50, workers=1)
    other = generate_rows(cfg.__class__(**{**cfg.__dict__, "seed": 7}), 0, 0, 50, workers=1)
    assert not np.array_equal(q.indptr, i.indptr) or not np.array_equal(q.indices, i.indices)
    assert not (np.array_equal(q.indptr, other.indptr) and np.array_equal(q.indices, other.indices))
