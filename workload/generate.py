"""Seeded synthetic CSR batches shaped like the workloads of the bulk-similarity
blog post ("Engineering practice for bulk similarity calculation over sparse
embeddings", sections 1 and 3.3): BM25/TF-IDF-like rows of ~43 nonzeros over a
1.2M-word dictionary, whose nonzeros cluster in the head of the dictionary.

The five workloads below give the dimension, the query and item counts, the
law of the nonzeros per row, the law of the indices and the law of the values.
Readings taken where the description is silent:

* "clipped" clamps the drawn count into [lo, hi]; it does not resample.
* Zipf(s) is the finite Zipf law on ranks 1..d with P(r) proportional to r^-s,
  and rank r maps to dimension r-1, so the hot dimensions are the low indices
  (the post says nonzeros concentrate in the dictionary prefix, section 3.2).
* "Without replacement" is successive sampling: draw i.i.d. from the law and
  keep the first nnz distinct values of the sequence.  The same rule gives
  uniform sampling without replacement when the law is uniform.
* The indices of a row are sorted ascending (CSR order); values are drawn after
  that, i.i.d., in CSR order.
* Rows are generated in blocks of BLOCK_ROWS rows.  Block b of side s
  (0 = queries, 1 = items) draws from PCG64 seeded with
  SeedSequence(seed, spawn_key=(s, b)), so any block can be regenerated alone
  and blocks can be drawn in parallel with identical results.

Nothing here computes a norm, a dot product or a cosine.
"""
from __future__ import annotations

import dataclasses
import functools
import math
import os
from typing import List, Optional, Tuple

import numpy as np

BLOCK_ROWS = 16384


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    """One synthetic workload: query set Q and item set I over dimension d."""

    name: str
    dim: int
    n_q: int
    n_i: int
    nnz_law: str  # "poisson" or "lognormal"
    nnz_center: float  # Poisson mean, or lognormal median
    nnz_sigma: float  # lognormal sigma (unused for poisson)
    nnz_lo: int
    nnz_hi: int
    index_law: str  # "zipf" or "uniform"
    zipf_s: float
    value_law: str  # "lognormal" (positive, TF-IDF-like) or "normal" (signed)
    seed: int = 0
    chunk_rows: int = 8192
    verify_rows: int = 0  # 0: verify the full matrix; else sampled query rows
    description: str = ""

    def n_rows(self, side: int) -> int:
        return self.n_q if side == 0 else self.n_i

    def scaled(self, n_q: int, n_i: int, name: Optional[str] = None) -> "WorkloadConfig":
        """Same laws, fewer rows (used for bounded CPU samples and small tests)."""
        return dataclasses.replace(self, n_q=n_q, n_i=n_i, name=name or f"{self.name}@{n_q}x{n_i}")


CONFIGS = {
    # Small case: the oracle computes the whole 1,000 x 10,000 matrix in seconds.
    "d65k_q1k_i10k": WorkloadConfig(
        name="d65k_q1k_i10k", dim=65_536, n_q=1_000, n_i=10_000,
        nnz_law="poisson", nnz_center=43, nnz_sigma=0.0, nnz_lo=1, nnz_hi=256,
        index_law="zipf", zipf_s=1.1, value_law="lognormal",
        description="d=65,536; 1,000 x 10,000; nnz~Poisson(43) in [1,256]; "
                    "Zipf(1.1) distinct indices; lognormal(0,1) values"),
    # The dictionary size and nnz of the post's e-commerce case (section 1),
    # 5,000 queries x 200,000 items: the throughput workload.
    "d1.2m_q5k_i200k": WorkloadConfig(
        name="d1.2m_q5k_i200k", dim=1_200_000, n_q=5_000, n_i=200_000,
        nnz_law="poisson", nnz_center=43, nnz_sigma=0.0, nnz_lo=1, nnz_hi=512,
        index_law="zipf", zipf_s=1.1, value_law="lognormal",
        description="d=1,200,000; 5,000 x 200,000; nnz~Poisson(43) in [1,512]; "
                    "Zipf(1.1) without replacement; lognormal(0,1) values"),
    "d500k_q50k_i500k_uniform": WorkloadConfig(
        name="d500k_q50k_i500k_uniform", dim=500_000, n_q=50_000, n_i=500_000,
        nnz_law="poisson", nnz_center=500, nnz_sigma=0.0, nnz_lo=1, nnz_hi=500_000,
        index_law="uniform", zipf_s=0.0, value_law="normal", verify_rows=256,
        description="d=500,000; 50,000 x 500,000; nnz~Poisson(500); uniform "
                    "without replacement; signed N(0,1) values"),
    "d1.2m_q50k_i2m": WorkloadConfig(
        name="d1.2m_q50k_i2m", dim=1_200_000, n_q=50_000, n_i=2_000_000,
        nnz_law="poisson", nnz_center=43, nnz_sigma=0.0, nnz_lo=1, nnz_hi=512,
        index_law="zipf", zipf_s=1.1, value_law="lognormal", verify_rows=256,
        description="d=1,200,000; 50,000 x 2,000,000; nnz~Poisson(43) in [1,512]; "
                    "Zipf(1.1); lognormal(0,1) values"),
    "d1.2m_q20k_i1m_heavy": WorkloadConfig(
        name="d1.2m_q20k_i1m_heavy", dim=1_200_000, n_q=20_000, n_i=1_000_000,
        nnz_law="lognormal", nnz_center=20, nnz_sigma=1.5, nnz_lo=1, nnz_hi=20_000,
        index_law="zipf", zipf_s=1.3, value_law="normal", verify_rows=256,
        description="d=1,200,000; 20,000 x 1,000,000; nnz~lognormal(median 20, "
                    "sigma 1.5) in [1,20,000]; Zipf(1.3) with hot dimensions; "
                    "signed N(0,1) values"),
}


@dataclasses.dataclass
class CsrBatch:
    """A CSR matrix: int64 indptr[n_rows+1], int32 indices[nnz], float32 values[nnz]."""

    indptr: np.ndarray
    indices: np.ndarray
    values: np.ndarray
    dim: int

    @property
    def n_rows(self) -> int:
        return int(self.indptr.shape[0] - 1)

    @property
    def nnz(self) -> int:
        return int(self.indptr[-1])

    def rows(self, begin: int, end: int) -> "CsrBatch":
        """Rows [begin, end) as a new CSR with indptr rebased to 0 (copies)."""
        lo, hi = int(self.indptr[begin]), int(self.indptr[end])
        return CsrBatch(self.indptr[begin:end + 1] - lo, self.indices[lo:hi].copy(),
                        self.values[lo:hi].copy(), self.dim)

    def take(self, rows: np.ndarray) -> "CsrBatch":
        """The listed rows, in the listed order, as a new CSR."""
        rows = np.asarray(rows, dtype=np.int64)
        lens = self.indptr[rows + 1] - self.indptr[rows]
        indptr = np.zeros(len(rows) + 1, dtype=np.int64)
        np.cumsum(lens, out=indptr[1:])
        starts = np.repeat(self.indptr[rows] - indptr[:-1], lens)
        flat = np.arange(indptr[-1], dtype=np.int64) + starts
        return CsrBatch(indptr, self.indices[flat], self.values[flat], self.dim)


@functools.lru_cache(maxsize=8)
def _zipf_cdf(dim: int, s: float) -> np.ndarray:
    w = np.arange(1, dim + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    cdf[-1] = 1.0
    return cdf


def _draw_indices(rng: np.random.Generator, cfg: WorkloadConfig, m: int) -> np.ndarray:
    if cfg.index_law == "zipf":
        u = rng.random(m)
        return np.searchsorted(_zipf_cdf(cfg.dim, cfg.zipf_s), u, side="right").astype(np.int64)
    if cfg.index_law == "uniform":
        return rng.integers(0, cfg.dim, size=m, dtype=np.int64)
    raise ValueError(f"unknown index law {cfg.index_law!r}")


def _draw_nnz(rng: np.random.Generator, cfg: WorkloadConfig, n: int) -> np.ndarray:
    if cfg.nnz_law == "poisson":
        k = rng.poisson(cfg.nnz_center, size=n).astype(np.int64)
    elif cfg.nnz_law == "lognormal":
        z = rng.standard_normal(n)
        k = np.rint(np.exp(math.log(cfg.nnz_center) + cfg.nnz_sigma * z))
        k = np.minimum(k, 2.0 ** 40).astype(np.int64)
    else:
        raise ValueError(f"unknown nnz law {cfg.nnz_law!r}")
    return np.clip(k, cfg.nnz_lo, min(cfg.nnz_hi, cfg.dim))


_POS_BITS = 24
_DIM_BITS = 22


def _successive_distinct(rng: np.random.Generator, cfg: WorkloadConfig,
                         need: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per row r, the first need[r] distinct values of an i.i.d. draw sequence.

    Returns (row, dim) pairs sorted by (row, dim).  Keys are packed into one
    int64 (row, dim and draw position) so that one sort orders them.
    """
    n = need.shape[0]
    d = cfg.dim
    if n >= (1 << 15) or d >= (1 << _DIM_BITS):
        raise ValueError("block too large for packed keys")
    pos_mask = (1 << _POS_BITS) - 1
    kept_rows: List[np.ndarray] = []
    kept_dims: List[np.ndarray] = []
    # Candidates of rows still short, carried over with their draw positions.
    c_row = np.zeros(0, np.int64)
    c_pos = np.zeros(0, np.int64)
    c_dim = np.zeros(0, np.int64)
    drawn = np.zeros(n, np.int64)
    found = np.zeros(n, np.int64)
    todo = np.arange(n, dtype=np.int64)
    factor = np.full(n, 1.25)
    while todo.size:
        deficit = need[todo] - found[todo]
        m_row = np.ceil(deficit * factor[todo]).astype(np.int64) + 4
        if int((drawn[todo] + m_row).max()) > pos_mask:
            raise ValueError("too many draws for one row")
        rows_new = np.repeat(todo, m_row)
        starts = np.repeat(np.cumsum(m_row) - m_row, m_row)
        pos_new = np.arange(rows_new.size, dtype=np.int64) - starts + np.repeat(drawn[todo], m_row)
        dims_new = _draw_indices(rng, cfg, int(rows_new.size))
        drawn[todo] += m_row
        row = np.concatenate([c_row, rows_new])
        pos = np.concatenate([c_pos, pos_new])
        dim = np.concatenate([c_dim, dims_new])
        # First occurrence of each (row, dim) in draw order.
        key = np.sort(((row * d + dim) << _POS_BITS) | pos)
        group = key >> _POS_BITS
        first = np.ones(key.size, bool)
        first[1:] = group[1:] != group[:-1]
        key = key[first]
        group = key >> _POS_BITS
        row, dim, pos = group // d, group % d, key & pos_mask
        # Keep the earliest need[r] distinct values of each row: order by
        # (row, pos) with dim carried in the low bits of the same key.
        key = np.sort((((row << _POS_BITS) | pos) << _DIM_BITS) | dim)
        dim = key & ((1 << _DIM_BITS) - 1)
        key >>= _DIM_BITS
        row, pos = key >> _POS_BITS, key & pos_mask
        bounds = np.searchsorted(row, todo)
        counts = np.diff(np.append(bounds, row.size))
        rank = np.arange(row.size, dtype=np.int64) - np.repeat(bounds, counts)
        keep = rank < need[row]
        row, pos, dim = row[keep], pos[keep], dim[keep]
        found[todo] = np.minimum(counts, need[todo])
        done_mask = found[todo] >= need[todo]
        done_rows = todo[done_mask]
        is_done = np.zeros(n, bool)
        is_done[done_rows] = True
        fin = is_done[row]
        kept_rows.append(row[fin])
        kept_dims.append(dim[fin])
        c_row, c_pos, c_dim = row[~fin], pos[~fin], dim[~fin]
        # Rows still short drew too few: draw more generously next time.
        still = todo[~done_mask]
        factor[still] = np.minimum(factor[still] * 2.0, 64.0)
        todo = still
    rows = np.concatenate(kept_rows) if kept_rows else np.zeros(0, np.int64)
    dims = np.concatenate(kept_dims) if kept_dims else np.zeros(0, np.int64)
    key = np.sort(rows * d + dims)
    return key // d, key % d


def generate_block(cfg: WorkloadConfig, side: int, block: int) -> CsrBatch:
    """Rows [block*BLOCK_ROWS, ...) of side 0 (queries) or 1 (items)."""
    n_rows = cfg.n_rows(side)
    r0 = block * BLOCK_ROWS
    n = min(BLOCK_ROWS, n_rows - r0)
    if n <= 0:
        raise ValueError("block out of range")
    ss = np.random.SeedSequence(cfg.seed, spawn_key=(side, block))
    rng = np.random.Generator(np.random.PCG64(ss))
    need = _draw_nnz(rng, cfg, n)
    rows, dims = _successive_distinct(rng, cfg, need)
    indptr = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=n), out=indptr[1:])
    nnz = int(indptr[-1])
    if cfg.value_law == "lognormal":
        values = rng.lognormal(0.0, 1.0, size=nnz).astype(np.float32)
    elif cfg.value_law == "normal":
        values = rng.standard_normal(nnz).astype(np.float32)
    else:
        raise ValueError(f"unknown value law {cfg.value_law!r}")
    return CsrBatch(indptr, dims.astype(np.int32), values, cfg.dim)


def _concat(parts: List[CsrBatch], dim: int) -> CsrBatch:
    if not parts:
        return CsrBatch(np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32), dim)
    offs = np.cumsum([0] + [p.nnz for p in parts])
    indptr = np.concatenate([parts[0].indptr[:1]] + [p.indptr[1:] + o for p, o in zip(parts, offs)])
    return CsrBatch(indptr.astype(np.int64), np.concatenate([p.indices for p in parts]),
                    np.concatenate([p.values for p in parts]), dim)


def _block_job(args):
    cfg, side, b = args
    return generate_block(cfg, side, b)


def generate_rows(cfg: WorkloadConfig, side: int, begin: int, end: int,
                  workers: int = 1) -> CsrBatch:
    """Rows [begin, end) of one side, identical whatever range is asked for."""
    n_rows = cfg.n_rows(side)
    if not 0 <= begin <= end <= n_rows:
        raise ValueError("row range out of bounds")
    if begin == end:
        return _concat([], cfg.dim)
    b0, b1 = begin // BLOCK_ROWS, (end - 1) // BLOCK_ROWS + 1
    jobs = [(cfg, side, b) for b in range(b0, b1)]
    if workers > 1 and len(jobs) > 1:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        with ctx.Pool(min(workers, len(jobs))) as pool:
            parts = pool.map(_block_job, jobs, chunksize=1)
    else:
        parts = [_block_job(j) for j in jobs]
    full = _concat(parts, cfg.dim)
    return full.rows(begin - b0 * BLOCK_ROWS, end - b0 * BLOCK_ROWS)


def default_workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def generate_side(cfg: WorkloadConfig, side: int, workers: Optional[int] = None) -> CsrBatch:
    n_rows = cfg.n_rows(side)
    if workers is None:
        workers = default_workers() if n_rows > 4 * BLOCK_ROWS else 1
    return generate_rows(cfg, side, 0, n_rows, workers=workers)


def make_pair(cfg: WorkloadConfig, workers: Optional[int] = None) -> Tuple[CsrBatch, CsrBatch]:
    """(Q, I) for a workload."""
    return generate_side(cfg, 0, workers), generate_side(cfg, 1, workers)


def sample_query_rows(n_q: int, k: int = 256, seed: int = 0) -> np.ndarray:
    """k distinct query rows, sorted, drawn from a stream separate from the data."""
    k = min(k, n_q)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(2,))))
    return np.sort(rng.choice(n_q, size=k, replace=False)).astype(np.int64)
