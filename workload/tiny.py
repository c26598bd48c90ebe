"""Small seeded CSR inputs for edge-case tests (no cosine arithmetic here)."""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np

from .generate import CsrBatch


def csr_from_rows(rows: Sequence[Tuple[Sequence[int], Sequence[float]]], dim: int) -> CsrBatch:
    """CSR from a list of (indices, values) rows, kept exactly as given."""
    indptr = np.zeros(len(rows) + 1, np.int64)
    for r, (idx, _) in enumerate(rows):
        indptr[r + 1] = indptr[r] + len(idx)
    indices = np.concatenate([np.asarray(i, np.int32) for i, _ in rows]) if rows else np.zeros(0, np.int32)
    values = np.concatenate([np.asarray(v, np.float32) for _, v in rows]) if rows else np.zeros(0, np.float32)
    return CsrBatch(indptr, indices.astype(np.int32), values.astype(np.float32), dim)


def random_csr(seed: int, n_rows: int, dim: int, density: float, value_law: str = "normal",
               zero_rows: int = 0, explicit_zeros: int = 0) -> Tuple[CsrBatch, np.ndarray]:
    """A random CSR and the same matrix as a dense float64 array.

    zero_rows rows are left empty and explicit_zeros stored entries are set
    to 0.0 (kept in the CSR), so both edge cases appear.
    """
    rng = np.random.default_rng(seed)
    mask = rng.random((n_rows, dim)) < density
    if zero_rows:
        mask[rng.choice(n_rows, size=min(zero_rows, n_rows), replace=False)] = False
    if value_law == "normal":
        vals = rng.standard_normal((n_rows, dim))
    elif value_law == "lognormal":
        vals = rng.lognormal(0.0, 1.0, (n_rows, dim))
    elif value_law == "integer":
        vals = rng.integers(-4, 5, (n_rows, dim)).astype(np.float64)
    else:
        raise ValueError(value_law)
    vals = vals.astype(np.float32)
    rr, cc = np.nonzero(mask)
    v = vals[rr, cc]
    if explicit_zeros and v.size:
        v[rng.choice(v.size, size=min(explicit_zeros, v.size), replace=False)] = 0.0
    indptr = np.zeros(n_rows + 1, np.int64)
    np.cumsum(np.bincount(rr, minlength=n_rows), out=indptr[1:])
    dense = np.zeros((n_rows, dim), np.float64)
    dense[rr, cc] = v
    return CsrBatch(indptr, cc.astype(np.int32), v.astype(np.float32), dim), dense
