"""Pins for the CPU oracle: each checks it against something other than itself.

* closed forms derived by hand from the cosine definition (tests/golden);
* dense float64 brute force on tiny inputs (a different computation: a dense
  matrix product over every dimension, zeros included);
* scipy.sparse products (the post's own comparison point, section 3.1) on
  samples of the synthetic workloads;
* invariants the definition fixes: S[x,x] = 1, symmetry, |S| <= 1, permutation
  equivariance, column-slice (chunk) invariance;
* and a planted-mistake check: the oracle built with a deliberate mistake
  (dropped term, wrong sign, wrong pointer advance, missing square root, one
  norm missing, transposed output) must fail at least one pin.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workload import CONFIGS, generate_rows
from workload.tiny import csr_from_rows, random_csr

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
MUTANTS = [1, 2, 3, 4, 5, 6]


def _dense_cosine(Qd, Id):
    nq = np.sqrt((Qd * Qd).sum(axis=1))
    ni = np.sqrt((Id * Id).sum(axis=1))
    den = np.outer(nq, ni)
    num = Qd @ Id.T
    with np.errstate(divide="ignore", invalid="ignore"):
        S = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
    return S


# ----------------------------------------------------------------- the pins
def pin_closed_forms(mutant=0):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        u = (c["u"]["indices"], c["u"]["values"])
        v = (c["v"]["indices"], c["v"]["values"])
        exp = float(Fraction(*c["expected"]))
        for a, b in ((u, v), (v, u)):
            A = csr_from_rows([a], c["dim"])
            B = csr_from_rows([b], c["dim"])
            got = oracle.cosine(A, B, f64=True, threads=1, mutant=mutant)[0, 0]
            if not abs(got - exp) <= 1e-15:
                return False, f"{c['name']}: {got} != {exp}"
    # All cases at once as a (n x n) matrix: the diagonal holds the pairs,
    # so a transposed or shifted output shows.
    us = [(c["u"]["indices"], c["u"]["values"]) for c in cases]
    vs = [(c["v"]["indices"], c["v"]["values"]) for c in cases]
    dim = max(c["dim"] for c in cases)
    S = oracle.cosine(csr_from_rows(us, dim), csr_from_rows(vs, dim), f64=True, threads=2,
                      mutant=mutant)
    exp = np.array([float(Fraction(*c["expected"])) for c in cases])
    if not np.allclose(np.diag(S), exp, rtol=0, atol=1e-15):
        return False, "diagonal of the batched closed forms"
    return True, ""


TINY_SHAPES = [(7, 9, 13, 0.4), (32, 32, 64, 0.3), (1, 20, 5, 0.6), (20, 1, 5, 0.6),
               (17, 23, 64, 0.05), (12, 12, 16, 0.9)]


def pin_dense_bruteforce(mutant=0):
    for seed, (nq, ni, d, dens) in enumerate(TINY_SHAPES):
        for law in ("normal", "lognormal", "integer"):
            Q, Qd = random_csr(100 + seed, nq, d, dens, law, zero_rows=1 if nq > 2 else 0,
                               explicit_zeros=2)
            I, Id = random_csr(200 + seed, ni, d, dens, law, zero_rows=1 if ni > 2 else 0,
                               explicit_zeros=2)
            ref = _dense_cosine(Qd, Id)
            got = oracle.cosine(Q, I, f64=True, threads=3, mutant=mutant)
            if got.shape != ref.shape or not np.allclose(got, ref, rtol=0, atol=1e-12):
                return False, f"dense brute force {nq}x{ni}x{d} {law}"
            got32 = oracle.cosine(Q, I, threads=1, mutant=mutant)
            ref32 = ref.astype(np.float32)
            ulps = np.abs(got32.view(np.int32).astype(np.int64) - ref32.view(np.int32).astype(np.int64))
            if ulps.max(initial=0) > 1:
                return False, f"fp32 rounding {nq}x{ni}x{d} {law}"
            dots = oracle.dot(Q, I, mutant=mutant)
            if not np.allclose(dots, Qd @ Id.T, rtol=1e-13, atol=1e-12):
                return False, f"dot {nq}x{ni}x{d} {law}"
    return True, ""


def pin_norms(mutant=0):
    for seed, (nq, _, d, dens) in enumerate(TINY_SHAPES):
        Q, Qd = random_csr(300 + seed, nq, d, dens, "lognormal", zero_rows=1, explicit_zeros=1)
        got = oracle.row_norms(Q, mutant=mutant)
        ref = np.linalg.norm(Qd, axis=1)
        if not np.allclose(got, ref, rtol=1e-14, atol=0):
            return False, "row norms vs numpy.linalg.norm"
    return True, ""


def _scipy_cosine(Q, I):
    sp = pytest.importorskip("scipy.sparse")
    A = sp.csr_matrix((Q.values.astype(np.float64), Q.indices, Q.indptr), shape=(Q.n_rows, Q.dim))
    B = sp.csr_matrix((I.values.astype(np.float64), I.indices, I.indptr), shape=(I.n_rows, I.dim))
    num = (A @ B.T).toarray()
    na = np.sqrt(np.asarray(A.multiply(A).sum(axis=1)).ravel())
    nb = np.sqrt(np.asarray(B.multiply(B).sum(axis=1)).ravel())
    den = np.outer(na, nb)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def pin_scipy(mutant=0):
    for name, nq, ni in (("d65k_q1k_i10k", 200, 1500), ("d1.2m_q5k_i200k", 60, 1200),
                         ("d1.2m_q20k_i1m_heavy", 40, 600), ("d500k_q50k_i500k_uniform", 30, 300)):
        cfg = CONFIGS[name]
        Q = generate_rows(cfg, 0, 0, nq)
        I = generate_rows(cfg, 1, 0, ni)
        ref = _scipy_cosine(Q, I)
        got = oracle.cosine(Q, I, f64=True, mutant=mutant)
        if not np.allclose(got, ref, rtol=0, atol=1e-12):
            return False, f"scipy.sparse on {name}"
    return True, ""


def pin_invariants(mutant=0):
    cfg = CONFIGS["d65k_q1k_i10k"]
    X = generate_rows(cfg, 1, 0, 150)
    S = oracle.cosine(X, X, f64=True, mutant=mutant)
    nz = np.diff(X.indptr) > 0
    if not np.allclose(np.diag(S)[nz], 1.0, rtol=0, atol=1e-14):
        return False, "S[x,x] = 1"
    if np.abs(S - S.T).max() > 1e-15:
        return False, "symmetry when Q = I"
    if np.abs(S).max() > 1 + 1e-15:
        return False, "|S| <= 1"
    perm = np.random.default_rng(5).permutation(X.n_rows)
    Sp = oracle.cosine(X, X.take(perm), f64=True, mutant=mutant)
    if not np.array_equal(Sp, S[:, perm]):
        return False, "item permutation permutes columns"
    parts = [oracle.cosine(X, X, i_begin=b, i_end=min(b + 64, X.n_rows), f64=True, mutant=mutant)
             for b in range(0, X.n_rows, 64)]
    if not np.array_equal(np.concatenate(parts, axis=1), S):
        return False, "column slices (chunks) equal the full matrix"
    return True, ""


ALL_PINS = [pin_closed_forms, pin_dense_bruteforce, pin_norms, pin_scipy, pin_invariants]


# ----------------------------------------------------------------- the tests
@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    ok, msg = pin(0)
    assert ok, msg


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_is_caught(oracle_lib, mutant):
    oracle.build(mutant)
    assert oracle.mutant_id(mutant) == mutant
    failed = []
    for pin in ALL_PINS:
        ok, msg = pin(mutant)
        if not ok:
            failed.append(f"{pin.__name__}: {msg}")
    assert failed, f"mutant {mutant} passed every pin"


def test_check_csr_rules(oracle_lib):
    good = csr_from_rows([([0, 3, 9], [1, 2, 3]), ([], []), ([2], [1])], 10)
    assert oracle.check_csr(good) == -1
    assert oracle.check_csr(csr_from_rows([([1], [1]), ([3, 2], [1, 1])], 10)) == 1
    assert oracle.check_csr(csr_from_rows([([1, 1], [1, 1])], 10)) == 0
    assert oracle.check_csr(csr_from_rows([([1, 10], [1, 1])], 10)) == 0
    assert oracle.check_csr(csr_from_rows([([-1, 2], [1, 1])], 10)) == 0


def test_oracle_threads_agree(oracle_lib):
    cfg = CONFIGS["d65k_q1k_i10k"]
    Q = generate_rows(cfg, 0, 0, 64)
    I = generate_rows(cfg, 1, 0, 500)
    a = oracle.cosine(Q, I, threads=1)
    b = oracle.cosine(Q, I, threads=7)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


def test_oracle_row_selection(oracle_lib):
    cfg = CONFIGS["d65k_q1k_i10k"]
    Q = generate_rows(cfg, 0, 0, 80)
    I = generate_rows(cfg, 1, 0, 300)
    rows = np.array([79, 3, 40, 3])
    full = oracle.cosine(Q, I)
    sel = oracle.cosine(Q, I, q_rows=rows, i_begin=17, i_end=250)
    assert np.array_equal(sel, full[rows, 17:250])


def test_oracle_empty_shapes(oracle_lib):
    Q = csr_from_rows([], 8)
    I = csr_from_rows([([1], [1.0])], 8)
    assert oracle.cosine(Q, I).shape == (0, 1)
    assert oracle.cosine(I, Q).shape == (1, 0)
