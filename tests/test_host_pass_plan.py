"""The split of a host pass under a device-memory limit (ss_plan_host_pass):
host-only logic, run on the CPU against the rules the header states.

A pass holds on the device a copy of each query tile and item batch (8 bytes
per row pointer, 8 per nonzero (10 with 16-bit host values, staged), 4 per
row for the inverse norms), two output
tiles of rows x min(chunk_rows, n_i) floats unless the output is written in
place, and two item batch slots.
"""
import ctypes

import numpy as np
import pytest

sec = pytest.importorskip("sparse_embedding_exact_gb300")
from sparse_embedding_exact_gb300 import _abi  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        _abi.load()
    except ImportError as e:
        pytest.skip(str(e))


def copy_bytes(ptr, r0, r1, half=False):
    # with 16-bit host values, a 2-byte staging copy per nonzero more
    return 8 * (r1 - r0 + 1) + (10 if half else 8) * int(ptr[r1] - ptr[r0]) + 4 * (r1 - r0)


def heavy_indptr(rng, n, median):
    lens = np.minimum(np.exp(rng.normal(np.log(median), 1.2, n)).astype(np.int64) + 1, 50_000)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def check_bounds(b, n):
    assert b[0] == 0 and b[-1] == n
    assert np.all(np.diff(b) > 0)


def check_plan(qp, ip, C, limit, direct, host_values="f32"):
    n_q, n_i = len(qp) - 1, len(ip) - 1
    qb, ib = sec.plan_host_pass(qp, ip, C, limit, direct, host_values)
    half = host_values != "f32"
    cb = lambda p, r0, r1: copy_bytes(p, r0, r1, half)  # noqa: E731
    check_bounds(qb, n_q)
    check_bounds(ib, n_i)
    W = min(C, n_i)
    out = lambda rows: 0 if direct else 8 * rows * W  # noqa: E731
    whole = cb(qp, 0, n_q) + out(n_q) + cb(ip, 0, n_i)
    if limit == 0 or whole <= limit:
        assert list(qb) == [0, n_q] and list(ib) == [0, n_i]
        return qb, ib
    if len(qb) == 2:
        assert cb(qp, 0, n_q) + out(n_q) <= limit // 2
        q_used = cb(qp, 0, n_q) + out(n_q)
    else:
        max_rows = n_q if direct else (limit // 4) // (8 * W)
        for t in range(len(qb) - 1):
            r0, r1 = qb[t], qb[t + 1]
            assert cb(qp, r0, r1) <= limit // 4 and r1 - r0 <= max_rows
            if r1 < n_q:  # greedy: one more row would not fit
                assert cb(qp, r0, r1 + 1) > limit // 4 or r1 + 1 - r0 > max_rows
        q_used = max(cb(qp, qb[t], qb[t + 1]) for t in range(len(qb) - 1)) + \
            out(int(np.diff(qb).max()))
    slot = (limit - q_used) // 2
    for k in range(len(ib) - 1):
        r0, r1 = ib[k], ib[k + 1]
        assert cb(ip, r0, r1) <= slot
        if r1 < n_i:
            if r1 - r0 >= C:  # whole chunks, and one chunk more would not fit
                assert (r1 - r0) % C == 0
                assert r0 + (r1 - r0) + C > n_i or cb(ip, r0, r1 + C) > slot
            else:
                assert cb(ip, r0, r1 + 1) > slot
    return qb, ib


def test_no_limit_and_a_limit_that_fits_keep_one_tile_and_one_batch():
    rng = np.random.default_rng(1)
    qp, ip = heavy_indptr(rng, 300, 20), heavy_indptr(rng, 7000, 40)
    for limit in (0, 10 ** 12):
        qb, ib = sec.plan_host_pass(qp, ip, 1024, limit)
        assert list(qb) == [0, 300] and list(ib) == [0, 7000]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("host_values", ["f32", "bf16"])
def test_plans_follow_the_stated_rules(seed, direct, host_values):
    rng = np.random.default_rng(100 + seed)
    n_q, n_i = int(rng.integers(1, 3000)), int(rng.integers(1, 40000))
    qp, ip = heavy_indptr(rng, n_q, 30), heavy_indptr(rng, n_i, 60)
    C = int(rng.choice([16, 1000, 8192]))
    W = min(C, n_i)
    whole = copy_bytes(qp, 0, n_q) + copy_bytes(ip, 0, n_i) + (0 if direct else 8 * n_q * W)
    tiled = 0
    for frac in (1.5, 1.0, 0.6, 0.3, 0.1, 0.03, 0.01):
        try:
            qb, ib = check_plan(qp, ip, C, int(whole * frac), direct, host_values)
            tiled += len(qb) > 2
        except _abi.SparseCosError as e:
            assert e.status == _abi.SS_ERR_LIMIT  # one row outgrew its share
    if not direct:
        assert tiled > 0 or n_q == 1


def test_every_range_stays_below_2_pow_31_nonzeros():
    # Row pointers alone (no data): four item rows of 2^30 nonzeros each.
    qp = np.array([0, 5], np.int64)
    ip = np.arange(5, dtype=np.int64) << 30
    qb, ib = sec.plan_host_pass(qp, ip, 8192, 1 << 50, True)
    assert list(qb) == [0, 1]
    assert list(ib) == [0, 1, 2, 3, 4]


def test_a_row_larger_than_its_share_is_a_limit_error():
    qp = np.array([0, 10, 20], np.int64)
    ip = np.array([0, 5, 100_000, 100_010], np.int64)
    with pytest.raises(_abi.SparseCosError) as e:
        sec.plan_host_pass(qp, ip, 2, 200_000, True)
    assert e.value.status == _abi.SS_ERR_LIMIT
    with pytest.raises(_abi.SparseCosError) as e:  # one query row's output tiles alone exceed a quarter
        sec.plan_host_pass(qp, ip, 2, 60, False)
    assert e.value.status == _abi.SS_ERR_LIMIT


def test_argument_errors():
    lib = _abi.load()
    qp = np.array([0, 1], np.int64)
    n1, n2 = ctypes.c_int64(-1), ctypes.c_int64(-1)
    P = qp.ctypes.data
    assert lib.ss_plan_host_pass(None, 1, P, 1, 8, 0, 0, 0, None, 0, ctypes.byref(n1), None, 0,
                                 ctypes.byref(n2)) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_plan_host_pass(P, 1, P, 1, 0, 0, 0, 0, None, 0, ctypes.byref(n1), None, 0,
                                 ctypes.byref(n2)) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_plan_host_pass(P, 1, P, 1, 8, -1, 0, 0, None, 0, ctypes.byref(n1), None, 0,
                                 ctypes.byref(n2)) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_plan_host_pass(P, 1, P, 1, 8, 0, 0, 3, None, 0, ctypes.byref(n1), None, 0,
                                 ctypes.byref(n2)) == _abi.SS_ERR_INVALID_ARG
    short = np.zeros(1, np.int64)
    assert lib.ss_plan_host_pass(P, 1, P, 1, 8, 0, 0, 0, short.ctypes.data, 1, ctypes.byref(n1), None, 0,
                                 ctypes.byref(n2)) == _abi.SS_ERR_INVALID_ARG
    assert n1.value == 1 and n2.value == 1  # counts are written all the same
    assert lib.ss_set_device_limit(None, 0) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_set_host_values(None, _abi.SS_VALUES_BF16) == _abi.SS_ERR_INVALID_ARG


def test_half_values_make_smaller_batches():
    rng = np.random.default_rng(5)
    qp, ip = heavy_indptr(rng, 50, 20), heavy_indptr(rng, 20000, 60)
    limit = copy_bytes(ip, 0, 20000) // 3
    _, ib32 = sec.plan_host_pass(qp, ip, 1000, limit, True, "f32")
    _, ib16 = sec.plan_host_pass(qp, ip, 1000, limit, True, "bf16")
    assert len(ib16) > len(ib32)
