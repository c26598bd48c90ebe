"""Failure handling on the GPU, made on the host (nothing here faults, traps
or hangs a GPU):

- allocation failures injected one at a time (ss_inject_alloc_failure) at
  every device and page-locked allocation of a whole run (handle creation,
  norms, the automatic choice, builds, scoring, top-k, the host pass): the
  call that meets one returns SS_ERR_OOM and the same handle then gives the
  oracle's cosines;
- a host pass whose deadline (1 ms) runs out before its first chunk is
  delivered returns SS_ERR_TIMEOUT; ss_check_device then waits for the work
  still in flight, and the same handle runs the pass again correctly.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from workload import CONFIGS, generate_rows, sample_query_rows  # noqa: E402

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


def _pipeline(sec, h, Q, I):
    """Norms, the full matrix, top-k, and a host pass through the ring."""
    q, i = sec.DeviceCsr.from_host(Q, "cuda"), sec.DeviceCsr.from_host(I, "cuda")
    inv_q, inv_i = h.row_norms(q), h.row_norms(i)
    S = h.score_all(q, inv_q, i, inv_i)
    vals, _ = h.topk_all(q, inv_q, i, inv_i, 4)
    tiles = np.empty((Q.n_rows, I.n_rows), np.float32)

    def consume(c, b, e, tile):
        tiles[:, b:e] = tile

    h.bulk_cosine_host(Q, I, consumer=consume, ring_depth=2)
    h.check_device()
    return S.cpu().numpy(), vals.cpu().numpy(), tiles


@pytest.mark.parametrize("algorithm", ["auto", "posting", "hybrid"])
def test_every_allocation_failure_leaves_a_usable_handle(sec, algorithm):
    from sparse_embedding_exact_gb300 import SparseCosError, _abi

    lib = _abi.load()
    cfg = CONFIGS["d65k_q1k_i10k"]
    Q, I = generate_rows(cfg, 0, 0, 70), generate_rows(cfg, 1, 0, 2500)
    ref = oracle.cosine(Q, I)
    ref_top = -np.sort(-ref, axis=1)[:, :4]
    fired_at = []
    for n in range(1, 200):
        lib.ss_inject_alloc_failure(n)
        h = None
        try:
            h = sec.SparseCosine(cfg.dim, chunk_rows=1024, algorithm=algorithm)
            out = _pipeline(sec, h, Q, I)
        except SparseCosError as e:
            assert e.status == _abi.SS_ERR_OOM, (n, str(e))
            out = None
        left = lib.ss_inject_alloc_failure(0)
        if out is not None and left > 0:  # the run made fewer than n allocations: all covered
            h.close()
            break
        fired_at.append(n)
        if h is None:  # the failure hit ss_create; nothing to reuse
            continue
        if out is None:  # the same handle, after the failure, gives the oracle's results
            out = _pipeline(sec, h, Q, I)
        S, top, tiles = out
        assert float(np.abs(S.astype(np.float64) - ref).max()) <= TOL, n
        assert float(np.abs(tiles.astype(np.float64) - ref).max()) <= TOL, n
        assert float(np.abs(top.astype(np.float64) - ref_top).max()) <= TOL, n
        h.close()
    else:
        pytest.fail("the run kept allocating")
    assert len(fired_at) >= 8, fired_at  # creation, workspace, builds, scoring, ring


def test_host_pass_timeout_then_the_handle_runs_again(sec):
    from sparse_embedding_exact_gb300 import SparseCosError, _abi

    # 20,000 query rows: each chunk's tile is 655 MB, whose copy alone takes
    # longer than the 1 ms deadline.
    cfg = CONFIGS["d1.2m_q5k_i200k"].scaled(20_000, 3 * 8192)
    Q, I = generate_rows(cfg, 0, 0, cfg.n_q), generate_rows(cfg, 1, 0, cfg.n_i)
    rows = sample_query_rows(Q.n_rows, 64, 5)
    got = np.full((len(rows), I.n_rows), np.nan, np.float32)

    def consume(c, b, e, tile):
        got[:, b:e] = tile[rows]

    with sec.SparseCosine(cfg.dim, chunk_rows=8192) as h:
        with pytest.raises(SparseCosError) as e:
            h.bulk_cosine_host(Q, I, consumer=consume, ring_depth=3, timeout_ms=1)
        assert e.value.status == _abi.SS_ERR_TIMEOUT
        h.check_device()  # waits for the pass's work still in flight; no device error
        h.bulk_cosine_host(Q, I, consumer=consume, ring_depth=3)
        h.check_device()
    ref = oracle.cosine(Q, I, q_rows=rows)
    assert float(np.abs(got.astype(np.float64) - ref).max()) <= TOL
