"""Full-size workloads on the GPU, in the launch configuration the benchmark
times (8,192-item chunks).

Every chunk is scored on the device.  The oracle checks 256 sampled query
rows against every item (the full matrix of the 1.2M-dimension workload is
checked in test_gpu_exactness.py), and properties that hold at any size are
checked on every entry: finite values and |S| <= 1 + tolerance.  The three
workloads too large to keep (100, 400 and 80 GB of scores) are also streamed
chunk by chunk into the page-locked host ring with stream verification on:
each chunk's checksum (the sum of the float32 bit patterns) is taken on the
device before its copy and must equal the host copy's, the sampled rows are
collected from the ring, and every entry of every delivered chunk is checked
for range.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from workload import CONFIGS, generate_side, sample_query_rows  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 2e-6
CHUNK = 8192


_DATA = {}


def _workload(name):
    """(Q, I) of a workload, generated once per test module."""
    if name not in _DATA:
        _DATA.clear()  # keep one workload in host memory at a time
        cfg = CONFIGS[name]
        _DATA[name] = (generate_side(cfg, 0), generate_side(cfg, 1))
    return _DATA[name]


@pytest.fixture(scope="module")
def sec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_embedding_exact_gb300 as sec
    from sparse_embedding_exact_gb300 import build

    build.build()
    sec._abi.load()
    return sec


def _bits_sum(t):
    return int(t.view(torch.int32).to(torch.int64).sum().item())


def _device_pass(sec, cfg, Q, I, rows):
    """Scores all chunks; returns sampled rows (host) and per-chunk stats."""
    with sec.SparseCosine(cfg.dim, chunk_rows=CHUNK) as h:
        q = sec.DeviceCsr.from_host(Q, "cuda")
        i = sec.DeviceCsr.from_host(I, "cuda")
        inv_q, inv_i = h.row_norms(q), h.row_norms(i)
        width = min(CHUNK, I.n_rows)
        buf = torch.empty((Q.n_rows, width), dtype=torch.float32, device="cuda")
        rows_d = torch.from_numpy(rows).cuda()
        sampled = torch.empty((len(rows), I.n_rows), dtype=torch.float32, device="cuda")
        max_abs = torch.zeros((), dtype=torch.float32, device="cuda")
        finite = torch.ones((), dtype=torch.bool, device="cuda")
        sums = []
        for b in range(0, I.n_rows, CHUNK):
            e = min(b + CHUNK, I.n_rows)
            idx = h.build_item_index(i, b, e)
            h.score_chunk(q, inv_q, idx, inv_i[b:], buf, width)
            tile = buf[:, : e - b]
            sampled[:, b:e] = tile.index_select(0, rows_d)
            max_abs = torch.maximum(max_abs, tile.abs().max())
            finite &= torch.isfinite(tile).all()
            sums.append(tile.view(torch.int32).to(torch.int64).sum())
        h.check_device()
        return (sampled.cpu().numpy(), float(max_abs.item()), bool(finite.item()),
                [int(s.item()) for s in sums])


@pytest.mark.parametrize("name", ["d1.2m_q5k_i200k", "d500k_q50k_i500k_uniform", "d1.2m_q50k_i2m",
                                  "d1.2m_q20k_i1m_heavy"])
def test_full_workload_sampled_rows(sec, name):
    cfg = CONFIGS[name]
    Q, I = _workload(name)
    rows = sample_query_rows(cfg.n_q, 256, cfg.seed)
    sampled, max_abs, finite, sums = _device_pass(sec, cfg, Q, I, rows)
    assert finite
    assert max_abs <= 1.0 + TOL
    assert len(sums) == -(-cfg.n_i // CHUNK)
    ref = oracle.cosine(Q, I, q_rows=rows)
    err = float(np.abs(sampled.astype(np.float64) - ref).max())
    assert err <= TOL, f"{name}: max abs error {err:.3e}"


@pytest.mark.parametrize("name", ["d500k_q50k_i500k_uniform", "d1.2m_q50k_i2m", "d1.2m_q20k_i1m_heavy"])
def test_streamed_workload_through_the_host_ring(sec, name):
    cfg = CONFIGS[name]
    Q, I = _workload(name)
    rows = sample_query_rows(cfg.n_q, 256, cfg.seed)
    sampled = np.full((len(rows), I.n_rows), np.nan, np.float32)
    seen, worst = [], [0.0]
    torch.set_num_threads(max(1, min(16, torch.get_num_threads())))

    def consume(c, b, e, tile):
        seen.append((c, b, e))
        sampled[:, b:e] = tile[rows]
        m = float(torch.from_numpy(tile).abs().max())  # NaN if any entry is NaN
        if not m == m:
            worst[0] = float("nan")
        elif worst[0] == worst[0]:
            worst[0] = max(worst[0], m)

    with sec.SparseCosine(cfg.dim, chunk_rows=CHUNK, verify_stream=True) as h:
        h.bulk_cosine_host(Q, I, consumer=consume, ring_depth=3)
        sums = h.stream_checksums()
    n_chunks = -(-cfg.n_i // CHUNK)
    assert [c for c, _, _ in seen] == list(range(n_chunks))
    assert [(b, e) for _, b, e in seen] == [(b, min(b + CHUNK, cfg.n_i)) for b in range(0, cfg.n_i, CHUNK)]
    assert len(sums) == n_chunks  # one verified checksum per chunk (device == host copy)
    assert worst[0] <= 1.0 + TOL  # every entry finite and in range
    ref = oracle.cosine(Q, I, q_rows=rows)
    err = float(np.abs(sampled.astype(np.float64) - ref).max())
    print(f"{name}: {n_chunks} chunks through the ring, sampled rows max |error| {err:.3e}")
    assert err <= TOL, f"{name}: max abs error {err:.3e}"


def test_host_ring_checksums_match_device(sec):
    cfg = CONFIGS["d1.2m_q5k_i200k"].scaled(2000, 60_000)
    Q, I = generate_side(cfg, 0), generate_side(cfg, 1)
    rows = sample_query_rows(cfg.n_q, 256, cfg.seed)
    _, _, _, dev_sums = _device_pass(sec, cfg, Q, I, rows)
    host_sums, host_rows = [], np.empty((len(rows), I.n_rows), np.float32)

    def consume(c, b, e, tile):
        host_sums.append(int(tile.view(np.int32).astype(np.int64).sum()))
        host_rows[:, b:e] = tile[rows]

    with sec.SparseCosine(cfg.dim, chunk_rows=CHUNK) as h:
        h.bulk_cosine_host(Q, I, consumer=consume, ring_depth=3)
    assert host_sums == dev_sums
    ref = oracle.cosine(Q, I, q_rows=rows)
    assert float(np.abs(host_rows.astype(np.float64) - ref).max()) <= TOL
