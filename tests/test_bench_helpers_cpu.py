"""Host helpers of bench.py: the roofline's algorithmic bytes, the captured
DRAM traffic that is dropped once the kernel's source changes, the peaks."""
import hashlib
import json
import os

import numpy as np

import bench
from workload.tiny import csr_from_rows


def test_chunk_algorithmic_bytes_by_hand(monkeypatch):
    monkeypatch.setattr(bench, "CHUNK", 2)
    Q = csr_from_rows([([0, 5], [1.0, 2.0]), ([5], [3.0])], dim=8)          # nnz 3, 2 rows
    I = csr_from_rows([([0, 1], [1.0, 1.0]), ([1, 7], [1.0, 1.0]), ([3], [1.0])], dim=8)
    got = bench.chunk_algorithmic_bytes(Q, I)
    q = 12 * 3 + 8 * 3
    # chunk 0: items 0-1, 4 nonzeros over dims {0, 1, 7}; chunk 1: item 2, 1 nonzero over {3}
    first = 4 * 2 * 2 + 6 * 4 + 4 * (3 + 1) + q + 4 * (2 + 2)
    second = 4 * 2 * 1 + 6 * 1 + 4 * (1 + 1) + q + 4 * (2 + 1)
    assert got == [first, second]


def test_captured_traffic_follows_the_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kernel": "k", "workload": "w", "source": "kernel.cu",
           "source_sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
           "dram_bytes_read": 100, "dram_bytes_write": 23}
    (tmp_path / "profiles" / "score_traffic.json").write_text(json.dumps({"records": [rec]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.captured_traffic("w", "k") == 123
    assert bench.captured_traffic("other", "k") is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.captured_traffic("w", "k") is None


def test_committed_traffic_records_name_existing_sources():
    path = os.path.join(bench.ROOT, "profiles", "score_traffic.json")
    with open(path) as f:
        recs = json.load(f)["records"]
    assert recs
    for rec in recs:
        assert os.path.exists(os.path.join(bench.ROOT, rec["source"]))
        assert rec["dram_bytes_read"] > 0 and rec["dram_bytes_write"] > 0
        assert os.path.exists(os.path.join(bench.ROOT, rec["capture"]))


def test_peaks_come_from_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6798.6}))
    assert bench.measured_peaks() == (6798.6, "measured")
    assert np.isfinite(bench.measured_peaks()[0])
