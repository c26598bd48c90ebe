#!/usr/bin/env python3
"""Throughput of exact bulk cosine similarity over CSR sparse embeddings.

One step = one pass of the whole path over one batch: row norms of Q and I,
then for every 8,192-item chunk the inverted index and the scoring kernel
(fused normalisation), leaving the full n_q x n_i float32 matrix in HBM.
`value` is pair-scores/s with the inputs resident in HBM; `e2e` is the same
metric through ss_bulk_cosine_host from pinned host buffers, with the input
copies and the device-to-host stream of the whole result inside the timed
region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) each rank scores its own item set against the same
queries (weak scaling: item rows [r*n_i, (r+1)*n_i) of one larger seeded set),
with no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import CONFIGS, generate_rows, generate_side, sample_query_rows  # noqa: E402

WORKLOAD = "d1.2m_q5k_i200k"
METRIC = "cosine pair-scores/sec"
UNIT = "pair-scores/s"
CHUNK = 8192
FLUSH_BYTES = 512 << 20  # > 129 MB L2
# Results larger than this stay on the device only chunk by chunk: two
# chunk-sized buffers alternate (every score is still computed and stored).
RESIDENT_OUTPUT_BYTES = 64 << 30
NOMINAL_HBM_GBS = 8000.0
# What the scores are computed in, per scoring algorithm of the handle.
ARITHMETIC = {
    0: "f32 (item tiles: fp32 products and sums)",
    1: "f32 (posting lists: fp32 products summed exactly in 2^-38 fixed point)",
    2: "f32 (hot dims: 2x fp16 split on tcgen05, fp32 accumulate; cold dims: exact 2^-28 fixed point)",
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD, choices=sorted(CONFIGS))
    p.add_argument("--algorithm", default="auto", choices=["auto", "hybrid", "posting", "tensor"],
                   help="scoring algorithm of the handle (auto: the library's choice per item matrix)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--topk", type=int, default=0,
                   help="also time the same step with the top-k epilogue (per query row, the k best items) "
                        "in place of storing the full matrix; reported under 'topk'")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target seconds of oracle work for the CPU baseline sample")
    p.add_argument("--ref-seconds", type=float, default=10.0,
                   help="target seconds of oracle work per step of the reference arm")
    p.add_argument("--n-queries", type=int, default=0,
                   help="use only the first N query rows (small profiling captures)")
    p.add_argument("--n-items", type=int, default=0,
                   help="use only the first N item rows (small profiling captures)")
    p.add_argument("--host-values", default="f32", choices=["f32", "bf16", "f16"],
                   help="value type of the host CSRs of the e2e leg (16-bit values are rounded from the "
                        "float32 workload, sent at 2 bytes a value and widened on the device)")
    p.add_argument("--device-limit", type=int, default=0,
                   help="device bytes the e2e host pass may hold for input copies and output tiles "
                        "(0: no limit); above it the pass streams item batches and tiles the queries")
    return p.parse_args()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def captured_traffic(workload, kernel):
    """DRAM bytes per scoring launch from a committed ncu capture of this
    workload and kernel, or None when there is none or the kernel's source
    has changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "score_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f)["records"]
    for rec in recs:
        if rec["workload"] != workload or rec["kernel"] != kernel:
            continue
        src = os.path.join(ROOT, rec["source"])
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])
    return None


def chunk_algorithmic_bytes(Q, I):
    """Bytes the scoring kernel must move per chunk (each item counted once).

    Output 4*n_q*C, the chunk's posting lists 6*nnz_c (16-bit item number +
    float32 value) plus 4*(touched dims + 1) list offsets, the query CSR
    12*nnz(Q) + 8*(n_q + 1), and the norms 4*(n_q + C).
    """
    out = []
    q_bytes = 12 * Q.nnz + 8 * (Q.n_rows + 1)
    for b in range(0, I.n_rows, CHUNK):
        e = min(b + CHUNK, I.n_rows)
        lo, hi = int(I.indptr[b]), int(I.indptr[e])
        touched = int(np.unique(I.indices[lo:hi]).size)
        c = e - b
        out.append(4 * Q.n_rows * c + 6 * (hi - lo) + 4 * (touched + 1) + q_bytes + 4 * (Q.n_rows + c))
    return out


def cpu_baseline(cfg, Q, I, seconds: float):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    import oracle

    oracle.build()
    cores = host_cores()
    probe_rows = sample_query_rows(cfg.n_q, 2, cfg.seed + 1)
    t0 = time.perf_counter()
    oracle.cosine(Q, I, q_rows=probe_rows, threads=2)
    per_row = max(time.perf_counter() - t0, 1e-4)  # one row on one thread
    k = int(max(2, min(cfg.n_q, seconds * cores / per_row)))
    rows = sample_query_rows(cfg.n_q, k, cfg.seed)
    t0 = time.perf_counter()
    oracle.cosine(Q, I, q_rows=rows[:k], threads=cores)
    dt = time.perf_counter() - t0
    pairs = k * I.n_rows
    return {"value": pairs / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{k} sampled query rows x all {I.n_rows} items ({pairs} pairs, "
                      f"{dt:.1f} s, {cores} threads)"}


def item_shard(cfg, rank: int, world: int):
    """Weak scaling: rank r scores item rows [r*n_i, (r+1)*n_i) of one seeded
    item set of world*n_i rows against the same queries (no data exchange)."""
    big = cfg.scaled(cfg.n_q, cfg.n_i * world, name=cfg.name)
    return big, rank * cfg.n_i, (rank + 1) * cfg.n_i


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    cfg = CONFIGS[args.workload]
    Q = generate_side(cfg, 0)
    I = generate_side(cfg, 1)
    import oracle

    oracle.build()
    cores = host_cores()
    # each step ~ref_seconds (10 s) of oracle work on all cores, so K + W steps end in minutes
    probe_rows = sample_query_rows(cfg.n_q, 2, cfg.seed + 1)
    t0 = time.perf_counter()
    oracle.cosine(Q, I, q_rows=probe_rows, threads=2)
    per_row = max(time.perf_counter() - t0, 1e-4)
    k = int(max(1, min(cfg.n_q, args.ref_seconds * cores / per_row)))
    rows = sample_query_rows(cfg.n_q, min(cfg.n_q, 4 * k), cfg.seed)
    times = []
    for s in range(args.warmup + args.steps):
        sel = rows[(s * k) % len(rows):][:k]
        if len(sel) < k:
            sel = rows[:k]
        t0 = time.perf_counter()
        oracle.cosine(Q, I, q_rows=sel, threads=cores)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    pairs = k * I.n_rows
    value = pairs / statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "n_q": cfg.n_q, "n_i": cfg.n_i, "dim": cfg.dim,
                   "step_sample": f"{k} sampled query rows x all {I.n_rows} items per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{k} sampled query rows x all {I.n_rows} items per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import sparse_embedding_exact_gb300 as sec
    from sparse_embedding_exact_gb300 import build

    build.build()
    cfg = CONFIGS[args.workload]
    if args.n_queries or args.n_items:
        cfg = cfg.scaled(args.n_queries or cfg.n_q, args.n_items or cfg.n_i)
    Q = generate_side(cfg, 0)
    if world > 1:
        big, b, e = item_shard(cfg, rank, world)
        I = generate_rows(big, 1, b, e, workers=max(1, host_cores() // world))
    else:
        I = generate_side(cfg, 1)

    # CPU baseline first (rank 0, N = 1 only), before the GPU work.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, Q, I, args.cpu_seconds)

    h = sec.SparseCosine(cfg.dim, chunk_rows=CHUNK, device=local, algorithm=args.algorithm)
    q = sec.DeviceCsr.from_host(Q, dev)
    it = sec.DeviceCsr.from_host(I, dev)
    n_q, n_i = Q.n_rows, I.n_rows
    resident = 4 * n_q * n_i <= RESIDENT_OUTPUT_BYTES
    if resident:
        out = torch.empty((n_q, n_i), dtype=torch.float32, device=dev)
    else:
        bufs = [torch.empty((n_q, CHUNK), dtype=torch.float32, device=dev) for _ in range(2)]
    inv_q = torch.empty(n_q, dtype=torch.float32, device=dev)
    inv_i = torch.empty(n_i, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    chunks = [(b, min(b + CHUNK, n_i)) for b in range(0, n_i, CHUNK)]
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in chunks]
    span = CHUNK * h.build_batch  # chunks whose indexes one build launch covers
    batches = [(b, min(b + span, n_i)) for b in range(0, n_i, span)]
    batch_chunks = [[c for c, (b, _) in enumerate(chunks) if bb <= b < be] for bb, be in batches]
    ev_build = [torch.cuda.Event(enable_timing=True) for _ in batches]

    def step(sampled=None):
        # Every step redoes the whole path: the hot set and the prepared
        # queries are derived again, not reused from the previous step.
        # Events (around the scoring calls, around the scoring kernel inside
        # them, before the build) go into the build batch `sampled` only:
        # each event costs GPU time, so timing every launch would slow the
        # step it measures.
        h.invalidate()
        h.row_norms(q, out=inv_q)
        h.row_norms(it, out=inv_i)
        c = 0
        for bi, (bb, be) in enumerate(batches):
            rec = bi == sampled
            if rec:
                ev_build[bi].record(stream)
            for b, e, idx in h.build_item_indexes(it, bb, be):
                if rec:
                    ev[c][0].record(stream)
                    h.profile_scorer(True)
                if resident:
                    h.score_chunk(q, inv_q, idx, inv_i[b:], out[:, b:], n_i)
                else:
                    h.score_chunk(q, inv_q, idx, inv_i[b:], bufs[c & 1], CHUNK)
                if rec:
                    h.profile_scorer(False)
                    ev[c][1].record(stream)
                c += 1
        return batch_chunks[sampled] if sampled is not None else []

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    h.check_device()
    index_stats = h.index_stats(h.build_item_index(it, *chunks[0]))

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    launches0 = h.kernel_launches()
    h.scorer_time()  # forget pairs recorded before the timed region
    step_ms, score_ms, build_ms, timed_chunks = [], [], [], []
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(args.steps):
        flush.fill_(1.0)  # evict L2 between timed steps
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        sb = k % len(batches)  # the batches take turns carrying the events
        t_start.record(stream)
        cs = step(sb)
        t_end.record(stream)
        torch.cuda.synchronize()
        step_ms.append(t_start.elapsed_time(t_end))
        score_ms.extend(ev[c][0].elapsed_time(ev[c][1]) for c in cs)
        timed_chunks.extend(cs)
        build_ms.append(ev_build[sb].elapsed_time(ev[cs[0]][0]))
    launches = h.kernel_launches() - launches0
    kernel_ms_total, kernel_launches = h.scorer_time()
    clocks = sampler.stop()
    h.check_device()

    ms = statistics.mean(step_ms)
    if world > 1:
        import torch.distributed as dist

        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = world * n_q * n_i / (ms / 1e3)

    # Roofline of the dominant kernel (the scoring kernel), timed by the
    # library's own events around each of its launches; the whole scoring
    # call (with its preparation kernels) is reported beside it.
    alg = chunk_algorithmic_bytes(Q, I)
    per_launch_bytes = statistics.mean(alg[c] for c in timed_chunks)
    call_s = statistics.mean(score_ms) / 1e3
    per_launch_s = (kernel_ms_total / kernel_launches / 1e3) if kernel_launches else call_s
    achieved = per_launch_bytes / per_launch_s / 1e9
    peak, peak_kind = measured_peaks()
    kernel = {0: "k_score_tiles", 1: "k_score_lists", 2: "k_tc_score"}[index_stats["algorithm"]]
    label = {0: " (item tiles)", 1: " (posting lists)", 2: " (tensor cores)"}[index_stats["algorithm"]]
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": captured_traffic(cfg.name, kernel),
            "kernel": kernel + label,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "frac_basis": "algorithmic bytes of one chunk (output + the chunk's lists + query CSR + norms) "
                          "over the scoring kernel's own launch time; call_frac: the same bytes over the "
                          "whole scoring call; output_hbm_gbs: the whole step's output bytes over its time",
            "bytes_per_launch": per_launch_bytes, "launch_ms": 1e3 * per_launch_s,
            "launches_timed": kernel_launches,
            "call_ms": 1e3 * call_s, "call_frac": per_launch_bytes / call_s / 1e9 / peak,
            "timing_sample": "events around one build batch of chunks per timed step (the batches "
                             "in turn); the other batches run without events",
            "score_share_of_step": statistics.mean(score_ms) * len(chunks) / max(statistics.mean(step_ms), 1e-9),
            "index_build_ms_per_launch": statistics.mean(build_ms),
            "index_build_chunks_per_launch": h.build_batch}

    topk = None
    if args.topk:
        # The same step (norms, hot set, builds, scoring) with the top-k
        # epilogue: every score is computed, only each row's k best are kept.
        def step_topk():
            h.invalidate()
            h.row_norms(q, out=inv_q)
            h.row_norms(it, out=inv_i)
            return h.topk_all(q, inv_q, it, inv_i, args.topk)

        for _ in range(args.warmup):
            step_topk()
        torch.cuda.synchronize()
        h.check_device()
        tk_ms = []
        for _ in range(args.steps):
            flush.fill_(1.0)
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            t_start.record(stream)
            step_topk()
            t_end.record(stream)
            torch.cuda.synchronize()
            tk_ms.append(t_start.elapsed_time(t_end))
        h.check_device()
        tms = statistics.mean(tk_ms)
        if world > 1:
            import torch.distributed as dist

            t = torch.tensor([tms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            tms = float(t.item())
        topk = {"k": args.topk, "value": world * n_q * n_i / (tms / 1e3), "unit": UNIT,
                "ms_per_step": tms, "api": "ss_topk_all"}

    e2e = None
    if not args.no_e2e:
        import torch as _t

        def pinned(a, dt):
            t = _t.from_numpy(np.ascontiguousarray(a, dtype=dt)).pin_memory()
            return t.numpy()

        class Host:
            pass

        def host_values(v):
            if args.host_values == "bf16":
                from workload.halfprec import to_bf16_bits
                return pinned(to_bf16_bits(v), np.uint16)
            if args.host_values == "f16":
                from workload.halfprec import to_f16_bits
                return pinned(to_f16_bits(v), np.uint16)
            return pinned(v, np.float32)

        def pin_csr(m):
            o = Host()
            o.indptr, o.indices, o.values, o.dim = (pinned(m.indptr, np.int64),
                                                  pinned(m.indices, np.int32),
                                                  host_values(m.values), m.dim)
            return o

        Qh, Ih = pin_csr(Q), pin_csr(I)
        h.set_device_limit(args.device_limit)
        if resident:  # the whole matrix lands in one page-locked host array
            out_h = _t.empty((n_q, n_i), dtype=_t.float32).pin_memory()
            api = "ss_bulk_cosine_host (pinned host CSR in, pinned host matrix out)"

            def host_pass():
                h.bulk_cosine_host(Qh, Ih, out=out_h, host_values=args.host_values)
        else:  # too large to keep: each chunk reaches the pinned ring, is handed over, dropped
            api = "ss_bulk_cosine_host (pinned host CSR in, each chunk to the pinned host ring)"

            def host_pass():
                h.bulk_cosine_host(Qh, Ih, consumer=lambda c, b, e, tile: 0, ring_depth=3,
                                   host_values=args.host_values)
        host_pass()  # warm-up
        e2e_steps = max(1, min(args.steps, 3))
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_pass()
        dt = (time.perf_counter() - t0) / e2e_steps
        if world > 1:
            import torch.distributed as dist

            t = torch.tensor([dt], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            dt = float(t.item())
        h2d = sum(a.nbytes for m in (Qh, Ih) for a in (m.indptr, m.indices, m.values))
        e2e = {"value": world * n_q * n_i / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(4 * n_q * n_i), "steps": e2e_steps,
               "api": api}
        if args.host_values != "f32":
            e2e["host_values"] = args.host_values
        if args.device_limit:
            qb, ib = sec.plan_host_pass(Q.indptr, I.indptr, CHUNK, args.device_limit, resident,
                                        args.host_values)
            e2e["device_limit"] = {"bytes": args.device_limit, "query_tiles": len(qb) - 1,
                                   "item_batches": len(ib) - 1}

    h.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ARITHMETIC[index_stats["algorithm"]], "data": "synthetic",
            "config": {"workload": cfg.name, "n_q": n_q, "n_i_per_gpu": n_i, "dim": cfg.dim,
                       "chunk_rows": CHUNK, "parallelism": f"items sharded x{world}",
                       "description": cfg.description,
                       "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MB write)",
                       "output_gb_per_step": 4 * n_q * n_i / 1e9,
                       "output_kept_on_device": "whole matrix" if resident else "two chunk buffers, reused"},
            "output_hbm_gbs": 4 * n_q * n_i / (ms / 1e3) / 1e9,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "topk": topk,
            "gpu_launches": int(launches),
            "clocks": clocks,
            "first_chunk_index": index_stats,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
