#!/usr/bin/env python3
"""Benchmark of the lattice-PIR database scan on GB300.

Default workload: the 64 GiB RowSel query pipeline (N = 4096, 3 RNS primes
below 2^29, D0 = 1024 x D1 = 1365 records, one query): forward NTT of the
query (2048 polynomials), the RowSel scan of the NTT-domain DB, inverse NTT of
the 2730 result polynomials.  One step = one query batch through all three
kernels; the encoded DB stays resident in HBM (encoded once, untimed).

Prints ONE JSON line (rank 0):
  value     DB GB/s scanned (logical DB bytes / step time), device-resident
            inputs, CUDA events on the launching stream, max over ranks;
  e2e       the same metric through the public API with the query coming
            from pinned host memory and the result going back to it;
  roofline  the RowSel kernel's algorithmic bytes / its average launch time
            against the measured HBM copy bandwidth, also as fractions of an
            in-run read-only stream over the DB and of the 8 TB/s spec;
  cpu_baseline  the oracle (plain C, all host cores) on a bounded sample.

--impl reference runs the oracle itself as the reference arm (each step a
bounded sample of the same workload on the host cores).
Multi-GPU (torchrun): every rank runs an independent replica (the scan does
not exchange data); value aggregates all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GIB = 1 << 30
WORKLOADS = {
    # name: ring, DB grid, batch, query domain
    "rowsel_64g": dict(N=4096, L=3, D0=1024, D1=1365, B=1, domain="coeff",
                       desc="RowSel 64 GiB NTT-form DB: N=4096, 3 RNS primes <2^29, D0=1024 x D1=1365 records, "
                            "B=1 query; step = NTT(query, 2048 polys) + RowSel scan + INTT(2730 result polys)"),
    "rowsel_6g": dict(N=4096, L=3, D0=256, D1=512, B=1, domain="ntt",
                      desc="RowSel 6 GiB: N=4096, 3 primes, D0=256 x D1=512, B=1, NTT-domain query"),
    "rowsel_24g_b16": dict(N=4096, L=3, D0=512, D1=1024, B=16, domain="ntt",
                           desc="RowSel 24 GiB: N=4096, 3 primes, D0=512 x D1=1024, B=16 queries, NTT-domain"),
    "rowsel_64g_b16": dict(N=4096, L=3, D0=1024, D1=1365, B=16, domain="ntt",
                           desc="RowSel 64 GiB: N=4096, 3 primes, D0=1024 x D1=1365, B=16 queries, NTT-domain"),
    "onion_64g": dict(kind="onion", N=4096, L=3, D0=1024, D1=1365, ell=5, w=18,
                      desc="OnionPIR server path per query over the 64 GiB DB: ExpandQuery of the row "
                           "ciphertext 1 -> 1024 and of the column ciphertext 1 -> 64 (55 gadget ciphertexts "
                           "of the 11 column bits), their conversion to 11 RGSW ciphertexts, RowSel "
                           "D0=1024 x D1=1365, ColTor 1365 -> 1 (N=4096, 3 primes, l=5)"),
    "onion_64g_b16": dict(kind="onion", N=4096, L=3, D0=1024, D1=1365, ell=5, w=18, B=16,
                          desc="OnionPIR server path for 16 clients per pass over the 64 GiB DB: 16 ExpandQuery "
                               "of the row ciphertexts 1 -> 1024 and of the column ciphertexts 1 -> 64 (batched "
                               "calls), 16 x 11 RGSW conversions (one batched call), one RowSel pass D0=1024 x "
                               "D1=1365 x 16 queries (tensor cores), 16 ColTor 1365 -> 1 (one batched call); "
                               "N=4096, 3 primes, l=5"),
    "expand_1024": dict(kind="expand", N=4096, L=3, stages=10, ell=5, w=18,
                        desc="ExpandQuery of one query ciphertext into the 1024 RowSel inputs of the 64 GiB DB: "
                             "N=4096, 3 primes, 10 stages of Subs, l=5 digits of 18 bits"),
    "coltor_1365": dict(kind="coltor", N=4096, L=3, n=1365, ell=5, w=18,
                        desc="ColTor over the 1365 RowSel output ciphertexts of one 64 GiB query: N=4096, "
                             "3 primes, 11 stages of RGSW-RLWE external products, l=5 digits of 18 bits"),
    # scalar-HE scan: byte DB x 64 query words mod 2^32 (tcgen05 fp16 path)
    "scalar_16g": dict(kind="scalar", R=131072, C=131072, B=64,
                       desc="Scalar-HE scan: DB 131072 x 131072 uint8 (16 GiB) x Q 131072 x 64 uint32, mod 2^32"),
    "scalar_16g_b1": dict(kind="scalar", R=131072, C=131072, B=1,
                          desc="Scalar-HE scan, one query: DB 131072 x 131072 uint8 (16 GiB) x Q 131072 uint32, "
                               "mod 2^32 (CUDA-core GEMV path)"),
    "scalar_2g_b1_prof": dict(kind="scalar", R=16384, C=131072, B=1,
                              desc="Scalar-HE scan profiling case, one query: DB 16384 x 131072 uint8 (2 GiB)"),
    "scalar_2g_prof": dict(kind="scalar", R=16384, C=131072, B=64,
                           desc="Scalar-HE scan profiling case: DB 16384 x 131072 uint8 (2 GiB), B=64"),
    # small case of the B=16 workload for profiler captures (3 GiB, tensor-core path)
    "rowsel_3g_b16_prof": dict(N=4096, L=3, D0=512, D1=128, B=16, domain="ntt",
                               desc="RowSel 3 GiB profiling case: N=4096, 3 primes, D0=512 x D1=128, B=16"),
    # ring-packing GEMM of expansion-based packing: the pages' 64 GiB configuration
    # (hint H of Dr = 256 x n = 1280 polynomials, 15 GiB), one client
    "exppack_15g": dict(kind="exppack", N=4096, L=3, n=1280, Dr=256, B=1,
                        desc="ExpPack GEMM H*C + (0|G): N=4096, 3 primes, hint Dr=256 x n=1280 polys (15 GiB), "
                             "B=1; step = lift+NTT(G, 256 polys) + the point-wise GEMM"),
    # the full-size workloads' per-point shapes on fewer evaluation points (a
    # smaller ring), for profiler captures of a few GB: traffic per point is
    # the same, so a full launch's traffic is the small launch's times the
    # ratio of points (12288 / 384 = 32, 12288 / 1536 = 8)
    "rowsel_64g_shape_2g_prof": dict(N=128, L=3, D0=1024, D1=1365, B=1, domain="ntt",
                                     desc="RowSel profiling case with the 64 GiB workload's point shape: N=128, "
                                          "3 primes (384 points), D0=1024 x D1=1365, B=1 (2.1 GB DB)"),
    "rowsel_64g_shape_2g_b16_prof": dict(N=128, L=3, D0=1024, D1=1365, B=16, domain="ntt",
                                         desc="RowSel profiling case with the 64 GiB workload's point shape: "
                                              "N=128, 3 primes (384 points), D0=1024 x D1=1365, B=16 (2.1 GB DB)"),
    "rowsel_24g_shape_3g_b16_prof": dict(N=512, L=3, D0=512, D1=1024, B=16, domain="ntt",
                                         desc="RowSel profiling case with the 24 GiB workload's point shape: "
                                              "N=512, 3 primes (1536 points), D0=512 x D1=1024, B=16 (3.2 GB DB)"),
    "exppack_15g_shape_2g_prof": dict(kind="exppack", N=512, L=3, n=1280, Dr=256, B=1,
                                      desc="ExpPack profiling case with the 15 GiB hint's point shape: N=512, "
                                           "3 primes (1536 points), hint Dr=256 x n=1280 (2.0 GB), B=1"),
    # small case of the 64 GiB pipeline for profiler captures (3 GiB, 2 column slabs)
    "rowsel_3g_prof": dict(N=4096, L=3, D0=256, D1=256, B=1, domain="coeff",
                           desc="RowSel 3 GiB profiling case: N=4096, 3 primes, D0=256 x D1=256, B=1, "
                                "NTT + RowSel + INTT"),
}
METRIC = "DB GB/s scanned & queries/s (RowSel, 64 GiB DB), % of GB300 HBM roofline"
SPEC_HBM_GBS = 8000.0   # nominal GB300 HBM3e bandwidth (context for the roofline fractions)
EXPPACK_METRIC = "ring-packing GEMM H*C + (0|G): hint GB/s scanned"
COLTOR_METRIC = "ColTor column tournaments per second (RGSW-RLWE external products)"
EXPAND_METRIC = "ExpandQuery expansions per second (Subs: automorphism + key switching)"
ONION_METRIC = "OnionPIR queries per second (ExpandQuery + RowSel + ColTor), 64 GiB DB"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="rowsel_64g", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiler runs)")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload only: skip the short timings of the other benchmark configurations")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float) -> float:
    """Largest value of x over all ranks (x itself without a process group).
    Works with NCCL (CUDA tensor) and gloo (CPU tensor) groups."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, steps: int, ms_total_max: float, world: int) -> float:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return world * units_per_rank * steps / (ms_total_max * 1e-3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def profile_traffic(kernel: str) -> dict:
    """DRAM bytes per launch from the committed ncu summary of `kernel`, with
    where they come from: {"traffic": bytes or None, "traffic_source": {...}}.
    The summary's `traffic_case:` line names the case the counters were taken
    on (and how they were scaled to a full launch, if they were)."""
    rel = os.path.join("profiles", "%s.md" % kernel)
    value, case = None, None
    try:
        for line in open(os.path.join(ROOT, rel)):
            if line.startswith("traffic_bytes_per_launch:"):
                v = line.split(":", 1)[1].strip()
                value = None if v in ("", "null") else float(v)
            elif line.startswith("traffic_case:"):
                case = line.split(":", 1)[1].strip()
    except OSError:
        return {"traffic": None, "traffic_source": None}
    return {"traffic": value, "traffic_source": {"profile": rel, "case": case}}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.f.name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU) leg
# Every oracle sample has a bounded size (host memory is not sized for the
# workloads) and is repeated until its time budget is spent.
SAMPLE_WORDS = 1 << 26   # at most 64 Mi DB (or hint) words per oracle sample


def sample_points(words_per_point: int) -> int:
    """Evaluation points (prime 0) of a sample: a multiple of 16 in [16, 4096]."""
    pts = SAMPLE_WORDS // max(1, words_per_point)
    return max(16, min(4096, pts // 16 * 16))


def repeat_for(fn, seconds: float):
    """Calls fn until `seconds` have passed (at least once): (calls, seconds taken)."""
    calls, t = 0, time.perf_counter()
    while True:
        fn()
        calls += 1
        dt = time.perf_counter() - t
        if dt >= seconds:
            return calls, dt


def calls_per_step(fn, seconds: float) -> int:
    """How many calls of fn fill about `seconds` (one timed call after a warm one)."""
    fn()
    t = time.perf_counter()
    fn()
    return max(1, int(round(seconds / max(time.perf_counter() - t, 1e-4))))


class RowselSample:
    """Oracle RowSel on a bounded sample of a workload: all D0 rows and B
    queries, one column per host thread, as many evaluation points of prime 0
    as the sample size allows."""

    def __init__(self, cfg):
        import oracle
        import synth
        N, D0, B = cfg["N"], cfg["D0"], cfg["B"]
        self.threads = oracle.default_threads()
        self.ncols = min(cfg["D1"], self.threads)
        self.pts = sample_points(D0 * self.ncols)
        self.q0 = oracle.primes(N, 1)[0]
        self.db = synth.residues(11, (D0, self.ncols, 1, self.pts), [self.q0], tid=synth.T_EXTRA)
        self.qu = synth.residues(12, (B, D0, 2, 1, self.pts), [self.q0], tid=synth.T_EXTRA)
        self.nbytes = D0 * self.ncols * self.pts * 4
        self.desc = ("oracle RowSel on %d of %d DB columns x %d of %d evaluation points, all %d rows, B=%d"
                     % (self.ncols, cfg["D1"], self.pts, cfg["L"] * N, D0, B))

    def __call__(self):
        import oracle
        oracle.rowsel(self.db, self.qu, [self.q0], threads=self.threads)


class ExppackSample:
    """Oracle ring-packing GEMM on a bounded sample: all n hint columns and B
    clients, one hint row per host thread, evaluation points of prime 0."""

    def __init__(self, cfg):
        import oracle
        import synth
        n, B = cfg["n"], cfg["B"]
        self.threads = oracle.default_threads()
        self.rows = min(cfg["Dr"], self.threads)
        self.pts = sample_points(n * self.rows)
        self.q0 = oracle.primes(cfg["N"], 1)[0]
        self.H = synth.residues(11, (self.rows, n, 1, self.pts), [self.q0], tid=synth.T_EXTRA)
        self.C = synth.residues(12, (B, n, 2, 1, self.pts), [self.q0], tid=synth.T_EXTRA)
        self.G = synth.residues(13, (B, self.rows, 1, self.pts), [self.q0], tid=synth.T_EXTRA)
        self.nbytes = self.rows * n * self.pts * 4
        self.desc = ("oracle ExpPack GEMM on %d of %d hint rows x %d of %d evaluation points, all n=%d, B=%d"
                     % (self.rows, cfg["Dr"], self.pts, cfg["L"] * cfg["N"], n, B))

    def __call__(self):
        import oracle
        oracle.exppack(self.H, self.C, self.G, [self.q0], threads=self.threads)


class ScalarSample:
    """Oracle scalar scan on a bounded sample: one DB row per host thread
    (all C columns) against the full query matrix."""

    def __init__(self, cfg):
        import oracle
        import synth
        R, C, B = cfg["R"], cfg["C"], cfg["B"]
        self.threads = oracle.default_threads()
        self.rows = min(R, self.threads)
        self.Q = synth.words(7, (C, B))
        self.db = synth.db_bytes(7, (self.rows, C))
        self.nbytes = self.rows * C
        self.desc = "oracle scalar scan on %d of %d DB rows x %d columns, B=%d" % (self.rows, R, C, B)

    def __call__(self):
        import oracle
        oracle.scalar_scan(self.db, self.Q, threads=self.threads)


class ColtorSample:
    """Oracle ColTor on a bounded sample: one tournament stage over two
    ciphertexts per host thread (one external product each), counted as the
    fraction of a whole tournament (n - 1 external products) it performs."""
    unit = "queries/s"

    def __init__(self, cfg):
        import oracle
        import synth
        N, L, n, ell = cfg["N"], cfg["L"], cfg["n"], cfg["ell"]
        self.ell, self.w = ell, cfg["w"]
        self.threads = oracle.default_threads()
        self.pairs = max(1, min((n + 1) // 2, self.threads))
        self.qs = oracle.primes(N, L)
        self.psis = [oracle.min_psi(q, N) for q in self.qs]
        self.C = synth.residues(11, (2 * ell, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.cts = synth.residues(12, (2 * self.pairs, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.nbytes = self.pairs / max(1, n - 1)      # tournaments per call
        self.desc = ("oracle ColTor stage over %d ciphertexts (%d external products of %d per tournament), "
                     "N=%d, L=%d, l=%d" % (2 * self.pairs, self.pairs, n - 1, N, L, ell))

    def __call__(self):
        import oracle
        oracle.coltor_stage(self.C, self.cts, self.qs, self.psis, self.ell, self.w, threads=self.threads)


class ExpandSample:
    """Oracle ExpandQuery on a bounded sample: one expansion stage over one
    ciphertext per host thread (one Subs each), counted as the fraction of a
    whole expansion (2^stages - 1 Subs operations) it performs."""
    unit = "queries/s"

    def __init__(self, cfg):
        import oracle
        import synth
        N, L, S, ell = cfg["N"], cfg["L"], cfg["stages"], cfg["ell"]
        self.ell, self.w, self.stage = ell, cfg["w"], S - 1
        self.threads = oracle.default_threads()
        self.M = max(1, min(1 << (S - 1), self.threads))
        self.qs = oracle.primes(N, L)
        self.psis = [oracle.min_psi(q, N) for q in self.qs]
        self.evk = synth.residues(13, (ell, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.cts = synth.residues(14, (self.M, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.nbytes = self.M / ((1 << S) - 1)          # expansions per call
        self.desc = ("oracle ExpandQuery stage over %d ciphertexts (%d Subs of %d per expansion), N=%d, L=%d, l=%d"
                     % (self.M, self.M, (1 << S) - 1, N, L, ell))

    def __call__(self):
        import oracle
        oracle.expand_stage(self.evk, self.cts, self.stage, self.qs, self.psis, self.ell, self.w,
                            threads=self.threads)


class RgswSample:
    """Oracle conversion of one client's expanded gadget ciphertexts into one
    RGSW ciphertext (ell key switches), counted as the fraction of a query's
    T = ceil(log2 D1) conversions it performs."""
    unit = "queries/s"

    def __init__(self, cfg):
        import oracle
        import synth
        N, L, ell, T = cfg["N"], cfg["L"], cfg["ell"], cfg["T"]
        self.ell, self.w = ell, cfg["w"]
        self.threads = 1
        self.qs = oracle.primes(N, L)
        self.psis = [oracle.min_psi(q, N) for q in self.qs]
        self.ksk = synth.residues(15, (ell, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.cts = synth.residues(16, (ell, 2, L, N), self.qs, tid=synth.T_EXTRA)
        self.nbytes = 1.0 / T                          # queries per call
        self.desc = "oracle RGSW conversion of one column bit (%d key switches; %d bits per query), N=%d, L=%d" % (
            ell, T, N, L)

    def __call__(self):
        import oracle
        oracle.rgsw_convert(self.ksk, self.cts, self.qs, self.psis, self.ell, self.w)


class OnionSample:
    """Oracle OnionPIR path, composed from bounded samples of its phases
    (ExpandQuery of the row and of the column ciphertext, the RGSW
    conversion of the column bits, RowSel over all D0 rows for the B
    queries, ColTor): a call runs one call of each phase's sample and times
    it; a query costs the sum over the phases of (time per call) / (queries
    per call), where a call covers the fraction of a query's expansion,
    conversion, DB scan or tournament its sample performs."""
    unit = "queries/s"

    def __init__(self, cfg):
        N, L, D0, D1, ell, w = cfg["N"], cfg["L"], cfg["D0"], cfg["D1"], cfg["ell"], cfg["w"]
        B = cfg.get("B", 1)
        S = D0.bit_length() - 1
        T = coltor_stages(D1)
        self.phases = [
            ExpandSample(dict(N=N, L=L, stages=S, ell=ell, w=w)),
            ExpandSample(dict(N=N, L=L, stages=column_stages(T, ell), ell=ell, w=w)),
            RgswSample(dict(N=N, L=L, ell=ell, w=w, T=T)),
            RowselSample(dict(N=N, L=L, D0=D0, D1=D1, B=B)),
            ColtorSample(dict(N=N, L=L, n=D1, ell=ell, w=w)),
        ]
        r = self.phases[3]
        # queries per call: expansions, conversions or tournaments per call,
        # or the scanned fraction of the DB times the B queries the scan serves
        self.per_call = [self.phases[0].nbytes, self.phases[1].nbytes, self.phases[2].nbytes,
                         r.nbytes / (D0 * D1 * L * N * 4) * B, self.phases[4].nbytes]
        self.threads = r.threads
        self.nbytes = 0.0
        self.reset()
        self.desc = "oracle OnionPIR path per query, composed of: " + "; ".join(x.desc for x in self.phases)

    def reset(self):
        self.spent = [0.0] * len(self.phases)
        self.calls = 0

    def __call__(self):
        for i, ph in enumerate(self.phases):
            t = time.perf_counter()
            ph()
            self.spent[i] += time.perf_counter() - t
        self.calls += 1

    def queries_per_s(self) -> float:
        per_query = sum(t / max(1, self.calls) / q for t, q in zip(self.spent, self.per_call))
        return 1.0 / per_query


def _rate(sample, units_per_s: float):
    """A sample's rate in its metric unit (GB/s unless the sample says otherwise)."""
    unit = getattr(sample, "unit", "GB/s")
    return (units_per_s / 1e9 if unit == "GB/s" else units_per_s), unit


def _sample_rate(sample, calls: int, dt: float):
    """Rate of `calls` calls of a sample taking dt seconds in its metric unit;
    a composed sample reports its own."""
    if hasattr(sample, "queries_per_s"):
        return sample.queries_per_s(), sample.unit
    return _rate(sample, sample.nbytes * calls / dt)


def oracle_baseline(sample, seconds: float):
    """cpu_baseline object: the sample repeated for about `seconds`."""
    sample()                                   # first touch of the inputs
    if hasattr(sample, "reset"):
        sample.reset()
    calls, dt = repeat_for(sample, seconds)
    value, unit = _sample_rate(sample, calls, dt)
    return {"value": value, "unit": unit, "cores": sample.threads, "kind": "oracle",
            "sample": "%s; %d calls in %.1f s" % (sample.desc, calls, dt), "seconds": round(dt, 2)}


def run_reference_sample(args, sample, metric, dtype, data, desc):
    """Reference arm: each step repeats the bounded oracle sample for about
    120 s / (steps + warmup) on all host cores."""
    per_step = 120.0 / max(1, args.steps + args.warmup)
    reps = calls_per_step(sample, per_step)

    def one_step():
        for _ in range(reps):
            sample()

    for _ in range(args.warmup):
        one_step()
    if hasattr(sample, "reset"):
        sample.reset()
    t = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = (time.perf_counter() - t) / max(1, args.steps)
    value, unit = _sample_rate(sample, reps * args.steps, dt * args.steps)
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": data, "config": {"workload": args.workload, "desc": desc},
        "cpu_baseline": {"value": value, "unit": unit, "cores": sample.threads, "kind": "oracle",
                         "sample": "per step %d calls of: %s" % (reps, sample.desc)},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, cfg):
    """Reference arm: the oracle as it stands, timed on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    kind = cfg.get("kind")
    if kind == "scalar":
        run_reference_sample(args, ScalarSample(cfg), "scalar-HE scan: DB GB/s scanned", "u8 x u32",
                             "synthetic", cfg["desc"])
    elif kind == "exppack":
        run_reference_sample(args, ExppackSample(cfg), EXPPACK_METRIC, "u32",
                             "synthetic (seeded SplitMix64 residues)", cfg["desc"])
    elif kind == "coltor":
        run_reference_sample(args, ColtorSample(cfg), COLTOR_METRIC, "u32",
                             "synthetic (seeded SplitMix64 residues)", cfg["desc"])
    elif kind == "expand":
        run_reference_sample(args, ExpandSample(cfg), EXPAND_METRIC, "u32",
                             "synthetic (seeded SplitMix64 residues)", cfg["desc"])
    elif kind == "onion":
        run_reference_sample(args, OnionSample(cfg), ONION_METRIC, "u32", "synthetic (seeded SplitMix64 residues)",
                             cfg["desc"])
    else:
        run_reference_sample(args, RowselSample(cfg), METRIC, "u32", "synthetic (seeded SplitMix64 residues)",
                             cfg["desc"])


# ---------------------------------------------------------------- GPU leg
def rowsel_passes(D0, B) -> int:
    """Query passes of one RowSel call (primes >= 2^26): 16 queries on the
    tensor cores while more than 8 remain, the rest on the CUDA cores as many
    as their on-chip query slice holds (112 KiB of 4-byte residues, 2
    polynomials per query)."""
    cap = 32
    while cap > 2 and D0 * cap * 4 > 112 * 1024:
        cap //= 2
    passes, left = 0, B
    while left:
        left -= min(left, 16) if left > 8 else min(left, cap // 2)
        passes += 1
    return passes


def coltor_stages(n) -> int:
    """Stages of a tournament over n ciphertexts: ceil(log2 n)."""
    s = 0
    while (1 << s) < n:
        s += 1
    return s


def column_stages(T, ell) -> int:
    """Expansion stages of the column ciphertext: its T * ell gadget values
    (ell per column bit) are coefficients 0 .. T ell - 1."""
    return coltor_stages(T * ell)


def coltor_algorithmic_bytes(n, L, N, ell) -> int:
    """Bytes a tournament must move at the least: every stage reads its input
    ciphertexts and its RGSW ciphertext and writes its outputs."""
    ct = 2 * L * N * 4
    total, cnt = 0, n
    while cnt > 1:
        nxt = (cnt + 1) // 2
        total += cnt * ct + 2 * ell * ct + nxt * ct
        cnt = nxt
    return total


def launches_per_step(cfg) -> int:
    """Kernels one step launches: per RowSel pass a query transpose, the scan
    and a result transpose; plus the query NTT and result INTT in coefficient
    form, or the lift + NTT of G for the ring-packing GEMM."""
    if cfg.get("kind") == "exppack":
        return 3 * rowsel_passes(cfg["n"], cfg["B"]) + 1
    if cfg.get("kind") == "coltor":
        return 4 * coltor_stages(cfg["n"])
    if cfg.get("kind") == "expand":
        return 4 * cfg["stages"]
    if cfg.get("kind") == "onion":
        # for all B clients: the batched row and column expansions, the batched
        # RGSW conversion, the RowSel passes and the batched tournament
        T = coltor_stages(cfg["D1"])
        return (4 * (cfg["D0"].bit_length() - 1) + 4 * column_stages(T, cfg["ell"]) + 4
                + 3 * rowsel_passes(cfg["D0"], cfg.get("B", 1)) + 4 * T)
    return 3 * rowsel_passes(cfg["D0"], cfg["B"]) + (2 if cfg["domain"] == "coeff" else 0)


def kernel_rooflines(coeff, q_bytes, o_bytes, ntt_fwd_ms, ntt_inv_ms, hbm_peak):
    """HBM fractions of the NTT kernels of the step (read + write of every residue)."""
    if not coeff:
        return None
    out = {}
    for name, nbytes, ms in (("ntt_fwd", 2 * q_bytes, ntt_fwd_ms), ("ntt_inv", 2 * o_bytes, ntt_inv_ms)):
        ach = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                     "algorithmic_bytes_per_launch": nbytes}
    return out


def run_scalar(args, cfg, emit=True):
    """Scalar-HE scan: one step = digit split of Q + the tensor-core scan."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    R, C, B = cfg["R"], cfg["C"], cfg["B"]
    ctx = pir.pir_ctx_create(4096, pir.pir_primes(4096, 1), local)
    db = torch.empty(R * C, dtype=torch.uint8, device="cuda")
    sd.fill_bytes(db, 7, synth.T_SCALAR_DB)
    Q = torch.empty(C * B, dtype=torch.int32, device="cuda")
    sd.fill_words(Q, 7, synth.T_SCALAR_Q)
    out = torch.empty(R * B, dtype=torch.int32, device="cuda")
    ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        pir.pir_scalar_scan(ctx, db, R, C, Q, B, out, ws, stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        pir.pir_scalar_scan(ctx, db, R, C, Q, B, out, ws, stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    ms = ms_total / args.steps
    if pir.pir_status(ctx):
        raise RuntimeError("device status word set")

    # end to end: the query matrix from pinned host memory, the results back
    q_host = torch.empty(Q.numel(), dtype=torch.int32, pin_memory=True)
    q_host.copy_(Q.cpu())
    o_host = [torch.empty(out.numel(), dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms = None
    if ke:
        # two scans in flight: query matrix i+1 in and results i-1 out during scan i
        Q2, out2 = [Q, torch.empty_like(Q)], [out, torch.empty_like(out)]
        e2e_ms = pipelined_ms(lambda k: Q2[k].copy_(q_host, non_blocking=True),
                              lambda k: pir.pir_scalar_scan(ctx, db, R, C, Q2[k], B, out2[k], ws, stream),
                              lambda k: o_host[k].copy_(out2[k], non_blocking=True), stream, ke)
    peaks, kind = measured_peaks()
    db_bytes = R * C
    if B <= 4:
        # CUDA-core GEMV: bound by the HBM read of the DB (+ Q and the output)
        algo = db_bytes + 4 * C * B + 4 * R * B
        gbs = algo / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": gbs / float(peaks["hbm_gbs"]), **profile_traffic("gemv_kernel_" + args.workload),
                "kernel": "gemv_kernel",
                "peak_source": "%s hbm_gbs (copy)" % kind, "algorithmic_bytes_per_launch": algo}
        dtype = "u8 x u32 (4-way byte dot products, u32 wrap-around)"
    else:
        flops = 2.0 * R * C * 4 * 64        # fp16 multiply-adds on 4 digit planes x 64 query slots
        tf = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": tf, "peak": float(peaks["bf16_tflops"]), "unit": "TFLOP/s",
                "frac": tf / float(peaks["bf16_tflops"]), **profile_traffic("scalar_kernel_" + args.workload),
                "kernel": "scalar_kernel",
                "peak_source": "%s bf16_tflops (fp16 dense rate is the same)" % kind,
                "hbm_frac": db_bytes / (ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"])}
        dtype = "u8 x u32 (fp16 digits, fp32 accumulate)"
    line = {
        "metric": "scalar-HE scan: DB GB/s scanned",
        "value": aggregate_throughput(db_bytes, args.steps, ms_total, world) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic: seeded SplitMix64 bytes U[0,256), words U[0,2^32)",
        "config": {"workload": args.workload, "desc": cfg["desc"], "R": R, "C": C, "B": B,
                   "l2": "inputs larger than L2 (DB %.1f GiB), no flush" % (db_bytes / GIB)},
        "queries_per_s": world * B * 1e3 / ms,
        "roofline": roof,
        "clocks": clk, "gpu_launches": 2 * args.steps, "cpu_baseline": None,
        "e2e": None if e2e_ms is None else {
            "value": db_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 4 * C * B,
            "d2h_bytes_per_step": 4 * R * B, "ms_per_step": e2e_ms,
            "how": "2 steps in flight: copy-in, compute and copy-out on three streams"},
    }
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_baseline(ScalarSample(cfg), args.cpu_seconds)
        if emit:
            print(json.dumps(line), flush=True)
    ctx.close()
    return line


def run_exppack(args, cfg):
    """Ring-packing GEMM: one step = lift + NTT of the scan output G, then
    H*C + (0|G) over the resident hint."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    N, L, n, Dr, B = cfg["N"], cfg["L"], cfg["n"], cfg["Dr"], cfg["B"]
    qs = pir.pir_primes(N, L)
    ctx = pir.pir_ctx_create(N, qs, local)
    P = L * N
    h_db = torch.empty(pir.pir_db_bytes(ctx, n, Dr) // 4, dtype=torch.int32, device="cuda")
    rows = max(1, min(n, (1 << 30) // (Dr * N * 4)))
    raw = torch.empty(rows * Dr * N, dtype=torch.int32, device="cuda")
    for k0 in range(0, n, rows):
        kc = min(rows, n - k0)
        sd.fill_words(raw[: kc * Dr * N], 7, synth.T_HINT, idx0=k0 * Dr * N)
        pir.pir_db_encode(ctx, raw[: kc * Dr * N], k0, kc, n, Dr, h_db)
    torch.cuda.synchronize()
    del raw
    graw = torch.empty(B * Dr * N, dtype=torch.int32, device="cuda")
    sd.fill_words(graw, 7, synth.T_SCAN_OUT)
    C = torch.empty(B * n * 2 * P, dtype=torch.int32, device="cuda")
    sd.fill_residues(C, 7, synth.T_SPECIAL, N, qs)
    G = torch.empty(B * Dr * P, dtype=torch.int32, device="cuda")
    out = torch.empty(B * Dr * 2 * P, dtype=torch.int32, device="cuda")
    ws = pir.rowsel_workspace(ctx, n, Dr, B)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        pir.pir_lift_ntt(ctx, graw, G, B * Dr, stream)
        if ev is not None:
            ev[1].record(stream)
        pir.pir_exppack(ctx, h_db, n, Dr, C, G, B, out, ws, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(kev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    lift_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in kev]))
    gemm_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in kev]))
    if pir.pir_status(ctx):
        raise RuntimeError("device status word set")

    hint_bytes = P * n * Dr * 4
    c_bytes, g_bytes, o_bytes, graw_bytes = B * n * 2 * P * 4, B * Dr * P * 4, B * Dr * 2 * P * 4, B * Dr * N * 4

    # end to end: C and the scan words from pinned host memory, the packed ciphertexts back
    c_host = torch.empty(C.numel(), dtype=torch.int32, pin_memory=True)
    c_host.copy_(C.cpu())
    g_host = torch.empty(graw.numel(), dtype=torch.int32, pin_memory=True)
    g_host.copy_(graw.cpu())
    o_host = [torch.empty(out.numel(), dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms = None
    if ke:
        # two steps in flight: C and the scan words of step i+1 in, the packed
        # ciphertexts of step i-1 out, while step i computes
        C2, g2, out2 = [C, torch.empty_like(C)], [graw, torch.empty_like(graw)], [out, torch.empty_like(out)]

        def copy_in(k):
            C2[k].copy_(c_host, non_blocking=True)
            g2[k].copy_(g_host, non_blocking=True)

        def compute(k):
            pir.pir_lift_ntt(ctx, g2[k], G, B * Dr, stream)
            pir.pir_exppack(ctx, h_db, n, Dr, C2[k], G, B, out2[k], ws, stream)

        e2e_ms = pipelined_ms(copy_in, compute, lambda k: o_host[k].copy_(out2[k], non_blocking=True), stream, ke)

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    algo = hint_bytes + c_bytes + g_bytes + o_bytes
    achieved = algo / (gemm_ms * 1e-3) / 1e9
    lift_bytes = graw_bytes + g_bytes
    result = None
    if rank == 0:
        line = {
            "metric": EXPPACK_METRIC, "value": aggregate_throughput(hint_bytes, args.steps, ms_total, world) / 1e9,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_total / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u32",
            "data": "synthetic: seeded SplitMix64 hint and scan words U[0,2^32), special-ct residues U[0,q_i)",
            "config": {"workload": args.workload, "desc": cfg["desc"], "hint_bytes": hint_bytes, "B": B,
                       "l2": "inputs larger than L2 (hint %.1f GiB), no flush" % (hint_bytes / GIB),
                       "parallelism": "replicas x%d" % world},
            "kernel_ms": {"lift_ntt": lift_ms, "exppack": gemm_ms},
            "kernels": {"lift_ntt": {"bound": "hbm", "unit": "GB/s", "peak": hbm_peak,
                                     "achieved": lift_bytes / (lift_ms * 1e-3) / 1e9,
                                     "frac": lift_bytes / (lift_ms * 1e-3) / 1e9 / hbm_peak,
                                     "algorithmic_bytes_per_launch": lift_bytes}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, **profile_traffic("rowsel_kernel_exppack_15g"),
                         "kernel": "rowsel_kernel (pir_exppack)", "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "algorithmic_bytes_per_launch": algo},
            "clocks": clk,
            "e2e": None if e2e_ms is None else {
                "value": hint_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": c_bytes + graw_bytes, "d2h_bytes_per_step": o_bytes, "ms_per_step": e2e_ms,
                "how": "2 steps in flight: copy-in, compute and copy-out on three streams"},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "cpu_baseline": None,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_baseline(ExppackSample(cfg), args.cpu_seconds)
        print(json.dumps(line), flush=True)
        result = line
    ctx.close()
    return result


def device_db(ctx, D0, D1, seed):
    """Seeded raw records generated on the device, encoded in row chunks."""
    import torch
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir
    N = ctx.N
    db = torch.empty(pir.pir_db_bytes(ctx, D0, D1) // 4, dtype=torch.int32, device="cuda")
    rows = max(1, min(D0, (1 << 30) // (D1 * N * 4)))
    raw = torch.empty(rows * D1 * N, dtype=torch.int32, device="cuda")
    for k0 in range(0, D0, rows):
        kc = min(rows, D0 - k0)
        r = raw[: kc * D1 * N]
        sd.fill_coeffs(r, seed, synth.T_DB_COEFF, idx0=k0 * D1 * N)
        pir.pir_db_encode(ctx, r, k0, kc, D0, D1, db)
    torch.cuda.synchronize()
    del raw
    return db


def ntt_rate(ctx, stream, polys=6830):
    """Rows per second of the library's 4096-point lift + forward NTT alone
    (polys x L rows, the size of a 1365-ciphertext ColTor's first digit batch)."""
    import torch
    from lattice_he_database_gb300 import pir
    N, L = ctx.N, len(ctx.qs)
    raw = torch.randint(0, 1 << 18, (polys * N,), dtype=torch.int32, device="cuda")
    out = torch.empty(polys * L * N, dtype=torch.int32, device="cuda")

    def run():
        pir.pir_lift_ntt(ctx, raw, out, polys, stream)

    run()
    ms = timed_ms(run, 10, stream)
    return polys * L / (ms * 1e-3)


def pipelined_ms(copy_in, compute, copy_out, stream, steps, warm=3):
    """Mean ms per step of a stream of steps with two in flight: step i's
    inputs are copied in on their own stream and step i-2's results copied
    out on another while `stream` computes step i-1; slot k = i % 2 holds one
    step's device buffers.  copy_in(k) and copy_out(k) enqueue on the current
    stream, compute(k) runs with `stream` current.  The timed region runs
    from the first copy-in to the last copy-out."""
    import torch
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    q_free, in_done, comp_done, out_free = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(4))

    def serve(n, t0):
        for i in range(t0, t0 + n):
            k = i % 2
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(q_free[k])
                copy_in(k)
                in_done[k].record(h2d)
            stream.wait_event(in_done[k])
            if i >= 2:
                stream.wait_event(out_free[k])
            with torch.cuda.stream(stream):
                compute(k)
            q_free[k].record(stream)
            comp_done[k].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(comp_done[k])
                copy_out(k)
                out_free[k].record(d2h)

    serve(warm, 0)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d)
    serve(steps, warm)
    e1.record(d2h)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def graph_of(step, stream):
    """A CUDA graph of one step (the library's launches on `stream`), for
    fixed-shape pipelines whose small stages are bound by launch latency."""
    import torch
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()
    return g


def timed_ms(fn, steps, stream):
    """Mean ms of `steps` calls of fn on `stream` (CUDA events)."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_coltor(args, cfg):
    """ColTor: one step = the whole tournament over n RowSel output
    ciphertexts (NTT form), S = ceil(log2 n) stages of four launches."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    N, L, n, ell, w = cfg["N"], cfg["L"], cfg["n"], cfg["ell"], cfg["w"]
    qs = pir.pir_primes(N, L)
    ctx = pir.pir_ctx_create(N, qs, local)
    P = L * N
    S = coltor_stages(n)
    cts = torch.empty(n * 2 * P, dtype=torch.int32, device="cuda")
    sd.fill_residues(cts, 7, synth.T_EXTRA, N, qs)
    Cs = torch.empty(max(S, 1) * 2 * ell * 2 * P, dtype=torch.int32, device="cuda")
    sd.fill_residues(Cs, 8, synth.T_EXTRA, N, qs)
    out = torch.empty(2 * P, dtype=torch.int32, device="cuda")
    ws = pir.coltor_workspace(ctx, n, ell)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step():
        pir.pir_coltor(ctx, Cs, ell, w, cts, n, out, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    eager_ms = timed_ms(step, args.steps, stream)      # one launch sequence per call, for comparison
    graph = graph_of(step, stream)

    def run():
        with torch.cuda.stream(stream):      # replay on the stream the events are recorded on
            graph.replay()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        run()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    if pir.pir_status(ctx):
        raise RuntimeError("device status word set")

    ct_bytes = n * 2 * P * 4
    o_bytes = 2 * P * 4
    cts_host = torch.empty(cts.numel(), dtype=torch.int32, pin_memory=True)
    cts_host.copy_(cts.cpu())
    o_host = [torch.empty(out.numel(), dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms = None
    if ke:
        # two tournaments in flight, each slot with its own buffers and graph
        cts2, out2 = [cts, torch.empty_like(cts)], [out, torch.empty_like(out)]
        graphs = [graph, graph_of(lambda: pir.pir_coltor(ctx, Cs, ell, w, cts2[1], n, out2[1], ws, stream), stream)]
        e2e_ms = pipelined_ms(lambda k: cts2[k].copy_(cts_host, non_blocking=True),
                              lambda k: graphs[k].replay(),
                              lambda k: o_host[k].copy_(out2[k], non_blocking=True), stream, ke)

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    ms_step = ms_total / args.steps
    ntt_alone = ntt_rate(ctx, stream)
    algo = coltor_algorithmic_bytes(n, L, N, ell)
    achieved = algo / (ms_step * 1e-3) / 1e9
    nntt = 0
    cnt = n
    while cnt > 1:
        pairs = (cnt + 1) // 2
        nntt += pairs * (2 * L + 2 * ell * L)
        cnt = pairs
    result = None
    if rank == 0:
        line = {
            "metric": COLTOR_METRIC, "value": world * args.steps / (ms_total * 1e-3), "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic: seeded SplitMix64 residues U[0,q_i) for the ciphertexts and RGSW rows",
            "config": {"workload": args.workload, "desc": cfg["desc"], "n": n, "stages": S, "ell": ell, "w": w,
                       "l2": "the first stage's digit NTTs (%.0f MB) exceed L2; no flush"
                             % (((n + 1) // 2) * 2 * ell * P * 4 / 1e6),
                       "parallelism": "replicas x%d" % world},
            "external_products_per_s": world * args.steps * (n - 1) / (ms_total * 1e-3),
            "launch": "one CUDA graph per tournament (the call's %d launches captured once, replayed)"
                      % launches_per_step(cfg),
            "eager_ms_per_step": eager_ms,
            "ntt_per_step": nntt, "ntt_per_s": nntt / (ms_step * 1e-3),
            "ntt": {"rows_per_s_in_step": nntt / (ms_step * 1e-3), "rows_per_s_standalone": ntt_alone,
                    "frac": nntt / (ms_step * 1e-3) / ntt_alone,
                    "note": "the step's transforms against the 4096-point lift + NTT kernel timed alone in this run"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, **profile_traffic("coltor_%s" % args.workload),
                         "kernel": "the tournament's five kernels per stage (NTT kernels dominate)",
                         "peak_source": "%s hbm_gbs (copy)" % peak_kind, "algorithmic_bytes_per_launch": algo},
            "clocks": clk,
            "e2e": None if e2e_ms is None else {
                "value": 1e3 / e2e_ms, "unit": "queries/s", "h2d_bytes_per_step": ct_bytes,
                "d2h_bytes_per_step": o_bytes, "ms_per_step": e2e_ms,
                "how": "2 steps in flight: copy-in, compute and copy-out on three streams"},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "cpu_baseline": None,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_baseline(ColtorSample(cfg), args.cpu_seconds)
        print(json.dumps(line), flush=True)
        result = line
    ctx.close()
    return result


def run_expand(args, cfg):
    """ExpandQuery: one step = the whole expansion of one query ciphertext
    (NTT form) into 2^stages ciphertexts, four launches per stage."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    N, L, S, ell, w = cfg["N"], cfg["L"], cfg["stages"], cfg["ell"], cfg["w"]
    qs = pir.pir_primes(N, L)
    ctx = pir.pir_ctx_create(N, qs, local)
    P = L * N
    ct = torch.empty(2 * P, dtype=torch.int32, device="cuda")
    sd.fill_residues(ct, 9, synth.T_EXTRA, N, qs)
    evks = torch.empty(S * ell * 2 * P, dtype=torch.int32, device="cuda")
    sd.fill_residues(evks, 10, synth.T_EXTRA, N, qs)
    out = torch.empty((1 << S) * 2 * P, dtype=torch.int32, device="cuda")
    ws = pir.expand_workspace(ctx, 1 << (S - 1), ell)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step():
        pir.pir_expand(ctx, evks, ell, w, S, ct, out, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    eager_ms = timed_ms(step, args.steps, stream)      # one launch sequence per call, for comparison
    graph = graph_of(step, stream)

    def run():
        with torch.cuda.stream(stream):      # replay on the stream the events are recorded on
            graph.replay()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        run()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    if pir.pir_status(ctx):
        raise RuntimeError("device status word set")

    ct_bytes = 2 * P * 4
    o_bytes = (1 << S) * 2 * P * 4
    ct_host = torch.empty(ct.numel(), dtype=torch.int32, pin_memory=True)
    ct_host.copy_(ct.cpu())
    o_host = [torch.empty(out.numel(), dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms = None
    if ke:
        # two expansions in flight, each slot with its own buffers and graph
        ct2, out2 = [ct, torch.empty_like(ct)], [out, torch.empty_like(out)]
        graphs = [graph, graph_of(lambda: pir.pir_expand(ctx, evks, ell, w, S, ct2[1], out2[1], ws, stream), stream)]
        e2e_ms = pipelined_ms(lambda k: ct2[k].copy_(ct_host, non_blocking=True),
                              lambda k: graphs[k].replay(),
                              lambda k: o_host[k].copy_(out2[k], non_blocking=True), stream, ke)

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    ms_step = ms_total / args.steps
    ntt_alone = ntt_rate(ctx, stream)
    # at the least every stage reads its inputs and key and writes its outputs
    algo = sum(((1 << j) * 3 + ell) * 2 * P * 4 for j in range(S))
    achieved = algo / (ms_step * 1e-3) / 1e9
    nsubs = (1 << S) - 1
    nntt = nsubs * (L + ell * L)
    result = None
    if rank == 0:
        line = {
            "metric": EXPAND_METRIC, "value": world * args.steps / (ms_total * 1e-3), "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic: seeded SplitMix64 residues U[0,q_i) for the query ciphertext and keys",
            "config": {"workload": args.workload, "desc": cfg["desc"], "stages": S, "outputs": 1 << S,
                       "ell": ell, "w": w,
                       "l2": "outputs %.0f MB exceed L2; no flush" % (o_bytes / 1e6),
                       "parallelism": "replicas x%d" % world},
            "subs_per_s": world * args.steps * nsubs / (ms_total * 1e-3),
            "launch": "one CUDA graph per expansion (the call's %d launches captured once, replayed)"
                      % launches_per_step(cfg),
            "eager_ms_per_step": eager_ms,
            "ntt_per_step": nntt, "ntt_per_s": nntt / (ms_step * 1e-3),
            "ntt": {"rows_per_s_in_step": nntt / (ms_step * 1e-3), "rows_per_s_standalone": ntt_alone,
                    "frac": nntt / (ms_step * 1e-3) / ntt_alone,
                    "note": "the step's transforms against the 4096-point lift + NTT kernel timed alone in this run"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, **profile_traffic("expand_%s" % args.workload),
                         "kernel": "the expansion's four kernels per stage (NTT kernels dominate)",
                         "peak_source": "%s hbm_gbs (copy)" % peak_kind, "algorithmic_bytes_per_launch": algo},
            "clocks": clk,
            "e2e": None if e2e_ms is None else {
                "value": 1e3 / e2e_ms, "unit": "queries/s", "h2d_bytes_per_step": ct_bytes,
                "d2h_bytes_per_step": o_bytes, "ms_per_step": e2e_ms,
                "how": "2 steps in flight: copy-in, compute and copy-out on three streams"},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "cpu_baseline": None,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_baseline(ExpandSample(cfg), args.cpu_seconds)
        print(json.dumps(line), flush=True)
        result = line
    ctx.close()
    return result


def run_onion(args, cfg):
    """The OnionPIR server path for B queries (B clients, each with its own
    keys): the B expansions of the row query ciphertext into D0 = 1024 and of
    the column query ciphertext into 64 (its first T ell = 55 outputs are the
    gadget ciphertexts of the T = 11 column bits), the conversion of those
    into T RGSW ciphertexts per client, one RowSel pass of the B queries over
    the resident 64 GiB DB, and the B tournaments of the D1 = 1365 results
    into one answer ciphertext each; every phase one (batched) call, all NTT
    form."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    N, L, D0, D1, ell, w = cfg["N"], cfg["L"], cfg["D0"], cfg["D1"], cfg["ell"], cfg["w"]
    B = cfg.get("B", 1)
    S, T = D0.bit_length() - 1, coltor_stages(D1)
    Sc = column_stages(T, ell)
    Mc = 1 << Sc
    qs = pir.pir_primes(N, L)
    ctx = pir.pir_ctx_create(N, qs, local)
    P = L * N
    qw = 2 * P                                           # words of a ciphertext
    db = device_db(ctx, D0, D1, seed=7)
    # per client and query: a row and a column query ciphertext; resident per
    # client (sent once): the expansion keys of S stages (the column
    # expansion takes the first Sc of them, stored again so that a batched
    # call finds client b's at b * Sc keys) and the key-switching key of s^2.
    # Two slots of per-query buffers so that two steps can be in flight.
    query = [torch.empty(B * qw, dtype=torch.int32, device="cuda") for _ in range(2)]
    colq = [torch.empty(B * qw, dtype=torch.int32, device="cuda") for _ in range(2)]
    sd.fill_residues(query[0], 11, synth.T_EXTRA, N, qs)
    sd.fill_residues(colq[0], 14, synth.T_EXTRA, N, qs)
    query[1].copy_(query[0])
    colq[1].copy_(colq[0])
    evks = torch.empty(B * S * ell * qw, dtype=torch.int32, device="cuda")
    sd.fill_residues(evks, 12, synth.T_EXTRA, N, qs)
    evks_c = evks.view(B, S * ell * qw)[:, : Sc * ell * qw].contiguous().view(-1)
    ksk = torch.empty(B * ell * qw, dtype=torch.int32, device="cuda")
    sd.fill_residues(ksk, 13, synth.T_EXTRA, N, qs)
    expanded = torch.empty(B * D0 * qw, dtype=torch.int32, device="cuda")
    col_exp = torch.empty(B * Mc * qw, dtype=torch.int32, device="cuda")
    rgsw = torch.empty(B * T * 2 * ell * qw, dtype=torch.int32, device="cuda")
    cols = torch.empty(B * D1 * qw, dtype=torch.int32, device="cuda")
    answer = [torch.empty(B * qw, dtype=torch.int32, device="cuda") for _ in range(2)]
    ws_e = pir.expand_workspace(ctx, B * D0 // 2, ell)
    ws_ec = pir.expand_workspace(ctx, B * Mc // 2, ell)
    ws_g = pir.rgsw_convert_workspace(ctx, T, B, ell)
    ws_r = pir.rowsel_workspace(ctx, D0, D1, B)
    ws_c = pir.coltor_batch_workspace(ctx, D1, B, ell)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def expand(k):
        pir.pir_expand_batch(ctx, evks, ell, w, S, query[k], B, expanded, ws_e, stream)

    def column(k):
        pir.pir_expand_batch(ctx, evks_c, ell, w, Sc, colq[k], B, col_exp, ws_ec, stream)
        pir.pir_rgsw_convert(ctx, ksk, ell, w, col_exp, T, B, rgsw, ws_g, stream, in_stride=Mc)

    def rowsel():
        pir.pir_rowsel(ctx, db, D0, D1, expanded, B, cols, ws_r, stream)

    def coltor(k):
        pir.pir_coltor_batch(ctx, rgsw, ell, w, cols, D1, B, answer[k], ws_c, stream)

    for _ in range(2):                        # first calls (kernel attributes, caches) outside the graphs
        expand(0)
        column(0)
        rowsel()
        coltor(0)
    g_expand = [graph_of(lambda: expand(0), stream), graph_of(lambda: expand(1), stream)]
    g_column = [graph_of(lambda: column(0), stream), graph_of(lambda: column(1), stream)]
    g_coltor = [graph_of(lambda: coltor(0), stream), graph_of(lambda: coltor(1), stream)]

    def step(ev=None, k=0):
        with torch.cuda.stream(stream):
            if ev is not None:
                ev[0].record(stream)
            g_expand[k].replay()              # the small expansion stages are bound by launch latency
            if ev is not None:
                ev[1].record(stream)
            g_column[k].replay()
            if ev is not None:
                ev[2].record(stream)
            rowsel()
            if ev is not None:
                ev[3].record(stream)
            g_coltor[k].replay()
            if ev is not None:
                ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(kev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    phase = [float(np.mean([e[k].elapsed_time(e[k + 1]) for e in kev])) for k in range(4)]
    if pir.pir_status(ctx):
        raise RuntimeError("device status word set")

    # end to end: every step's row and column query ciphertexts in from
    # pinned host memory, the answers out; two steps in flight
    q_host = torch.empty(query[0].numel(), dtype=torch.int32, pin_memory=True)
    q_host.copy_(query[0].cpu())
    c_host = torch.empty(colq[0].numel(), dtype=torch.int32, pin_memory=True)
    c_host.copy_(colq[0].cpu())
    a_host = [torch.empty(answer[0].numel(), dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms = None
    if ke:
        def copy_in(k):
            query[k].copy_(q_host, non_blocking=True)
            colq[k].copy_(c_host, non_blocking=True)

        e2e_ms = pipelined_ms(copy_in, lambda k: step(None, k),
                              lambda k: a_host[k].copy_(answer[k], non_blocking=True), stream, ke)

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    logical_db = P * D0 * D1 * 4
    ms_step = ms_total / args.steps
    db_gbs = logical_db / (phase[2] * 1e-3) / 1e9
    on_tensor = 8 < B <= 16
    result = None
    if rank == 0:
        line = {
            "metric": ONION_METRIC, "value": world * B * args.steps / (ms_total * 1e-3), "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic: seeded SplitMix64 DB coefficients U[0,2^16), query and key residues U[0,q_i)",
            "config": {"workload": args.workload, "desc": cfg["desc"], "logical_db_bytes": logical_db, "B": B,
                       "l2": "inputs larger than L2 (DB %.1f GiB), no flush" % (logical_db / GIB),
                       "parallelism": "replicas x%d" % world},
            "phase_ms": {"expand": phase[0], "column_expand_and_rgsw": phase[1], "rowsel": phase[2],
                         "coltor": phase[3]},
            "launch": "the batched row expansion, column expansion + RGSW conversion and ColTor calls each "
                      "replayed as one CUDA graph; RowSel launched directly",
            "db_gbs_in_rowsel": db_gbs,
            "roofline": {"bound": "hbm", "achieved": db_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": db_gbs / hbm_peak, "traffic": None, "traffic_source": None,
                         "kernel": "rowsel_tc_kernel (the DB scan, %d queries per pass)" % B if on_tensor
                                   else "rowsel_kernel (the DB scan)",
                         "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "algorithmic_bytes_per_launch": logical_db},
            "clocks": clk,
            "e2e": None if e2e_ms is None else {
                "value": B * 1e3 / e2e_ms, "unit": "queries/s", "h2d_bytes_per_step": B * 2 * qw * 4,
                "d2h_bytes_per_step": B * qw * 4, "ms_per_step": e2e_ms,
                "how": "row and column query ciphertexts in, answers out; expansion and key-switching keys "
                       "resident; 2 steps in flight on three streams"},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "cpu_baseline": None,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = oracle_baseline(OnionSample(cfg), args.cpu_seconds)
        print(json.dumps(line), flush=True)
        result = line
    ctx.close()
    return result


def run_ours(args, cfg, emit=True):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import synth
    import synth.device as sd
    from lattice_he_database_gb300 import pir

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")

    N, L, D0, D1, B = cfg["N"], cfg["L"], cfg["D0"], cfg["D1"], cfg["B"]
    qs = pir.pir_primes(N, L)
    ctx = pir.pir_ctx_create(N, qs, local)
    P = L * N
    db = device_db(ctx, D0, D1, seed=7)
    stream = torch.cuda.Stream()
    srv = pir.RowselServer(ctx, db, D0, D1, B, stream=stream)
    sd.fill_residues(srv.q_coef, 7, synth.T_QUERY, N, qs)
    torch.cuda.synchronize()

    logical_db = P * D0 * D1 * 4
    q_bytes = B * D0 * 2 * P * 4
    o_bytes = B * D1 * 2 * P * 4
    coeff = cfg["domain"] == "coeff"

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if coeff:
            pir.pir_ntt_fwd(ctx, srv.q_coef, srv.q_ntt, B * D0 * 2, stream)
        if ev is not None:
            ev[1].record(stream)
        pir.pir_rowsel(ctx, db, D0, D1, srv.q_ntt if coeff else srv.q_coef, B, srv.o_ntt, srv.ws, stream)
        if ev is not None:
            ev[2].record(stream)
        if coeff:
            pir.pir_ntt_inv(ctx, srv.o_ntt, srv.o_coef, B * D1 * 2, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0.record(stream)
    for i in range(args.steps):
        step(kev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ntt_fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in kev]))
    rowsel_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in kev]))
    ntt_inv_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in kev]))
    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps
    status = pir.pir_status(ctx)
    if status:
        raise RuntimeError("device status word set: %d" % status)

    # in-run read-only stream over the encoded DB (the ceiling of a pure read)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd.read_probe(db, sink, stream)
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(3):
        sd.read_probe(db, sink, stream)
    r1.record(stream)
    torch.cuda.synchronize()
    read_probe_gbs = 3 * db.numel() * 4 / (r0.elapsed_time(r1) * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host query in, result out.
    # Coefficient-form workloads use the pipelined query server (copies of
    # the neighbouring queries overlap each scan); NTT-form ones the plain
    # sequence copy-in -> RowSel -> copy-out on one stream.
    q_host = torch.empty(srv.q_words, dtype=torch.int32, pin_memory=True)
    q_host.copy_(srv.q_coef.cpu())
    o_host = [torch.empty(srv.o_words, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    ke = 0 if args.no_e2e else max(1, min(args.e2e_steps, args.steps))
    e2e_ms, e2e_how = None, None
    if ke and coeff:
        server = pir.PirServer(ctx, db, D0, D1, B)

        def serve(n, t0):
            for i in range(t0, t0 + n):
                if i >= 2:
                    server.wait(i - 2)          # its result buffer is reused now
                server.submit(q_host, o_host[i % 2])
            server.wait(t0 + n - 1)

        serve(3, 0)                              # warm-up
        torch.cuda.synchronize()
        server.mark(0)
        serve(ke, 3)
        server.mark(1)
        e2e_ms = server.elapsed_ms() / ke
        e2e_how = "pir_server: 2 queries in flight, copies on their own streams"
        server.close()
    elif ke:
        # two slots: query i+1 is copied in and result i-1 copied out (own
        # streams, the copy engines) while RowSel scans query i
        q_dev = [srv.q_coef, torch.empty_like(srv.q_coef)]
        o_dev = [srv.o_ntt, torch.empty_like(srv.o_ntt)]
        e2e_ms = pipelined_ms(lambda k: q_dev[k].copy_(q_host, non_blocking=True),
                              lambda k: pir.pir_rowsel(ctx, db, D0, D1, q_dev[k], B, o_dev[k], srv.ws, stream),
                              lambda k: o_host[k].copy_(o_dev[k], non_blocking=True), stream, ke)
        e2e_how = "2 queries in flight: copy-in, RowSel and copy-out on three streams"

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    algo_bytes = logical_db + q_bytes + o_bytes       # the RowSel kernel's algorithmic bytes per launch
    achieved = algo_bytes / (rowsel_ms * 1e-3) / 1e9
    # passes of 9..16 queries run on the tensor cores (primes >= 2^26 here)
    on_tensor = 8 < B <= 16
    kernel = "rowsel_tc_kernel" if on_tensor else "rowsel_kernel"
    tensor = None
    if on_tensor:
        # 16 digit-plane products per multiply-add, fp16 inputs, 2 flops each
        flops = 2.0 * 16 * (2 * B) * D0 * D1 * P
        tf = flops / (rowsel_ms * 1e-3) / 1e12
        tensor = {"achieved": tf, "peak": float(peaks["bf16_tflops"]), "unit": "TFLOP/s",
                  "frac": tf / float(peaks["bf16_tflops"]), "algorithmic_flops_per_launch": flops}

    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = oracle_baseline(RowselSample(cfg), args.cpu_seconds)
        value = aggregate_throughput(logical_db, args.steps, ms_total, world) / 1e9
        result = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32",
            "data": "synthetic: seeded SplitMix64 DB coefficients U[0,2^16), query residues U[0,q_i)",
            "config": {"workload": args.workload, "desc": cfg["desc"], "logical_db_bytes": logical_db,
                       "encoded_db_bytes": pir.pir_db_bytes(ctx, D0, D1), "B": B,
                       "l2": "inputs larger than L2 (DB %.1f GiB >> 129 MB L2), no flush" % (logical_db / GIB),
                       "parallelism": "replicas x%d" % world},
            "queries_per_s": world * B * args.steps / (ms_total * 1e-3),
            "kernel_ms": {"ntt_fwd": ntt_fwd_ms, "rowsel": rowsel_ms, "ntt_inv": ntt_inv_ms},
            "kernels": kernel_rooflines(coeff, q_bytes, o_bytes, ntt_fwd_ms, ntt_inv_ms, hbm_peak),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, **profile_traffic("%s_%s" % (kernel, args.workload)),
                         "kernel": kernel, "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "algorithmic_bytes_per_launch": algo_bytes, "tensor": tensor,
                         "read_probe_gbs": read_probe_gbs, "frac_of_read_probe": achieved / read_probe_gbs,
                         "spec_gbs": SPEC_HBM_GBS, "frac_of_spec": achieved / SPEC_HBM_GBS},
            "clocks": clk,
            "e2e": None if e2e_ms is None else {
                "value": logical_db / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": q_bytes,
                "d2h_bytes_per_step": o_bytes, "ms_per_step": e2e_ms, "how": e2e_how},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "cpu_baseline": cpu,
        }
        if emit:
            print(json.dumps(result), flush=True)
    ctx.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


# The other benchmark configurations, timed briefly after the headline one in
# the default run (one GPU), so that their numbers come from the same run:
# the tiny RowSel, the 6 GiB single query, the 24 GiB 16-query batch on the
# tensor cores and the 16 GiB x 64 scalar scan.
OTHER_CONFIGS = ["tiny", "rowsel_6g", "rowsel_24g_b16", "scalar_16g"]
WORKLOADS["tiny"] = dict(N=4096, L=2, D0=16, D1=16, B=1, domain="ntt",
                         desc="Tiny RowSel: N=4096, 2 primes, D0=16 x D1=16, B=1, NTT-domain query (L2-resident)")


def other_configs(args):
    """Short timings (20 steps, CUDA events) of OTHER_CONFIGS."""
    out = {}
    for name in OTHER_CONFIGS:
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup = name, 20, 3
        sub.no_cpu_baseline, sub.no_e2e = True, True
        cfg = WORKLOADS[name]
        line = (run_scalar if cfg.get("kind") == "scalar" else run_ours)(sub, cfg, emit=False)
        if line is None:
            continue
        r = line["roofline"]
        entry = {"desc": cfg["desc"], "value": line["value"], "unit": line["unit"], "ms_per_step": line["ms_per_step"],
                 "steps": 20, "kernel": r.get("kernel"), "bound": r["bound"], "roofline_frac": r["frac"],
                 "roofline_unit": r["unit"], "achieved": r["achieved"], "peak": r["peak"],
                 "clocks": line.get("clocks")}
        if r.get("hbm_frac") is not None:
            entry["hbm_frac"] = r["hbm_frac"]
        if r.get("tensor"):
            entry["tensor_frac"] = r["tensor"]["frac"]
        if "queries_per_s" in line:
            entry["queries_per_s"] = line["queries_per_s"]
        out[name] = entry
    return out


def main():
    args = parse()
    cfg = WORKLOADS[args.workload]
    if (args.impl == "ours" and args.workload == "rowsel_64g" and not args.no_configs
            and int(os.environ.get("WORLD_SIZE", "1")) == 1):
        line = run_ours(args, cfg, emit=False)
        if line is not None:
            line["other_configs"] = other_configs(args)
            print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, cfg)
    elif cfg.get("kind") == "scalar":
        run_scalar(args, cfg)
    elif cfg.get("kind") == "exppack":
        run_exppack(args, cfg)
    elif cfg.get("kind") == "coltor":
        run_coltor(args, cfg)
    elif cfg.get("kind") == "expand":
        run_expand(args, cfg)
    elif cfg.get("kind") == "onion":
        run_onion(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
