"""The bench's CPU-baseline samples stay bounded whatever the host's core
count, and each one runs the oracle.

The samples used to be sized by a time calibration alone; on a host with
many cores that grew the 64 GiB workload's sample to its whole 1365-column
slice (~22 GB of residues plus temporaries) and the host ran out of memory.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


@pytest.mark.parametrize("threads", [8, 72, 288])
@pytest.mark.parametrize("workload", ["rowsel_64g", "rowsel_24g_b16", "exppack_15g"])
def test_sample_words_bounded(monkeypatch, workload, threads):
    monkeypatch.setattr(oracle, "default_threads", lambda: threads)
    cfg = bench.WORKLOADS[workload]
    if cfg.get("kind") == "exppack":
        rows = min(cfg["Dr"], threads)
        pts = bench.sample_points(cfg["n"] * rows)
        words = rows * cfg["n"] * pts
    else:
        ncols = min(cfg["D1"], threads)
        pts = bench.sample_points(cfg["D0"] * ncols)
        words = cfg["D0"] * ncols * pts
    assert pts % 16 == 0 and 16 <= pts <= 4096
    assert words <= max(bench.SAMPLE_WORDS, 16 * (cfg.get("D0") or cfg["n"]) * threads)


def test_samples_run_on_small_shapes(monkeypatch):
    monkeypatch.setattr(oracle, "default_threads", lambda: 2)
    rs = bench.RowselSample(dict(N=4096, L=3, D0=8, D1=5, B=2))
    rs()
    assert rs.nbytes == 8 * 2 * rs.pts * 4 and "2 of 5 DB columns" in rs.desc
    ex = bench.ExppackSample(dict(N=4096, L=3, n=6, Dr=3, B=1))
    ex()
    assert ex.nbytes == 2 * 6 * ex.pts * 4
    sc = bench.ScalarSample(dict(R=100, C=256, B=3))
    sc()
    assert sc.nbytes == 2 * 256
    line = bench.oracle_baseline(sc, 0.05)
    assert line["kind"] == "oracle" and line["cores"] == 2 and line["value"] > 0
    ct = bench.ColtorSample(dict(N=16, L=3, n=11, ell=5, w=18))
    ct()
    assert ct.pairs == 2 and abs(ct.nbytes - 2 / 10) < 1e-12
    line = bench.oracle_baseline(ct, 0.05)
    assert line["unit"] == "queries/s" and line["value"] > 0


@pytest.mark.parametrize("threads", [8, 72, 288])
def test_coltor_sample_bounded(monkeypatch, threads):
    monkeypatch.setattr(oracle, "default_threads", lambda: threads)
    cfg = bench.WORKLOADS["coltor_1365"]
    pairs = max(1, min((cfg["n"] + 1) // 2, threads))
    assert pairs <= 288 and 2 * pairs * 2 * cfg["L"] * cfg["N"] * 4 < 300 * 1024 * 1024


def test_launch_counts_of_the_workloads():
    """The bench's gpu_launches claim per step, counted by hand from the
    library's call structure: a RowSel pass is three launches (query
    transpose, scan, result transpose), a coefficient-form query adds its NTT
    and the result INTT, an expansion or tournament stage is four launches
    (INTT, decomposition, lift + NTT, MAC), the RGSW conversion is four more
    (INTT, decomposition, lift + NTT, MAC), ring packing adds the lift + NTT
    of G.  Batched expansions, conversions and tournaments launch per stage,
    not per client.  OnionPIR: the row expansion (10 stages), the column
    expansion (6 stages: 11 bits x 5 gadget values = 55 <= 64 outputs), the
    conversion, the RowSel pass and the tournament (11 stages)."""
    import bench
    W = bench.WORKLOADS
    assert bench.launches_per_step(W["rowsel_64g"]) == 3 + 2
    assert bench.launches_per_step(W["rowsel_24g_b16"]) == 3            # one pass of 16 on the tensor cores
    assert bench.launches_per_step(W["expand_1024"]) == 4 * 10
    assert bench.launches_per_step(W["coltor_1365"]) == 4 * 11
    assert bench.column_stages(11, 5) == 6
    assert bench.launches_per_step(W["onion_64g"]) == 4 * 10 + 4 * 6 + 4 + 3 + 4 * 11
    assert bench.launches_per_step(W["onion_64g_b16"]) == 4 * 10 + 4 * 6 + 4 + 3 + 4 * 11
    assert bench.launches_per_step(W["exppack_15g"]) == 3 + 1
    # pass planning: 16 per pass on the tensor cores while more than 8 remain,
    # then the CUDA cores (16 queries fit the on-chip slice for D0 <= 896)
    assert bench.rowsel_passes(1024, 16) == 1
    assert bench.rowsel_passes(1024, 17) == 2
    assert bench.rowsel_passes(600, 40) == 3          # 16 + 16 + 8
    assert bench.rowsel_passes(512, 8) == 1           # CUDA cores, 8 of 16
    assert bench.rowsel_passes(4096, 8) == 4          # D0 = 4096: 4 polynomials (2 queries) per CUDA-core pass


def test_onion_sample_composes_the_phases(monkeypatch):
    """The composed OnionPIR sample: each phase covers the fraction of a
    query its sample performs (expansions, conversions and tournaments per
    call, the scanned fraction of the DB times B), and a query costs the sum
    of each phase's time per call over its queries per call."""
    monkeypatch.setattr(oracle, "default_threads", lambda: 2)
    N, L, D0, D1, B = 64, 3, 16, 11, 2
    on = bench.OnionSample(dict(N=N, L=L, D0=D0, D1=D1, ell=5, w=18, B=B))
    e, ec, g, r, c = on.phases
    assert abs(on.per_call[0] - 2 / 15) < 1e-12                # 2 of the 15 Subs of a 16-way expansion
    assert abs(on.per_call[1] - 2 / 31) < 1e-12                # column: 4 bits x 5 values -> 32 outputs, 31 Subs
    assert abs(on.per_call[2] - 1 / 4) < 1e-12                 # one of the 4 bits' conversions
    assert abs(on.per_call[3] - r.nbytes / (D0 * D1 * L * N * 4) * B) < 1e-12
    assert abs(on.per_call[4] - 2 / 10) < 1e-12                # 2 of the 10 external products
    on()
    on()
    assert on.calls == 2 and all(t > 0 for t in on.spent)
    want = 1.0 / sum(t / 2 / q for t, q in zip(on.spent, on.per_call))
    assert abs(on.queries_per_s() - want) < 1e-9 * want
    line = bench.oracle_baseline(on, 0.05)
    assert line["unit"] == "queries/s" and line["value"] > 0 and line["cores"] == 2
