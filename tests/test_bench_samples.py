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
