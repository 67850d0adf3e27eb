"""Repeated launches: every pipelined kernel gives the same result and a clean
status word launch after launch.

The kernels' producer/consumer rings use mbarrier parity waits, which are
only sound while no party can run two phases ahead on a slot; a rare slip
shows up as a bounded wait that gives up (PIR_STATUS_TIMEOUT) or as a result
that changes between launches.  Medium sizes, many launches each: the
tensor-core RowSel (16 queries), the CUDA-core RowSel with row-split partial
sums (one query), and the scalar scan on the tensor cores (64 queries).
The first result of each is also checked against the oracle on a few
columns or rows.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev, to_host_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


@pytest.mark.parametrize("D0,D1,B,launches", [
    (512, 64, 16, 40),     # tensor cores: 8192 points, 2 tiles per slab
    (1100, 40, 16, 20),    # tensor cores, three K segments per point
    (256, 72, 1, 60),      # CUDA cores, ksplit = 8 partial sums per output
])
def test_rowsel_repeated(pir, D0, D1, B, launches):
    import torch
    N, L = 4096, 2
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(41, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    query = synth.residues(42, (B, D0, 2, L, N), qs)
    q_t = to_dev(query)
    ws = pir.rowsel_workspace(ctx, D0, D1, B)
    first = pir.empty_u32(B * D1 * 2 * L * N)
    pir.pir_rowsel(ctx, db, D0, D1, q_t, B, first, ws)
    out = torch.empty_like(first)
    for _ in range(launches):
        out.fill_(-1)
        pir.pir_rowsel(ctx, db, D0, D1, q_t, B, out, ws)
        assert torch.equal(out, first)
    assert pir.pir_status(ctx) == 0
    cols = np.array([0, D1 // 2, D1 - 1])
    enc = oracle.encode_records(raw[:, cols], qs, psis)
    want = oracle.rowsel(enc, query, qs)
    got = to_host_u32(first).reshape(B, D1, 2, L, N)[:, cols]
    assert np.array_equal(got, want)


def test_scalar_repeated(pir):
    import torch
    R, C, B, launches = 4096, 16384, 64, 80
    ctx = pir.pir_ctx_create(4096, pir.pir_primes(4096, 1))
    dbh = synth.db_bytes(43, (R, C))
    Qh = synth.words(43, (C, B))
    db, Q = to_dev(dbh), to_dev(Qh)
    ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
    first = pir.empty_u32(R * B)
    pir.pir_scalar_scan(ctx, db, R, C, Q, B, first, ws)
    out = torch.empty_like(first)
    for _ in range(launches):
        out.fill_(-1)
        pir.pir_scalar_scan(ctx, db, R, C, Q, B, out, ws)
        assert torch.equal(out, first)
    assert pir.pir_status(ctx) == 0
    rows = np.array([0, 1777, R - 1])
    assert np.array_equal(to_host_u32(first).reshape(R, B)[rows], oracle.scalar_scan(dbh[rows], Qh))
