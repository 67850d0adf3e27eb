"""GPU parity: the pipelined query server (pir_server_*), host queries in,
host results out, against the oracle's NTT -> RowSel -> INTT for every query
of a stream (slots reused, copies overlapping the scans)."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


@pytest.mark.parametrize("N,L,D0,D1,B,nq", [
    (64, 2, 33, 130, 2, 5),      # CUDA-core RowSel, two slabs
    (16, 2, 40, 20, 12, 4),      # tensor-core RowSel (24 polynomials per pass)
    (4096, 3, 8, 5, 1, 3),       # the pages' ring
])
def test_server_stream_matches_oracle(pir, N, L, D0, D1, B, nq):
    import torch
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs((N + D0) % 251, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    srv = pir.PirServer(ctx, db, D0, D1, B)
    P = L * N
    queries = [synth.residues((D1 + i) % 251, (B, D0, 2, L, N), qs) for i in range(nq)]
    q_host = [torch.from_numpy(q.view(np.int32).reshape(-1)).pin_memory() for q in queries]
    o_host = [torch.full((B * D1 * 2 * P,), -1, dtype=torch.int32).pin_memory() for _ in range(nq)]
    srv.mark(0)
    tickets = [srv.submit(q_host[i], o_host[i]) for i in range(nq)]
    srv.mark(1)
    assert tickets == list(range(nq))
    srv.wait(nq - 1)
    assert srv.elapsed_ms() > 0
    enc = oracle.encode_records(raw, qs, psis)
    for i in range(nq):
        want = oracle.ntt_polys(oracle.rowsel(enc, oracle.ntt_polys(queries[i], qs, psis), qs), qs, psis,
                                inverse=True)
        got = o_host[i].numpy().view(np.uint32).reshape(B, D1, 2, L, N)
        assert np.array_equal(got, want), i
    with pytest.raises(pir.PirError):
        srv.wait(nq)                     # not submitted
    srv.close()
    assert pir.pir_status(ctx) == 0


def test_server_alternating_result_buffers(pir):
    """Two host result buffers reused in turn (wait for ticket t before
    submitting t + 2), as a serving loop runs."""
    import torch
    N, L, D0, D1, B, nq = 64, 3, 17, 9, 1, 7
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(3, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    enc = oracle.encode_records(raw, qs, psis)
    srv = pir.PirServer(ctx, db, D0, D1, B)
    P = L * N
    out = [torch.empty(B * D1 * 2 * P, dtype=torch.int32).pin_memory() for _ in range(2)]
    qh = [torch.empty(B * D0 * 2 * P, dtype=torch.int32).pin_memory() for _ in range(2)]
    queries = [synth.residues(40 + i, (B, D0, 2, L, N), qs) for i in range(nq)]
    for i in range(nq):
        if i >= 2:
            srv.wait(i - 2)
            want = oracle.ntt_polys(oracle.rowsel(enc, oracle.ntt_polys(queries[i - 2], qs, psis), qs), qs, psis,
                                    inverse=True)
            assert np.array_equal(out[i % 2].numpy().view(np.uint32).reshape(want.shape), want), i - 2
        qh[i % 2].copy_(torch.from_numpy(queries[i].view(np.int32).reshape(-1)))
        srv.submit(qh[i % 2], out[i % 2])
    srv.close()
