"""The bounded-wait recovery path, exercised without faulting the GPU.

Every device wait of the RowSel scans gives up after a limit, sets
PIR_STATUS_TIMEOUT in the context's status word, stops computing, drains its
own bulk copies in flight and returns, so the context stays usable.  Here a
test hook makes the first CTA of the scan never issue the copy of its last
DB chunk (a wait that nothing will ever satisfy), with the context's wait
limit shortened to 1 ms: on the CUDA cores (1 and 3 queries) and on the
tensor cores (9 queries, two K segments per point).  The launch must return promptly
with the status bit set; the next launch on the same context, with the hook
off and the default limit, must be bit-exact against the oracle with a clean
status word.
"""
import time

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


@pytest.mark.parametrize("D0,D1,B", [(16, 16, 1), (300, 40, 3), (520, 8, 9)])
def test_withheld_copy_times_out_and_context_recovers(pir, D0, D1, B):
    import torch
    N, L = 4096, 2
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(61, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    query = synth.residues(62, (B, D0, 2, L, N), qs)
    q_t = to_dev(query)
    ws = pir.rowsel_workspace(ctx, D0, D1, B)
    out = pir.empty_u32(B * D1 * 2 * L * N)
    torch.cuda.synchronize()
    assert pir.pir_status(ctx) == 0

    pir.pir_ctx_set_wait_limit(ctx, 1_000_000)
    pir.pir_ctx_set_test_hook(ctx, pir.PIR_HOOK_WITHHOLD_LAST_COPY)
    t0 = time.perf_counter()
    pir.pir_rowsel(ctx, db, D0, D1, q_t, B, out, ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert pir.pir_status(ctx) & pir.PIR_STATUS_TIMEOUT      # reported, and cleared by the read
    assert elapsed < 1.0, elapsed                             # the 1 ms limit, not the 2 s default

    pir.pir_ctx_set_test_hook(ctx, pir.PIR_HOOK_NONE)
    pir.pir_ctx_set_wait_limit(ctx, 0)
    out.fill_(-1)
    pir.pir_rowsel(ctx, db, D0, D1, q_t, B, out, ws)
    torch.cuda.synchronize()
    assert pir.pir_status(ctx) == 0
    enc = oracle.encode_records(raw, qs, psis)
    want = oracle.rowsel(enc, query, qs)
    assert np.array_equal(to_host_u32(out).reshape(B, D1, 2, L, N), want)


def test_diagnostic_setters_validate(pir):
    ctx = pir.pir_ctx_create(4096, oracle.primes(4096, 1))
    with pytest.raises(pir.PirError):
        pir.pir_ctx_set_wait_limit(ctx, 3_000_000_000)       # above the 2 s default
    with pytest.raises(pir.PirError):
        pir.pir_ctx_set_test_hook(ctx, 7)
    pir.pir_ctx_set_wait_limit(ctx, 0)
    pir.pir_ctx_set_test_hook(ctx, pir.PIR_HOOK_NONE)
