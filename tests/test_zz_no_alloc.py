"""The allocation-free scalar scan (pir_scalar_scan_noalloc).

Callers that cannot allocate device memory while they run the scan -- code
running while a framework's caching allocator owns the device pool, plugin
or serving paths handed only their input and output buffers, loops where a
cudaMalloc and its implicit synchronisation are not acceptable -- use this
entry point; it keeps the split-query scratch in a static device array.

The test calls it through the C ABI several times in a row, with different
shapes and data, and checks every result against the oracle (sampled rows)
and bit-exactly against the regular pir_scalar_scan with its own workspace,
so a stale scratch from an earlier call would show up in a later one.  The
cases cover both scratch layouts: the tensor-core digit blocks (B > 4) and
the GEMV plane words (B <= 4), each after a call of the other kind.  Kept in
a file collected last.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev, to_host_u32

pytestmark = pytest.mark.gpu

# (R, C, B, seed): largest allowed C first, then a smaller shape, then the
# GEMV route through the same scratch after a tensor-core call, and back.
CASES = [(384, 16384, 64, 21), (300, 16384, 3, 23), (200, 4096, 7, 22), (257, 8192, 1, 24), (130, 4096, 4, 25)]


def test_noalloc_matches_oracle_and_workspace_entry_point():
    import torch
    ensure_built()
    from lattice_he_database_gb300 import pir
    ctx = pir.pir_ctx_create(4096, pir.pir_primes(4096, 1))
    rng = np.random.default_rng(5)
    for R, C, B, seed in CASES:
        db_h = synth.db_bytes(seed, (R, C))
        Q_h = synth.words(seed, (C, B))
        db, Q = to_dev(db_h), to_dev(Q_h)
        ref = pir.empty_u32(R * B)
        ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
        pir.pir_scalar_scan(ctx, db, R, C, Q, B, ref, ws)
        got = pir.empty_u32(R * B)
        got.fill_(-1)
        pir.pir_scalar_scan_noalloc(ctx, db, R, C, Q, B, got)
        torch.cuda.synchronize()
        g = to_host_u32(got).reshape(R, B)
        assert np.array_equal(g, to_host_u32(ref).reshape(R, B)), (R, C, B)
        rows = np.unique(np.concatenate([[0, R - 1], rng.integers(0, R, 24)]))
        assert np.array_equal(g[rows], oracle.scalar_scan(db_h[rows], Q_h)), (R, C, B)
        assert pir.pir_status(ctx) == 0
    # C beyond the static scratch is rejected on the host
    with pytest.raises(pir.PirError) as e:
        big = torch.zeros(128 * 16448, dtype=torch.uint8, device="cuda")
        pir.pir_scalar_scan_noalloc(ctx, big, 128, 16448, pir.empty_u32(16448 * 64), 64, pir.empty_u32(128 * 64))
    assert e.value.code == pir.PIR_ERR_UNSUPPORTED
