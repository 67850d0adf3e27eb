"""The allocation-free scalar scan (pir_scalar_scan_noalloc).

For callers that cannot allocate device memory when they run the scan, the
library keeps the split-query scratch in a static device array.  This test
calls that entry point through the C ABI twice in a row, with different
shapes and data, and checks each result bit-exactly against the regular
pir_scalar_scan with its own workspace, so a stale scratch from the first
call would show up in the second.  Kept in a file collected last.
"""
import numpy as np
import pytest

import synth
from tests.helpers import ensure_built, to_dev, to_host_u32

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    ensure_built()
    from lattice_he_database_gb300 import pir
    ctx = pir.pir_ctx_create(4096, pir.pir_primes(4096, 1))
    cases = [(384, 16384, 64, 21), (200, 4096, 7, 22)]   # largest allowed C first, then a smaller one
    for R, C, B, seed in cases:
        db = to_dev(synth.db_bytes(seed, (R, C)))
        Q = to_dev(synth.words(seed, (C, B)))
        ref = pir.empty_u32(R * B)
        ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
        pir.pir_scalar_scan(ctx, db, R, C, Q, B, ref, ws)
        got = pir.empty_u32(R * B)
        got.fill_(-1)
        pir.pir_scalar_scan_noalloc(ctx, db, R, C, Q, B, got)
        torch.cuda.synchronize()
        assert np.array_equal(to_host_u32(got), to_host_u32(ref)), (R, C, B)
        assert pir.pir_status(ctx) == 0
    # C beyond the static scratch is rejected on the host
    with pytest.raises(pir.PirError) as e:
        big = torch.zeros(128 * 16448, dtype=torch.uint8, device="cuda")
        pir.pir_scalar_scan_noalloc(ctx, big, 128, 16448, pir.empty_u32(16448 * 64), 64, pir.empty_u32(128 * 64))
    assert e.value.code == pir.PIR_ERR_UNSUPPORTED
