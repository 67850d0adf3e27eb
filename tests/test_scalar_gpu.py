"""GPU parity: the scalar-HE scan (byte DB x 32-bit query words mod 2^32).

Bit-exact against the oracle on small shapes (ragged row tiles, partial
accumulator chunks, B < 64, more row tiles than SMs), on adversarial values that put every partial
sum of the fp16/fp32 tensor-core path at its largest magnitude, on the
CUDA-core GEMV used for B <= 4 (ragged tiles and boxes, row tiles split
between CTAs, wrapping byte-plane sums), and on sampled rows of the full
131072 x 131072 DB with B = 64 and B = 1.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import SCALAR, ensure_built, to_dev, to_host_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    ensure_built()
    from lattice_he_database_gb300 import pir
    ctx = pir.pir_ctx_create(4096, pir.pir_primes(4096, 1))
    return pir, ctx


def _run(pir, ctx, db, Q):
    import torch
    R, C = db.shape
    B = Q.shape[1]
    out = pir.empty_u32(R * B)
    out.fill_(-1)
    ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
    pir.pir_scalar_scan(ctx, to_dev(db), R, C, to_dev(Q), B, out, ws)
    got = to_host_u32(out).reshape(R, B)
    assert pir.pir_status(ctx) == 0
    return got


@pytest.mark.parametrize("R,C,B", [
    (128, 64, 64),       # one tile, one stage
    (128, 512, 64),      # exactly one accumulator chunk
    (256, 1088, 64),     # two tiles, 2 chunks + a partial one
    (300, 640, 64),      # ragged last tile (rows zero-filled by TMA)
    (128, 1024, 5),      # B < 64
    (257, 192, 1),       # B = 1, ragged
    (64, 8192, 64),      # one ragged row tile over 16 accumulator chunks
    (20000, 1088, 33),   # more row tiles than SMs (a second, partial wave), B < 64
])
def test_scalar_scan_small(env, R, C, B):
    pir, ctx = env
    db = synth.db_bytes((R + C + B) % 251, (R, C))
    Q = synth.words((R + C + B + 1) % 251, (C, B))
    assert np.array_equal(_run(pir, ctx, db, Q), oracle.scalar_scan(db, Q))


@pytest.mark.parametrize("R,C,B", [
    (1, 64, 1),          # one row, half a box (columns zero-filled by TMA)
    (256, 128, 1),       # exactly one unit
    (300, 1088, 2),      # ragged row tile and column box
    (1000, 8192, 3),     # many units: CTA ranges split row tiles (atomic partial sums)
    (513, 4160, 4),      # B = 4, ragged both ways
    (40000, 192, 1),     # more row tiles than CTAs, 2 boxes per tile
])
def test_scalar_gemv_small_batches(env, R, C, B):
    """B <= 4: the CUDA-core GEMV path."""
    pir, ctx = env
    db = synth.db_bytes((R + C + B) % 251, (R, C))
    Q = synth.words((R + C + 2 * B) % 251, (C, B))
    assert np.array_equal(_run(pir, ctx, db, Q), oracle.scalar_scan(db, Q))


@pytest.mark.parametrize("B", [1, 4])
def test_scalar_gemv_wraparound(env, B):
    """All-255 DB times all-ones words: every byte-plane sum wraps past 2^32
    (C * 255 * 255 > 2^32 at C = 131072) and only its low bits may survive."""
    pir, ctx = env
    R, C = 300, 131072
    db = np.full((R, C), 255, np.uint8)
    Q = np.full((C, B), 0xFFFFFFFF, np.uint32)
    got = _run(pir, ctx, db, Q)
    assert (got == (255 * 0xFFFFFFFF * C) % (1 << 32)).all()


def test_scalar_gemv_one_hot(env):
    pir, ctx = env
    R, C, B = 700, 4096, 4
    db = synth.db_bytes(19, (R, C))
    Q = np.zeros((C, B), np.uint32)
    cols = [0, 127, 128, C - 1]
    for b, c in enumerate(cols):
        Q[c, b] = 0x01000001            # byte planes 0 and 3: db + (db << 24)
    got = _run(pir, ctx, db, Q)
    for b, c in enumerate(cols):
        v = db[:, c].astype(np.uint64)
        assert np.array_equal(got[:, b], ((v + (v << 24)) % (1 << 32)).astype(np.uint32))


@pytest.mark.parametrize("qword", [0x7F7F7F80, 0x7F7F7F7F, 0xFFFFFFFF, 0x80808080])
def test_scalar_scan_extreme_digits(env, qword):
    """DB all 255 with words whose balanced digits are all -128 (0x7F7F7F80) or
    all +127 (0x7F7F7F7F): every chunk sum is +-512*255*128, just below 2^24."""
    pir, ctx = env
    R, C, B = 128, 2048, 64
    db = np.full((R, C), 255, np.uint8)
    Q = np.full((C, B), qword, np.uint32)
    got = _run(pir, ctx, db, Q)
    assert (got == (255 * qword * C) % (1 << 32)).all()
    assert np.array_equal(got, oracle.scalar_scan(db, Q))


def test_scalar_scan_one_hot(env):
    pir, ctx = env
    R, C, B = 256, 1024, 64
    db = synth.db_bytes(9, (R, C))
    Q = np.zeros((C, B), np.uint32)
    for b in range(B):
        Q[(b * 37) % C, b] = 1
    got = _run(pir, ctx, db, Q)
    for b in range(B):
        assert np.array_equal(got[:, b], db[:, (b * 37) % C].astype(np.uint32))


def test_scalar_scan_rejects_bad_shapes(env):
    import torch
    pir, ctx = env
    db = torch.zeros(128 * 100, dtype=torch.uint8, device="cuda")
    Q = pir.empty_u32(100 * 64)
    out = pir.empty_u32(128 * 64)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(pir.PirError):     # C not a multiple of 64
        pir.pir_scalar_scan(ctx, db, 128, 100, Q, 64, out, ws)
    with pytest.raises(pir.PirError):     # B > 64
        pir.pir_scalar_scan(ctx, db, 128, 64, Q, 65, out, ws)
    with pytest.raises(pir.PirError):     # workspace too small
        pir.pir_scalar_scan(ctx, db, 128, 64 * 64, Q, 64, out, ws[: 1024])


@pytest.mark.parametrize("B", [SCALAR["B"], 1])
def test_scalar_scan_full_size_sampled_rows(env, B):
    """131072 x 131072 byte DB (16 GiB), 64 queries (tensor path) and one
    query (CUDA-core GEMV): sampled rows vs the oracle."""
    import torch
    import synth.device as sd
    pir, ctx = env
    R, C = SCALAR["R"], SCALAR["C"]
    seed = 7
    db_t = torch.empty(R * C, dtype=torch.uint8, device="cuda")
    sd.fill_bytes(db_t, seed, synth.T_SCALAR_DB)
    Q_t = pir.empty_u32(C * B)
    sd.fill_words(Q_t, seed, synth.T_SCALAR_Q)
    out = pir.empty_u32(R * B)
    ws = torch.empty(pir.pir_scalar_workspace_bytes(C, B), dtype=torch.uint8, device="cuda")
    pir.pir_scalar_scan(ctx, db_t, R, C, Q_t, B, out, ws)
    got = to_host_u32(out).reshape(R, B)
    assert pir.pir_status(ctx) == 0
    rows = np.array([0, 1, 127, 128, 65535, 65536, R - 129, R - 1])
    db_rows = np.stack([synth.db_bytes(seed, (C,), offset=int(r) * C) for r in rows])
    Q = synth.words(seed, (C, B))
    assert np.array_equal(got[rows], oracle.scalar_scan(db_rows, Q))
    del db_t
    torch.cuda.empty_cache()
