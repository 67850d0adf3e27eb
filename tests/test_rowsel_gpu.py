"""GPU parity: DB encoding and the RowSel scan against the oracle (bit-exact).

Small shapes are compared element by element (several column slabs, ragged
row chunks and column tails, multi-pass batches).  The full-size workloads
(6 GiB, 24 GiB with B = 16, 64 GiB with the query NTT and output INTT) are
checked on sampled DB columns, all evaluation points, all queries.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import (CONFIGS, ensure_built, gather_db_device, make_device_db, oracle_db_columns, to_dev,
                           to_host_u32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


def _small_case(pir, N, L, D0, D1, B, seed):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(seed, (D0, D1, N))
    db_t = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    db_t.fill_(-1)  # poison: every word must be written
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db_t)
    query = synth.residues(seed + 1, (B, D0, 2, L, N), qs)
    return ctx, qs, psis, raw, db_t, query


@pytest.mark.parametrize("N,L,D0,D1,B", [
    (64, 2, 3, 5, 1),        # single slab, ragged width
    (64, 3, 33, 130, 1),     # 2 slabs (128 + 4), ragged row chunk (32 + 1)
    (256, 2, 70, 257, 2),    # 3 slabs, 3 chunks
    (16, 1, 5, 128, 3),      # exact slab, odd B
    (64, 2, 40, 200, 5),     # padded polynomial count (M = 10 -> 16)
    (16, 2, 9, 44, 16),      # M = 32
    (16, 2, 9, 44, 17),      # two passes (16 + 1)
    (16, 2, 512, 300, 16),   # tensor-core path: D0 = 512, 3 slabs (128 + 128 + 44)
    (64, 3, 100, 37, 12),    # tensor-core path, padded polynomials (24 of 32), ragged rows
    (16, 2, 1000, 44, 16),   # tensor-core path, two K segments (512 + 488)
    (16, 2, 1536, 40, 12),   # tensor-core path, three full K segments
    (16, 1, 600, 130, 17),   # two passes: tensor cores (512 + 88 rows, 2 slabs), then 1 query on CUDA cores
    (16, 2, 513, 9, 9),      # tensor-core path, second segment of a single row
    (16, 2, 130, 200, 16),   # tensor-core path, last slab of 72 columns: a full and a ragged 64-column tile
    (16, 2, 64, 100, 10),    # tensor-core path, one 100-column slab (64 + 36), 20 of 32 polynomials
])
def test_encode_and_rowsel_small(pir, N, L, D0, D1, B):
    ctx, qs, psis, raw, db_t, query = _small_case(pir, N, L, D0, D1, B, seed=(N + D0 + D1 + B) % 251)
    # the encoded DB holds NTT(record) at its documented position
    enc = oracle.encode_records(raw, qs, psis)               # [D0][D1][L][N]
    ks, ns = np.meshgrid(np.arange(D0), np.arange(D1), indexing="ij")
    got_db = gather_db_device(db_t, N, L, D0, D1, ks.reshape(-1), ns.reshape(-1))
    assert np.array_equal(got_db, enc.reshape(D0 * D1, L * N))
    D1p = (D1 + 3) // 4 * 4
    if D1p > D1:  # padding columns are zero
        kp, npd = np.meshgrid(np.arange(D0), np.arange(D1, D1p), indexing="ij")
        assert (gather_db_device(db_t, N, L, D0, D1, kp.reshape(-1), npd.reshape(-1)) == 0).all()
    out = pir.empty_u32(B * D1 * 2 * L * N)
    out.fill_(-1)
    pir.pir_rowsel(ctx, db_t, D0, D1, to_dev(query), B, out, pir.rowsel_workspace(ctx, D0, D1, B))
    got = to_host_u32(out).reshape(B, D1, 2, L, N)
    assert np.array_equal(got, oracle.rowsel(enc, query, qs))
    assert pir.pir_status(ctx) == 0


def test_rowsel_one_hot_returns_record(pir):
    """Selection invariant: a one-hot query returns DB[i*][n] exactly after the INTT."""
    N, L, D0, D1 = 4096, 3, 40, 131
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(5, (D0, D1, N))
    db_t = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db_t)
    for istar in (0, 17, D0 - 1):
        q = np.zeros((1, D0, 2, L, N), np.uint32)
        q[0, istar, 0] = 1       # the constant polynomial 1: all ones in NTT form
        out = pir.empty_u32(D1 * 2 * L * N)
        pir.pir_rowsel(ctx, db_t, D0, D1, to_dev(q), 1, out, pir.rowsel_workspace(ctx, D0, D1, 1))
        pir.pir_ntt_inv(ctx, out, out, D1 * 2)
        got = to_host_u32(out).reshape(D1, 2, L, N)
        for l in range(L):
            assert np.array_equal(got[:, 0, l], raw[istar])
        assert (got[:, 1] == 0).all()
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("B,D0", [(1, 1000), (2, 1000), (4, 1000), (8, 1000), (16, 1000), (16, 512)])
def test_rowsel_max_residues(pir, B, D0):
    """All residues q-1 (largest products, longest lazy chains) for every split
    of rows and polynomials across warps, and on the tensor-core path
    (B = 16, D0 = 512): out = D0 mod q."""
    N, L, D1 = 64, 3, 9
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    P = L * N
    D1p = (D1 + 3) // 4 * 4
    # an encoded DB with every word q_l - 1 (written directly in the layout)
    words = np.empty((P, D0 * D1p), np.uint32)
    for l in range(L):
        words[l * N:(l + 1) * N] = qs[l] - 1
    db_t = to_dev(words.reshape(-1))
    query = np.broadcast_to(np.array(qs, np.uint32).reshape(1, 1, 1, L, 1) - 1, (B, D0, 2, L, N)).copy()
    out = pir.empty_u32(B * D1 * 2 * P)
    out.fill_(-1)
    pir.pir_rowsel(ctx, db_t, D0, D1, to_dev(query), B, out, pir.rowsel_workspace(ctx, D0, D1, B))
    got = to_host_u32(out).reshape(B, D1, 2, L, N)
    for l in range(L):
        assert (got[..., l, :] == D0 % qs[l]).all()
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("D0", [512, 1024, 1100])
def test_rowsel_tensor_path_digit_extremes(pir, D0):
    """Tensor-core path at its exactness limit: DB words 0x1EFFFFFF (three
    bytes 255) against query words 0x1F7F7F80 (balanced digits -128, -128,
    -128, 32) over a 512-row K segment puts every digit-plane sum at
    512 * 255 * 128, just below 2^24; out = D0 * a * b mod q, with the
    segments' residues added for D0 > 512."""
    N, L, D1, B = 64, 3, 33, 16
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    P = L * N
    D1p = (D1 + 3) // 4 * 4
    a, b = 0x1F7F7F80, 0x1EFFFFFF
    assert a < min(qs) and b < min(qs)
    db_t = to_dev(np.full(P * D0 * D1p, b, np.uint32))
    query = np.full((B, D0, 2, L, N), a, np.uint32)
    out = pir.empty_u32(B * D1 * 2 * P)
    out.fill_(-1)
    pir.pir_rowsel(ctx, db_t, D0, D1, to_dev(query), B, out, pir.rowsel_workspace(ctx, D0, D1, B))
    got = to_host_u32(out).reshape(B, D1, 2, L, N)
    for l in range(L):
        assert (got[..., l, :] == (D0 * a * b) % qs[l]).all()
    assert pir.pir_status(ctx) == 0


def _primes_between(N, L, lo, hi):
    qs = oracle.primes(N, L, bound=hi)
    assert len(qs) == L and all(lo <= q < hi for q in qs), qs
    return qs


@pytest.mark.parametrize("lo,hi", [(1 << 26, (1 << 26) + (1 << 20)), (1 << 25, 1 << 26)])
def test_rowsel_b16_prime_sizes(pir, lo, hi):
    """A 16-query pass with the smallest primes the tensor-core epilogue
    supports (just above 2^26) and with primes below 2^26 (which take the
    CUDA-core kernel): random residues compared element by element, and the
    largest partial sums of the epilogue's quotient estimate (DB words with
    three low bytes 255, query words with balanced digits -128, -128, -128)."""
    N, L, D0, D1, B = 64, 2, 512, 40, 16
    qs = _primes_between(N, L, lo, hi)
    ctx = pir.pir_ctx_create(N, qs)
    P = L * N
    D1p = (D1 + 3) // 4 * 4
    psis = [oracle.min_psi(q, N) for q in qs]
    raw = synth.coeffs(31, (D0, D1, N))
    db_t = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db_t)
    enc = oracle.encode_records(raw, qs, psis)
    query = synth.residues(32, (B, D0, 2, L, N), qs)
    out = pir.empty_u32(B * D1 * 2 * P)
    out.fill_(-1)
    pir.pir_rowsel(ctx, db_t, D0, D1, to_dev(query), B, out, pir.rowsel_workspace(ctx, D0, D1, B))
    got = to_host_u32(out).reshape(B, D1, 2, L, N)
    assert np.array_equal(got, oracle.rowsel(enc, query, qs))
    # extremes, written directly in the (single-slab) DB layout [p][k][n]:
    # every DB word b_l, every query word a_l (per prime)
    db_words = np.empty((P, D0 * D1p), np.uint32)
    qext = np.empty((B, D0, 2, L, N), np.uint32)
    want = []
    for l, q in enumerate(qs):
        top = q >> 24
        b = (top - 1) * (1 << 24) + 0xFFFFFF if (top - 1) * (1 << 24) + 0xFFFFFF < q else q - 1
        a = top * (1 << 24) - 0x808080
        assert 0 <= a < q and 0 <= b < q
        db_words[l * N:(l + 1) * N] = b
        qext[..., l, :] = a
        want.append(D0 * a * b % q)
    out.fill_(-1)
    pir.pir_rowsel(ctx, to_dev(db_words.reshape(-1)), D0, D1, to_dev(qext), B, out,
                   pir.rowsel_workspace(ctx, D0, D1, B))
    got = to_host_u32(out).reshape(B, D1, 2, L, N)
    for l in range(L):
        assert (got[..., l, :] == want[l]).all()
    assert pir.pir_status(ctx) == 0


def test_rowsel_rejects_bad_arguments(pir):
    qs = oracle.primes(64, 2)
    ctx = pir.pir_ctx_create(64, qs)
    db = pir.empty_u32(pir.pir_db_bytes(ctx, 4, 4) // 4)
    q = pir.empty_u32(4 * 2 * 2 * 64)
    out = pir.empty_u32(4 * 2 * 2 * 64)
    ws = pir.rowsel_workspace(ctx, 4, 4, 1)
    for args in [(0, 4, 1), (4, 0, 1), (4, 4, 0)]:
        with pytest.raises(pir.PirError):
            pir.pir_rowsel(ctx, db, args[0], args[1], q, args[2], out, ws)
    with pytest.raises(pir.PirError):
        pir.pir_rowsel(ctx, db, 4, 4, q[1:], 1, out, ws)
    with pytest.raises(pir.PirError):                 # workspace too small
        pir.pir_rowsel(ctx, db, 4, 4, q, 1, out, ws[:16])
    with pytest.raises(pir.PirError):                 # D0 beyond the on-chip query slice
        pir.pir_rowsel(ctx, db, 14337, 4, q, 1, out, ws)
    with pytest.raises(pir.PirError):
        pir.pir_db_encode(ctx, q, 3, 2, 4, 4, db)   # k0 + kcnt > D0


# ------------------------------------------------------------------ full-size workloads
def _full_size(pir, name, sample_cols):
    import torch
    import synth.device as sd
    cfg = CONFIGS[name]
    N, L, D0, D1, B = cfg["N"], cfg["L"], cfg["D0"], cfg["D1"], cfg["B"]
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    seed = 7
    db_t = make_device_db(ctx, D0, D1, seed)
    P = L * N
    qwords = B * D0 * 2 * P
    q_t = torch.empty(qwords, dtype=torch.int32, device="cuda")
    sd.fill_residues(q_t, seed, synth.T_QUERY, N, qs)
    query = to_host_u32(q_t).reshape(B, D0, 2, L, N)
    out = pir.empty_u32(B * D1 * 2 * P)
    if cfg["query_domain"] == "coeff":
        # the serving path: NTT(query) -> RowSel -> INTT(result)
        srv = pir.RowselServer(ctx, db_t, D0, D1, B)
        res = srv.answer_device(q_t)
        q_ntt_gpu = to_host_u32(srv.q_ntt).reshape(query.shape)
        q_ntt = oracle.ntt_polys(query, qs, psis)
        assert np.array_equal(q_ntt_gpu, q_ntt)
        out_ntt = to_host_u32(srv.o_ntt).reshape(B, D1, 2, L, N)
        out_coef = to_host_u32(res).reshape(B, D1, 2, L, N)
    else:
        q_ntt = query
        pir.pir_rowsel(ctx, db_t, D0, D1, q_t, B, out, pir.rowsel_workspace(ctx, D0, D1, B))
        out_ntt = to_host_u32(out).reshape(B, D1, 2, L, N)
        out_coef = None
    assert pir.pir_status(ctx) == 0
    cols = np.array(sample_cols, np.uint32)
    # the DB words of the sampled columns (a few rows) match the oracle encoding
    enc = oracle_db_columns(qs, psis, N, D0, D1, seed, cols)    # [D0][ncols][L][N]
    for k in (0, D0 - 1):
        got = gather_db_device(db_t, N, L, D0, D1, [k] * len(cols), cols)
        assert np.array_equal(got, enc[k].reshape(len(cols), P))
    want = oracle.rowsel(enc, q_ntt, qs, cols=np.arange(len(cols)))   # [B][ncols][2][L][N]
    assert np.array_equal(out_ntt[:, cols.astype(np.int64)], want)
    if out_coef is not None:
        want_coef = oracle.ntt_polys(want, qs, psis, inverse=True)
        assert np.array_equal(out_coef[:, cols.astype(np.int64)], want_coef)
    del db_t
    torch.cuda.empty_cache()


def test_full_tiny_exact(pir):
    """16 x 16 records, 2 primes: every output compared."""
    _full_size(pir, "tiny", sample_cols=list(range(16)))


def test_full_rowsel_6g(pir):
    _full_size(pir, "rowsel_6g", sample_cols=[0, 127, 128, 300, 511])


def test_full_rowsel_24g_b16(pir):
    _full_size(pir, "rowsel_24g_b16", sample_cols=[0, 513, 1023])


def test_full_rowsel_64g_b16(pir):
    """16 queries over the 64 GiB DB: tensor cores, two K segments per point."""
    _full_size(pir, "rowsel_64g_b16", sample_cols=[0, 700, 1364])


def test_full_rowsel_64g_with_ntt(pir):
    _full_size(pir, "rowsel_64g", sample_cols=[0, 1279, 1280, 1364])
