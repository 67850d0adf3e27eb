"""The OnionPIR server path end to end on the GPU: ExpandQuery -> RowSel ->
ColTor (GPIR section 2: the three phases), under a ternary secret with
noise-free encryptions and keys, so every step is exact mod q.

The client's query encrypts X^(i*); the expansion gives D0 ciphertexts of
which only i* decrypts to a nonzero constant (2^S); RowSel's point-wise GEMM
with the encoded DB gives, for every column n, a ciphertext of
2^S DB[i*][n]; ColTor with RGSW encryptions of the bits of j* keeps column
j*.  The decryption of the final ciphertext must equal 2^S DB[i*][j*].

In the one-ciphertext form (GPIR section 2: the query carries both indices)
the same query also carries, in coefficients D0 .. D0 + T ell - 1, the
gadget values b_s g_u of the bits b_s of j* pre-scaled by 2^-S; the
expansion turns them into the gadget ciphertexts of each bit and
pir_rgsw_convert, with a key-switching key of s^2, into the RGSW
ciphertexts ColTor takes.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev, to_host_u32
from tests.test_expand_oracle import Keys, _mul, _qcol, _rand, _signed, _sub

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


def _rgsw(K, bit):
    """RGSW(bit) = Z + bit * (I_2 x g): rows of Z encrypt 0 under s (noise-free), NTT form."""
    L, N, ell = len(K.qs), K.N, K.ell
    C = np.zeros((2 * ell, 2, L, N), dtype=np.uint32)
    for r in range(2 * ell):
        a = _rand(K.rng, K.qs, N)
        C[r, 0] = _sub(np.zeros_like(a), _mul(a, K.sN, K.qs), K.qs)
        C[r, 1] = a
    for u in range(ell):
        for l, q in enumerate(K.qs):
            g = bit * pow(2, K.w * u, q) % q
            C[u, 0, l] = (C[u, 0, l].astype(np.uint64) + g) % q
            C[ell + u, 1, l] = (C[ell + u, 1, l].astype(np.uint64) + g) % q
    return C


@pytest.mark.parametrize("D0,D1,istar,jstar", [(16, 11, 5, 7), (64, 40, 63, 0), (1024, 24, 700, 17)])
def test_query_returns_the_selected_record(pir, D0, D1, istar, jstar):
    N, L, ell, w = 4096, 3, 5, 18
    K = Keys(N, L, ell, w, seed=D0 + D1)
    ctx = pir.pir_ctx_create(N, K.qs)
    S = D0.bit_length() - 1
    assert 1 << S == D0
    # the DB: D0 x D1 records of 16-bit coefficients, encoded on the GPU
    raw = synth.coeffs(D0 % 251, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    # client: Enc(X^i*), evaluation keys, RGSW bits of j*
    mono = np.zeros(N, dtype=np.int64)
    mono[istar] = 1
    query = K.encrypt(_signed(mono, K.qs))
    evks = np.stack([K.evk(N // (1 << j) + 1) for j in range(S)])
    T = oracle.coltor_stages(D1)
    rgsw = np.stack([_rgsw(K, (jstar >> s) & 1) for s in range(T)])
    # server: ExpandQuery -> RowSel -> ColTor, all on the GPU
    expanded = pir.empty_u32(D0 * 2 * L * N)
    pir.pir_expand(ctx, to_dev(evks), ell, w, S, to_dev(query), expanded, pir.expand_workspace(ctx, D0 // 2, ell))
    cols = pir.empty_u32(D1 * 2 * L * N)
    pir.pir_rowsel(ctx, db, D0, D1, expanded, 1, cols, pir.rowsel_workspace(ctx, D0, D1, 1))
    answer = pir.empty_u32(2 * L * N)
    pir.pir_coltor(ctx, to_dev(rgsw), ell, w, cols, D1, answer, pir.coltor_workspace(ctx, D1, ell))
    assert pir.pir_status(ctx) == 0
    # client: decrypt
    got = K.decrypt(to_host_u32(answer).reshape(2, L, N))
    want = _signed(raw[istar, jstar].astype(np.int64) << S, K.qs)
    assert np.array_equal(got, want)


def test_batch_of_clients_on_the_tensor_path(pir):
    """Ten clients, each with its own secret, keys, record and column, served
    together: one batched expansion, one RowSel pass of B = 10 queries (the
    tensor cores: primes >= 2^26, 8 < B <= 16) and one batched tournament.
    Every answer decrypts under its own client's secret to 2^S DB[i*_b][j*_b]."""
    N, L, ell, w, D0, D1, B = 4096, 3, 5, 18, 16, 11, 10
    S, T = 4, oracle.coltor_stages(D1)
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(77, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    P = L * N
    clients, queries, evks, rgsws = [], [], [], []
    for b in range(B):
        K = Keys(N, L, ell, w, seed=500 + b)
        istar, jstar = (5 * b + 3) % D0, (7 * b + 2) % D1
        mono = np.zeros(N, dtype=np.int64)
        mono[istar] = 1
        queries.append(K.encrypt(_signed(mono, K.qs)))
        evks.append(np.stack([K.evk(N // (1 << j) + 1) for j in range(S)]))
        rgsws.append(np.stack([_rgsw(K, (jstar >> s) & 1) for s in range(T)]))
        clients.append((K, istar, jstar))
    expanded = pir.empty_u32(B * D0 * 2 * P)
    pir.pir_expand_batch(ctx, to_dev(np.stack(evks)), ell, w, S, to_dev(np.stack(queries)), B, expanded,
                         pir.expand_workspace(ctx, B * D0 // 2, ell))
    cols = pir.empty_u32(B * D1 * 2 * P)
    pir.pir_rowsel(ctx, db, D0, D1, expanded, B, cols, pir.rowsel_workspace(ctx, D0, D1, B))
    answers = pir.empty_u32(B * 2 * P)
    pir.pir_coltor_batch(ctx, to_dev(np.stack(rgsws)), ell, w, cols, D1, B, answers,
                         pir.coltor_batch_workspace(ctx, D1, B, ell))
    assert pir.pir_status(ctx) == 0
    got = to_host_u32(answers).reshape(B, 2, L, N)
    for b, (K, istar, jstar) in enumerate(clients):
        assert np.array_equal(K.decrypt(got[b]), _signed(raw[istar, jstar].astype(np.int64) << S, K.qs)), b


def _ksk(K):
    """Key-switching key: noise-free encryptions of s^2 g_v, v < ell."""
    N = K.N
    full = np.convolve(K.s.astype(np.int64), K.s.astype(np.int64))
    s2 = full[:N].copy()
    s2[: len(full) - N] -= full[N:]
    rows = []
    for v in range(K.ell):
        g = np.array([pow(2, K.w * v, q) for q in K.qs], dtype=np.uint64).reshape(-1, 1)
        rows.append(K.encrypt(((_signed(s2, K.qs).astype(np.uint64) * g) % _qcol(K.qs)).astype(np.uint32)))
    return np.stack(rows)


def _one_ciphertext_query(K, D0, T, istar, jstar, S):
    """[L][N] plaintext residues: X^(i*) in the first D0 coefficients, and
    2^-S b_s g_u at D0 + s ell + u for the bits b_s of j*."""
    m = np.zeros((len(K.qs), K.N), dtype=np.uint32)
    m[:, istar] = 1
    for s in range(T):
        if (jstar >> s) & 1:
            for u in range(K.ell):
                for l, q in enumerate(K.qs):
                    m[l, D0 + s * K.ell + u] = pow(2, K.w * u, q) * pow(pow(2, S, q), -1, q) % q
    return m


@pytest.mark.parametrize("D0,D1,istar,jstar", [(16, 11, 9, 6), (64, 40, 1, 39)])
def test_one_query_ciphertext_with_converted_rgsw(pir, D0, D1, istar, jstar):
    N, L, ell, w = 4096, 3, 5, 18
    K = Keys(N, L, ell, w, seed=3 * D0 + D1)
    ctx = pir.pir_ctx_create(N, K.qs)
    T = oracle.coltor_stages(D1)
    S = (D0 + T * ell - 1).bit_length()          # expansion outputs cover the row and the column part
    raw = synth.coeffs(D0 + 1, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    query = K.encrypt(_one_ciphertext_query(K, D0, T, istar, jstar, S))
    evks = np.stack([K.evk(N // (1 << j) + 1) for j in range(S)])
    expanded = pir.empty_u32((1 << S) * 2 * L * N)
    pir.pir_expand(ctx, to_dev(evks), ell, w, S, to_dev(query), expanded, pir.expand_workspace(ctx, 1 << (S - 1), ell))
    P2 = 2 * L * N
    rgsw = pir.empty_u32(T * 2 * ell * P2)
    pir.pir_rgsw_convert(ctx, to_dev(_ksk(K)), ell, w, expanded[D0 * P2:(D0 + T * ell) * P2], T, 1, rgsw,
                         pir.rgsw_convert_workspace(ctx, T, 1, ell))
    cols = pir.empty_u32(D1 * P2)
    pir.pir_rowsel(ctx, db, D0, D1, expanded[: D0 * P2], 1, cols, pir.rowsel_workspace(ctx, D0, D1, 1))
    answer = pir.empty_u32(P2)
    pir.pir_coltor(ctx, rgsw, ell, w, cols, D1, answer, pir.coltor_workspace(ctx, D1, ell))
    assert pir.pir_status(ctx) == 0
    got = K.decrypt(to_host_u32(answer).reshape(2, L, N))
    assert np.array_equal(got, _signed(raw[istar, jstar].astype(np.int64) << S, K.qs))


def test_batch_of_one_ciphertext_queries_on_the_tensor_path(pir):
    """Nine clients, each sending one query ciphertext (row and column
    index), their own expansion keys and key-switching key: one batched
    expansion, one batched conversion to RGSW, one RowSel pass of B = 9
    queries on the tensor cores, one batched tournament."""
    N, L, ell, w, D0, D1, B = 4096, 3, 5, 18, 16, 11, 9
    T = oracle.coltor_stages(D1)
    S = (D0 + T * ell - 1).bit_length()
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.coeffs(91, (D0, D1, N))
    db = pir.empty_u32(pir.pir_db_bytes(ctx, D0, D1) // 4)
    pir.pir_db_encode(ctx, to_dev(raw), 0, D0, D0, D1, db)
    P2 = 2 * L * N
    clients, queries, evks, ksks = [], [], [], []
    for b in range(B):
        K = Keys(N, L, ell, w, seed=900 + b)
        istar, jstar = (3 * b + 1) % D0, (5 * b + 4) % D1
        queries.append(K.encrypt(_one_ciphertext_query(K, D0, T, istar, jstar, S)))
        evks.append(np.stack([K.evk(N // (1 << j) + 1) for j in range(S)]))
        ksks.append(_ksk(K))
        clients.append((K, istar, jstar))
    M = 1 << S
    expanded = pir.empty_u32(B * M * P2)
    pir.pir_expand_batch(ctx, to_dev(np.stack(evks)), ell, w, S, to_dev(np.stack(queries)), B, expanded,
                         pir.expand_workspace(ctx, B * M // 2, ell))
    ex = expanded.view(B, M * P2)
    rows = ex[:, : D0 * P2].contiguous()                       # [B][D0] RowSel queries
    rgsw = pir.empty_u32(B * T * 2 * ell * P2)
    # client b's T ell gadget ciphertexts sit at b M + D0 in the expansion output
    pir.pir_rgsw_convert(ctx, to_dev(np.stack(ksks)), ell, w, expanded[D0 * P2:], T, B, rgsw,
                         pir.rgsw_convert_workspace(ctx, T, B, ell), in_stride=M)
    cols = pir.empty_u32(B * D1 * P2)
    pir.pir_rowsel(ctx, db, D0, D1, rows, B, cols, pir.rowsel_workspace(ctx, D0, D1, B))
    answers = pir.empty_u32(B * P2)
    pir.pir_coltor_batch(ctx, rgsw, ell, w, cols, D1, B, answers, pir.coltor_batch_workspace(ctx, D1, B, ell))
    assert pir.pir_status(ctx) == 0
    got = to_host_u32(answers).reshape(B, 2, L, N)
    for b, (K, istar, jstar) in enumerate(clients):
        assert np.array_equal(K.decrypt(got[b]), _signed(raw[istar, jstar].astype(np.int64) << S, K.qs)), b
