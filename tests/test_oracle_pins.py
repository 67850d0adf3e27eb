"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something the pages or mathematics fix:
page parameters (tests/golden/page_parameters.json), closed forms, library
routines (sympy primality/orders, numpy convolution and matmul), invariants
(inverse transforms, the one-hot selection of PIR) and brute force in Python
integers on tiny inputs.  The cases are chosen so that a dropped term, a
wrong sign, a wrong index order or a transposed operand fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
sympy = pytest.importorskip("sympy")


def brv(j, bits):
    return int(format(j, "0%db" % bits)[::-1], 2) if bits else 0


def page_params():
    with open(os.path.join(GOLDEN, "page_parameters.json")) as f:
        return json.load(f)


# ------------------------------------------------------------------ generator
def test_splitmix64_reference_vector():
    """Published SplitMix64 outputs from state 0 (state advances by gamma first)."""
    want = [int(l, 16) for l in open(os.path.join(GOLDEN, "splitmix64_seed0.txt"))
            if l.strip() and not l.startswith("#")]
    # our splitmix64(x) mixes x + gamma, i.e. the state after k+1 steps is gamma*(k+1)
    g = 0x9E3779B97F4A7C15
    states = np.array([(g * k) % (1 << 64) for k in range(3)], dtype=np.uint64)
    got = [int(v) for v in synth.splitmix64(states)]
    assert got == want


def test_generator_ranges_and_addressing():
    qs = [536813569, 536690689]
    r = synth.residues(7, (3, 2, 2, 16), qs)
    assert (r[..., 0, :] < qs[0]).all() and (r[..., 1, :] < qs[1]).all()
    c = synth.coeffs(7, (4, 5, 16))
    assert c.max() < (1 << 16)
    # explicit-index regeneration agrees with the bulk generator
    rec = synth.raw_records(7, 5, 16, [2, 3], [1, 4])
    assert np.array_equal(rec, c[np.ix_([2, 3], [1, 4])])
    idx = np.array([5, 17, 63], dtype=np.uint64)
    assert np.array_equal(synth.residues_at(7, idx, 16, qs), r.reshape(-1)[idx.astype(np.int64)])


# ------------------------------------------------------------------ parameters
def test_primes_match_page_parameters():
    P = page_params()
    N, L = P["N"], P["num_rns"]
    qs = oracle.primes(N, L, 1 << P["prime_bound_log2"])
    assert len(qs) == L
    assert qs == sorted(qs, reverse=True) and len(set(qs)) == L
    for q in qs:
        assert sympy.isprime(q)
        assert q % (2 * N) == 1
        assert q < (1 << P["prime_bound_log2"])
    # they are the largest such primes: no prime = 1 mod 2N lies above the smallest one
    lo = qs[-1]
    cands = [x for x in range(lo, 1 << 29, 2 * N) if sympy.isprime(x)]
    assert sorted(cands, reverse=True) == qs
    # q = q0*q1*q2 is about 2^87
    assert abs(math.log2(math.prod(qs)) - P["log2_q_approx"]) < 0.5
    # lazy reduction claim: 32 products of residues below 2^29 fit a 64-bit accumulator
    assert P["lazy_terms"] * (max(qs) - 1) ** 2 < (1 << 64)


def test_primes_small_bound_brute_force():
    for N, bound in [(16, 5000), (64, 100000)]:
        want = sorted([x for x in range(2, bound) if x % (2 * N) == 1 and sympy.isprime(x)],
                      reverse=True)[:4]
        assert oracle.primes(N, 4, bound) == want
        for q in want:
            assert oracle.is_prime(q)
        assert not oracle.is_prime(want[0] * 3)


def test_psi_is_smallest_primitive_root():
    for N, q in [(4096, 536813569), (4096, 536690689), (4096, 536641537), (16, 4513), (64, 7937)]:
        psi = oracle.min_psi(q, N)
        assert pow(psi, N, q) == q - 1
        assert sympy.n_order(psi, q) == 2 * N
        # independent construction: all primitive 2N-th roots are g^((q-1)/2N * odd)
        g = sympy.primitive_root(q)
        base = pow(g, (q - 1) // (2 * N), q)
        roots = [pow(base, e, q) for e in range(1, 2 * N, 2)]
        assert psi == min(roots)


def test_powmod_invmod():
    q = 536813569
    for a in [1, 2, 12345, q - 1]:
        assert oracle.invmod(a, q) == pow(a, -1, q)
        assert oracle.powmod(a, 1 << 40, q) == pow(a, 1 << 40, q)


# ------------------------------------------------------------------ NTT
SMALL = [(16, 4513), (64, 7937), (256, 536813569)]


@pytest.mark.parametrize("N,q", SMALL)
def test_ntt_closed_forms(N, q):
    psi = oracle.min_psi(q, N)
    bits = N.bit_length() - 1
    one = np.zeros(N, np.uint32)
    one[0] = 1
    assert (oracle.ntt_direct(one, q, psi) == 1).all()
    for k in [1, 3, N - 1]:
        xk = np.zeros(N, np.uint32)
        xk[k] = 1
        want = [pow(psi, (2 * brv(j, bits) + 1) * k, q) for j in range(N)]
        assert oracle.ntt_direct(xk, q, psi).tolist() == want
        assert oracle.ntt_iter(xk, q, psi).tolist() == want


@pytest.mark.parametrize("N,q", SMALL)
def test_ntt_is_evaluation_at_odd_roots(N, q):
    """out[j] = a(psi^(2 brv(j)+1)): polynomial evaluation by sympy."""
    psi = oracle.min_psi(q, N)
    bits = N.bit_length() - 1
    rng = np.random.default_rng(N)
    a = rng.integers(0, q, N, dtype=np.uint64).astype(np.uint32)
    x = sympy.symbols("x")
    poly = sympy.Poly(list(reversed([int(v) for v in a])), x, modulus=q)
    out = oracle.ntt_direct(a, q, psi)
    for j in [0, 1, N // 2, N - 1]:
        root = pow(psi, 2 * brv(j, bits) + 1, q)
        assert int(poly.eval(root)) % q == int(out[j])


@pytest.mark.parametrize("N,q", SMALL + [(4096, 536641537)])
def test_ntt_iter_equals_direct_and_inverts(N, q):
    psi = oracle.min_psi(q, N)
    rng = np.random.default_rng(q)
    a = rng.integers(0, q, N, dtype=np.uint64).astype(np.uint32)
    d = oracle.ntt_direct(a, q, psi)
    assert np.array_equal(oracle.ntt_iter(a, q, psi), d)
    assert np.array_equal(oracle.intt_iter(d, q, psi), a)
    if N <= 256:
        assert np.array_equal(oracle.intt_direct(d, q, psi), a)
        assert np.array_equal(oracle.ntt_direct(oracle.intt_direct(a, q, psi), q, psi), a)


def _negacyclic_numpy(a, b, q):
    """Linear convolution by numpy (exact, object dtype), folded with X^N = -1."""
    N = len(a)
    full = np.convolve(np.array(a, dtype=object), np.array(b, dtype=object))
    c = [0] * N
    for t, v in enumerate(full):
        if t < N:
            c[t] += v
        else:
            c[t - N] -= v
    return [int(v) % q for v in c]


@pytest.mark.parametrize("N,q", SMALL)
def test_schoolbook_against_numpy_convolution(N, q):
    rng = np.random.default_rng(N + 1)
    a = rng.integers(0, q, N, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, q, N, dtype=np.uint64).astype(np.uint32)
    assert oracle.negacyclic_mul(a, b, q).tolist() == _negacyclic_numpy(a, b, q)
    # X^k * a is a negacyclic shift (closed form)
    k = 3
    xk = np.zeros(N, np.uint32)
    xk[k] = 1
    want = [(int(a[t - k]) if t >= k else (q - int(a[t - k + N])) % q) for t in range(N)]
    assert oracle.negacyclic_mul(xk, a, q).tolist() == want


@pytest.mark.parametrize("N,q", SMALL + [(4096, 536813569)])
def test_ntt_convolution_theorem(N, q):
    """INTT(NTT(a) . NTT(b)) = a*b in Z_q[X]/(X^N+1)   (VIPIR 2.3)."""
    psi = oracle.min_psi(q, N)
    rng = np.random.default_rng(2 * N + 3)
    a = rng.integers(0, q, N, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, 1 << 16, N, dtype=np.uint64).astype(np.uint32)
    pw = (oracle.ntt_iter(a, q, psi).astype(np.uint64) * oracle.ntt_iter(b, q, psi)) % q
    prod = oracle.intt_iter(pw.astype(np.uint32), q, psi)
    want = oracle.negacyclic_mul(a, b, q) if N <= 256 else np.array(_negacyclic_numpy(a, b, q))
    assert np.array_equal(prod, np.asarray(want, dtype=np.uint32))


def test_ntt_polys_batched_matches_rows():
    N, qs = 64, [7937, 7681]
    psis = [oracle.min_psi(q, N) for q in qs]
    polys = synth.residues(3, (5, 2, N), qs)
    fw = oracle.ntt_polys(polys, qs, psis)
    for i in range(5):
        for l in range(2):
            assert np.array_equal(fw[i, l], oracle.ntt_direct(polys[i, l], qs[l], psis[l]))
    assert np.array_equal(oracle.ntt_polys(fw, qs, psis, inverse=True), polys)


def test_encode_records_lift_and_transform():
    N, qs = 64, [7937, 7681]
    psis = [oracle.min_psi(q, N) for q in qs]
    raw = synth.coeffs(4, (3, N)) % 7000           # below both primes
    enc = oracle.encode_records(raw, qs, psis)
    for r in range(3):
        for l in range(2):
            assert np.array_equal(enc[r, l], oracle.ntt_direct(raw[r], qs[l], psis[l]))
    const = np.full((1, N), 0, np.uint32)
    const[0, 0] = 1234
    assert (oracle.encode_records(const, qs, psis) == 1234).all()


# ------------------------------------------------------------------ RowSel
def _tiny_rowsel_setup(seed, N=16, qs=(4513, 4481), D0=3, D1=2, B=2):
    qs = list(qs)
    psis = [oracle.min_psi(q, N) for q in qs]
    raw = synth.coeffs(seed, (D0, D1, N)) % min(qs)
    db = oracle.encode_records(raw, qs, psis)                  # [D0][D1][L][N]
    query = synth.residues(seed, (B, D0, 2, len(qs), N), qs)   # NTT form
    return qs, psis, raw, db, query


def test_rowsel_bruteforce_python_ints():
    qs, psis, raw, db, query = _tiny_rowsel_setup(11)
    B, D0, _, L, N = query.shape
    D1 = db.shape[1]
    out = oracle.rowsel(db, query, qs)
    for b in range(B):
        for n in range(D1):
            for c in range(2):
                for l in range(L):
                    for j in range(N):
                        s = sum(int(query[b, k, c, l, j]) * int(db[k, n, l, j]) for k in range(D0))
                        assert out[b, n, c, l, j] == s % qs[l]


def test_rowsel_d0_one_is_negacyclic_product():
    """D0 = 1: each output polynomial is query_c * record in R_q (schoolbook)."""
    qs, psis, raw, db, query = _tiny_rowsel_setup(12, N=64, qs=(7937, 7681), D0=1, D1=3, B=1)
    out = oracle.rowsel(db, query, qs)
    qcoef = oracle.ntt_polys(query, qs, psis, inverse=True)
    ocoef = oracle.ntt_polys(out, qs, psis, inverse=True)
    for n in range(3):
        for c in range(2):
            for l in range(2):
                want = oracle.negacyclic_mul(qcoef[0, 0, c, l], raw[0, n] % qs[l], qs[l])
                assert np.array_equal(ocoef[0, n, c, l], want)


def test_rowsel_one_hot_selects_record():
    """One-hot query (row i* holds ct = (1, 0), the rest (0, 0)) returns DB[i*][n] exactly."""
    N, qs, D0, D1 = 64, [7937, 7681], 5, 4
    qs_, psis, raw, db, _ = _tiny_rowsel_setup(13, N=N, qs=qs, D0=D0, D1=D1, B=1)
    for istar in [0, 3]:
        query = np.zeros((1, D0, 2, 2, N), np.uint32)
        query[0, istar, 0] = 1                       # NTT of the constant 1 is all ones
        out = oracle.rowsel(db, query, qs)
        assert np.array_equal(out[0, :, 0], db[istar])
        assert (out[0, :, 1] == 0).all()
        coef = oracle.ntt_polys(out, qs, psis, inverse=True)
        for l in range(2):
            assert np.array_equal(coef[0, :, 0, l], raw[istar])


def test_rowsel_max_residues_closed_form():
    """All inputs q-1: sum of D0 products (q-1)^2 = 1 mod q, so out = D0 mod q."""
    N, qs, D0, D1, B = 16, [536813569, 536690689], 1024, 2, 1
    L = len(qs)
    qcol = np.array(qs, np.uint32).reshape(1, 1, L, 1)
    db = np.broadcast_to(qcol - 1, (D0, D1, L, N)).copy()
    query = np.broadcast_to(np.array(qs, np.uint32).reshape(1, 1, 1, L, 1) - 1,
                            (B, D0, 2, L, N)).copy()
    out = oracle.rowsel(db, query, qs)
    for l in range(L):
        assert (out[..., l, :] == D0 % qs[l]).all()


def test_rowsel_linear_and_column_subset():
    qs, psis, raw, db, query = _tiny_rowsel_setup(14, D1=5, B=1)
    q2 = synth.residues(15, query.shape, qs)
    qarr = np.array(qs, np.uint64).reshape(1, 1, 1, -1, 1)
    s = ((query.astype(np.uint64) + q2) % qarr).astype(np.uint32)
    o1, o2, o3 = oracle.rowsel(db, query, qs), oracle.rowsel(db, q2, qs), oracle.rowsel(db, s, qs)
    qa = np.array(qs, np.uint64).reshape(1, 1, 1, -1, 1)
    assert np.array_equal(o3, ((o1.astype(np.uint64) + o2) % qa).astype(np.uint32))
    cols = np.array([4, 0, 2], np.uint32)
    assert np.array_equal(oracle.rowsel(db, query, qs, cols=cols), o1[:, cols.astype(int)])


def test_encode_records_lifts_full_32bit_words():
    """Plain 32-bit words (the scan output that becomes G, the hint that
    becomes H) are lifted as integers: the transform of w equals the sum of
    the transforms of its base-2^16 halves, w = lo + 2^16 hi, mod q."""
    N, qs = 64, [7937, 7681]
    psis = [oracle.min_psi(q, N) for q in qs]
    w = synth.words(21, (3, N))
    w[0, :4] = [0xFFFFFFFF, 0x80000000, 7937, 7681 * 7937]
    lo, hi = w & 0xFFFF, w >> 16
    e, elo, ehi = (oracle.encode_records(a, qs, psis) for a in (w, lo, hi))
    for l, q in enumerate(qs):
        want = (elo[:, l].astype(np.int64) + (1 << 16) % q * ehi[:, l].astype(np.int64)) % q
        assert np.array_equal(e[:, l], want)
        # and the constant term of the inverse is the word itself mod q
        back = oracle.ntt_polys(e, qs, psis, inverse=True)
        assert np.array_equal(back[:, l], (w.astype(np.int64) % q).astype(np.uint32))


# ------------------------------------------------------------------ ExpPack GEMM
def _tiny_exppack(seed, N=16, qs=(4513, 4481), Dr=3, n=4, B=2):
    qs = list(qs)
    L = len(qs)
    H = synth.residues(seed, (Dr, n, L, N), qs)
    C = synth.residues(seed + 1, (B, n, 2, L, N), qs)
    G = synth.residues(seed + 2, (B, Dr, L, N), qs)
    return qs, H, C, G


def test_exppack_bruteforce_python_ints():
    """out[b][r][c] = sum_k H[r][k] C[b][k][c] + [c == 1] G[b][r], point-wise mod q."""
    qs, H, C, G = _tiny_exppack(31)
    Dr, n, L, N = H.shape
    B = C.shape[0]
    out = oracle.exppack(H, C, G, qs)
    assert out.shape == (B, Dr, 2, L, N)
    for b in range(B):
        for r in range(Dr):
            for c in range(2):
                for l in range(L):
                    for j in range(N):
                        s = sum(int(H[r, k, l, j]) * int(C[b, k, c, l, j]) for k in range(n))
                        s += int(G[b, r, l, j]) if c == 1 else 0
                        assert out[b, r, c, l, j] == s % qs[l]


def test_exppack_zero_specials_returns_zero_and_g():
    """C = 0 leaves the trivial ciphertexts (0, G_b) for every hint row."""
    qs, H, C, G = _tiny_exppack(32)
    out = oracle.exppack(H, np.zeros_like(C), G, qs)
    assert (out[:, :, 0] == 0).all()
    assert np.array_equal(out[:, :, 1], G)


def test_exppack_packed_ciphertext_decrypts_to_g_minus_hs():
    """The packing's purpose as a closed form.  With RLWE secret z and special
    ciphertexts C_k = (a_k, -a_k z - s_k) (noise-free encryptions of -s_k,
    ciphertext (c0, c1) decrypting as c1 + c0 z), the row-r output decrypts to
    G_r - sum_k s_k H[r][k] in R_q: the LWE decryption b - <a, s> of the
    scan result, for all N coefficients at once.  Products are checked in the
    coefficient domain with the schoolbook negacyclic product."""
    N, qs, Dr, n, B = 32, [7937, 7681], 3, 5, 2
    L = len(qs)
    psis = [oracle.min_psi(q, N) for q in qs]
    rng = np.random.default_rng(33)
    Hc = rng.integers(0, 1 << 32, (Dr, n, N), dtype=np.uint64).astype(np.uint32)   # hint words
    Gc = rng.integers(0, 1 << 32, (B, Dr, N), dtype=np.uint64).astype(np.uint32)   # scan words
    z = rng.integers(0, 3, N).astype(np.int64) - 1                               # ternary secret
    s = rng.integers(0, 3, (B, n)).astype(np.int64) - 1                          # LWE secrets
    a = rng.integers(0, 1 << 20, (B, n, N)).astype(np.int64)
    C = np.zeros((B, n, 2, L, N), np.uint32)
    for l, q in enumerate(qs):
        zq = (z % q).astype(np.uint32)
        for b in range(B):
            for k in range(n):
                ak = (a[b, k] % q).astype(np.uint32)
                az = oracle.negacyclic_mul(ak, zq, q).astype(np.int64)
                c1 = (-az) % q
                c1[0] = (c1[0] - s[b, k]) % q
                C[b, k, 0, l] = ak
                C[b, k, 1, l] = c1.astype(np.uint32)
    H = oracle.encode_records(Hc, qs, psis)                  # [Dr][n][L][N]
    G = oracle.encode_records(Gc, qs, psis)                  # [B][Dr][L][N]
    Cn = oracle.ntt_polys(C, qs, psis)
    out = oracle.ntt_polys(oracle.exppack(H, Cn, G, qs), qs, psis, inverse=True)
    for l, q in enumerate(qs):
        zq = (z % q).astype(np.uint32)
        for b in range(B):
            for r in range(Dr):
                dec = (out[b, r, 1, l].astype(np.int64)
                       + oracle.negacyclic_mul(out[b, r, 0, l], zq, q)) % q
                want = Gc[b, r].astype(np.int64)
                for k in range(n):
                    want = want - s[b, k] * Hc[r, k].astype(np.int64)
                assert np.array_equal(dec, want % q)


# ------------------------------------------------------------------ scalar scan
def test_scalar_scan_against_numpy_matmul():
    R, C, B = 37, 300, 5
    db = synth.db_bytes(1, (R, C))
    Q = synth.words(1, (C, B))
    want = (db.astype(np.uint64) @ Q.astype(np.uint64)) % (1 << 32)   # exact: C*2^40 < 2^64
    assert np.array_equal(oracle.scalar_scan(db, Q), want.astype(np.uint32))


def test_scalar_scan_wraparound_closed_form():
    R, C, B = 4, 70000, 3
    db = np.full((R, C), 255, np.uint8)
    Q = np.full((C, B), 0xFFFFFFFF, np.uint32)
    assert (oracle.scalar_scan(db, Q) == (255 * 0xFFFFFFFF * C) % (1 << 32)).all()


def test_scalar_scan_one_hot_column_and_byte_split():
    R, C, B = 9, 64, 4
    db = synth.db_bytes(2, (R, C))
    Q = synth.words(2, (C, B))
    cstar = 17
    Q1 = np.zeros_like(Q)
    Q1[cstar, 2] = 1
    out = oracle.scalar_scan(db, Q1)
    assert np.array_equal(out[:, 2], db[:, cstar].astype(np.uint32)) and (out[:, [0, 1, 3]] == 0).all()
    # VIPIR 4.1 byte split: sum_i 2^(8i) * (A * B_i) = A * B  mod 2^32
    acc = np.zeros((R, B), np.uint64)
    for i in range(4):
        Bi = ((Q >> np.uint32(8 * i)) & np.uint32(0xFF)).astype(np.uint32)
        acc += oracle.scalar_scan(db, Bi).astype(np.uint64) << np.uint64(8 * i)
    assert np.array_equal((acc % (1 << 32)).astype(np.uint32), oracle.scalar_scan(db, Q))
