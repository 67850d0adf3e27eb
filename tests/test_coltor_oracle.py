"""Pins of the ColTor oracle (gadget decomposition, RGSW-RLWE external
product, tournament stage) against facts that do not come from the oracle:

* Dcp: the digits rebuild every residue as a Python big integer
  (sum_u d_u 2^(w u) = x_l mod q_l, below Q, every digit below 2^w);
* the external product with a noise-free RGSW encryption of m -- rows
  C[u] = (m g_u, 0), C[ell + u] = (0, m g_u), g_u = 2^(w u) -- is exactly
  m * ct: the identity for m = 1, a negacyclic shift for m = X^k (written
  out directly in coefficient form);
* a stage with RGSW(0) keeps the even ciphertexts, with RGSW(1) takes the
  odd ones (a missing partner counts as zero); the whole tournament with the
  bits of j* returns ct[j*];
* on tiny rings the product equals a brute-force evaluation: big-integer
  CRT digits, the O(N^2) NTT definition and the point-wise sums (two and
  four primes);
* the product is linear in C.

GPIR sections 2-3 (ColTor, Dcp, l = 5) and VIPIR 3.6 step 7 / section 5
(q ~ 2^87 in three RNS primes) are the passages these readings follow.
"""
import numpy as np
import pytest

import oracle


def _setup(N, L):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    return qs, psis


def _Q(qs):
    Q = 1
    for q in qs:
        Q *= q
    return Q


def _ntt(polys, qs, psis):
    return oracle.ntt_polys(np.ascontiguousarray(polys, dtype=np.uint32), qs, psis)


def _trivial_rgsw(m_ntt, qs, ell, w):
    """Noise-free RGSW of m (m_ntt [L][N], NTT form): Z = 0, C = m * (I_2 x g)."""
    L, N = m_ntt.shape
    C = np.zeros((2 * ell, 2, L, N), dtype=np.uint32)
    for u in range(ell):
        for l, q in enumerate(qs):
            g = pow(2, w * u, q)
            row = (m_ntt[l].astype(np.uint64) * g % q).astype(np.uint32)
            C[u, 0, l] = row
            C[ell + u, 1, l] = row
    return C


def _random_cts(rng, n, qs, N):
    L = len(qs)
    cts = np.empty((n, 2, L, N), dtype=np.uint32)
    for l, q in enumerate(qs):
        cts[:, :, l] = rng.integers(0, q, size=(n, 2, N), dtype=np.uint64).astype(np.uint32)
    return cts


@pytest.mark.parametrize("L,ell,w", [(3, 5, 18), (2, 4, 15), (1, 1, 29), (3, 3, 29), (4, 6, 20), (4, 4, 29)])
def test_dcp_rebuilds_every_residue(L, ell, w):
    N = 4096
    qs, _ = _setup(N, L)
    Q = _Q(qs)
    assert Q.bit_length() <= ell * w
    rng = np.random.default_rng(L * 100 + ell)
    x = np.empty((L, N), dtype=np.uint32)
    for l, q in enumerate(qs):
        x[l] = rng.integers(0, q, size=N, dtype=np.uint64).astype(np.uint32)
    x[:, 0] = 0                                        # X = 0
    x[:, 1] = [q - 1 for q in qs]                      # X = Q - 1
    x[:, 2] = 1                                        # X = 1
    d = oracle.dcp(x, qs, ell, w)
    assert d.shape == (ell, N) and (d.astype(np.uint64) < (1 << w)).all()
    for t in range(0, N, 7):
        X = sum(int(d[u, t]) << (w * u) for u in range(ell))
        assert X < Q
        assert all(X % q == int(x[l, t]) for l, q in enumerate(qs)), t
    assert int(d[:, 0].sum()) == 0 and int(d[0, 2]) == 1 and int(d[1:, 2].sum()) == 0
    top = sum(int(d[u, 1]) << (w * u) for u in range(ell))
    assert top == Q - 1


@pytest.mark.parametrize("N,L,ell,w", [(64, 3, 5, 18), (4096, 3, 5, 18), (256, 2, 4, 15), (64, 4, 6, 20)])
def test_ext_product_with_rgsw_of_one_is_identity(N, L, ell, w):
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(N + L)
    ct = _random_cts(rng, 1, qs, N)[0]                 # coefficient form
    one = np.ones((L, N), dtype=np.uint32)             # NTT(1): every point 1
    C = _trivial_rgsw(one, qs, ell, w)
    got = oracle.ext_product(C, ct, qs, psis, ell, w)
    assert np.array_equal(got, _ntt(ct, qs, psis))


def _negacyclic_shift(a, k, q):
    """X^k * a(X) mod X^N + 1, coefficient form, written out directly."""
    N = a.shape[-1]
    out = np.zeros_like(a)
    for t in range(N):
        s = t + k
        if s < N:
            out[..., s] = a[..., t]
        else:
            out[..., s - N] = (q - a[..., t].astype(np.int64)) % q
    return out


@pytest.mark.parametrize("k", [1, 5, 63])
def test_ext_product_with_rgsw_of_monomial_shifts(k):
    N, L, ell, w = 64, 3, 5, 18
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(k)
    ct = _random_cts(rng, 1, qs, N)[0]
    mono = np.zeros((L, N), dtype=np.uint32)
    mono[:, k] = 1
    C = _trivial_rgsw(_ntt(mono, qs, psis), qs, ell, w)
    got = oracle.ext_product(C, ct, qs, psis, ell, w)
    want = np.empty_like(ct)
    for l, q in enumerate(qs):
        want[:, l] = _negacyclic_shift(ct[:, l], k, q)
    assert np.array_equal(got, _ntt(want, qs, psis))


@pytest.mark.parametrize("n", [2, 7, 8])
def test_stage_selects_by_the_encrypted_bit(n):
    N, L, ell, w = 64, 3, 5, 18
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(n)
    cts = _random_cts(rng, n, qs, N)                   # NTT form
    zero = np.zeros((L, N), dtype=np.uint32)
    one = np.ones((L, N), dtype=np.uint32)
    keep = oracle.coltor_stage(_trivial_rgsw(zero, qs, ell, w), cts, qs, psis, ell, w)
    take = oracle.coltor_stage(_trivial_rgsw(one, qs, ell, w), cts, qs, psis, ell, w)
    assert keep.shape == ((n + 1) // 2, 2, L, N)
    assert np.array_equal(keep, cts[0::2])
    assert np.array_equal(take[: n // 2], cts[1::2])
    if n % 2:
        assert not take[-1].any()                      # the missing partner is zero


@pytest.mark.parametrize("n,jstar", [(11, 0), (11, 6), (11, 10), (16, 13), (1, 0)])
def test_tournament_returns_the_selected_ciphertext(n, jstar):
    N, L, ell, w = 16, 3, 5, 18
    qs, psis = _setup(N, L)
    cts = _random_cts(np.random.default_rng(n * 31 + jstar), n, qs, N)
    S = oracle.coltor_stages(n)
    Cs = np.stack([_trivial_rgsw(np.full((L, N), (jstar >> s) & 1, dtype=np.uint32), qs, ell, w)
                   for s in range(max(S, 1))])
    assert np.array_equal(oracle.coltor(Cs, cts, qs, psis, ell, w), cts[jstar])


@pytest.mark.parametrize("L,ell,w", [(2, 4, 15), (4, 6, 20)])   # four primes: Q ~ 2^116, Q/q_l above 2^64
def test_ext_product_brute_force_tiny(L, ell, w):
    N = 16
    qs, psis = _setup(N, L)
    Q = _Q(qs)
    assert Q.bit_length() <= ell * w
    rng = np.random.default_rng(3)
    ct = _random_cts(rng, 1, qs, N)[0]
    C = np.empty((2 * ell, 2, L, N), dtype=np.uint32)
    for l, q in enumerate(qs):
        C[:, :, l] = rng.integers(0, q, size=(2 * ell, 2, N), dtype=np.uint64).astype(np.uint32)
    got = oracle.ext_product(C, ct, qs, psis, ell, w)
    # big-integer CRT (explicit basis), digits, the O(N^2) NTT definition, point-wise sums
    basis = [(Q // q) * pow(Q // q, -1, q) for q in qs]
    want = np.zeros((2, L, N), dtype=object)
    for cin in range(2):
        X = [sum(int(ct[cin, l, t]) * basis[l] for l in range(L)) % Q for t in range(N)]
        for u in range(ell):
            digit = np.array([(X[t] >> (w * u)) & ((1 << w) - 1) for t in range(N)], dtype=np.uint64)
            for l, q in enumerate(qs):
                dn = oracle.ntt_direct((digit % q).astype(np.uint32), q, psis[l])
                for c in range(2):
                    want[c, l] += dn.astype(object) * C[cin * ell + u, c, l].astype(object)
    for l, q in enumerate(qs):
        want[:, l] %= q
    assert np.array_equal(got, want.astype(np.uint32))


def test_ext_product_is_linear_in_the_rgsw_rows():
    N, L, ell, w = 64, 3, 5, 18
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(9)
    ct = _random_cts(rng, 1, qs, N)[0]
    C1 = np.stack([_random_cts(rng, 2, qs, N)[:, 0] for _ in range(2 * ell)])     # [2ell][2][L][N]
    C2 = np.stack([_random_cts(rng, 2, qs, N)[:, 0] for _ in range(2 * ell)])
    q = np.asarray(qs, dtype=np.uint64).reshape(1, 1, L, 1)
    Cs = ((C1.astype(np.uint64) + C2) % q).astype(np.uint32)
    a = oracle.ext_product(C1, ct, qs, psis, ell, w).astype(np.uint64)
    b = oracle.ext_product(C2, ct, qs, psis, ell, w).astype(np.uint64)
    qq = np.asarray(qs, dtype=np.uint64).reshape(1, L, 1)
    assert np.array_equal(oracle.ext_product(Cs, ct, qs, psis, ell, w), ((a + b) % qq).astype(np.uint32))


def test_swapped_rows_break_the_identity():
    """A plausible indexing slip (digits of ct_0 meeting the rows of ct_1)
    fails the identity pin: the pin is sensitive to the row layout."""
    N, L, ell, w = 64, 3, 5, 18
    qs, psis = _setup(N, L)
    ct = _random_cts(np.random.default_rng(4), 1, qs, N)[0]
    C = _trivial_rgsw(np.ones((L, N), dtype=np.uint32), qs, ell, w)
    swapped = np.concatenate([C[ell:], C[:ell]])
    assert not np.array_equal(oracle.ext_product(swapped, ct, qs, psis, ell, w), _ntt(ct, qs, psis))
