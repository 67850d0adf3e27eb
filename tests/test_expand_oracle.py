"""Pins of the ExpandQuery oracle (automorphism, Subs, expansion stages)
against facts that do not come from the oracle:

* sigma_k(X^t) = +-X^(t k mod 2N) written out directly; sigma_k is a ring
  homomorphism (checked with the pinned negacyclic product) and
  sigma_k . sigma_k' = sigma_(k k' mod 2N); in NTT form it permutes the slots
  (slot j holds the value at psi^(2 brv(j) + 1), so sigma_k moves slot
  pi(j) with 2 brv(pi(j)) + 1 = k (2 brv(j) + 1) mod 2N into slot j);
* with a ternary secret s, noise-free encryptions and noise-free evaluation
  keys evk[u] = (-a_u s + sigma_k(s) g_u, a_u): Dec(Subs(ct, k)) =
  sigma_k(Dec(ct)) exactly, for the Galois elements of the expansion and
  others;
* after S expansion stages, ciphertext r decrypts to
  2^S * sum_{t = r mod 2^S} m_t X^(t - r): each output carries its own
  coefficient of the query plaintext (the tree's defining property).
* with random keys and ciphertexts on a 16-point ring, Subs and whole
  expansion stages equal the definitions evaluated with Python integers
  (O(N^2) NTT and inverse, the automorphism written out, big-integer CRT
  digits), up to four primes (Q/q_l above 2^64).

GPIR sections 2-3 (ExpandQuery, Subs, evk; Subs decomposes only the a
polynomial) are the passages the oracle follows.
"""
import numpy as np
import pytest

import oracle


def _setup(N, L):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    return qs, psis


def _ntt(x, qs, psis):
    return oracle.ntt_polys(np.ascontiguousarray(x, dtype=np.uint32), qs, psis)


def _intt(x, qs, psis):
    return oracle.ntt_polys(np.ascontiguousarray(x, dtype=np.uint32), qs, psis, inverse=True)


def _qcol(qs):
    return np.asarray(qs, dtype=np.uint64).reshape(-1, 1)


def _rand(rng, qs, N, lead=()):
    out = np.empty(tuple(lead) + (len(qs), N), dtype=np.uint32)
    for l, q in enumerate(qs):
        out[..., l, :] = rng.integers(0, q, size=tuple(lead) + (N,), dtype=np.uint64).astype(np.uint32)
    return out


def _signed(v, qs):
    """[L][N] coefficient residues of a small signed polynomial."""
    return np.stack([np.asarray(v, dtype=np.int64) % q for q in qs]).astype(np.uint32)


def _mul(a, b, qs):
    return ((a.astype(np.uint64) * b) % _qcol(qs)).astype(np.uint32)


def _add(a, b, qs):
    return ((a.astype(np.uint64) + b) % _qcol(qs)).astype(np.uint32)


def _sub(a, b, qs):
    return ((a.astype(np.uint64) + _qcol(qs) - b) % _qcol(qs)).astype(np.uint32)


class Keys:
    """A ternary secret, noise-free encryption / decryption and evaluation keys (NTT form)."""

    def __init__(self, N, L, ell, w, seed):
        self.N, self.ell, self.w = N, ell, w
        self.qs, self.psis = _setup(N, L)
        self.rng = np.random.default_rng(seed)
        self.s = self.rng.integers(-1, 2, size=N)
        self.sN = _ntt(_signed(self.s, self.qs), self.qs, self.psis)

    def encrypt(self, m_coeff):
        a = _rand(self.rng, self.qs, self.N)
        c0 = _sub(_ntt(m_coeff, self.qs, self.psis), _mul(a, self.sN, self.qs), self.qs)
        return np.stack([c0, a])

    def decrypt(self, ct):
        return _intt(_add(ct[0], _mul(ct[1], self.sN, self.qs), self.qs), self.qs, self.psis)

    def evk(self, k):
        ss = _ntt(oracle.automorph(_signed(self.s, self.qs), k, self.qs), self.qs, self.psis)
        rows = []
        for u in range(self.ell):
            a = _rand(self.rng, self.qs, self.N)
            g = np.array([pow(2, self.w * u, q) for q in self.qs], dtype=np.uint64).reshape(-1, 1)
            b = _add(_sub(np.zeros_like(a), _mul(a, self.sN, self.qs), self.qs),
                     ((ss.astype(np.uint64) * g) % _qcol(self.qs)).astype(np.uint32), self.qs)
            rows.append(np.stack([b, a]))
        return np.stack(rows)


@pytest.mark.parametrize("N,k", [(16, 17), (16, 9), (64, 65), (64, 3), (64, 127), (4096, 4097), (4096, 2049)])
def test_automorphism_closed_form_and_homomorphism(N, k):
    qs, psis = _setup(N, 2)
    rng = np.random.default_rng(N + k)
    for t in (0, 1, N // 2, N - 1):
        mono = np.zeros((2, N), dtype=np.uint32)
        mono[:, t] = 1
        e = t * k % (2 * N)
        want = np.zeros((2, N), dtype=np.uint32)
        if e < N:
            want[:, e] = 1
        else:
            want[:, e - N] = [q - 1 for q in qs]
        assert np.array_equal(oracle.automorph(mono, k, qs), want)
    if N <= 64:
        a, b = _rand(rng, qs, N), _rand(rng, qs, N)
        ab = np.stack([oracle.negacyclic_mul(a[l], b[l], q) for l, q in enumerate(qs)])
        sa, sb = oracle.automorph(a, k, qs), oracle.automorph(b, k, qs)
        sab = np.stack([oracle.negacyclic_mul(sa[l], sb[l], q) for l, q in enumerate(qs)])
        assert np.array_equal(oracle.automorph(ab, k, qs), sab)
        k2 = 2 * N - 1
        assert np.array_equal(oracle.automorph(oracle.automorph(a, k, qs), k2, qs),
                              oracle.automorph(a, k * k2 % (2 * N), qs))


@pytest.mark.parametrize("k", [65, 33, 5])
def test_automorphism_permutes_ntt_slots(k):
    N = 64
    qs, psis = _setup(N, 3)
    a = _rand(np.random.default_rng(k), qs, N)
    bits = 6
    slot_of = {2 * oracle.bitrev(j, bits) + 1: j for j in range(N)}
    pi = [slot_of[(k * (2 * oracle.bitrev(j, bits) + 1)) % (2 * N)] for j in range(N)]
    want = _ntt(a, qs, psis)[:, pi]
    assert np.array_equal(_ntt(oracle.automorph(a, k, qs), qs, psis), want)


@pytest.mark.parametrize("N,L,ell,w,k", [(64, 3, 5, 18, 65), (64, 3, 5, 18, 33), (64, 3, 5, 18, 3),
                                         (256, 2, 4, 15, 129), (4096, 3, 5, 18, 4097), (64, 4, 6, 20, 17)])
def test_subs_decrypts_to_the_automorphism(N, L, ell, w, k):
    K = Keys(N, L, ell, w, seed=N + k)
    m = _signed(K.rng.integers(-1000, 1000, size=N), K.qs)
    ct = K.encrypt(m)
    assert np.array_equal(K.decrypt(ct), m)
    sub = oracle.subs(K.evk(k), ct, k, K.qs, K.psis, ell, w)
    assert np.array_equal(K.decrypt(sub), oracle.automorph(m, k, K.qs))


@pytest.mark.parametrize("N,S,support", [(64, 4, 16), (64, 3, 64), (256, 5, 256)])
def test_expansion_separates_the_coefficients(N, S, support):
    L, ell, w = 3, 5, 18
    K = Keys(N, L, ell, w, seed=S * 7 + N)
    coeffs = np.zeros(N, dtype=np.int64)
    coeffs[:support] = K.rng.integers(-500, 500, size=support)
    ct = K.encrypt(_signed(coeffs, K.qs))
    evks = np.stack([K.evk(N // (1 << j) + 1) for j in range(S)])
    out = oracle.expand(evks, ct, S, K.qs, K.psis, ell, w)
    assert out.shape == (1 << S, 2, L, N)
    for r in range(1 << S):
        want = np.zeros(N, dtype=np.int64)
        for t in range(r, N, 1 << S):
            want[t - r] = coeffs[t] << S
        assert np.array_equal(K.decrypt(out[r]), _signed(want, K.qs)), r


def _subs_brute(evk, ct, k, qs, psis, ell, w):
    """Subs(ct, k) on a tiny ring from the definitions: the O(N^2) inverse and
    forward NTT, the automorphism as t -> t k mod 2N with X^N = -1 written
    out, big-integer CRT digits, point-wise sums."""
    L, N = ct.shape[1], ct.shape[2]
    Q = 1
    for q in qs:
        Q *= q
    basis = [(Q // q) * pow(Q // q, -1, q) for q in qs]

    def coef(poly):            # [L][N] NTT form -> [L][N] Python ints, coefficient form
        return [[int(v) for v in oracle.intt_direct(poly[l], q, psis[l])] for l, q in enumerate(qs)]

    def sigma(c):              # coefficient form, per prime
        out = [[0] * N for _ in qs]
        for l, q in enumerate(qs):
            for t in range(N):
                e = t * k % (2 * N)
                if e < N:
                    out[l][e] = (out[l][e] + c[l][t]) % q
                else:
                    out[l][e - N] = (out[l][e - N] - c[l][t]) % q
        return out

    def ntt(c):                # [L][N] ints -> [L][N] uint32, NTT form
        return np.stack([oracle.ntt_direct(np.array(c[l], dtype=np.uint32), q, psis[l]) for l, q in enumerate(qs)])

    s0, s1 = sigma(coef(ct[0])), sigma(coef(ct[1]))
    X = [sum(s1[l][t] * basis[l] for l in range(L)) % Q for t in range(N)]
    acc = np.zeros((2, L, N), dtype=object)
    for u in range(ell):
        d = [(x >> (w * u)) & ((1 << w) - 1) for x in X]
        dn = ntt([[v % q for v in d] for q in qs]).astype(object)
        for c in range(2):
            acc[c] += dn * evk[u, c].astype(object)
    acc[0] += ntt(s0).astype(object)
    for l, q in enumerate(qs):
        acc[:, l] %= q
    return acc.astype(np.uint32)


@pytest.mark.parametrize("L,ell,w,k", [(2, 4, 15, 17), (2, 4, 15, 5), (3, 5, 18, 9), (4, 6, 20, 31)])
def test_subs_brute_force_tiny(L, ell, w, k):
    """Random (not noise-free) keys and ciphertexts: the oracle's Subs equals
    the definitions evaluated with Python integers."""
    N = 16
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(L * 100 + k)
    evk = _rand(rng, qs, N, (ell, 2))
    ct = _rand(rng, qs, N, (2,))
    assert np.array_equal(oracle.subs(evk, ct, k, qs, psis, ell, w), _subs_brute(evk, ct, k, qs, psis, ell, w))


@pytest.mark.parametrize("j,M", [(0, 1), (1, 3), (3, 2)])
def test_expand_stage_brute_force_tiny(j, M):
    """Stage j over M random ciphertexts: out[i] = ct_i + Subs(ct_i, N/2^j + 1)
    and out[i + M] = (ct_i - Subs) . NTT(X^(-2^j)), with X^(-2^j) written out
    as -X^(N - 2^j) and transformed by the O(N^2) definition."""
    N, L, ell, w = 16, 2, 4, 15
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(10 * j + M)
    evk = _rand(rng, qs, N, (ell, 2))
    cts = _rand(rng, qs, N, (M, 2))
    k = N // (1 << j) + 1
    mono = np.stack([oracle.ntt_direct(np.array([0] * (N - (1 << j)) + [q - 1] + [0] * ((1 << j) - 1),
                                                dtype=np.uint32), q, psis[l]) for l, q in enumerate(qs)])
    got = oracle.expand_stage(evk, cts, j, qs, psis, ell, w)
    for i in range(M):
        S = _subs_brute(evk, cts[i], k, qs, psis, ell, w)
        assert np.array_equal(got[i], _add(cts[i], S, qs)), i
        diff = _sub(cts[i], S, qs)
        assert np.array_equal(got[i + M], np.stack([_mul(diff[c], mono, qs) for c in range(2)])), i
