"""Pins of the oracle's conversion of expanded gadget ciphertexts into RGSW
ciphertexts (oracle.rgsw_convert), against facts that do not come from it:

* with a ternary secret s, noise-free ciphertexts ct_u of m g_u and a
  noise-free key-switching key ksk[v] of s^2 g_v, the rows of the result
  decrypt exactly to m g_u (rows u) and to m s g_u (rows ell + u), with the
  product m s written out as a numpy convolution folded by X^N = -1;
* the result is a working RGSW ciphertext for the external product: it
  multiplies a noise-free ciphertext's plaintext by m (m = 0, 1, X^3, a
  small random polynomial), through the already pinned orc_ext_product;
* with random (not noise-free) inputs on a 16-point ring the oracle equals
  the definition evaluated with Python integers (O(N^2) inverse and forward
  NTT, big-integer CRT digits, point-wise sums), two to four primes.

The conversion is a reading: the pages say only that the expanded query
yields the RGSW ciphertexts of the column tournament (GPIR section 2).
"""
import numpy as np
import pytest

import oracle
from tests.test_expand_oracle import Keys, _intt, _qcol, _rand, _setup, _signed


def _negacyclic_np(a, b):
    """Signed product a * b in Z[X]/(X^N + 1) by numpy convolution (int64)."""
    N = len(a)
    full = np.convolve(np.asarray(a, dtype=np.int64), np.asarray(b, dtype=np.int64))
    out = full[:N].copy()
    out[: len(full) - N] -= full[N:]
    return out


def _gadget(K, u):
    return np.array([pow(2, K.w * u, q) for q in K.qs], dtype=np.uint64).reshape(-1, 1)


def _enc_scaled(K, m_signed, u):
    """Noise-free ciphertext of m g_u (m a small signed coefficient vector)."""
    m = (_signed(m_signed, K.qs).astype(np.uint64) * _gadget(K, u)) % _qcol(K.qs)
    return K.encrypt(m.astype(np.uint32))


def _ksk(K):
    s2 = _negacyclic_np(K.s, K.s)
    return np.stack([_enc_scaled(K, s2, v) for v in range(K.ell)])


@pytest.mark.parametrize("N,L,ell,w", [(64, 3, 5, 18), (256, 2, 4, 15), (64, 4, 6, 20), (4096, 3, 5, 18)])
def test_rows_decrypt_to_m_g_and_m_s_g(N, L, ell, w):
    K = Keys(N, L, ell, w, seed=N + L)
    for m in (np.eye(1, N, 0, dtype=np.int64)[0], np.eye(1, N, 5, dtype=np.int64)[0],
              K.rng.integers(-3, 4, size=N)):
        cts = np.stack([_enc_scaled(K, m, u) for u in range(ell)])
        C = oracle.rgsw_convert(_ksk(K), cts, K.qs, K.psis, ell, w)
        ms = _negacyclic_np(m, K.s)
        for u in range(ell):
            g = _gadget(K, u)
            assert np.array_equal(C[u], cts[u])
            want_u = ((_signed(m, K.qs).astype(np.uint64) * g) % _qcol(K.qs)).astype(np.uint32)
            want_s = ((_signed(ms, K.qs).astype(np.uint64) * g) % _qcol(K.qs)).astype(np.uint32)
            assert np.array_equal(K.decrypt(C[u]), want_u), u
            assert np.array_equal(K.decrypt(C[ell + u]), want_s), u


@pytest.mark.parametrize("N,L,ell,w", [(64, 3, 5, 18), (256, 3, 5, 18)])
def test_converted_rgsw_multiplies_in_the_external_product(N, L, ell, w):
    K = Keys(N, L, ell, w, seed=3 * N)
    ksk = _ksk(K)
    msg = K.rng.integers(-1000, 1000, size=N)
    ct = K.encrypt(_signed(msg, K.qs))
    ct_coef = np.stack([_intt(ct[c], K.qs, K.psis) for c in range(2)])
    for m in (np.zeros(N, dtype=np.int64), np.eye(1, N, 0, dtype=np.int64)[0], np.eye(1, N, 3, dtype=np.int64)[0],
              K.rng.integers(-2, 3, size=N)):
        cts = np.stack([_enc_scaled(K, m, u) for u in range(ell)])
        C = oracle.rgsw_convert(ksk, cts, K.qs, K.psis, ell, w)
        out = oracle.ext_product(C, ct_coef, K.qs, K.psis, ell, w)
        assert np.array_equal(K.decrypt(out), _signed(_negacyclic_np(m, msg), K.qs))


def _convert_brute(ksk, cts, qs, psis, ell, w):
    L, N = cts.shape[2], cts.shape[3]
    Q = 1
    for q in qs:
        Q *= q
    basis = [(Q // q) * pow(Q // q, -1, q) for q in qs]

    def ntt(c):
        return np.stack([oracle.ntt_direct(np.array(c[l], dtype=np.uint32), q, psis[l]) for l, q in enumerate(qs)])

    out = np.zeros((2 * ell, 2, L, N), dtype=np.uint32)
    for u in range(ell):
        out[u] = cts[u]
        c1 = [[int(v) for v in oracle.intt_direct(cts[u, 1, l], q, psis[l])] for l, q in enumerate(qs)]
        X = [sum(c1[l][t] * basis[l] for l in range(L)) % Q for t in range(N)]
        acc = np.zeros((2, L, N), dtype=object)
        acc[1] += cts[u, 0].astype(object)
        for v in range(ell):
            d = [(x >> (w * v)) & ((1 << w) - 1) for x in X]
            dn = ntt([[x % q for x in d] for q in qs]).astype(object)
            for c in range(2):
                acc[c] += dn * ksk[v, c].astype(object)
        for l, q in enumerate(qs):
            acc[:, l] %= q
        out[ell + u] = acc.astype(np.uint32)
    return out


@pytest.mark.parametrize("L,ell,w", [(2, 4, 15), (3, 5, 18), (4, 6, 20)])
def test_brute_force_tiny(L, ell, w):
    N = 16
    qs, psis = _setup(N, L)
    rng = np.random.default_rng(40 + L)
    ksk = _rand(rng, qs, N, (ell, 2))
    cts = _rand(rng, qs, N, (ell, 2))
    assert np.array_equal(oracle.rgsw_convert(ksk, cts, qs, psis, ell, w), _convert_brute(ksk, cts, qs, psis, ell, w))
