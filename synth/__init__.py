"""Seeded synthetic inputs for the lattice-PIR scan (host side).

A counter-based generator: element ``idx`` of input tensor ``tid`` under seed
``seed`` is

    v = splitmix64((tid << 56) ^ (seed << 48) ^ idx)

where splitmix64(x) is the output function of Steele, Lea and Flood's
SplitMix64 ("Fast splittable pseudorandom number generators", OOPSLA 2014)
applied to the state x + 0x9E3779B97F4A7C15.  Any element can be regenerated
on its own, so the oracle can rebuild one record of a 64 GiB database without
holding it.  The device half (synth.cu) implements the same function.

Derived values (the workloads' value distributions):
  * DB coefficient   v & 0xFFFF          uniform in [0, 2^16)
  * RNS residue      v mod q_l           uniform mod q_l (bias < 2^-34)
  * DB byte          v & 0xFF            uniform in [0, 256)
  * query word       v >> 32             uniform over Z_2^32

This module holds no arithmetic of the PIR method itself.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids
T_DB_COEFF = 1     # raw DB polynomial coefficients [D0][D1][N]
T_QUERY = 2        # query ciphertexts [B][D0][2][L][N]
T_SCALAR_DB = 3    # scalar-HE DB bytes [R][C]
T_SCALAR_Q = 4     # scalar-HE query words [C][B]
T_EXTRA = 5        # anything else a test needs
T_HINT = 6         # ring-packing hint words, record order [n][Dr][N] (record (k, r) = H[r][k])
T_SCAN_OUT = 7     # INT32 scan results read as polynomials [B][Dr][N]
T_SPECIAL = 8      # expanded special ciphertexts [B][n][2][L][N] (NTT form)


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output for state x + golden gamma (vectorised, uint64)."""
    z = np.asarray(x, dtype=np.uint64) + GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def keys(seed: int, tid: int, idx) -> np.ndarray:
    assert 0 <= seed < 256 and 0 <= tid < 256
    idx = np.asarray(idx, dtype=np.uint64)
    return (np.uint64(tid) << np.uint64(56)) ^ (np.uint64(seed) << np.uint64(48)) ^ idx


def values(seed: int, tid: int, idx) -> np.ndarray:
    return splitmix64(keys(seed, tid, idx))


def _flat_idx(shape, offset=0):
    n = int(np.prod(shape)) if len(shape) else 1
    return np.arange(offset, offset + n, dtype=np.uint64).reshape(shape)


def coeffs(seed: int, shape, offset: int = 0, tid: int = T_DB_COEFF) -> np.ndarray:
    """Polynomial coefficients uniform in [0, 2^16), uint32."""
    v = values(seed, tid, _flat_idx(shape, offset))
    return (v & np.uint64(0xFFFF)).astype(np.uint32)


def residues(seed: int, shape, qs, offset: int = 0, tid: int = T_QUERY) -> np.ndarray:
    """RNS residues for an array whose last two axes are [L][N]; row l is mod qs[l]."""
    L, N = shape[-2], shape[-1]
    assert L == len(qs)
    idx = _flat_idx(shape, offset)
    v = values(seed, tid, idx)
    l = (idx // np.uint64(N)) % np.uint64(L)
    qv = np.asarray(qs, dtype=np.uint64)[l.astype(np.int64)]
    return (v % qv).astype(np.uint32)


def residues_at(seed: int, idx: np.ndarray, N: int, qs, tid: int = T_QUERY) -> np.ndarray:
    """Residues for explicit flat indices of an [..., L, N] array."""
    idx = np.asarray(idx, dtype=np.uint64)
    v = values(seed, tid, idx)
    l = (idx // np.uint64(N)) % np.uint64(len(qs))
    qv = np.asarray(qs, dtype=np.uint64)[l.astype(np.int64)]
    return (v % qv).astype(np.uint32)


def coeffs_at(seed: int, idx: np.ndarray, tid: int = T_DB_COEFF) -> np.ndarray:
    v = values(seed, tid, np.asarray(idx, dtype=np.uint64))
    return (v & np.uint64(0xFFFF)).astype(np.uint32)


def db_bytes(seed: int, shape, offset: int = 0, tid: int = T_SCALAR_DB) -> np.ndarray:
    v = values(seed, tid, _flat_idx(shape, offset))
    return (v & np.uint64(0xFF)).astype(np.uint8)


def words(seed: int, shape, offset: int = 0, tid: int = T_SCALAR_Q) -> np.ndarray:
    v = values(seed, tid, _flat_idx(shape, offset))
    return (v >> np.uint64(32)).astype(np.uint32)


def raw_records(seed: int, D1: int, N: int, ks, ns) -> np.ndarray:
    """Coefficients of DB records (k, n) for k in ks, n in ns: shape [len(ks)][len(ns)][N].

    Record (k, n) of a D0 x D1 DB occupies flat indices ((k*D1 + n)*N + t).
    """
    ks = np.asarray(ks, dtype=np.uint64).reshape(-1, 1, 1)
    ns = np.asarray(ns, dtype=np.uint64).reshape(1, -1, 1)
    t = np.arange(N, dtype=np.uint64).reshape(1, 1, -1)
    idx = (ks * np.uint64(D1) + ns) * np.uint64(N) + t
    return coeffs_at(seed, idx)


def words_at(seed: int, idx: np.ndarray, tid: int) -> np.ndarray:
    """The 32-bit words of tensor `tid` at the given flat indices (same values as `words`)."""
    v = values(seed, tid, np.asarray(idx, dtype=np.uint64))
    return (v >> np.uint64(32)).astype(np.uint32)


def hint_records(seed: int, Dr: int, N: int, ks, rs) -> np.ndarray:
    """Hint polynomials H[r][k] (plain words) for k in ks, r in rs: [len(ks)][len(rs)][N].

    Record (k, r) of the n x Dr hint grid occupies flat indices ((k*Dr + r)*N + t).
    """
    ks = np.asarray(ks, dtype=np.uint64).reshape(-1, 1, 1)
    rs = np.asarray(rs, dtype=np.uint64).reshape(1, -1, 1)
    t = np.arange(N, dtype=np.uint64).reshape(1, 1, -1)
    return words_at(seed, (ks * np.uint64(Dr) + rs) * np.uint64(N) + t, T_HINT)
