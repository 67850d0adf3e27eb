"""CPU oracle for the lattice-PIR database scan (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
and its Python binding never do.  The oracle shares no code with the CUDA path.

Every function restates a definition from the pages (see oracle.c):
  * VIPIR (CSDN translation), sections 2.2-2.5, 4.1-4.3: RNS primes, the
    negacyclic NTT, the INT8 x INT32 scan mod 2^32;
  * GPIR (arXiv 2604.04696), section 2: RowSel as point-wise GEMMs
    M_out[p,m,n] = sum_k M_in0[p,m,k] * M_in1[p,k,n] mod q;
  * GPIR sections 2-3 and VIPIR 3.6 step 7: ColTor, the column tournament of
    RGSW-RLWE external products with the gadget decomposition Dcp (l = 5);
  * GPIR sections 2-3: ExpandQuery, the expansion tree of Subs operations
    (automorphism and key switching of the a polynomial);
  * GPIR section 2 (the expanded query also yields the RGSW ciphertexts of
    the column bits): the conversion of the expanded gadget ciphertexts
    RLWE'(m) into RGSW(m) with a key-switching key of s^2 (a reading).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_u32p = ctypes.POINTER(ctypes.c_uint32)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into liboracle.so (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.orc_powmod.restype = ctypes.c_uint32
        L.orc_powmod.argtypes = [ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint32]
        L.orc_invmod.restype = ctypes.c_uint32
        L.orc_invmod.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        L.orc_is_prime.restype = ctypes.c_int
        L.orc_is_prime.argtypes = [ctypes.c_uint32]
        L.orc_primes.restype = ctypes.c_int
        L.orc_primes.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _u32p]
        L.orc_min_psi.restype = ctypes.c_uint32
        L.orc_min_psi.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        L.orc_bitrev.restype = ctypes.c_uint32
        L.orc_bitrev.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        for name in ("orc_ntt_direct", "orc_intt_direct"):
            f = getattr(L, name)
            f.restype = None
            f.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p]
        for name in ("orc_ntt_iter", "orc_intt_iter"):
            f = getattr(L, name)
            f.restype = None
            f.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _u32p]
        L.orc_negacyclic_mul.restype = None
        L.orc_negacyclic_mul.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, _u32p]
        L.orc_ntt_polys.restype = None
        L.orc_ntt_polys.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint64,
                                    _u32p, _u32p, ctypes.c_int, ctypes.c_int]
        L.orc_encode_records.restype = None
        L.orc_encode_records.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p,
                                         ctypes.c_uint64, _u32p, _u32p, ctypes.c_int]
        L.orc_rowsel.restype = None
        L.orc_rowsel.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, ctypes.c_uint32,
                                 ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32,
                                 _u32p, _u32p, ctypes.c_int]
        L.orc_dcp.restype = None
        L.orc_dcp.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, ctypes.c_uint32, ctypes.c_uint32,
                              _u32p, _u32p]
        L.orc_ext_product.restype = None
        L.orc_ext_product.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32,
                                      ctypes.c_uint32, _u32p, _u32p, _u32p]
        L.orc_coltor_stage.restype = None
        L.orc_coltor_stage.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32,
                                       ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint64, _u32p, ctypes.c_int]
        L.orc_automorph.restype = None
        L.orc_automorph.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, ctypes.c_uint32, _u32p, _u32p]
        L.orc_subs.restype = None
        L.orc_subs.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32, ctypes.c_uint32,
                               ctypes.c_uint32, _u32p, _u32p, _u32p]
        L.orc_rgsw_convert.restype = None
        L.orc_rgsw_convert.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32,
                                       ctypes.c_uint32, _u32p, _u32p, _u32p]
        L.orc_expand_stage.restype = None
        L.orc_expand_stage.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint32,
                                       ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p, ctypes.c_uint64, _u32p,
                                       ctypes.c_int]
        L.orc_scalar_scan.restype = None
        L.orc_scalar_scan.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32, _u8p,
                                      _u32p, _u32p, ctypes.c_int]
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _p32(a: np.ndarray):
    assert a.dtype == np.uint32 and a.flags["C_CONTIGUOUS"], (a.dtype, a.flags)
    return a.ctypes.data_as(_u32p)


def _p8(a: np.ndarray):
    assert a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_u8p)


# --------------------------------------------------------------- parameters
def is_prime(q: int) -> bool:
    return bool(lib().orc_is_prime(q))


def primes(N: int, count: int, bound: int = 1 << 29) -> list[int]:
    """The `count` largest primes < bound with q = 1 mod 2N, descending."""
    out = np.zeros(count, dtype=np.uint32)
    n = lib().orc_primes(N, count, bound, _p32(out))
    return [int(x) for x in out[:n]]


def min_psi(q: int, N: int) -> int:
    """Smallest g with g^N = -1 mod q (a primitive 2N-th root of unity)."""
    return int(lib().orc_min_psi(q, N))


def powmod(b: int, e: int, q: int) -> int:
    return int(lib().orc_powmod(b, e, q))


def invmod(a: int, q: int) -> int:
    return int(lib().orc_invmod(a, q))


def bitrev(x: int, bits: int) -> int:
    return int(lib().orc_bitrev(x, bits))


# --------------------------------------------------------------- NTT
def ntt_direct(a: np.ndarray, q: int, psi: int) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint32)
    out = np.empty_like(a)
    lib().orc_ntt_direct(q, psi, a.size, _p32(a), _p32(out))
    return out


def intt_direct(a: np.ndarray, q: int, psi: int) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint32)
    out = np.empty_like(a)
    lib().orc_intt_direct(q, psi, a.size, _p32(a), _p32(out))
    return out


def ntt_iter(a: np.ndarray, q: int, psi: int) -> np.ndarray:
    out = np.array(a, dtype=np.uint32, copy=True, order="C")
    lib().orc_ntt_iter(q, psi, out.size, _p32(out))
    return out


def intt_iter(a: np.ndarray, q: int, psi: int) -> np.ndarray:
    out = np.array(a, dtype=np.uint32, copy=True, order="C")
    lib().orc_intt_iter(q, psi, out.size, _p32(out))
    return out


def negacyclic_mul(a: np.ndarray, b: np.ndarray, q: int) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint32)
    b = np.ascontiguousarray(b, dtype=np.uint32)
    c = np.empty_like(a)
    lib().orc_negacyclic_mul(q, a.size, _p32(a), _p32(b), _p32(c))
    return c


def ntt_polys(polys: np.ndarray, qs, psis, inverse: bool = False, threads: int | None = None) -> np.ndarray:
    """Transform an array [..., L, N] of RNS polynomials (row l uses qs[l])."""
    polys = np.ascontiguousarray(polys, dtype=np.uint32)
    L, N = polys.shape[-2], polys.shape[-1]
    cnt = polys.size // (L * N)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty_like(polys)
    lib().orc_ntt_polys(N, L, _p32(q), _p32(ps), cnt, _p32(polys), _p32(out), int(inverse),
                        threads or default_threads())
    return out


def encode_records(raw: np.ndarray, qs, psis, threads: int | None = None) -> np.ndarray:
    """raw [..., N] plain 32-bit coefficients, each lifted mod q_l -> NTT form [..., L, N]."""
    raw = np.ascontiguousarray(raw, dtype=np.uint32)
    N = raw.shape[-1]
    cnt = raw.size // N
    L = len(qs)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty(raw.shape[:-1] + (L, N), dtype=np.uint32)
    lib().orc_encode_records(N, L, _p32(q), _p32(ps), cnt, _p32(raw), _p32(out),
                             threads or default_threads())
    return out


# --------------------------------------------------------------- RowSel
def rowsel(db: np.ndarray, query: np.ndarray, qs, cols=None, threads: int | None = None) -> np.ndarray:
    """db [D0][D1][L][N], query [B][D0][2][L][N] -> out [B][len(cols)][2][L][N]."""
    db = np.ascontiguousarray(db, dtype=np.uint32)
    query = np.ascontiguousarray(query, dtype=np.uint32)
    D0, D1, L, N = db.shape
    B = query.shape[0]
    assert query.shape == (B, D0, 2, L, N), (query.shape, db.shape)
    if cols is None:
        cols = np.arange(D1, dtype=np.uint32)
    cols = np.ascontiguousarray(cols, dtype=np.uint32)
    q = np.asarray(qs, dtype=np.uint32)
    out = np.empty((B, cols.size, 2, L, N), dtype=np.uint32)
    lib().orc_rowsel(N, L, _p32(q), D0, D1, B, _p32(db), _p32(query), cols.size, _p32(cols),
                     _p32(out), threads or default_threads())
    return out


def exppack(H: np.ndarray, C: np.ndarray, G: np.ndarray, qs, threads: int | None = None) -> np.ndarray:
    """Ring-packing GEMM of expansion-based packing (VIPIR 3.5.2): out = H*C + (0|G).

    H [Dr][n][L][N], C [B][n][2][L][N], G [B][Dr][L][N] (NTT form) ->
    out [B][Dr][2][L][N] with out[b][r][c] = sum_k H[r][k] * C[b][k][c] point-wise,
    plus G[b][r] on c = 1 (the polynomial carrying the message), mod q_l.
    The product is the RowSel sum with the DB record (k, r) := H[r][k].
    """
    H = np.ascontiguousarray(H, dtype=np.uint32)
    Dr, n, L, N = H.shape
    db = np.ascontiguousarray(H.transpose(1, 0, 2, 3))           # record (k, r)
    out = rowsel(db, C, qs, threads=threads)                       # [B][Dr][2][L][N]
    q = np.asarray(qs, dtype=np.uint64).reshape(1, 1, -1, 1)
    out[:, :, 1] = ((out[:, :, 1].astype(np.uint64) + np.asarray(G, dtype=np.uint64)) % q).astype(np.uint32)
    return out


# --------------------------------------------------------------- scalar scan
def scalar_scan(db_rows: np.ndarray, Q: np.ndarray, threads: int | None = None) -> np.ndarray:
    """db_rows [R'][C] uint8, Q [C][B] uint32 -> [R'][B] uint32 (mod 2^32)."""
    db_rows = np.ascontiguousarray(db_rows, dtype=np.uint8)
    Q = np.ascontiguousarray(Q, dtype=np.uint32)
    R, C = db_rows.shape
    assert Q.shape[0] == C
    B = Q.shape[1]
    out = np.empty((R, B), dtype=np.uint32)
    lib().orc_scalar_scan(R, C, B, _p8(db_rows), _p32(Q), _p32(out), threads or default_threads())
    return out


# --------------------------------------------------------------- ColTor
def dcp(x: np.ndarray, qs, ell: int, w: int) -> np.ndarray:
    """Gadget decomposition of one RNS polynomial x [L][N] (coefficient form):
    digits [ell][N] with CRT(x[:, t]) = sum_u d[u][t] * 2^(w u)."""
    x = np.ascontiguousarray(x, dtype=np.uint32)
    L, N = x.shape
    q = np.asarray(qs, dtype=np.uint32)
    d = np.empty((ell, N), dtype=np.uint32)
    lib().orc_dcp(N, L, _p32(q), ell, w, _p32(x), _p32(d))
    return d


def ext_product(C: np.ndarray, ct: np.ndarray, qs, psis, ell: int, w: int) -> np.ndarray:
    """RGSW C [2 ell][2][L][N] (NTT form) times RLWE ct [2][L][N] (coefficient
    form) -> [2][L][N] NTT form."""
    C = np.ascontiguousarray(C, dtype=np.uint32)
    ct = np.ascontiguousarray(ct, dtype=np.uint32)
    _, _, L, N = C.shape
    assert C.shape == (2 * ell, 2, L, N) and ct.shape == (2, L, N)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty((2, L, N), dtype=np.uint32)
    lib().orc_ext_product(N, L, _p32(q), _p32(ps), ell, w, _p32(C), _p32(ct), _p32(out))
    return out


def coltor_stage(C: np.ndarray, cts: np.ndarray, qs, psis, ell: int, w: int,
                 threads: int | None = None) -> np.ndarray:
    """One tournament stage: cts [n][2][L][N] (NTT form) -> [ceil(n/2)][2][L][N],
    out_i = ct_2i + C (x) (ct_2i+1 - ct_2i), a missing partner being zero."""
    C = np.ascontiguousarray(C, dtype=np.uint32)
    cts = np.ascontiguousarray(cts, dtype=np.uint32)
    n, _, L, N = cts.shape
    assert C.shape == (2 * ell, 2, L, N)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty(((n + 1) // 2, 2, L, N), dtype=np.uint32)
    lib().orc_coltor_stage(N, L, _p32(q), _p32(ps), ell, w, _p32(C), _p32(cts), n, _p32(out),
                           threads or default_threads())
    return out


def coltor_stages(n: int) -> int:
    """Stages of a tournament over n ciphertexts: ceil(log2 n)."""
    s = 0
    while (1 << s) < n:
        s += 1
    return s


def coltor(Cs: np.ndarray, cts: np.ndarray, qs, psis, ell: int, w: int, threads: int | None = None) -> np.ndarray:
    """The whole tournament: stage s uses Cs[s]; cts [n][2][L][N] -> [2][L][N]."""
    cur = np.ascontiguousarray(cts, dtype=np.uint32)
    for s in range(coltor_stages(cur.shape[0])):
        cur = coltor_stage(Cs[s], cur, qs, psis, ell, w, threads)
    return cur[0].copy()


# --------------------------------------------------------------- ExpandQuery
def automorph(a: np.ndarray, k: int, qs) -> np.ndarray:
    """sigma_k(a) = a(X^k) for a [L][N] in coefficient form (k odd)."""
    a = np.ascontiguousarray(a, dtype=np.uint32)
    L, N = a.shape
    q = np.asarray(qs, dtype=np.uint32)
    out = np.empty_like(a)
    lib().orc_automorph(N, L, _p32(q), k, _p32(a), _p32(out))
    return out


def subs(evk: np.ndarray, ct: np.ndarray, k: int, qs, psis, ell: int, w: int) -> np.ndarray:
    """Subs(ct, k) with evk [ell][2][L][N]; ct and result [2][L][N], NTT form."""
    evk = np.ascontiguousarray(evk, dtype=np.uint32)
    ct = np.ascontiguousarray(ct, dtype=np.uint32)
    _, L, N = ct.shape
    assert evk.shape == (ell, 2, L, N)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty_like(ct)
    lib().orc_subs(N, L, _p32(q), _p32(ps), ell, w, k, _p32(evk), _p32(ct), _p32(out))
    return out


def expand_stage(evk: np.ndarray, cts: np.ndarray, j: int, qs, psis, ell: int, w: int,
                 threads: int | None = None) -> np.ndarray:
    """Stage j of the expansion: cts [M][2][L][N] -> [2M][2][L][N] (NTT form)."""
    evk = np.ascontiguousarray(evk, dtype=np.uint32)
    cts = np.ascontiguousarray(cts, dtype=np.uint32)
    M, _, L, N = cts.shape
    assert evk.shape == (ell, 2, L, N) and (1 << j) < N
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty((2 * M, 2, L, N), dtype=np.uint32)
    lib().orc_expand_stage(N, L, _p32(q), _p32(ps), ell, w, j, _p32(evk), _p32(cts), M, _p32(out),
                           threads or default_threads())
    return out


def expand(evks: np.ndarray, ct: np.ndarray, stages: int, qs, psis, ell: int, w: int,
           threads: int | None = None) -> np.ndarray:
    """ExpandQuery: one ciphertext [2][L][N] -> 2^stages ciphertexts; stage j uses evks[j]."""
    cur = np.ascontiguousarray(ct, dtype=np.uint32)[None]
    for j in range(stages):
        cur = expand_stage(evks[j], cur, j, qs, psis, ell, w, threads)
    return cur


def rgsw_convert(ksk: np.ndarray, cts: np.ndarray, qs, psis, ell: int, w: int) -> np.ndarray:
    """RGSW(m) [2 ell][2][L][N] from RLWE'(m) = cts [ell][2][L][N] (ciphertexts of
    m g_u) and the key-switching key ksk [ell][2][L][N] (ciphertexts of s^2 g_v),
    all NTT form: rows u are cts[u], rows ell + u = (0, c0_u) + sum_v
    NTT(Dcp_v(c1_u)) . ksk[v]."""
    ksk = np.ascontiguousarray(ksk, dtype=np.uint32)
    cts = np.ascontiguousarray(cts, dtype=np.uint32)
    _, _, L, N = cts.shape
    assert cts.shape == (ell, 2, L, N) and ksk.shape == (ell, 2, L, N)
    q = np.asarray(qs, dtype=np.uint32)
    ps = np.asarray(psis, dtype=np.uint32)
    out = np.empty((2 * ell, 2, L, N), dtype=np.uint32)
    lib().orc_rgsw_convert(N, L, _p32(q), _p32(ps), ell, w, _p32(ksk), _p32(cts), _p32(out))
    return out
