"""Shared setup for the parity tests: workloads, device inputs, oracle samples."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# The workloads (N = 4096; the largest primes < 2^29 with q = 1 mod 8192).
PRIMES3 = oracle.primes(4096, 3)
CONFIGS = {
    "tiny": dict(N=4096, L=2, D0=16, D1=16, B=1, query_domain="ntt"),
    "rowsel_6g": dict(N=4096, L=3, D0=256, D1=512, B=1, query_domain="ntt"),
    "rowsel_24g_b16": dict(N=4096, L=3, D0=512, D1=1024, B=16, query_domain="ntt"),
    "rowsel_64g": dict(N=4096, L=3, D0=1024, D1=1365, B=1, query_domain="coeff"),
    "rowsel_64g_b16": dict(N=4096, L=3, D0=1024, D1=1365, B=16, query_domain="ntt"),
}
SCALAR = dict(R=131072, C=131072, B=64)


def primes_for(N, L):
    return oracle.primes(N, L)


def psis_for(N, qs):
    return [oracle.min_psi(q, N) for q in qs]


def ensure_built():
    from lattice_he_database_gb300 import build as b
    import synth.device as sd
    b.build()
    sd.build()
    oracle.build()


def to_dev(a: np.ndarray, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    if a.dtype == np.uint8:
        return torch.from_numpy(a).to(device)
    raise TypeError(a.dtype)


def to_host_u32(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def make_device_db(ctx, D0, D1, seed, chunk_rows=None):
    """Generate raw records on the device (seeded) and encode them; returns the DB tensor."""
    import torch
    import synth.device as sd
    from lattice_he_database_gb300 import pir
    N = ctx.N
    nbytes = pir.pir_db_bytes(ctx, D0, D1)
    db = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    if chunk_rows is None:
        chunk_rows = max(1, min(D0, (1 << 30) // (D1 * N * 4)))
    raw = torch.empty(chunk_rows * D1 * N, dtype=torch.int32, device="cuda")
    for k0 in range(0, D0, chunk_rows):
        kc = min(chunk_rows, D0 - k0)
        r = raw[: kc * D1 * N]
        sd.fill_coeffs(r, seed, synth.T_DB_COEFF, idx0=k0 * D1 * N)
        pir.pir_db_encode(ctx, r, k0, kc, D0, D1, db)
    del raw
    return db


def oracle_db_columns(qs, psis, N, D0, D1, seed, cols):
    """Oracle NTT-form records for all rows k and the given columns: [D0][len(cols)][L][N]."""
    raw = synth.raw_records(seed, D1, N, np.arange(D0), cols)
    return oracle.encode_records(raw, qs, psis)


def gather_db_device(db_t, N, L, D0, D1, ks, ns):
    """Read encoded-DB words for all points p and the given (k, n) pairs: [len][L*N]."""
    import torch
    from lattice_he_database_gb300 import pir
    P = L * N
    p = np.arange(P).reshape(1, P)
    off = pir.db_layout_offset(N, L, D0, D1, p, np.asarray(ks).reshape(-1, 1), np.asarray(ns).reshape(-1, 1))
    idx = torch.from_numpy(off.reshape(-1)).to(db_t.device)
    return db_t[idx].cpu().numpy().view(np.uint32).reshape(len(ks), P)
