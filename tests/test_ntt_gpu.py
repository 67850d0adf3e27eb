"""GPU parity: batched RNS negacyclic NTT / INTT against the oracle (bit-exact)."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev, to_host_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


CASES = [(16, 2, 37), (64, 1, 5), (256, 3, 17), (1024, 2, 9), (4096, 3, 7), (4096, 2, 33)]


@pytest.mark.parametrize("N,L,cnt", CASES)
def test_ntt_fwd_inv_match_oracle(pir, N, L, cnt):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    assert pir.pir_ctx_psi(ctx) == psis
    a = synth.residues((N + L) % 251, (cnt, L, N), qs)
    want = oracle.ntt_polys(a, qs, psis)
    d_in = to_dev(a)
    d_out = pir.empty_u32(a.size)
    pir.pir_ntt_fwd(ctx, d_in, d_out, cnt)
    got = to_host_u32(d_out).reshape(a.shape)
    assert np.array_equal(got, want)
    # inverse, in place
    pir.pir_ntt_inv(ctx, d_out, d_out, cnt)
    assert np.array_equal(to_host_u32(d_out).reshape(a.shape), a)
    # inverse of arbitrary residues against the oracle inverse
    b = synth.residues((N + L + 1) % 251, (cnt, L, N), qs)
    d_b = to_dev(b)
    pir.pir_ntt_inv(ctx, d_b, d_b, cnt)
    assert np.array_equal(to_host_u32(d_b).reshape(b.shape), oracle.ntt_polys(b, qs, psis, inverse=True))
    assert pir.pir_status(ctx) == 0


def test_ntt_extreme_values_and_noop(pir):
    N, L = 4096, 3
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    a = np.broadcast_to(np.array(qs, np.uint32).reshape(1, L, 1) - 1, (2, L, N)).copy()
    a[1] = 0
    a[1, :, 0] = np.array(qs) - 1
    d = to_dev(a)
    pir.pir_ntt_fwd(ctx, d, d, 2)
    assert np.array_equal(to_host_u32(d).reshape(a.shape), oracle.ntt_polys(a, qs, psis))
    pir.pir_ntt_fwd(ctx, d, d, 0)  # cnt = 0: no-op
    with pytest.raises(pir.PirError):
        pir.pir_ntt_fwd(ctx, d.view(-1)[1:], d, 1)  # misaligned input
    assert pir.pir_status(ctx) == 0


def test_ntt_convolution_on_gpu(pir):
    """INTT(NTT(a) . NTT(b)) on the GPU equals the schoolbook product (N = 256)."""
    N, L = 256, 2
    qs = oracle.primes(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    a = synth.residues(91, (1, L, N), qs)
    b = synth.coeffs(92, (1, 1, N))
    b = np.repeat(b, L, axis=1)
    da, db = to_dev(a), to_dev(b)
    pir.pir_ntt_fwd(ctx, da, da, 1)
    pir.pir_ntt_fwd(ctx, db, db, 1)
    A = to_host_u32(da).reshape(L, N).astype(np.uint64)
    Bv = to_host_u32(db).reshape(L, N).astype(np.uint64)
    prod = (A * Bv) % np.array(qs, np.uint64).reshape(L, 1)
    dp = to_dev(prod.astype(np.uint32))
    pir.pir_ntt_inv(ctx, dp, dp, 1)
    got = to_host_u32(dp).reshape(L, N)
    for l in range(L):
        assert np.array_equal(got[l], oracle.negacyclic_mul(a[0, l], b[0, l] % qs[l], qs[l]))


def test_device_generator_matches_host():
    import torch
    import synth.device as sd
    ensure_built()
    qs = oracle.primes(4096, 3)
    t = torch.empty(3 * 4096 * 5, dtype=torch.int32, device="cuda")
    sd.fill_residues(t, 3, synth.T_QUERY, 4096, qs, idx0=4096 * 3 * 7)
    want = synth.residues(3, (12, 3, 4096), qs)[7:].reshape(-1)
    assert np.array_equal(to_host_u32(t), want)
    sd.fill_coeffs(t, 4, synth.T_DB_COEFF, idx0=123)
    assert np.array_equal(to_host_u32(t), synth.coeffs(4, (t.numel(),), offset=123))
    sd.fill_words(t, 5, synth.T_SCALAR_Q, idx0=99)
    assert np.array_equal(to_host_u32(t), synth.words(5, (t.numel(),), offset=99))
    b = torch.empty(4096, dtype=torch.uint8, device="cuda")
    sd.fill_bytes(b, 6, synth.T_SCALAR_DB, idx0=4096 * 3)
    assert np.array_equal(b.cpu().numpy(), synth.db_bytes(6, (4096,), offset=4096 * 3))
