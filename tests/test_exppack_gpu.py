"""GPU parity: the ring-packing GEMM H*C + (0|G) and the lift + NTT of G (bit-exact).

The hint H (plain 32-bit words) is encoded with pir_db_encode as an n x Dr
grid of records (record (k, r) = H[r][k]); G (plain words) goes through
pir_lift_ntt; C holds NTT-form residues.  Small shapes are compared in full;
the 15 GiB hint of the pages' 64 GiB configuration (n = 1280, Dr = 256) is
checked on sampled hint rows, all evaluation points.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, gather_db_device, to_dev, to_host_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


@pytest.mark.parametrize("N,L,cnt", [(16, 1, 1), (64, 3, 7), (256, 2, 33), (4096, 3, 5), (2048, 2, 3)])
def test_lift_ntt_matches_oracle(pir, N, L, cnt):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    raw = synth.words((N + cnt) % 251, (cnt, N), tid=synth.T_SCAN_OUT)
    raw[0, :3] = [0xFFFFFFFF, qs[0], 0]
    out = pir.empty_u32(cnt * L * N)
    out.fill_(-1)
    pir.pir_lift_ntt(ctx, to_dev(raw), out, cnt)
    assert np.array_equal(to_host_u32(out).reshape(cnt, L, N), oracle.encode_records(raw, qs, psis))
    assert pir.pir_status(ctx) == 0


def test_lift_ntt_rejects_overlap(pir):
    qs = oracle.primes(64, 2)
    ctx = pir.pir_ctx_create(64, qs)
    buf = pir.empty_u32(4 * 2 * 64)
    with pytest.raises(pir.PirError):
        pir.pir_lift_ntt(ctx, buf[:4 * 64], buf, 4)        # in place is not allowed: sizes differ
    with pytest.raises(pir.PirError):
        pir.pir_lift_ntt(ctx, buf[1:], buf, 1)             # unaligned


def _exppack_case(pir, N, L, n, Dr, B, seed):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    hraw = synth.words(seed, (n, Dr, N), tid=synth.T_HINT)            # record (k, r) = H[r][k]
    graw = synth.words(seed, (B, Dr, N), tid=synth.T_SCAN_OUT)
    C = synth.residues(seed, (B, n, 2, L, N), qs, tid=synth.T_SPECIAL)
    h_db = pir.empty_u32(pir.pir_db_bytes(ctx, n, Dr) // 4)
    pir.pir_db_encode(ctx, to_dev(hraw), 0, n, n, Dr, h_db)
    G = pir.empty_u32(B * Dr * L * N)
    pir.pir_lift_ntt(ctx, to_dev(graw), G, B * Dr)
    out = pir.empty_u32(B * Dr * 2 * L * N)
    out.fill_(-1)
    pir.pir_exppack(ctx, h_db, n, Dr, to_dev(C), G, B, out, pir.rowsel_workspace(ctx, n, Dr, B))
    got = to_host_u32(out).reshape(B, Dr, 2, L, N)
    H = oracle.encode_records(hraw, qs, psis).transpose(1, 0, 2, 3)  # [Dr][n][L][N]
    Gn = oracle.encode_records(graw, qs, psis)                        # [B][Dr][L][N]
    assert np.array_equal(to_host_u32(G).reshape(B, Dr, L, N), Gn)
    want = oracle.exppack(H, C, Gn, qs)
    assert np.array_equal(got, want)
    assert pir.pir_status(ctx) == 0
    return ctx, h_db


@pytest.mark.parametrize("N,L,n,Dr,B", [
    (64, 3, 33, 5, 1),       # one slab, ragged width, ragged row chunk
    (16, 2, 40, 130, 3),     # two slabs (128 + 4), odd B
    (64, 2, 100, 37, 12),    # tensor-core path (B = 12 -> 24 polynomials), padded polynomials
    (16, 2, 512, 44, 16),    # tensor-core path at its largest n
    (16, 1, 9, 20, 17),      # two passes (16 + 1): G joins each pass's results
    (4096, 3, 20, 3, 2),     # the pages' ring
])
def test_exppack_small(pir, N, L, n, Dr, B):
    _exppack_case(pir, N, L, n, Dr, B, seed=(N + n + Dr + B) % 251)


def test_exppack_rejects_missing_addend(pir):
    qs = oracle.primes(64, 2)
    ctx = pir.pir_ctx_create(64, qs)
    h = pir.empty_u32(pir.pir_db_bytes(ctx, 4, 4) // 4)
    C = pir.empty_u32(4 * 2 * 2 * 64)
    out = pir.empty_u32(4 * 2 * 2 * 64)
    ws = pir.rowsel_workspace(ctx, 4, 4, 1)
    assert pir.lib().pir_exppack(ctx, h.data_ptr(), 4, 4, C.data_ptr(), None, 1, out.data_ptr(),
                                 ws.data_ptr(), ws.numel() * ws.element_size(), None) == pir.PIR_ERR_ARG
    with pytest.raises(pir.PirError):                      # unaligned G
        pir.pir_exppack(ctx, h, 4, 4, C, out[1:], 1, out, ws)


def test_exppack_full_15g_hint(pir):
    """n = 1280, Dr = 256, L = 3, N = 4096: a 15 GiB hint, one client; the
    output ciphertexts of sampled hint rows (both slabs, the last row) against
    the oracle at every evaluation point."""
    import torch
    import synth.device as sd
    N, L, n, Dr, B, seed = 4096, 3, 1280, 256, 1, 9
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    ctx = pir.pir_ctx_create(N, qs)
    h_db = torch.empty(pir.pir_db_bytes(ctx, n, Dr) // 4, dtype=torch.int32, device="cuda")
    rows = 256
    raw = torch.empty(rows * Dr * N, dtype=torch.int32, device="cuda")
    for k0 in range(0, n, rows):
        sd.fill_words(raw, seed, synth.T_HINT, idx0=k0 * Dr * N)
        pir.pir_db_encode(ctx, raw, k0, rows, n, Dr, h_db)
    del raw
    graw = torch.empty(B * Dr * N, dtype=torch.int32, device="cuda")
    sd.fill_words(graw, seed, synth.T_SCAN_OUT)
    C = torch.empty(B * n * 2 * L * N, dtype=torch.int32, device="cuda")
    sd.fill_residues(C, seed, synth.T_SPECIAL, N, qs)
    G = pir.empty_u32(B * Dr * L * N)
    pir.pir_lift_ntt(ctx, graw, G, B * Dr)
    out = pir.empty_u32(B * Dr * 2 * L * N)
    pir.pir_exppack(ctx, h_db, n, Dr, C, G, B, out, pir.rowsel_workspace(ctx, n, Dr, B))
    got = to_host_u32(out).reshape(B, Dr, 2, L, N)
    assert pir.pir_status(ctx) == 0
    rs = np.array([0, 127, 128, 255])
    hraw = synth.hint_records(seed, Dr, N, np.arange(n), rs)        # [n][len(rs)][N]
    H = oracle.encode_records(hraw, qs, psis)                        # [n][len(rs)][L][N]
    for k in (0, n - 1):                                             # the encoded hint itself
        assert np.array_equal(gather_db_device(h_db, N, L, n, Dr, [k] * len(rs), rs), H[k].reshape(len(rs), -1))
    # oracle inputs from the host generator (the device fills must agree with it)
    Gn = oracle.encode_records(synth.words(seed, (B, Dr, N), tid=synth.T_SCAN_OUT)[:, rs], qs, psis)
    Ch = synth.residues(seed, (B, n, 2, L, N), qs, tid=synth.T_SPECIAL)
    want = oracle.exppack(H.transpose(1, 0, 2, 3), Ch, Gn, qs)
    assert np.array_equal(got[:, rs], want)
    del h_db
    torch.cuda.empty_cache()
