"""GPU parity: ExpandQuery (automorphism, Subs, expansion stages) against the
oracle, bit-exact.

Random evaluation keys and ciphertexts (seeded residues) for single stages at
several ring sizes, stage indices and ciphertext counts; whole expansions;
the 1024-ciphertext expansion that feeds a D0 = 1024 RowSel; and, with a
ternary secret and noise-free keys, the decryption of the GPU's outputs:
ciphertext r carries coefficient r of the query plaintext times 2^S.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import ensure_built, to_dev, to_host_u32
from tests.test_expand_oracle import Keys, _signed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


def _setup(pir, N, L):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    return pir.pir_ctx_create(N, qs), qs, psis


@pytest.mark.parametrize("N,L,ell,w,j,M", [
    (4096, 3, 5, 18, 0, 1),
    (4096, 3, 5, 18, 3, 8),
    (4096, 3, 5, 18, 11, 3),    # the last stage a 4096-ring has
    (4096, 2, 4, 15, 5, 2),
    (256, 2, 4, 15, 2, 5),
    (64, 3, 5, 18, 5, 4),
    (16, 1, 1, 29, 1, 3),
    (4096, 4, 6, 20, 2, 3),     # four primes: Q ~ 2^116
])
def test_stage_matches_oracle(pir, N, L, ell, w, j, M):
    ctx, qs, psis = _setup(pir, N, L)
    evk = synth.residues(60 + j, (ell, 2, L, N), qs)
    cts = synth.residues(70 + M, (M, 2, L, N), qs)
    out = pir.empty_u32(2 * M * 2 * L * N)
    out.fill_(-1)
    pir.pir_expand_stage(ctx, to_dev(evk), ell, w, j, to_dev(cts), M, out, pir.expand_workspace(ctx, M, ell))
    got = to_host_u32(out).reshape(2 * M, 2, L, N)
    assert np.array_equal(got, oracle.expand_stage(evk, cts, j, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("N,L,S", [(4096, 3, 1), (4096, 3, 4), (256, 2, 6)])
def test_expansion_matches_oracle(pir, N, L, S):
    ell, w = (5, 18) if L == 3 else (4, 15)
    ctx, qs, psis = _setup(pir, N, L)
    evks = synth.residues(90 + S, (S, ell, 2, L, N), qs)
    ct = synth.residues(100 + S, (2, L, N), qs)
    out = pir.empty_u32((1 << S) * 2 * L * N)
    pir.pir_expand(ctx, to_dev(evks), ell, w, S, to_dev(ct), out, pir.expand_workspace(ctx, 1 << (S - 1), ell))
    got = to_host_u32(out).reshape(1 << S, 2, L, N)
    assert np.array_equal(got, oracle.expand(evks, ct, S, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


def test_expansion_full_size(pir):
    """1024 ciphertexts (10 stages), the RowSel input of a D0 = 1024 DB."""
    N, L, ell, w, S = 4096, 3, 5, 18, 10
    ctx, qs, psis = _setup(pir, N, L)
    evks = synth.residues(120, (S, ell, 2, L, N), qs)
    ct = synth.residues(121, (2, L, N), qs)
    out = pir.empty_u32((1 << S) * 2 * L * N)
    pir.pir_expand(ctx, to_dev(evks), ell, w, S, to_dev(ct), out, pir.expand_workspace(ctx, 1 << (S - 1), ell))
    got = to_host_u32(out).reshape(1 << S, 2, L, N)
    assert np.array_equal(got, oracle.expand(evks, ct, S, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("N,S", [(4096, 10), (64, 6)])
def test_expansion_decrypts_to_coefficients(pir, N, S):
    """Noise-free keys under a ternary secret: the GPU's output r decrypts to
    2^S * sum_{t = r mod 2^S} m_t X^(t - r)."""
    L, ell, w = 3, 5, 18
    K = Keys(N, L, ell, w, seed=S + N)
    ctx = pir.pir_ctx_create(N, K.qs)
    coeffs = K.rng.integers(-300, 300, size=N)
    ct = K.encrypt(_signed(coeffs, K.qs))
    evks = np.stack([K.evk(N // (1 << j) + 1) for j in range(S)])
    out = pir.empty_u32((1 << S) * 2 * L * N)
    pir.pir_expand(ctx, to_dev(evks), ell, w, S, to_dev(ct), out, pir.expand_workspace(ctx, 1 << (S - 1), ell))
    got = to_host_u32(out).reshape(1 << S, 2, L, N)
    for r in sorted({0, 1, 5, (1 << S) - 1, (1 << S) // 3}):
        want = np.zeros(N, dtype=np.int64)
        for t in range(r, N, 1 << S):
            want[t - r] = int(coeffs[t]) << S
        assert np.array_equal(K.decrypt(got[r]), _signed(want, K.qs)), r
    assert pir.pir_status(ctx) == 0


def test_expand_rejects_bad_arguments(pir):
    import torch
    N, L = 64, 3
    ctx, qs, _ = _setup(pir, N, L)
    evk = pir.empty_u32(7 * 5 * 2 * L * N)
    cts = pir.empty_u32(2 * 2 * L * N)
    out = pir.empty_u32(8 * 2 * L * N)
    ws = pir.expand_workspace(ctx, 4, 5)
    with pytest.raises(pir.PirError):                 # j = log2 N
        pir.pir_expand_stage(ctx, evk, 5, 18, 6, cts, 2, out, ws)
    with pytest.raises(pir.PirError):                 # more stages than log2 N
        pir.pir_expand(ctx, evk, 5, 18, 7, cts, out, ws)
    with pytest.raises(pir.PirError):                 # digits do not cover Q
        pir.pir_expand_stage(ctx, evk, 5, 17, 0, cts, 2, out, ws)
    with pytest.raises(pir.PirError):                 # workspace too small
        pir.pir_expand(ctx, evk, 5, 18, 4, cts, out, ws[:64])
    with pytest.raises(pir.PirError):                 # out overlaps in
        pir.pir_expand_stage(ctx, evk, 5, 18, 0, cts, 2, cts, ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace
        pir.pir_expand_stage(ctx, evk, 5, 18, 0, cts, 2, ws[: 4 * 2 * L * N * 4].view(torch.int32), ws)
    with pytest.raises(pir.PirError):                 # in inside the workspace
        pir.pir_expand_stage(ctx, evk, 5, 18, 0, ws[: cts.numel() * 4].view(torch.int32), 2, out, ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace (whole expansion)
        pir.pir_expand(ctx, evk, 5, 18, 2, cts, ws[: 4 * 2 * L * N * 4].view(torch.int32), ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace (batch of two clients)
        pir.pir_expand_batch(ctx, evk, 5, 18, 1, cts, 2, ws[: 4 * 2 * L * N * 4].view(torch.int32), ws)
    assert pir.pir_expand_workspace_bytes(ctx, 0, 5) == 0


@pytest.mark.parametrize("N,L,S,G", [(4096, 3, 3, 3), (4096, 3, 1, 4), (256, 2, 4, 3)])
def test_batch_matches_oracle_per_client(pir, N, L, S, G):
    """G expansions in one call, each with its own query and keys, equal the
    oracle's expansion of each client; client b's outputs are contiguous."""
    ell, w = (5, 18) if L == 3 else (4, 15)
    ctx, qs, psis = _setup(pir, N, L)
    evks = synth.residues(130 + S + G, (G, S, ell, 2, L, N), qs)
    cts = synth.residues(140 + S + G, (G, 2, L, N), qs)
    out = pir.empty_u32(G * (1 << S) * 2 * L * N)
    out.fill_(-1)
    pir.pir_expand_batch(ctx, to_dev(evks), ell, w, S, to_dev(cts), G, out,
                         pir.expand_workspace(ctx, G << (S - 1), ell))
    got = to_host_u32(out).reshape(G, 1 << S, 2, L, N)
    for b in range(G):
        assert np.array_equal(got[b], oracle.expand(evks[b], cts[b], S, qs, psis, ell, w)), b
    assert pir.pir_status(ctx) == 0


def test_batch_of_16_full_size(pir):
    """16 expansions into 1024 ciphertexts each (the RowSel input of 16
    queries over the 64 GiB DB): every client equals its own single call, the
    last client equals the oracle."""
    N, L, ell, w, S, G = 4096, 3, 5, 18, 10, 16
    ctx, qs, psis = _setup(pir, N, L)
    P = L * N
    evks = synth.residues(150, (G, S, ell, 2, L, N), qs)
    cts = synth.residues(151, (G, 2, L, N), qs)
    e_dev, c_dev = to_dev(evks).reshape(-1), to_dev(cts).reshape(-1)      # flat, sliced per client
    out = pir.empty_u32(G * (1 << S) * 2 * P)
    pir.pir_expand_batch(ctx, e_dev, ell, w, S, c_dev, G, out, pir.expand_workspace(ctx, G << (S - 1), ell))
    ws = pir.expand_workspace(ctx, 1 << (S - 1), ell)
    one = pir.empty_u32((1 << S) * 2 * P)
    for b in range(G):
        pir.pir_expand(ctx, e_dev[b * S * ell * 2 * P:(b + 1) * S * ell * 2 * P], ell, w, S,
                       c_dev[b * 2 * P:(b + 1) * 2 * P], one, ws)
        assert bool((out[b * (1 << S) * 2 * P:(b + 1) * (1 << S) * 2 * P] == one).all()), b
    got = to_host_u32(out[(G - 1) * (1 << S) * 2 * P:]).reshape(1 << S, 2, L, N)
    assert np.array_equal(got, oracle.expand(evks[G - 1], cts[G - 1], S, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


def test_batch_rejects_bad_arguments(pir):
    N, L = 64, 3
    ctx, qs, _ = _setup(pir, N, L)
    evks = pir.empty_u32(2 * 3 * 5 * 2 * L * N)
    cts = pir.empty_u32(2 * 2 * L * N)
    out = pir.empty_u32(2 * 8 * 2 * L * N)
    with pytest.raises(pir.PirError):                 # G = 0
        pir.pir_expand_batch(ctx, evks, 5, 18, 3, cts, 0, out, pir.expand_workspace(ctx, 8, 5))
    with pytest.raises(pir.PirError):                 # workspace for one expansion only
        pir.pir_expand_batch(ctx, evks, 5, 18, 3, cts, 2, out, pir.expand_workspace(ctx, 4, 5))
