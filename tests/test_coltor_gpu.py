"""GPU parity: ColTor (gadget decomposition, RGSW-RLWE external product,
tournament stages) against the oracle, bit-exact.

Random RGSW rows and ciphertexts (seeded residues) at several ring sizes and
gadget shapes, odd ciphertext counts (the missing partner is zero), stages
of a few pairs and of several hundred (grids past one CTA per SM), the whole
tournament, the 1365-ciphertext list one 64 GiB RowSel query produces, the
noise-free selection of ct[j*] at that size, and batches of tournaments
(one per client) in one call.
"""
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


def _setup(pir, N, L):
    qs = oracle.primes(N, L)
    psis = [oracle.min_psi(q, N) for q in qs]
    return pir.pir_ctx_create(N, qs), qs, psis


def _trivial_rgsw(bit, qs, N, ell, w):
    """Noise-free RGSW of a constant bit, NTT form: C[u] = (bit g_u, 0), C[ell+u] = (0, bit g_u)."""
    L = len(qs)
    C = np.zeros((2 * ell, 2, L, N), dtype=np.uint32)
    for u in range(ell):
        for l, q in enumerate(qs):
            C[u, 0, l] = C[ell + u, 1, l] = bit * pow(2, w * u, q)
    return C


@pytest.mark.parametrize("N,L,ell,w,n", [
    (4096, 3, 5, 18, 2),
    (4096, 3, 5, 18, 7),      # odd: the last ciphertext meets zero
    (4096, 3, 3, 29, 16),     # fewer, wider digits
    (256, 2, 4, 15, 9),
    (64, 1, 1, 29, 5),        # one prime, one digit: Dcp is the identity
    (16, 2, 16, 4, 3),        # many narrow digits (the top ones zero)
    # several hundred pairs: grids past one CTA per SM
    (4096, 3, 5, 18, 333),    # odd count
    (4096, 3, 3, 29, 400),
    (4096, 2, 4, 15, 400),
    (4096, 1, 1, 29, 400),
    (4096, 3, 16, 6, 320),    # sixteen digits
    (4096, 4, 6, 20, 5),      # four primes: Q ~ 2^116, Q/q_l above 2^64
    (256, 4, 4, 29, 9),
])
def test_stage_matches_oracle(pir, N, L, ell, w, n):
    ctx, qs, psis = _setup(pir, N, L)
    C = synth.residues(100 + n % 97, (2 * ell, 2, L, N), qs)
    cts = synth.residues(200 + n % 53, (n, 2, L, N), qs)
    out = pir.empty_u32(((n + 1) // 2) * 2 * L * N)
    out.fill_(-1)
    pir.pir_coltor_stage(ctx, to_dev(C), ell, w, to_dev(cts), n, out, pir.coltor_workspace(ctx, n, ell))
    got = to_host_u32(out).reshape((n + 1) // 2, 2, L, N)
    assert np.array_equal(got, oracle.coltor_stage(C, cts, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("n", [1, 2, 37])
def test_tournament_matches_oracle(pir, n):
    N, L, ell, w = 4096, 3, 5, 18
    ctx, qs, psis = _setup(pir, N, L)
    S = oracle.coltor_stages(n)
    Cs = synth.residues(30 + n, (max(S, 1), 2 * ell, 2, L, N), qs)
    cts = synth.residues(80 + n, (n, 2, L, N), qs)
    out = pir.empty_u32(2 * L * N)
    pir.pir_coltor(ctx, to_dev(Cs), ell, w, to_dev(cts), n, out, pir.coltor_workspace(ctx, n, ell))
    got = to_host_u32(out).reshape(2, L, N)
    assert np.array_equal(got, oracle.coltor(Cs, cts, qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


def test_tournament_full_size(pir):
    """The 1365 ciphertexts of one 64 GiB RowSel query (D1 = 1365): 11 stages,
    random RGSW rows, compared with the oracle; then noise-free RGSW bits of
    j* = 1000 select ct[1000] exactly."""
    import torch
    N, L, ell, w, n = 4096, 3, 5, 18, 1365
    ctx, qs, psis = _setup(pir, N, L)
    S = oracle.coltor_stages(n)
    assert S == 11
    Cs = synth.residues(51, (S, 2 * ell, 2, L, N), qs)
    cts = synth.residues(52, (n, 2, L, N), qs)
    cts_d = to_dev(cts)
    ws = pir.coltor_workspace(ctx, n, ell)
    out = pir.empty_u32(2 * L * N)
    pir.pir_coltor(ctx, to_dev(Cs), ell, w, cts_d, n, out, ws)
    assert np.array_equal(to_host_u32(out).reshape(2, L, N), oracle.coltor(Cs, cts, qs, psis, ell, w))
    jstar = 1000
    sel = np.stack([_trivial_rgsw((jstar >> s) & 1, qs, N, ell, w) for s in range(S)])
    out2 = torch.empty_like(out)
    pir.pir_coltor(ctx, to_dev(sel), ell, w, cts_d, n, out2, ws)
    assert np.array_equal(to_host_u32(out2).reshape(2, L, N), cts[jstar])
    assert pir.pir_status(ctx) == 0


def test_coltor_rejects_bad_arguments(pir):
    import torch
    N, L = 64, 3
    ctx, qs, _ = _setup(pir, N, L)
    C = pir.empty_u32(2 * 5 * 2 * L * N)
    cts = pir.empty_u32(4 * 2 * L * N)
    out = pir.empty_u32(2 * 2 * L * N)
    ws = pir.coltor_workspace(ctx, 4, 5)
    with pytest.raises(pir.PirError):                 # 5 digits of 17 bits do not cover Q ~ 2^87
        pir.pir_coltor_stage(ctx, C, 5, 17, cts, 4, out, ws)
    with pytest.raises(pir.PirError):                 # ell = 0
        pir.pir_coltor_stage(ctx, C, 0, 18, cts, 4, out, ws)
    with pytest.raises(pir.PirError):                 # workspace too small
        pir.pir_coltor_stage(ctx, C, 5, 18, cts, 4, out, ws[:64])
    with pytest.raises(pir.PirError):                 # out overlaps in
        pir.pir_coltor_stage(ctx, C, 5, 18, cts, 4, cts, ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace
        pir.pir_coltor_stage(ctx, C, 5, 18, cts, 4, ws[: out.numel() * 4].view(torch.int32), ws)
    with pytest.raises(pir.PirError):                 # in inside the workspace
        pir.pir_coltor_stage(ctx, C, 5, 18, ws[: cts.numel() * 4].view(torch.int32), 4, out, ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace (whole tournament)
        pir.pir_coltor(ctx, C, 5, 18, cts, 4, ws[: (out.numel() // 2) * 4].view(torch.int32), ws)
    with pytest.raises(pir.PirError):                 # n = 0
        pir.pir_coltor(ctx, C, 5, 18, cts, 0, out, ws)
    assert pir.pir_coltor_workspace_bytes(ctx, 0, 5) == 0


def test_graph_replay_matches_eager(pir):
    """A pir_coltor / pir_expand call captured into a CUDA graph and replayed
    gives the eager call's results (the bench replays such graphs)."""
    import torch
    N, L, ell, w = 4096, 3, 5, 18
    ctx, qs, _ = _setup(pir, N, L)
    stream = torch.cuda.Stream()
    n = 300
    S = oracle.coltor_stages(n)
    Cs = to_dev(synth.residues(61, (S, 2 * ell, 2, L, N), qs))
    cts = to_dev(synth.residues(62, (n, 2, L, N), qs))
    ws = pir.coltor_workspace(ctx, n, ell)
    eager, replay = pir.empty_u32(2 * L * N), pir.empty_u32(2 * L * N)
    pir.pir_coltor(ctx, Cs, ell, w, cts, n, eager, ws, stream)
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        pir.pir_coltor(ctx, Cs, ell, w, cts, n, replay, ws, stream)
    replay.fill_(-1)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(replay, eager)
    Sx = 7
    evks = to_dev(synth.residues(63, (Sx, ell, 2, L, N), qs))
    ct = to_dev(synth.residues(64, (2, L, N), qs))
    wsx = pir.expand_workspace(ctx, 1 << (Sx - 1), ell)
    e_out, r_out = pir.empty_u32((1 << Sx) * 2 * L * N), pir.empty_u32((1 << Sx) * 2 * L * N)
    pir.pir_expand(ctx, evks, ell, w, Sx, ct, e_out, wsx, stream)
    g2 = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g2, stream=stream):
        pir.pir_expand(ctx, evks, ell, w, Sx, ct, r_out, wsx, stream)
    r_out.fill_(-1)
    with torch.cuda.stream(stream):
        g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(r_out, e_out)
    assert pir.pir_status(ctx) == 0


@pytest.mark.parametrize("N,L,ell,w,n,G", [
    (4096, 3, 5, 18, 11, 3),     # odd n: every tournament's last pair meets zero
    (4096, 3, 5, 18, 2, 4),
    (256, 2, 4, 15, 9, 3),       # the operation-level path (N != 4096)
    (4096, 3, 5, 18, 1, 2),      # no stage: a copy per client
])
def test_batch_matches_oracle_per_client(pir, N, L, ell, w, n, G):
    """G tournaments in one call, each with its own RGSW ciphertexts, equal
    the oracle's tournament of each client on its own inputs."""
    ctx, qs, psis = _setup(pir, N, L)
    S = oracle.coltor_stages(n)
    Cs = synth.residues(40 + n + G, (G, max(S, 1), 2 * ell, 2, L, N), qs)
    cts = synth.residues(90 + n + G, (G, n, 2, L, N), qs)
    out = pir.empty_u32(G * 2 * L * N)
    out.fill_(-1)
    C_dev = to_dev(np.ascontiguousarray(Cs[:, :S])) if S else to_dev(Cs)
    pir.pir_coltor_batch(ctx, C_dev, ell, w, to_dev(cts), n, G, out,
                         pir.coltor_batch_workspace(ctx, n, G, ell))
    got = to_host_u32(out).reshape(G, 2, L, N)
    for b in range(G):
        assert np.array_equal(got[b], oracle.coltor(Cs[b, :max(S, 1)], cts[b], qs, psis, ell, w)), b
    assert pir.pir_status(ctx) == 0


def test_batch_of_16_full_size(pir):
    """16 tournaments over 1365 ciphertexts (a 16-query RowSel output of the
    64 GiB DB): every client equals its own single-tournament call, and the
    last client equals the oracle."""
    N, L, ell, w, n, G = 4096, 3, 5, 18, 1365, 16
    ctx, qs, psis = _setup(pir, N, L)
    S = oracle.coltor_stages(n)
    P = L * N
    Cs = synth.residues(61, (G, S, 2 * ell, 2, L, N), qs)
    cts = synth.residues(62, (G, n, 2, L, N), qs)
    C_dev, cts_dev = to_dev(Cs).reshape(-1), to_dev(cts).reshape(-1)      # flat, sliced per client
    out = pir.empty_u32(G * 2 * P)
    pir.pir_coltor_batch(ctx, C_dev, ell, w, cts_dev, n, G, out, pir.coltor_batch_workspace(ctx, n, G, ell))
    got = to_host_u32(out).reshape(G, 2, L, N)
    ws = pir.coltor_workspace(ctx, n, ell)
    one = pir.empty_u32(2 * P)
    for b in range(G):
        pir.pir_coltor(ctx, C_dev[b * S * 2 * ell * 2 * P:(b + 1) * S * 2 * ell * 2 * P], ell, w,
                       cts_dev[b * n * 2 * P:(b + 1) * n * 2 * P], n, one, ws)
        assert np.array_equal(got[b], to_host_u32(one).reshape(2, L, N)), b
    assert np.array_equal(got[G - 1], oracle.coltor(Cs[G - 1], cts[G - 1], qs, psis, ell, w))
    assert pir.pir_status(ctx) == 0


def test_batch_rejects_bad_arguments(pir):
    import torch
    N, L = 64, 3
    ctx, qs, _ = _setup(pir, N, L)
    C = pir.empty_u32(2 * 10 * 2 * L * N)
    cts = pir.empty_u32(2 * 4 * 2 * L * N)
    out = pir.empty_u32(2 * 2 * L * N)
    ws = pir.coltor_batch_workspace(ctx, 4, 2, 5)
    with pytest.raises(pir.PirError):                 # G = 0
        pir.pir_coltor_batch(ctx, C, 5, 18, cts, 4, 0, out, ws)
    with pytest.raises(pir.PirError):                 # workspace for one tournament only
        pir.pir_coltor_batch(ctx, C, 5, 18, cts, 4, 2, out, pir.coltor_workspace(ctx, 4, 5))
    with pytest.raises(pir.PirError):                 # out overlaps in
        pir.pir_coltor_batch(ctx, C, 5, 18, cts, 4, 2, cts[8 * L * N:], ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace
        pir.pir_coltor_batch(ctx, C, 5, 18, cts, 4, 2, ws[: out.numel() * 4].view(torch.int32), ws)
    assert pir.pir_coltor_batch_workspace_bytes(ctx, 4, 0, 5) == 0
    assert pir.pir_coltor_batch_workspace_bytes(ctx, 4, 1, 5) == pir.pir_coltor_workspace_bytes(ctx, 4, 5)
