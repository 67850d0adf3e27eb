"""GPU parity of pir_rgsw_convert (RGSW ciphertexts from the expanded gadget
ciphertexts) against oracle.rgsw_convert, bit for bit: random inputs and
keys, several clients with their own keys, N = 4096 (the library's 4096-point
kernels) and smaller rings (the generic ones), two to four primes; and the
host-side argument checks."""
import numpy as np
import pytest

import oracle
from tests.helpers import ensure_built, to_dev, to_host_u32
from tests.test_expand_oracle import _rand, _setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pir():
    ensure_built()
    from lattice_he_database_gb300 import pir as p
    return p


@pytest.mark.parametrize("N,L,ell,w,n,G,pad", [(4096, 3, 5, 18, 3, 2, 0), (4096, 3, 5, 18, 11, 1, 0),
                                               (4096, 3, 5, 18, 2, 3, 7), (256, 2, 4, 15, 2, 3, 0),
                                               (256, 2, 4, 15, 2, 3, 5), (64, 4, 6, 20, 1, 1, 0),
                                               (16, 2, 4, 15, 5, 2, 0)])
def test_convert_matches_oracle(pir, N, L, ell, w, n, G, pad):
    """pad > 0: client b's gadget ciphertexts start at b (n ell + pad)
    (a strided input, as a batched expansion's output is)."""
    qs, psis = _setup(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    rng = np.random.default_rng(N + n + G + pad)
    ksk = _rand(rng, qs, N, (G, ell, 2))
    cts = _rand(rng, qs, N, (G, n, ell, 2))
    stride = n * ell + pad
    src = _rand(rng, qs, N, (G, stride, 2))
    src[:, : n * ell] = cts.reshape(G, n * ell, 2, L, N)
    out = pir.empty_u32(G * n * 2 * ell * 2 * L * N)
    out.fill_(-1)
    pir.pir_rgsw_convert(ctx, to_dev(ksk), ell, w, to_dev(src), n, G, out, pir.rgsw_convert_workspace(ctx, n, G, ell),
                         in_stride=stride if pad else 0)
    got = to_host_u32(out).reshape(G, n, 2 * ell, 2, L, N)
    assert pir.pir_status(ctx) == 0
    for b in range(G):
        for r in sorted({0, n - 1}):
            assert np.array_equal(got[b, r], oracle.rgsw_convert(ksk[b], cts[b, r], qs, psis, ell, w)), (b, r)


def test_convert_rejects_bad_arguments(pir):
    import torch
    N, L, ell = 64, 3, 5
    qs, _ = _setup(N, L)
    ctx = pir.pir_ctx_create(N, qs)
    ksk = pir.empty_u32(ell * 2 * L * N)
    cts = pir.empty_u32(2 * ell * 2 * L * N)
    out = pir.empty_u32(2 * 2 * ell * 2 * L * N)
    ws = pir.rgsw_convert_workspace(ctx, 2, 1, ell)
    with pytest.raises(pir.PirError):                 # digits do not cover Q
        pir.pir_rgsw_convert(ctx, ksk, ell, 17, cts, 2, 1, out, ws)
    with pytest.raises(pir.PirError):                 # n = 0
        pir.pir_rgsw_convert(ctx, ksk, ell, 18, cts, 0, 1, out, ws)
    with pytest.raises(pir.PirError):                 # workspace too small
        pir.pir_rgsw_convert(ctx, ksk, ell, 18, cts, 2, 1, out, ws[:64])
    with pytest.raises(pir.PirError):                 # out overlaps in
        pir.pir_rgsw_convert(ctx, ksk, ell, 18, cts, 2, 1, cts, ws)
    with pytest.raises(pir.PirError):                 # out inside the workspace
        pir.pir_rgsw_convert(ctx, ksk, ell, 18, cts, 2, 1, ws[: out.numel() * 4].view(torch.int32), ws)
    with pytest.raises(pir.PirError):                 # client stride below n ell
        pir.pir_rgsw_convert(ctx, ksk, ell, 18, cts, 2, 1, out, ws, in_stride=2 * ell - 1)
    assert pir.pir_rgsw_convert_workspace_bytes(ctx, 0, 1, ell) == 0
    assert pir.pir_rgsw_convert_workspace_bytes(ctx, 2, 0, ell) == 0
