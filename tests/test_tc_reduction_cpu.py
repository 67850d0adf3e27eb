"""Host check of the tensor-core RowSel epilogue's modular reduction.

The kernel reduces W = sum_j 2^(8j) S_j mod q, where the S_j are the exact
integer sums of one query digit plane against the four DB byte planes
(|S_j| <= 128 * 255 * D0 for j < 3, the top byte of a residue below q
bounding S_3), without 64-bit arithmetic:

    lo = sum_j S_j << 8j              (wrapping 32-bit)
    wf = fma(S_3, 2^24, fma(S_2, 2^16, fma(S_1, 2^8, S_0)))   (fp32)
    k  = round_to_int(wf * fp32(1/q))
    r  = lo - k*q (signed 32-bit), + q if negative, - q if >= q

This test replays those fp32 operations bit-exactly on the CPU (an fma is
one rounding of the exact float64 value, which holds all the digits here)
and checks r == W mod q for the largest partial sums the kernel can see,
for primes from 2^26 (the smallest the kernel accepts) to 2^29.
"""
import numpy as np
import pytest

import oracle


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def epilogue_reduce(S, q):
    """The kernel's reduction for an array S of shape [..., 4] (int64)."""
    S = np.asarray(S, dtype=np.int64)
    lo = np.zeros(S.shape[:-1], dtype=np.uint64)
    wf = np.zeros(S.shape[:-1], dtype=np.float32)
    for j in range(4):
        lo = (lo + ((S[..., j].astype(np.uint64) & 0xFFFFFFFF) << np.uint64(8 * j))) & np.uint64(0xFFFFFFFF)
        # fmaf(x, 2^(8j), wf): exact product and sum in float64 (< 2^53), one rounding to fp32
        wf = _f32(S[..., j].astype(np.float64) * float(1 << (8 * j)) + wf.astype(np.float64))
    qinv = np.float32(1.0) / np.float32(q)
    k = np.rint((wf * qinv).astype(np.float32)).astype(np.int64)          # __float2int_rn
    r = ((lo.astype(np.int64) - k * q) & 0xFFFFFFFF).astype(np.int64)
    r = np.where(r >= 1 << 31, r - (1 << 32), r)                            # signed 32-bit
    r = np.where(r < 0, r + q, r)
    r = np.where(r >= q, r - q, r)
    return r


def _bounds(q, D0):
    top = (q - 1) >> 24
    return np.array([128 * 255 * D0, 128 * 255 * D0, 128 * 255 * D0, 128 * top * D0], dtype=np.int64)


@pytest.mark.parametrize("q", [None, "min", "mid", "max"])
def test_reduction_exact_on_extremes(q):
    N = 4096
    if q is None:
        q = oracle.primes(N, 1, bound=(1 << 26) + (1 << 22))[0]     # just above 2^26
    elif q == "min":
        q = oracle.primes(N, 1, bound=(1 << 26) + (1 << 24))[0]
    elif q == "mid":
        q = oracle.primes(N, 1, bound=1 << 28)[0]
    else:
        q = oracle.primes(N, 1)[0]                                   # largest below 2^29
    assert q >= 1 << 26
    D0 = 512
    b = _bounds(q, D0)
    rng = np.random.default_rng(q & 0xFFFF)
    # every sign pattern of the extreme partial sums, then random values inside the bounds
    corners = np.array([[s0, s1, s2, s3] for s0 in (-1, 1) for s1 in (-1, 1) for s2 in (-1, 1) for s3 in (-1, 1)])
    S = np.concatenate([corners * b, (corners * b) // 3,
                        rng.integers(-b, b + 1, size=(200000, 4), dtype=np.int64)])
    W = (S * (np.int64(1) << (8 * np.arange(4, dtype=np.int64)))).sum(axis=1)
    want = np.mod(W, q)
    got = epilogue_reduce(S, q)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (q, S[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_reduction_needs_the_prime_bound():
    """Below the bound the quotient estimate can be off by more than one:
    with q just below 2^16, some sums inside the same bounds are reduced
    wrongly (a fraction of a percent), which is why passes with smaller
    primes take the CUDA-core kernel."""
    q = oracle.primes(16, 1, bound=1 << 16)[0]
    D0 = 512
    b = np.array([128 * 255 * D0] * 3 + [0], dtype=np.int64)
    S = np.random.default_rng(5).integers(-b, b + 1, size=(20000, 4), dtype=np.int64)
    W = (S * (np.int64(1) << (8 * np.arange(4, dtype=np.int64)))).sum(axis=1)
    assert (epilogue_reduce(S, q) != np.mod(W, q)).any()
