"""Host check of the tensor-core RowSel epilogue's modular reduction.

The kernel reduces W = sum_j 2^(8j) S_j mod q, where the S_j are the exact
integer sums of one query digit plane against the four DB byte planes
(|S_j| <= 128 * 255 * D0 for j < 3, the top byte of a residue below q
bounding S_3), without 64-bit arithmetic:

    lo = sum_j S_j << 8j              (wrapping 32-bit)
    wf = fma(S_3, 2^24, fma(S_2, 2^16, fma(S_1, 2^8, S_0)))   (fp32)
    k  = round_to_int(wf * fp32(1/q))
    r  = lo - k*q + q                 (wrapping 32-bit; must be in [0, 2^32))
    u  = Shoup product r * (2^(8i) mod q), in [0, 2q)
and the four digit planes i of one output are summed (below 8q) and
reduced by conditional subtractions of 4q, 2q and q.

This test replays those operations bit-exactly on the CPU (an fma is one
rounding of the exact float64 value, which holds all the digits here) and
checks every step's range and the final residue against the exact value,
for the largest partial sums the kernel can see and primes from 2^26 (the
smallest the kernel accepts) to 2^29.
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
    signed = ((lo.astype(np.int64) - k * q) & 0xFFFFFFFF).astype(np.int64)
    signed = np.where(signed >= 1 << 31, signed - (1 << 32), signed)        # W - k*q as signed 32-bit
    return signed + q                                                        # the kernel's r (unsigned)


def shoup(y, w, q):
    """Shoup product of 32-bit y by w < q: y*w mod q in [0, 2q)."""
    wp = (w << 32) // q
    y = np.asarray(y, dtype=object)
    return np.array([(int(v) * w - ((int(v) * wp) >> 32) * q) & 0xFFFFFFFF for v in y.ravel()],
                    dtype=np.int64).reshape(y.shape)


def epilogue_output(S4, q):
    """Full epilogue for S4 of shape [..., 4 planes, 4 byte planes]: the output residue."""
    x = np.zeros(S4.shape[:-2], dtype=np.int64)
    for i in range(4):
        r = epilogue_reduce(S4[..., i, :], q)
        assert (r > 0).all() and (r < 1 << 31).all()
        u = shoup(r, pow(2, 8 * i, q), q)
        assert (u < 2 * q).all()
        x = x + u
    assert (x < 8 * q).all()
    for c in (4, 2, 1):
        x = np.where(x >= c * q, x - c * q, x)
    return x


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
    r = epilogue_reduce(S, q)
    # r is congruent to W, positive and below 2q + 0.7q (a valid Shoup input)
    assert (np.mod(r - W, q) == 0).all() and (r > 0).all() and (r < 3 * q).all()
    # the whole output path on groups of four planes
    S4 = S[: (S.shape[0] // 4) * 4][:4000].reshape(-1, 4, 4)
    W4 = (S4 * (np.int64(1) << (8 * np.arange(4, dtype=np.int64)))).sum(axis=2)
    want = np.array([sum(int(W4[g, i]) << (8 * i) for i in range(4)) % q for g in range(W4.shape[0])])
    got = epilogue_output(S4, q)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (q, got[bad[:5]], want[bad[:5]])


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
    r = epilogue_reduce(S, q)
    assert ((np.mod(r - W, q) != 0) | (r <= 0) | (r >= 3 * q)).any()
