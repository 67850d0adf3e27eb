"""Host check of the tensor-core RowSel epilogue's modular reduction.

The kernel reduces W = sum_j 2^(8j) S_j mod q, where the S_j are the exact
integer sums of one query digit plane i against the four DB byte planes
over a K segment of at most 512 rows (|S_j| <= 128 * 255 * 512 for i, j < 3;
the top query digit (<= 32) bounds plane 3, the top byte of a residue
below q bounds S_3), without 64-bit arithmetic.  The DB bytes enter the
tensor cores as fp16 subnormals b * 2^-24, so the accumulators hold
x_j = S_j * 2^-24 (exact in fp32):

    lo = sum_j t_j << 8j              (wrapping 32-bit), where t_j is
         x_j * 2^24 converted to an integer, or, for j = 3 (|S_3| < 2^22),
         the fp32 bits of x_3 + 0.75, which are 0x3F400000 + S_3
    wf = fma(x_3, 2^48, fma(x_2, 2^40, fma(x_1, 2^32, x_0 * 2^24)))   (fp32)
    kb = fp32 bits of fma(wf, fp32(1/q), 1.5 * 2^23) = 0x4B400000 + k,
         k = wf / q rounded to an integer
    r  = lo - kb*q + (q + 0x4B400000*q - the magic offset in lo)
         (wrapping 32-bit; equals W - k*q + q, which must lie in [0, 2^32))
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


MAGIC = 12582912.0          # 1.5 * 2^23
MAGIC_BITS = 0x4B400000
SMAGIC = 0.75               # 1.5 * 2^-1
SMAGIC_BITS = 0x3F400000
M32 = 0xFFFFFFFF


def _scaled(S):
    """The accumulator value S * 2^-24 as fp32 (exact for |S| < 2^24)."""
    S = np.asarray(S, dtype=np.int64)
    assert (np.abs(S) < 1 << 24).all()
    x = _f32(S.astype(np.float64) / float(1 << 24))
    assert (x.astype(np.float64) * float(1 << 24) == S).all()
    return x


def _smagic_bits(S):
    """fp32 bits of S * 2^-24 + 0.75 for integers |S| <= 2^22 (then 0x3F400000 + S)."""
    S = np.asarray(S, dtype=np.int64)
    assert (np.abs(S) <= 1 << 22).all()
    x = _scaled(S)
    bits = _f32(x.astype(np.float64) + SMAGIC).view(np.uint32).astype(np.int64)
    assert (bits == SMAGIC_BITS + S).all()
    return bits


def epilogue_reduce(S, q, plane=0, strict=True):
    """The kernel's reduction of digit plane `plane` for S of shape [..., 4] (int64):
    the 32-bit value r that goes into the Shoup product.  A quotient outside
    the magic conversion's range fails the call (strict) or gives r = -1."""
    S = np.asarray(S, dtype=np.int64)
    lo = np.zeros(S.shape[:-1], dtype=np.int64)
    wf = np.zeros(S.shape[:-1], dtype=np.float32)
    for j in range(4):
        x = _scaled(S[..., j])
        if j == 3:
            t = _smagic_bits(S[..., j])
        else:   # __float2int_rn(x * 2^24): the product is exact, so the conversion returns S
            t = np.rint(x.astype(np.float64) * float(1 << 24)).astype(np.int64) & M32
        lo = (lo + (t << (8 * j))) & M32
        # fmaf(x, 2^(8j+24), wf): exact product and sum in float64 (< 2^53), one rounding to fp32
        wf = _f32(x.astype(np.float64) * float(1 << (8 * j + 24)) + wf.astype(np.float64))
    qinv = np.float32(1.0) / np.float32(q)
    # fmaf(wf, qinv, 1.5 * 2^23): the product is exact in float64 and the result lies in
    # [2^23, 2^24), where fp32 steps by 1, so its one rounding is that of wf*qinv to an integer
    k = np.rint(wf.astype(np.float64) * np.float64(qinv)).astype(np.int64)
    k_ok = np.abs(k) < 1 << 22
    assert k_ok.all() or not strict
    kb = MAGIC_BITS + k
    off = (SMAGIC_BITS << 24) & M32
    rc = (q + MAGIC_BITS * q - off) & M32
    return np.where(k_ok, (lo - kb * q + rc) & M32, -1)


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
        r = epilogue_reduce(S4[..., i, :], q, plane=i)
        assert (r > 0).all() and (r < 1 << 31).all()
        u = shoup(r, pow(2, 8 * i, q), q)
        assert (u < 2 * q).all()
        x = x + u
    assert (x < 8 * q).all()
    for c in (4, 2, 1):
        x = np.minimum(x, (x - c * q) & M32)     # x - cq wraps above x when x < cq
    return x


def _bounds(q, D0, plane):
    """Largest |S_j| of digit plane `plane` over D0 rows: query digits |d| <= 128
    (the top digit of a residue below q: <= (q - 1 + 0x808080) >> 24), DB bytes
    <= 255 (the top byte: <= (q - 1) >> 24)."""
    d = 128 if plane < 3 else (q - 1 + 0x808080) >> 24
    top = (q - 1) >> 24
    return np.array([d * 255 * D0, d * 255 * D0, d * 255 * D0, d * top * D0], dtype=np.int64)


def _sums(b, rng, n):
    """Every sign pattern of the extreme partial sums, a third of them, then random values."""
    corners = np.array([[s0, s1, s2, s3] for s0 in (-1, 1) for s1 in (-1, 1) for s2 in (-1, 1) for s3 in (-1, 1)])
    return np.concatenate([corners * b, (corners * b) // 3, rng.integers(-b, b + 1, size=(n, 4), dtype=np.int64)])


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
    D0 = 512                                                         # rows of one K segment
    rng = np.random.default_rng(q & 0xFFFF)
    pw = np.int64(1) << (8 * np.arange(4, dtype=np.int64))
    for plane in range(4):
        S = _sums(_bounds(q, D0, plane), rng, 50000)
        W = (S * pw).sum(axis=1)
        r = epilogue_reduce(S, q, plane)
        # r is congruent to W (so W - kq + q did not leave [0, 2^32)), positive and below 3q
        assert (np.mod(r - W, q) == 0).all() and (r > 0).all() and (r < 3 * q).all(), plane
    # the whole output path on groups of four planes
    S4 = np.stack([_sums(_bounds(q, D0, i), rng, 4000)[:4000] for i in range(4)], axis=1)   # [g][i][j]
    W4 = (S4 * pw).sum(axis=2)
    want = np.array([sum(int(W4[g, i]) << (8 * i) for i in range(4)) % q for g in range(W4.shape[0])])
    got = epilogue_output(S4, q)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (q, got[bad[:5]], want[bad[:5]])


def test_top_byte_sums_fit_the_magic_conversion():
    """The fp32 magic-constant conversion (x + 0.75 with ulp 2^-24) is exact only
    for |S| <= 2^22: every query digit plane against the top DB byte (<= 31 for
    residues below 2^29) over 512 rows stays below it; the other byte planes reach
    2^24 and take the exact conversion, and every sum stays below 2^24 (exact
    accumulators and exact scaling)."""
    q = oracle.primes(4096, 1)[0]
    assert q < 1 << 29
    assert max(_bounds(q, 512, i)[3] for i in range(4)) < 1 << 22
    assert _bounds(q, 512, 0)[0] >= 1 << 22          # the lower byte planes need the exact conversion
    assert max(_bounds(q, 512, i).max() for i in range(4)) < 1 << 24


def test_reduction_needs_the_prime_bound():
    """Below the bound the quotient estimate fails: with q just below 2^16
    some sums inside the same bounds have a quotient beyond the magic
    conversion's range or one off by more than one, which is why passes with
    smaller primes take the CUDA-core kernel."""
    q = oracle.primes(16, 1, bound=1 << 16)[0]
    D0 = 512
    b = np.array([128 * 255 * D0] * 3 + [0], dtype=np.int64)
    S = np.random.default_rng(5).integers(-b, b + 1, size=(20000, 4), dtype=np.int64)
    W = (S * (np.int64(1) << (8 * np.arange(4, dtype=np.int64)))).sum(axis=1)
    r = epilogue_reduce(S, q, strict=False)
    assert ((r < 0) | (np.mod(r - W, q) != 0) | (r <= 0) | (r >= 3 * q)).any()
