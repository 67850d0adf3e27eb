// ntt_core.cuh — negacyclic NTT of rows held in shared memory.
//
// VIPIR section 2.3: the NTT of each row of the L x N residue matrix turns a
// product in Z_q[X]/(X^N+1) into a point-wise product mod q_i; section 4.3:
// for N = 2^12 the whole transform fits on chip, so one kernel does it.
//
// Forward: in-place Cooley-Tukey on natural-order input with twiddles
// psi^brv(m+i), giving out[j] = sum_t a[t] psi^((2 brv(j)+1) t) (bit-reversed
// order).  Inverse: Gentleman-Sande with psi^-brv(m+i), natural-order output,
// then the factor N^-1.  Butterflies use Shoup products with Harvey's lazy
// ranges: forward values live in [0, 4q), inverse values in [0, 2q); q < 2^29
// keeps 4q below 2^32.  The 4096-point forward rounds go further (see
// fwd_round16).  Twiddles are read as {w, Shoup companion} pairs, one 8-byte
// load per butterfly.
//
// Stages are processed three at a time in registers: a thread loads 8
// elements spaced by the smallest butterfly distance of the round, runs the
// three butterfly levels, and writes them back; rounds are separated by
// __syncthreads.
#pragma once

#include "common.cuh"

// Forward CT butterfly, Harvey form: x, y in [0, 4q) -> [0, 4q).
__device__ __forceinline__ void ct_bfly(uint32_t &x, uint32_t &y, uint32_t w, uint32_t wp, uint32_t q,
                                        uint32_t q2) {
    uint32_t a = x >= q2 ? x - q2 : x;          // [0, 2q)
    uint32_t t = shoup_mul(y, w, wp, q);         // [0, 2q)
    x = a + t;                                   // [0, 4q)
    y = a - t + q2;                              // (0, 4q)
}

// Inverse GS butterfly, Harvey form: x, y in [0, 2q) -> [0, 2q).
__device__ __forceinline__ void gs_bfly(uint32_t &x, uint32_t &y, uint32_t w, uint32_t wp, uint32_t q,
                                        uint32_t q2) {
    uint32_t u = x + y;
    u = u >= q2 ? u - q2 : u;                    // [0, 2q)
    uint32_t v = x - y + q2;                     // (0, 4q)
    x = u;
    y = shoup_mul(v, w, wp, q);                  // [0, 2q)
}

// One forward round of R stages (s0 .. s0+R-1) on a group of G = 2^R
// elements e_i = g + i*tlow, where tlow = N >> (s0+R) is the butterfly
// distance of the last stage and `high` the group's index bits above the
// round's R bits (so e = (high << (log2 tlow + R)) | (i << log2 tlow) | low).
template <int R>
__device__ __forceinline__ void fwd_round_group(uint32_t *row, uint32_t g, uint32_t tlow, uint32_t s0,
                                                uint32_t high, const uint2 *__restrict__ T, uint32_t q) {
    constexpr int G = 1 << R;
    uint32_t x[G];
#pragma unroll
    for (int i = 0; i < G; ++i) x[i] = row[g + i * tlow];
    const uint32_t q2 = 2 * q;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int d = G >> (r + 1);
        const uint32_t m = 1u << (s0 + r);
#pragma unroll
        for (int i = 0; i < G; ++i) {
            if (i & d) continue;
            uint32_t blk = (high << r) | (uint32_t)(i >> (R - r));
            const uint2 w = __ldg(T + m + blk);
            ct_bfly(x[i], x[i + d], w.x, w.y, q, q2);
        }
    }
#pragma unroll
    for (int i = 0; i < G; ++i) row[g + i * tlow] = x[i];
}

// One inverse round of R stages s_hi, s_hi-1, .., s_hi-R+1 on a group of
// G = 2^R elements e_i = g + i*tlow, tlow = N >> (s_hi+1) the distance of the
// first (smallest) stage.
template <int R>
__device__ __forceinline__ void inv_round_group(uint32_t *row, uint32_t g, uint32_t tlow, uint32_t s_hi,
                                                uint32_t high, const uint2 *__restrict__ T, uint32_t q) {
    constexpr int G = 1 << R;
    uint32_t x[G];
#pragma unroll
    for (int i = 0; i < G; ++i) x[i] = row[g + i * tlow];
    const uint32_t q2 = 2 * q;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int d = 1 << r;
        const uint32_t m = 1u << (s_hi - r);
#pragma unroll
        for (int i = 0; i < G; ++i) {
            if (i & d) continue;
            uint32_t blk = (high << (R - 1 - r)) | (uint32_t)(i >> (r + 1));
            const uint2 w = __ldg(T + m + blk);
            gs_bfly(x[i], x[i + d], w.x, w.y, q, q2);
        }
    }
#pragma unroll
    for (int i = 0; i < G; ++i) row[g + i * tlow] = x[i];
}

// Transform `nrows` rows of length N held contiguously in shared memory
// (row r at sm + r*N, using prime prime_of(r)), cooperatively by all threads
// of the block.  Leaves forward results in [0, 4q) and inverse results in
// [0, 2q) *without* the N^-1 factor; callers finish the reduction.
template <bool FWD, typename PrimeOf>
__device__ void ntt_rows_smem(uint32_t *sm, uint32_t nrows, const RnsParams &P, PrimeOf prime_of) {
    const uint32_t N = P.N, logN = P.logN;
    const uint32_t nthr = blockDim.x, tid = threadIdx.x;
    uint32_t done = 0;  // stages completed
    while (done < logN) {
        const uint32_t R = (logN - done) >= 3 ? 3 : (logN - done);
        const uint32_t lg = logN - R;  // log2(groups per row)
        // forward: stages s0 = done .. done+R-1; inverse: s_hi = logN-1-done .. down
        const uint32_t log_tlow = FWD ? (logN - done - R) : done;
        const uint32_t tlow = 1u << log_tlow;
        for (uint32_t v = tid; v < (nrows << lg); v += nthr) {
            const uint32_t r = v >> lg, vv = v & ((1u << lg) - 1);
            const uint32_t l = prime_of(r);
            const uint32_t q = P.q[l];
            const uint2 *T = tw_pairs(P.tw, l, N, FWD ? TW_FWD : TW_INV);
            const uint32_t low = vv & (tlow - 1), high = vv >> log_tlow;
            const uint32_t g = (high << (log_tlow + R)) | low;
            uint32_t *row = sm + (size_t)r * N;
            if (FWD) {
                if (R == 3) fwd_round_group<3>(row, g, tlow, done, high, T, q);
                else if (R == 2) fwd_round_group<2>(row, g, tlow, done, high, T, q);
                else fwd_round_group<1>(row, g, tlow, done, high, T, q);
            } else {
                const uint32_t s_hi = logN - 1 - done;
                if (R == 3) inv_round_group<3>(row, g, tlow, s_hi, high, T, q);
                else if (R == 2) inv_round_group<2>(row, g, tlow, s_hi, high, T, q);
                else inv_round_group<1>(row, g, tlow, s_hi, high, T, q);
            }
        }
        __syncthreads();
        done += R;
    }
}

// Final reductions.
__device__ __forceinline__ uint32_t fwd_final(uint32_t x, uint32_t q) {  // [0,4q) -> [0,q)
    x = x >= 2 * q ? x - 2 * q : x;
    return x >= q ? x - q : x;
}

__device__ __forceinline__ uint32_t inv_final(uint32_t x, uint32_t ninv, uint32_t ninv_shoup,
                                              uint32_t q) {  // [0,2q) * N^-1 -> [0,q)
    uint32_t y = shoup_mul(x, ninv, ninv_shoup, q);
    return y >= q ? y - q : y;
}

// N = 4096: 256 threads x 16 elements, three rounds of four butterfly stages.
// The first round reads its 16 elements straight from global memory
// (coalesced: element t + 256 i for the forward, 16t .. 16t+15 for the
// inverse) and the last round writes straight back, so a row crosses shared
// memory only twice; in shared memory it is placed by Swz4096 (below).  Early-round twiddles are the same for all threads of a
// warp (broadcast loads); the butterflies are branch-free.
constexpr int kN4 = 4096, kT4 = 256;

// Placement of a 4096-point row in shared memory.  With a = 256 hi + 16 mid
// + lo (4-bit digits), element a sits at
//     256 hi + 16 (mid ^ (hi & 1)) + (lo ^ mid),
// a bijection under which each access pattern of the three radix-16 rounds,
// over the 32 threads t of a warp, hits 32 distinct banks:
//     t + 256 i                    at e_(i & 1) + 256 i     (col)
//     256 (t>>4) + (t&15) + 16 i   at b1 ^ 17 i             (mid)
//     16 t + i                     at b2 ^ i                (row)
// (in natural placement the second pattern is a 2-way and the vectorised
// third a 4-way bank conflict).
struct Swz4096 {
    uint32_t e0, e1, b1, b2;
    __device__ __forceinline__ explicit Swz4096(uint32_t t) {
        const uint32_t hi = t >> 4, lo = t & 15;
        e0 = (hi << 4) | (lo ^ hi);
        e1 = ((hi ^ 1) << 4) | (lo ^ hi);
        b1 = (hi << 8) | ((hi & 1) << 4) | lo;
        b2 = (hi << 8) | ((lo ^ (hi & 1)) << 4) | lo;
    }
    __device__ __forceinline__ uint32_t col(int i) const { return ((i & 1) ? e1 : e0) + 256u * (uint32_t)i; }
    __device__ __forceinline__ uint32_t mid(int i) const { return b1 ^ (17u * (uint32_t)i); }
    __device__ __forceinline__ uint32_t row(int i) const { return b2 ^ (uint32_t)i; }
};

__device__ __forceinline__ uint32_t umin32(uint32_t a, uint32_t b) { return a < b ? a : b; }

// The 4096-point forward rounds reduce the upper butterfly input only at
// stages 3, 5, 7, 9 and 11.  A CT butterfly without reduction maps x in
// [0, B) and any 32-bit y to x + t and x - t + 2q in [0, B + 2q) (t, the
// Shoup product, lies in [0, 2q)), and the lower input is never reduced (a
// Shoup product accepts any 32-bit value).  From inputs below 2q the bound
// after stage s is 4q, 6q, 8q for s = 0, 1, 2; at a reducing stage x < 8q
// drops below 4q by one conditional subtraction of 4q, so the bound
// alternates 6q, 8q.  8q < 2^32 for q < 2^29, and outputs leave below 6q
// (fwd_final6).
__host__ __device__ constexpr bool fwd_reduces(uint32_t s) { return s >= 3 && (s & 1); }

__device__ __forceinline__ void ct_bfly_lazy(uint32_t &x, uint32_t &y, uint2 w, uint32_t q, bool reduce) {
    const uint32_t a = reduce ? umin32(x, x - 4 * q) : x;
    const uint32_t t = shoup_mul(y, w.x, w.y, q);
    x = a + t;
    y = a - t + 2 * q;
}

// One forward round of 4 stages (s0..s0+3, s0 a compile-time constant at
// every call) on x[16] = elements g + tlow*i.
__device__ __forceinline__ void fwd_round16(uint32_t (&x)[16], uint32_t s0, uint32_t high,
                                            const uint2 *__restrict__ T, uint32_t q) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = 16 >> (r + 1);
        const uint32_t m = 1u << (s0 + r);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & d) continue;
            const uint2 w = __ldg(T + m + ((high << r) | (uint32_t)(i >> (4 - r))));
            ct_bfly_lazy(x[i], x[i + d], w, q, fwd_reduces(s0 + r));
        }
    }
}

// fwd_round16 on two rows of the same prime at once: each twiddle pair is
// loaded once for both, and the two rows' butterflies are independent work.
__device__ __forceinline__ void fwd_round16x2(uint32_t (&x)[16], uint32_t (&y)[16], uint32_t s0, uint32_t high,
                                              const uint2 *__restrict__ T, uint32_t q) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = 16 >> (r + 1);
        const uint32_t m = 1u << (s0 + r);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & d) continue;
            const uint2 w = __ldg(T + m + ((high << r) | (uint32_t)(i >> (4 - r))));
            ct_bfly_lazy(x[i], x[i + d], w, q, fwd_reduces(s0 + r));
            ct_bfly_lazy(y[i], y[i + d], w, q, fwd_reduces(s0 + r));
        }
    }
}

// Final reduction of the 4096-point forward outputs: [0, 6q) -> [0, q).
__device__ __forceinline__ uint32_t fwd_final6(uint32_t x, uint32_t q) {
    x = umin32(x, x - 4 * q);
    x = umin32(x, x - 2 * q);
    return umin32(x, x - q);
}

// One inverse round of 4 stages s_hi..s_hi-3 on x[16] = elements g + tlow*i.
__device__ __forceinline__ void inv_round16(uint32_t (&x)[16], uint32_t s_hi, uint32_t high,
                                            const uint2 *__restrict__ T, uint32_t q) {
    const uint32_t q2 = 2 * q;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = 1 << r;
        const uint32_t m = 1u << (s_hi - r);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & d) continue;
            const uint2 w = __ldg(T + m + ((high << (3 - r)) | (uint32_t)(i >> (r + 1))));
            const uint32_t u = x[i] + x[i + d];
            const uint32_t v = x[i] - x[i + d] + q2;
            x[i] = umin32(u, u - q2);                            // [0, 2q)
            x[i + d] = shoup_mul(v, w.x, w.y, q);                // [0, 2q)
        }
    }
}

// inv_round16 on two rows of the same prime (shared twiddle loads).
__device__ __forceinline__ void inv_round16x2(uint32_t (&x)[16], uint32_t (&y)[16], uint32_t s_hi, uint32_t high,
                                              const uint2 *__restrict__ T, uint32_t q) {
    const uint32_t q2 = 2 * q;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = 1 << r;
        const uint32_t m = 1u << (s_hi - r);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & d) continue;
            const uint2 w = __ldg(T + m + ((high << (3 - r)) | (uint32_t)(i >> (r + 1))));
            const uint32_t u = x[i] + x[i + d];
            const uint32_t v = x[i] - x[i + d] + q2;
            x[i] = umin32(u, u - q2);
            x[i + d] = shoup_mul(v, w.x, w.y, q);
            const uint32_t a = y[i] + y[i + d];
            const uint32_t b = y[i] - y[i + d] + q2;
            y[i] = umin32(a, a - q2);
            y[i + d] = shoup_mul(b, w.x, w.y, q);
        }
    }
}

// The three inverse rounds of a 4096-point transform on one row whose
// first-round inputs (16 consecutive values per thread, in [0, 2q)) are in
// x; the results (natural order, times N^-1, canonical) go to dst.
__device__ __forceinline__ void inv4096_rounds(uint32_t (&x)[16], uint32_t *sm, const uint2 *__restrict__ T,
                                               uint32_t q, uint32_t ni, uint32_t nis, uint32_t *dst) {
    const uint32_t t = threadIdx.x;
    const Swz4096 z(t);
    inv_round16(x, 11, t, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) sm[z.row(k)] = x[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] = sm[z.mid(k)];
    inv_round16(x, 7, t >> 4, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) sm[z.mid(k)] = x[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] = sm[z.col(k)];
    inv_round16(x, 3, 0, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) dst[t + 256 * k] = inv_final(x[k], ni, nis, q);
}

// The three inverse rounds of a 4096-point transform on two rows of one
// prime whose first-round inputs (16 consecutive values per thread, in
// [0, 2q)) are already in x and y; the results (natural order, times N^-1,
// canonical) go to dst0 and dst1 (dst1 skipped when !two).
__device__ __forceinline__ void inv4096x2_rounds(uint32_t (&x)[16], uint32_t (&y)[16], uint32_t *sa, uint32_t *sb,
                                                 const uint2 *__restrict__ T, uint32_t q, uint32_t ni, uint32_t nis,
                                                 uint32_t *dst0, uint32_t *dst1, bool two) {
    const uint32_t t = threadIdx.x;
    const Swz4096 z(t);
    inv_round16x2(x, y, 11, t, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        sa[z.row(k)] = x[k];
        sb[z.row(k)] = y[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        x[k] = sa[z.mid(k)];
        y[k] = sb[z.mid(k)];
    }
    inv_round16x2(x, y, 7, t >> 4, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        sa[z.mid(k)] = x[k];
        sb[z.mid(k)] = y[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        x[k] = sa[z.col(k)];
        y[k] = sb[z.col(k)];
    }
    inv_round16x2(x, y, 3, 0, T, q);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        dst0[t + 256 * k] = inv_final(x[k], ni, nis, q);
        if (two) dst1[t + 256 * k] = inv_final(y[k], ni, nis, q);
    }
}
