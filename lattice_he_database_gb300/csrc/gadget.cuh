// gadget.cuh — the gadget decomposition Dcp shared by ColTor and ExpandQuery.
//
// GPIR section 3 (Dcp, l = 5 digits at q ~ 2^87): every coefficient's CRT
// value X in [0, Q), Q = q_0 ... q_{L-1}, is written in base 2^w with ell
// unsigned digits, least significant first.  X = sum_l [x_l (Q/q_l)^-1]_{q_l}
// (Q/q_l) lies in [0, L*Q) and is brought into [0, Q) by at most L - 1
// subtractions of Q.  Optionally the digits are those of sigma_k(x) =
// x(X^k), the automorphism of Subs: output coefficient p reads input
// coefficient t = p k^-1 mod 2N, negated when t >= N (X^N = -1).
#pragma once

#include <cstring>

#include "common.cuh"

namespace {

typedef unsigned __int128 u128;

constexpr uint32_t GD_THREADS = 256;
constexpr uint32_t GD_MAX_ELL = 16;

// a[l] for a small runtime l without indexing the parameter array (which
// would copy it to local memory).
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[PIR_MAX_RNS], uint32_t l) {
    T r = a[0];
#pragma unroll
    for (uint32_t k = 1; k < PIR_MAX_RNS; ++k) r = l == k ? a[k] : r;
    return r;
}

struct DcpArgs {
    const uint32_t *x;      // [polys][L][N] coefficient form (row stride x_stride words per polynomial)
    uint32_t *d;            // [polys][ell][N]
    uint64_t polys, x_stride;
    uint32_t N, L, ell, w;
    uint32_t kinv;          // 1: the digits of x itself; otherwise of sigma_k(x), kinv = k^-1 mod 2N
    uint32_t q[PIR_MAX_RNS];
    uint32_t hinv[PIR_MAX_RNS];      // (Q/q_l)^-1 mod q_l
    uint32_t hinv_shoup[PIR_MAX_RNS];
    uint64_t M_lo[PIR_MAX_RNS], M_hi[PIR_MAX_RNS];   // Q/q_l
    uint64_t Q_lo, Q_hi;
};

__device__ __forceinline__ u128 crt_value(const DcpArgs &A, const uint32_t (&r)[PIR_MAX_RNS], u128 Q) {
    u128 X = 0;
#pragma unroll
    for (uint32_t l = 0; l < PIR_MAX_RNS; ++l) {
        if (l < A.L) {
            const uint32_t q = A.q[l];
            uint32_t y = shoup_mul(r[l], A.hinv[l], A.hinv_shoup[l], q);
            y = y >= q ? y - q : y;
            X += (u128)y * A.M_lo[l] + ((u128)((uint64_t)y * A.M_hi[l]) << 64);
        }
    }
#pragma unroll
    for (uint32_t l = 1; l < PIR_MAX_RNS; ++l)
        if (l < A.L) X = X >= Q ? X - Q : X;
    return X;
}

// One thread per four consecutive output coefficients; EC = ell when known
// at compile time (the digit loop unrolled), else 0.
template <uint32_t EC>
__global__ void __launch_bounds__(GD_THREADS) gadget_dcp_kernel(const DcpArgs A) {
    pdl_wait();
    const uint64_t total4 = A.polys * A.N / 4;
    const u128 Q = ((u128)A.Q_hi << 64) | A.Q_lo;
    const u128 mask = A.w >= 32 ? (u128)0xffffffffu : (((u128)1 << A.w) - 1);
    for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total4;
         e += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t p0 = e * 4;
        const uint64_t pi = p0 / A.N, p = p0 - pi * A.N;
        const uint32_t *xp = A.x + pi * A.x_stride;
        uint32_t r[4][PIR_MAX_RNS];
        if (A.kinv == 1) {
            const uint64_t pol = policy_evict_first();   // the coefficient rows are read once
#pragma unroll
            for (uint32_t l = 0; l < PIR_MAX_RNS; ++l) {
                const uint4 v = l < A.L ? ld_policy(xp + (uint64_t)l * A.N + p, pol) : make_uint4(0, 0, 0, 0);
                r[0][l] = v.x; r[1][l] = v.y; r[2][l] = v.z; r[3][l] = v.w;
            }
        } else {
            const uint32_t twoN = 2 * A.N;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t t0 = (uint32_t)(((uint64_t)(p + c) * A.kinv) & (twoN - 1));
                const bool neg = t0 >= A.N;
                const uint32_t t = neg ? t0 - A.N : t0;
#pragma unroll
                for (uint32_t l = 0; l < PIR_MAX_RNS; ++l) {
                    uint32_t v = 0;
                    if (l < A.L) {
                        v = xp[(uint64_t)l * A.N + t];
                        const uint32_t q = A.q[l];
                        v = neg && v ? q - v : v;
                    }
                    r[c][l] = v;
                }
            }
        }
        // digits from a two-word window: after each digit the 128-bit value
        // moves right by w (1 <= w <= 32, so both shifts stay below 64)
        uint64_t lo[4], hi[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const u128 X = crt_value(A, r[c], Q);
            lo[c] = (uint64_t)X;
            hi[c] = (uint64_t)(X >> 64);
        }
        const uint32_t m32 = (uint32_t)mask, w = A.w, wr = 64 - A.w;
        const uint32_t ell = EC ? EC : A.ell;
        uint32_t *dp = A.d + pi * ell * A.N + p;
#pragma unroll (EC ? EC : 1)
        for (uint32_t u = 0; u < ell; ++u) {
            *reinterpret_cast<uint4 *>(dp + (uint64_t)u * A.N) =
                make_uint4((uint32_t)lo[0] & m32, (uint32_t)lo[1] & m32, (uint32_t)lo[2] & m32, (uint32_t)lo[3] & m32);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                lo[c] = (lo[c] >> w) | (hi[c] << wr);
                hi[c] >>= w;
            }
        }
    }
}

// Bit length of Q = q_0 ... q_{L-1}.
uint32_t gadget_bits_of_Q(const pir_ctx *ctx) {
    u128 Q = 1;
    for (uint32_t l = 0; l < ctx->L; ++l) Q *= ctx->q[l];
    uint32_t b = 0;
    while (b < 128 && (Q >> b) != 0) ++b;
    return b;
}

// ell digits of w bits must cover [0, Q); digits are 32-bit words.
bool gadget_params_ok(const pir_ctx *ctx, uint32_t ell, uint32_t w) {
    return ctx && ell >= 1 && ell <= GD_MAX_ELL && w >= 1 && w <= 32 && (uint64_t)ell * w >= gadget_bits_of_Q(ctx);
}

// Kernel arguments for the digits of `polys` polynomials at x (stride
// x_stride words apart) into d, with the CRT constants of the context.
DcpArgs gadget_dcp_args(const pir_ctx *ctx, const uint32_t *x, uint64_t x_stride, uint32_t *d, uint64_t polys,
                        uint32_t ell, uint32_t w, uint32_t kinv) {
    DcpArgs A;
    memset(&A, 0, sizeof(A));
    A.x = x;
    A.d = d;
    A.polys = polys;
    A.x_stride = x_stride;
    A.N = ctx->N;
    A.L = ctx->L;
    A.ell = ell;
    A.w = w;
    A.kinv = kinv;
    u128 Q = 1;
    for (uint32_t l = 0; l < ctx->L; ++l) Q *= ctx->q[l];
    A.Q_lo = (uint64_t)Q;
    A.Q_hi = (uint64_t)(Q >> 64);
    for (uint32_t l = 0; l < ctx->L; ++l) {
        const uint32_t q = ctx->q[l];
        const u128 M = Q / q;
        uint64_t inv = 1, b = (uint64_t)(M % q), e = q - 2;   // (Q/q_l)^-1 by Fermat: q_l is prime
        for (; e; e >>= 1) {
            if (e & 1) inv = inv * b % q;
            b = b * b % q;
        }
        A.q[l] = q;
        A.hinv[l] = (uint32_t)inv;
        A.hinv_shoup[l] = (uint32_t)((inv << 32) / q);
        A.M_lo[l] = (uint64_t)M;
        A.M_hi[l] = (uint64_t)(M >> 64);
    }
    return A;
}

uint64_t gadget_grid(const pir_ctx *ctx, uint64_t work) {
    const uint64_t g = (work + GD_THREADS - 1) / GD_THREADS;
    const uint64_t cap = (uint64_t)ctx->num_sms * 64;
    return g < 1 ? 1 : (g < cap ? g : cap);
}

int gadget_dcp_launch(const pir_ctx *ctx, const DcpArgs &A, cudaStream_t st) {
    if (A.ell == 5)
        pdl_launch(gadget_dcp_kernel<5>, dim3((unsigned)gadget_grid(ctx, A.polys * A.N / 4)), dim3(GD_THREADS), 0, st, A);
    else
        pdl_launch(gadget_dcp_kernel<0>, dim3((unsigned)gadget_grid(ctx, A.polys * A.N / 4)), dim3(GD_THREADS), 0, st, A);
    return cudaGetLastError() == cudaSuccess ? PIR_OK : PIR_ERR_CUDA;
}

}  // namespace
