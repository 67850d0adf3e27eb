// expand.cu — ExpandQuery: the expansion tree of Subs operations.
//
// GPIR section 2 (ExpandQuery: every depth of the expansion tree is a stage
// with its own evaluation key evk, up to log N stages) and section 3 (Subs
// operates on the a polynomial only).  Stage j, Galois element k = N/2^j + 1,
// over M ciphertexts ct = (c0, c1) in NTT form (decrypting as c0 + c1 s):
//     S_i      = Subs(ct_i, k) = (sigma_k(c0), 0)
//                + sum_u NTT(Dcp_u(sigma_k(c1))) . evk_j[u]
//     out[i]     = ct_i + S_i
//     out[i + M] = (ct_i - S_i) . NTT(X^(-2^j))
// so that after S stages ciphertext r carries coefficient r of the query's
// plaintext (times 2^S).  sigma_k(a)(X) = a(X^k): in coefficient form a
// move of coefficient t to t k mod 2N with a sign, in NTT form a permutation
// of the evaluation slots (slot j holds the value at zeta_j =
// psi^(2 brv(j) + 1), and sigma_k(a)(zeta_j) = a(zeta_j^k)).
//
// Per stage, four launches:
//   1. expand_intt_a4096_kernel  inverse NTT of every c1 (N = 4096; other N:
//      a strided copy and the library's inverse NTT)
//   2. gadget_dcp_kernel         digits of sigma_k(c1) (the automorphism as a
//      gather with signs)
//   3. lift + forward NTT of the digits (the library's NTT kernel)
//   4. expand_mac_kernel         the key switch, sigma_k(c0) by slot
//      permutation, and both outputs with the monomial's NTT
//
// RGSW ciphertexts from the expansion (pir_rgsw_convert; a reading, the pages
// say only that the expanded query also yields the RGSW ciphertexts of the
// column tournament): the expansion outputs ct_u = RLWE(m g_u), u < ell, are
// the rows u of RGSW(m); rows ell + u = (0, c0_u) + sum_v NTT(Dcp_v(c1_u)) .
// ksk[v] with ksk[v] = RLWE(s^2 g_v), which decrypt to s (c0_u + c1_u s) =
// m s g_u.  The same four launches as a stage, without the automorphism:
// inverse NTT of c1, Dcp, lift + NTT of the digits, rgsw_mac_kernel.
//
// Batches: G expansions (one per client, each with its own keys) run as one
// expansion of G*M ciphertexts per stage; global ciphertext g belongs to
// client b = g / M, and client b's outputs i and i + M go to b*2M + i and
// b*2M + i + M, so after the last stage client b's 2^S ciphertexts are
// contiguous (the layout RowSel takes for a batch of queries).
#include <cstring>

#include "common.cuh"
#include "gadget.cuh"
#include "ntt_core.cuh"

extern "C" int pir_ntt_inv(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream);
extern "C" int pir_lift_ntt(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, void *stream);

namespace {

struct InttAArgs {
    const uint32_t *in;     // ciphertext i at in + ((i / per) * stride + i % per) * 2 L N words
    uint32_t *coef;         // [M][L][N]
    const uint32_t *tw;
    uint64_t M, per, stride;   // per = stride = M for a contiguous [M][2][L][N] input
    uint32_t L;
    uint32_t q[PIR_MAX_RNS], ninv[PIR_MAX_RNS], ninv_shoup[PIR_MAX_RNS];
};

// N = 4096: one CTA per (ciphertexts 2i' and 2i'+1, prime l) transforms
// both c1 rows with shared twiddles; rounds as in the library's inverse.
__global__ void __launch_bounds__(kT4) expand_intt_a4096_kernel(const __grid_constant__ InttAArgs A) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sa[kN4];
    __shared__ __align__(16) uint32_t sb[kN4];
    const uint64_t i0 = 2 * (blockIdx.x / A.L), i1 = i0 + 1;
    const uint32_t l = blockIdx.x % A.L;
    const bool two = i1 < A.M;
    const uint32_t q = A.q[l];
    const uint2 *T = tw_pairs(A.tw, l, kN4, TW_INV);
    const uint64_t j0 = (i0 / A.per) * A.stride + i0 % A.per, j1 = (i1 / A.per) * A.stride + i1 % A.per;
    const uint32_t *s0 = A.in + ((2 * j0 + 1) * A.L + l) * kN4;
    const uint32_t *s1 = A.in + ((2 * j1 + 1) * A.L + l) * kN4;
    const uint32_t t = threadIdx.x;
    uint32_t x[16], y[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(s0 + 16 * t + k);
        const uint4 v = two ? *reinterpret_cast<const uint4 *>(s1 + 16 * t + k) : make_uint4(0, 0, 0, 0);
        x[k] = u.x; x[k + 1] = u.y; x[k + 2] = u.z; x[k + 3] = u.w;
        y[k] = v.x; y[k + 1] = v.y; y[k + 2] = v.z; y[k + 3] = v.w;
    }
    inv4096x2_rounds(x, y, sa, sb, T, q, A.ninv[l], A.ninv_shoup[l], A.coef + (i0 * A.L + l) * kN4,
                     A.coef + (i1 * A.L + l) * kN4, two);
}

// The same, one ciphertext's c1 row (ciphertext i, prime l) per CTA: for
// small stages, where each CTA's chain of rounds sets the stage's latency.
__global__ void __launch_bounds__(kT4) expand_intt_a4096_row_kernel(const __grid_constant__ InttAArgs A) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sm[kN4];
    const uint64_t i = blockIdx.x / A.L;
    const uint32_t l = blockIdx.x % A.L;
    const uint32_t q = A.q[l];
    const uint2 *T = tw_pairs(A.tw, l, kN4, TW_INV);
    const uint64_t j = (i / A.per) * A.stride + i % A.per;
    const uint32_t *src = A.in + ((2 * j + 1) * A.L + l) * kN4;
    const uint32_t t = threadIdx.x;
    uint32_t x[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(src + 16 * t + k);
        x[k] = u.x; x[k + 1] = u.y; x[k + 2] = u.z; x[k + 3] = u.w;
    }
    inv4096_rounds(x, sm, T, q, A.ninv[l], A.ninv_shoup[l], A.coef + (i * A.L + l) * kN4);
}

struct ExpMacArgs {
    const uint32_t *in;     // [G][M][2][L][N]
    const uint32_t *dn;     // [G][M][ell][L][N] NTT of the digits of sigma_k(c1)
    const uint32_t *evk;    // client b's stage key [ell][2][L][N] at evk + b * evk_stride
    uint32_t *out;          // [G][2M][2][L][N]
    const uint32_t *xpow;   // the stage's NTT(X^(-2^j)), [L][N]
    uint64_t M, GM, evk_stride;
    uint32_t N, logN, L, ell, k;
    uint32_t q[PIR_MAX_RNS];
    uint64_t mu[PIR_MAX_RNS];
};

__device__ __forceinline__ uint32_t brv(uint32_t x, uint32_t logN) { return __brev(x) >> (32 - logN); }

__device__ __forceinline__ uint32_t addq(uint32_t a, uint32_t b, uint32_t q) {
    const uint32_t r = a + b;
    return r >= q ? r - q : r;
}

__device__ __forceinline__ uint32_t subq(uint32_t a, uint32_t b, uint32_t q) {
    const uint32_t r = a + q - b;
    return r >= q ? r - q : r;
}

// Four consecutive slots per thread.  The ell <= 16 key-switch products of
// residues below 2^29 sum below 2^62 without reduction.
// EC = ell when known at compile time (ell = 5: the digit loop unrolled), else 0.
template <uint32_t EC>
__global__ void __launch_bounds__(GD_THREADS) expand_mac_kernel(const ExpMacArgs A) {
    pdl_wait();
    const uint64_t LN = (uint64_t)A.L * A.N;
    const uint64_t total4 = A.GM * LN / 4;
    const uint32_t twoN = 2 * A.N;
    const uint64_t pol_first = policy_evict_first();   // the digit transforms are read once
    for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total4;
         e += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t e0 = e * 4;
        const uint64_t i = e0 / LN, pt = e0 - i * LN;    // pt = l * N + slot
        const uint32_t l = (uint32_t)(pt / A.N), s0 = (uint32_t)(pt - (uint64_t)l * A.N);
        const uint32_t q = pick(A.q, l);
        const uint64_t mu = pick(A.mu, l);
        const uint32_t b = (uint32_t)i / (uint32_t)A.M;         // G * M < 2^31 (checked on the host)
        const uint64_t ib = i - (uint64_t)b * A.M;
        const uint32_t *dp = A.dn + i * A.ell * LN + pt;
        const uint32_t *kp = A.evk + b * A.evk_stride + pt;
        uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, b0 = 0, b1 = 0, b2 = 0, b3 = 0;
        const uint32_t ell = EC ? EC : A.ell;
#pragma unroll (EC ? 5 : 4)
        for (uint32_t u = 0; u < ell; ++u) {
            const uint4 d = ld_policy(dp + (uint64_t)u * LN, pol_first);
            const uint4 k0 = __ldg(reinterpret_cast<const uint4 *>(kp + (uint64_t)(2 * u) * LN));
            const uint4 k1 = __ldg(reinterpret_cast<const uint4 *>(kp + (uint64_t)(2 * u + 1) * LN));
            a0 += (uint64_t)d.x * k0.x; a1 += (uint64_t)d.y * k0.y; a2 += (uint64_t)d.z * k0.z; a3 += (uint64_t)d.w * k0.w;
            b0 += (uint64_t)d.x * k1.x; b1 += (uint64_t)d.y * k1.y; b2 += (uint64_t)d.z * k1.z; b3 += (uint64_t)d.w * k1.w;
        }
        const uint64_t ks0[4] = {a0, a1, a2, a3}, ks1[4] = {b0, b1, b2, b3};
        const uint32_t *c0 = A.in + i * 2 * LN + (uint64_t)l * A.N;
        const uint32_t *c1 = c0 + LN;
        const uint4 xm = __ldg(reinterpret_cast<const uint4 *>(A.xpow + pt));   // NTT(X^(-2^j)) at the 4 slots
        const uint32_t xmv[4] = {xm.x, xm.y, xm.z, xm.w};
        const uint4 v0 = *reinterpret_cast<const uint4 *>(c0 + s0);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(c1 + s0);
        const uint32_t x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
        uint32_t o0[4], o1[4], p0[4], p1[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t slot = s0 + c;
            const uint32_t odd = 2 * brv(slot, A.logN) + 1;
            // sigma_k(c0) at this slot: c0 at the slot of zeta^k
            const uint32_t ek = (uint32_t)(((uint64_t)A.k * odd) & (twoN - 1));
            const uint32_t src = brv((ek - 1) >> 1, A.logN);
            const uint32_t S0 = addq(c0[src], barrett64(ks0[c], q, mu), q);
            const uint32_t S1 = barrett64(ks1[c], q, mu);
            const uint32_t m = xmv[c];
            o0[c] = addq(x0[c], S0, q);
            o1[c] = addq(x1[c], S1, q);
            p0[c] = barrett64((uint64_t)subq(x0[c], S0, q) * m, q, mu);
            p1[c] = barrett64((uint64_t)subq(x1[c], S1, q) * m, q, mu);
        }
        uint32_t *out1 = A.out + ((uint64_t)b * 2 * A.M + ib) * 2 * LN + pt;
        uint32_t *out2 = out1 + A.M * 2 * LN;
        *reinterpret_cast<uint4 *>(out1) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<uint4 *>(out1 + LN) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *reinterpret_cast<uint4 *>(out2) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
        *reinterpret_cast<uint4 *>(out2 + LN) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
    }
}

struct RgswMacArgs {
    const uint32_t *in;     // gadget ciphertexts: client b's n * ell at in + b * in_stride * 2 L N words
    const uint32_t *dn;     // [M][ell][L][N] NTT of the digits of c1
    const uint32_t *ksk;    // client b's key [ell][2][L][N] at ksk + b * ksk_stride
    uint32_t *out;          // [G * n][2 ell][2][L][N]
    uint64_t M, per_client, in_stride, ksk_stride;   // per_client = n * ell input ciphertexts
    uint32_t N, L, ell;
    uint32_t q[PIR_MAX_RNS];
    uint64_t mu[PIR_MAX_RNS];
};

// Four consecutive slots per thread: input ciphertext i = (RGSW r, row u)
// goes to row u of RGSW r unchanged and, key-switched, to row ell + u.
__global__ void __launch_bounds__(GD_THREADS) rgsw_mac_kernel(const RgswMacArgs A) {
    pdl_wait();
    const uint64_t LN = (uint64_t)A.L * A.N;
    const uint64_t total4 = A.M * LN / 4;
    for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total4;
         e += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t e0 = e * 4;
        const uint64_t i = e0 / LN, pt = e0 - i * LN;    // pt = l * N + slot
        const uint32_t l = (uint32_t)(pt / A.N);
        const uint32_t q = pick(A.q, l);
        const uint64_t mu = pick(A.mu, l);
        const uint32_t b = (uint32_t)i / (uint32_t)A.per_client;   // M < 2^31 (checked on the host)
        const uint32_t *dp = A.dn + i * A.ell * LN + pt;
        const uint32_t *kp = A.ksk + b * A.ksk_stride + pt;
        uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, b0 = 0, b1 = 0, b2 = 0, b3 = 0;
#pragma unroll 4
        for (uint32_t u = 0; u < A.ell; ++u) {
            const uint4 d = *reinterpret_cast<const uint4 *>(dp + (uint64_t)u * LN);
            const uint4 k0 = __ldg(reinterpret_cast<const uint4 *>(kp + (uint64_t)(2 * u) * LN));
            const uint4 k1 = __ldg(reinterpret_cast<const uint4 *>(kp + (uint64_t)(2 * u + 1) * LN));
            a0 += (uint64_t)d.x * k0.x; a1 += (uint64_t)d.y * k0.y; a2 += (uint64_t)d.z * k0.z; a3 += (uint64_t)d.w * k0.w;
            b0 += (uint64_t)d.x * k1.x; b1 += (uint64_t)d.y * k1.y; b2 += (uint64_t)d.z * k1.z; b3 += (uint64_t)d.w * k1.w;
        }
        const uint64_t src = (uint64_t)b * A.in_stride + (i - (uint64_t)b * A.per_client);
        const uint4 v0 = *reinterpret_cast<const uint4 *>(A.in + src * 2 * LN + pt);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(A.in + src * 2 * LN + LN + pt);
        const uint64_t r = i / A.ell, u = i - r * A.ell;
        uint32_t *row_u = A.out + (r * 2 * A.ell + u) * 2 * LN + pt;
        uint32_t *row_s = A.out + (r * 2 * A.ell + A.ell + u) * 2 * LN + pt;
        *reinterpret_cast<uint4 *>(row_u) = v0;
        *reinterpret_cast<uint4 *>(row_u + LN) = v1;
        *reinterpret_cast<uint4 *>(row_s) =
            make_uint4(barrett64(a0, q, mu), barrett64(a1, q, mu), barrett64(a2, q, mu), barrett64(a3, q, mu));
        *reinterpret_cast<uint4 *>(row_s + LN) =
            make_uint4(addq(v0.x, barrett64(b0, q, mu), q), addq(v0.y, barrett64(b1, q, mu), q),
                       addq(v0.z, barrett64(b2, q, mu), q), addq(v0.w, barrett64(b3, q, mu), q));
    }
}

uint64_t align64(uint64_t words) { return (words + 63) / 64 * 64; }

// Workspace (words) for stages of at most Mmax input ciphertexts: c1 in
// coefficient form, the digits, their NTTs, and the two buffers the stage
// outputs alternate between (stage j writes 2^(j+1) ciphertexts).
struct ExLayout {
    uint64_t coef, dig, dn, ping, pong, total;
};

ExLayout ex_layout(const pir_ctx *ctx, uint64_t Mmax, uint32_t ell) {
    const uint64_t LN = (uint64_t)ctx->L * ctx->N;
    ExLayout x;
    x.coef = 0;
    x.dig = x.coef + align64(Mmax * LN);
    x.dn = x.dig + align64(Mmax * ell * (uint64_t)ctx->N);
    x.ping = x.dn + align64(Mmax * ell * LN);
    x.pong = x.ping + align64(Mmax * 2 * LN);
    x.total = x.pong + align64(Mmax * 2 * LN);
    return x;
}

// k^-1 mod 2N for odd k (Newton iteration on 2-adic inverses).
uint32_t inv_mod_2n(uint32_t k, uint32_t twoN) {
    uint32_t x = k;                 // correct to 3 bits for odd k
    for (int it = 0; it < 5; ++it) x *= 2 - k * x;
    return x & (twoN - 1);
}

// The a polynomial c1 of each of the GM ciphertexts in `in` (NTT form) in
// coefficient form, coef [GM][L][N]; ciphertext i is at in + ((i / per) *
// stride + i % per) * 2 L N words (per = stride = GM: contiguous).
int c1_to_coef(pir_ctx *ctx, const uint32_t *in, uint64_t GM, uint32_t *coef, cudaStream_t st,
               uint64_t per = 0, uint64_t stride = 0) {
    const uint64_t LN = (uint64_t)ctx->L * ctx->N;
    if (per == 0) per = stride = GM;
    if (ctx->N == (uint32_t)kN4) {
        InttAArgs ia;
        memset(&ia, 0, sizeof(ia));
        ia.in = in;
        ia.coef = coef;
        ia.tw = ctx->d_tw;
        ia.L = ctx->L;
        for (uint32_t l = 0; l < ctx->L; ++l) {
            ia.q[l] = ctx->q[l];
            ia.ninv[l] = ctx->ninv[l];
            ia.ninv_shoup[l] = ctx->ninv_shoup[l];
        }
        if ((GM + 1) / 2 * ctx->L > 0x7fffffffull) return PIR_ERR_ARG;
        ia.M = GM;
        ia.per = per;
        ia.stride = stride;
        if ((GM + 1) / 2 * ctx->L >= (uint64_t)ctx->num_sms)
            pdl_launch(expand_intt_a4096_kernel, dim3((unsigned)((GM + 1) / 2 * ctx->L)), dim3(kT4), 0, st, ia);
        else   // a small stage: one row per CTA
            pdl_launch(expand_intt_a4096_row_kernel, dim3((unsigned)(GM * ctx->L)), dim3(kT4), 0, st, ia);
        return cudaGetLastError() == cudaSuccess ? PIR_OK : PIR_ERR_CUDA;
    }
    for (uint64_t b = 0; b < GM / per; ++b)   // one strided copy of the c1 rows per block of `per`
        if (cudaMemcpy2DAsync(coef + b * per * LN, LN * 4, in + (b * stride * 2 + 1) * LN, 2 * LN * 4, LN * 4, per,
                              cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return PIR_ERR_CUDA;
    return pir_ntt_inv(ctx, coef, coef, GM, st);
}

// Stage j of G expansions: in [G][M], out [G][2M]; client b's key at
// evk + b * evk_stride.
int one_stage(pir_ctx *ctx, const uint32_t *evk, uint64_t evk_stride, uint32_t ell, uint32_t w, uint32_t j,
              const uint32_t *in, uint64_t M, uint64_t G, uint32_t *out, uint32_t *ws, const ExLayout &lay,
              cudaStream_t st) {
    const uint64_t LN = (uint64_t)ctx->L * ctx->N, GM = G * M;
    uint32_t *coef = ws + lay.coef, *dig = ws + lay.dig, *dn = ws + lay.dn;
    const uint32_t k = (ctx->N >> j) + 1;
    int rc = PIR_OK;

    rc = c1_to_coef(ctx, in, GM, coef, st);
    if (rc) return rc;

    rc = gadget_dcp_launch(ctx, gadget_dcp_args(ctx, coef, LN, dig, GM, ell, w, inv_mod_2n(k, 2 * ctx->N)), st);
    if (rc) return rc;
    rc = lift_ntt_digits(ctx, dig, dn, GM * ell, w, st);
    if (rc) return rc;

    ExpMacArgs ma;
    memset(&ma, 0, sizeof(ma));
    ma.in = in;
    ma.dn = dn;
    ma.evk = evk;
    ma.out = out;
    ma.xpow = ctx->d_xpow + (size_t)j * ctx->L * ctx->N;
    ma.M = M;
    ma.GM = GM;
    ma.evk_stride = evk_stride;
    ma.N = ctx->N;
    ma.logN = ctx->logN;
    ma.L = ctx->L;
    ma.ell = ell;
    ma.k = k;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        ma.q[l] = ctx->q[l];
        ma.mu[l] = ctx->mu[l];
    }
    if (ell == 5)
        pdl_launch(expand_mac_kernel<5>, dim3((unsigned)gadget_grid(ctx, GM * LN / 4)), dim3(GD_THREADS), 0, st, ma);
    else
        pdl_launch(expand_mac_kernel<0>, dim3((unsigned)gadget_grid(ctx, GM * LN / 4)), dim3(GD_THREADS), 0, st, ma);
    return launch_status(cudaGetLastError());
}

bool overlaps(const void *a, uint64_t abytes, const void *b, uint64_t bbytes) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bbytes && y < x + abytes;
}

}  // namespace

extern "C" uint64_t pir_expand_workspace_bytes(const pir_ctx *ctx, uint64_t M, uint32_t ell) {
    if (!ctx || M == 0 || M > (1ull << 31) || ell == 0 || ell > GD_MAX_ELL) return 0;
    return ex_layout(ctx, M, ell).total * 4;
}

extern "C" int pir_expand_stage(pir_ctx *ctx, const uint32_t *evk, uint32_t ell, uint32_t w, uint32_t j,
                                const uint32_t *in, uint64_t M, uint32_t *out, void *workspace,
                                uint64_t workspace_bytes, void *stream) {
    if (!ctx || !evk || !in || !out || !workspace || M == 0 || M > (1ull << 31)) return PIR_ERR_ARG;
    if (!gadget_params_ok(ctx, ell, w) || j >= ctx->logN) return PIR_ERR_ARG;
    if (!aligned16(evk) || !aligned16(in) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    const ExLayout lay = ex_layout(ctx, M, ell);
    if (workspace_bytes < lay.total * 4) return PIR_ERR_ARG;
    const uint64_t ctb = 2ull * ctx->L * ctx->N * 4;
    if (overlaps(in, M * ctb, out, 2 * M * ctb)) return PIR_ERR_ARG;
    // the stage keeps its digits and coefficient-form rows in the workspace while it reads in and writes out
    if (overlaps(workspace, lay.total * 4, in, M * ctb) || overlaps(workspace, lay.total * 4, out, 2 * M * ctb))
        return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    return one_stage(ctx, evk, 0, ell, w, j, in, M, 1, out, static_cast<uint32_t *>(workspace), lay,
                     (cudaStream_t)stream);
}

extern "C" int pir_expand_batch(pir_ctx *ctx, const uint32_t *evks, uint32_t ell, uint32_t w, uint32_t stages,
                                const uint32_t *ct, uint64_t G, uint32_t *out, void *workspace,
                                uint64_t workspace_bytes, void *stream) {
    if (!ctx || !evks || !ct || !out || !workspace || stages == 0 || stages > ctx->logN) return PIR_ERR_ARG;
    if (G == 0 || G >= (1ull << 31) >> (stages - 1)) return PIR_ERR_ARG;     // G * 2^(stages-1) < 2^31
    if (!gadget_params_ok(ctx, ell, w)) return PIR_ERR_ARG;
    if (!aligned16(evks) || !aligned16(ct) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    const uint64_t Mmax = 1ull << (stages - 1);
    const ExLayout lay = ex_layout(ctx, G * Mmax, ell);
    if (workspace_bytes < lay.total * 4) return PIR_ERR_ARG;
    const uint64_t ctw = 2ull * ctx->L * ctx->N;
    if (overlaps(ct, G * ctw * 4, out, G * (2 * Mmax) * ctw * 4)) return PIR_ERR_ARG;
    // the stages ping-pong through the workspace while the first reads ct and the last writes out
    if (overlaps(workspace, lay.total * 4, ct, G * ctw * 4) || overlaps(workspace, lay.total * 4, out, G * (2 * Mmax) * ctw * 4))
        return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *ws = static_cast<uint32_t *>(workspace);
    const uint64_t key = (uint64_t)ell * ctw;       // words of one stage's evaluation key
    const uint64_t stride = stages * key;           // words of one client's keys
    const uint32_t *cur = ct;
    for (uint32_t j = 0; j < stages; ++j) {
        const uint64_t M = 1ull << j;
        uint32_t *dst = j + 1 == stages ? out : ws + ((j & 1) ? lay.pong : lay.ping);
        const int rc = one_stage(ctx, evks + j * key, stride, ell, w, j, cur, M, G, dst, ws, lay, st);
        if (rc) return rc;
        cur = dst;
    }
    return PIR_OK;
}

extern "C" int pir_expand(pir_ctx *ctx, const uint32_t *evks, uint32_t ell, uint32_t w, uint32_t stages,
                          const uint32_t *ct, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                          void *stream) {
    return pir_expand_batch(ctx, evks, ell, w, stages, ct, 1, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- RGSW conversion
namespace {

// Workspace (words) of pir_rgsw_convert over M gadget ciphertexts.
struct RgLayout {
    uint64_t coef, dig, dn, total;
};

RgLayout rg_layout(const pir_ctx *ctx, uint64_t M, uint32_t ell) {
    const uint64_t LN = (uint64_t)ctx->L * ctx->N;
    RgLayout r;
    r.coef = 0;
    r.dig = align64(M * LN);
    r.dn = r.dig + align64(M * ell * (uint64_t)ctx->N);
    r.total = r.dn + align64(M * ell * LN);
    return r;
}

}  // namespace

extern "C" uint64_t pir_rgsw_convert_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint64_t G, uint32_t ell) {
    if (!ctx || n == 0 || G == 0 || ell == 0 || ell > GD_MAX_ELL || n > (1ull << 31) || G > (1ull << 31) ||
        n * G * ell >= (1ull << 31))
        return 0;
    return rg_layout(ctx, n * G * ell, ell).total * 4;
}

extern "C" int pir_rgsw_convert(pir_ctx *ctx, const uint32_t *ksk, uint32_t ell, uint32_t w, const uint32_t *in,
                                uint64_t in_stride, uint64_t n, uint64_t G, uint32_t *out, void *workspace,
                                uint64_t workspace_bytes, void *stream) {
    if (!ctx || !ksk || !in || !out || !workspace || n == 0 || G == 0) return PIR_ERR_ARG;
    if (!gadget_params_ok(ctx, ell, w) || n > (1ull << 31) || G > (1ull << 31) || n * G * ell >= (1ull << 31))
        return PIR_ERR_ARG;
    if (in_stride == 0) in_stride = n * ell;
    if (in_stride < n * ell || in_stride > (1ull << 31) || (G - 1) * in_stride + n * ell >= (1ull << 31))
        return PIR_ERR_ARG;
    if (!aligned16(ksk) || !aligned16(in) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    const uint64_t M = n * G * ell, LN = (uint64_t)ctx->L * ctx->N;
    const RgLayout lay = rg_layout(ctx, M, ell);
    if (workspace_bytes < lay.total * 4) return PIR_ERR_ARG;
    const uint64_t in_b = ((G - 1) * in_stride + n * ell) * 2 * LN * 4, out_b = 2 * M * 2 * LN * 4,
                   ws_b = lay.total * 4;
    if (overlaps(in, in_b, out, out_b) || overlaps(workspace, ws_b, in, in_b) || overlaps(workspace, ws_b, out, out_b))
        return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *ws = static_cast<uint32_t *>(workspace);
    uint32_t *coef = ws + lay.coef, *dig = ws + lay.dig, *dn = ws + lay.dn;
    int rc = c1_to_coef(ctx, in, M, coef, st, n * ell, in_stride);
    if (rc) return rc;
    rc = gadget_dcp_launch(ctx, gadget_dcp_args(ctx, coef, LN, dig, M, ell, w, 1), st);
    if (rc) return rc;
    rc = lift_ntt_digits(ctx, dig, dn, M * ell, w, st);
    if (rc) return rc;
    RgswMacArgs ma;
    memset(&ma, 0, sizeof(ma));
    ma.in = in;
    ma.dn = dn;
    ma.ksk = ksk;
    ma.out = out;
    ma.M = M;
    ma.per_client = n * ell;
    ma.in_stride = in_stride;
    ma.ksk_stride = (uint64_t)ell * 2 * LN;
    ma.N = ctx->N;
    ma.L = ctx->L;
    ma.ell = ell;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        ma.q[l] = ctx->q[l];
        ma.mu[l] = ctx->mu[l];
    }
    pdl_launch(rgsw_mac_kernel, dim3((unsigned)gadget_grid(ctx, M * LN / 4)), dim3(GD_THREADS), 0, st, ma);
    return launch_status(cudaGetLastError());
}
