// coltor.cu — ColTor: the column tournament of RGSW-RLWE external products.
//
// GPIR section 2 (the ColTor phase of the OnionPIR family) and section 3
// (Dcp, l = 5 digits); VIPIR 3.6 step 7 (RGSW-RLWE external products for the
// folding after the first dimension) and section 5 (q ~ 2^87 in three RNS
// primes).  One stage maps n ciphertexts (NTT form) to ceil(n/2):
//     out_i = ct_2i + C (x) (ct_2i+1 - ct_2i)          (a missing partner is 0)
// with the external product of the RGSW ciphertext C = [2 ell][2] RLWE rows
//     C (x) ct = sum_u NTT(Dcp_u(ct_0)) . C[u] + NTT(Dcp_u(ct_1)) . C[ell + u],
// where Dcp_u is digit u of each coefficient's CRT value X in [0, Q) in base
// 2^w (unsigned digits, least significant first) and "." is the point-wise
// product mod q_l.
//
// Per stage, four launches (five for N != 4096); every intermediate goes
// through HBM (for n = 1365 ciphertexts the first stage's digit NTTs alone
// are 336 MB, far past L2), and the 2L inverse plus 2 ell L forward NTTs per
// pair bound the stage:
//   1. coltor_diff_intt4096_kernel  d_i = INTT(ct_2i+1 - ct_2i), [R][2][L][N]
//      (other N: coltor_diff_kernel, then the library's inverse NTT in place)
//   2. gadget_dcp_kernel    CRT value of each coefficient -> ell digits, [R][2][ell][N]
//   3. lift + forward NTT of the digits (the library's NTT kernel) -> [R][2][ell][L][N]
//   4. coltor_mac_kernel    out_i = ct_2i + sum_v D_v . C[v], lazy 64-bit sums
// The difference, decomposition and MAC kernels move four words per thread
// and memory access; all three are bound by HBM.  The decomposition is
// shared with ExpandQuery (gadget.cuh).
//
// Batches: G tournaments of n ciphertexts each (one per client, each with
// its own RGSW ciphertexts) run as one tournament of G*ceil(n/2) pairs per
// stage; global pair g belongs to tournament b = g / Rp (Rp = ceil(n/2)
// pairs per tournament), and the stage output [G][Rp] is the next stage's
// input [G][n' = Rp].
#include <cstring>

#include "common.cuh"
#include "gadget.cuh"
#include "ntt_core.cuh"

extern "C" int pir_ntt_inv(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream);
extern "C" int pir_lift_ntt(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, void *stream);

namespace {

constexpr uint32_t CT_THREADS = 256;

struct DiffArgs {
    const uint32_t *in;
    uint32_t *diff;
    uint64_t n, R, Rp;      // input ciphertexts per tournament, pairs in all, pairs per tournament
    uint32_t N, L;
    uint32_t q[PIR_MAX_RNS];
};

// Index of the even ciphertext of global pair g (tournament g / Rp).
__device__ __forceinline__ uint64_t even_ct(uint64_t g, uint64_t Rp, uint64_t n, bool &has_odd) {
    const uint32_t b = (uint32_t)g / (uint32_t)Rp;          // g < 2^31 (checked on the host)
    const uint64_t i = g - (uint64_t)b * Rp;
    has_odd = 2 * i + 1 < n;
    return (uint64_t)b * n + 2 * i;
}

// d_i = ct_2i+1 - ct_2i mod q_l, four words per thread.
__global__ void __launch_bounds__(CT_THREADS) coltor_diff_kernel(const DiffArgs A) {
    pdl_wait();
    const uint64_t ct_words = 2ull * A.L * A.N;          // one ciphertext
    const uint64_t total4 = A.R * ct_words / 4;
    for (uint64_t v = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; v < total4;
         v += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t w0 = v * 4;
        const uint64_t i = w0 / ct_words, r = w0 - i * ct_words;
        const uint32_t q = pick(A.q, (uint32_t)((r / A.N) % A.L));
        bool has_odd;
        const uint64_t ce = even_ct(i, A.Rp, A.n, has_odd);
        const uint4 e = *reinterpret_cast<const uint4 *>(A.in + ce * ct_words + r);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (has_odd) o = *reinterpret_cast<const uint4 *>(A.in + (ce + 1) * ct_words + r);
        uint4 d;
        d.x = o.x + q - e.x; d.x = d.x >= q ? d.x - q : d.x;
        d.y = o.y + q - e.y; d.y = d.y >= q ? d.y - q : d.y;
        d.z = o.z + q - e.z; d.z = d.z >= q ? d.z - q : d.z;
        d.w = o.w + q - e.w; d.w = d.w >= q ? d.w - q : d.w;
        *reinterpret_cast<uint4 *>(A.diff + w0) = d;
    }
}

struct DiffInttArgs {
    const uint32_t *in;
    uint32_t *diff;
    const uint32_t *tw;     // [L][2][N] twiddle pairs (tw_pairs)
    uint64_t n, Rp;         // ciphertexts and pairs per tournament
    uint32_t L;
    uint32_t q[PIR_MAX_RNS], ninv[PIR_MAX_RNS], ninv_shoup[PIR_MAX_RNS];
};

// N = 4096: one CTA per (pair i, prime l) transforms both difference rows
// (polynomials c = 0, 1) with shared twiddles; the first inverse round loads
// ct_2i+1 - ct_2i + q (in (0, 2q), the inverse butterflies' input range)
// instead of a stored difference.  Rounds as in the library's inverse.
__global__ void __launch_bounds__(kT4) coltor_diff_intt4096_kernel(const __grid_constant__ DiffInttArgs A) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sa[kN4];
    __shared__ __align__(16) uint32_t sb[kN4];
    const uint64_t i = blockIdx.x / A.L;
    const uint32_t l = blockIdx.x % A.L;
    const uint64_t LN = (uint64_t)A.L * kN4;
    const uint32_t q = A.q[l];
    const uint2 *T = tw_pairs(A.tw, l, kN4, TW_INV);
    bool has_odd;
    const uint64_t ce = even_ct(i, A.Rp, A.n, has_odd);
    const uint32_t *ev = A.in + ce * 2 * LN + (uint64_t)l * kN4;             // polynomial 0 of ct_2i
    const uint32_t *od = A.in + (ce + 1) * 2 * LN + (uint64_t)l * kN4;       // polynomial 0 of ct_2i+1
    const uint32_t t = threadIdx.x;
    uint32_t x[16], y[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const uint4 e0 = *reinterpret_cast<const uint4 *>(ev + 16 * t + k);
        const uint4 e1 = *reinterpret_cast<const uint4 *>(ev + LN + 16 * t + k);
        const uint4 o0 = has_odd ? *reinterpret_cast<const uint4 *>(od + 16 * t + k) : make_uint4(0, 0, 0, 0);
        const uint4 o1 = has_odd ? *reinterpret_cast<const uint4 *>(od + LN + 16 * t + k) : make_uint4(0, 0, 0, 0);
        x[k] = o0.x + q - e0.x; x[k + 1] = o0.y + q - e0.y; x[k + 2] = o0.z + q - e0.z; x[k + 3] = o0.w + q - e0.w;
        y[k] = o1.x + q - e1.x; y[k + 1] = o1.y + q - e1.y; y[k + 2] = o1.z + q - e1.z; y[k + 3] = o1.w + q - e1.w;
    }
    uint32_t *dst = A.diff + i * 2 * LN + (uint64_t)l * kN4;
    inv4096x2_rounds(x, y, sa, sb, T, q, A.ninv[l], A.ninv_shoup[l], dst, dst + LN, true);
}

// The same, one difference row (pair i, polynomial c, prime l) per CTA: for
// small stages, where a CTA per (pair, prime) would leave SMs idle and each
// CTA's chain of rounds sets the stage's latency.
__global__ void __launch_bounds__(kT4) coltor_diff_intt4096_row_kernel(const __grid_constant__ DiffInttArgs A) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sm[kN4];
    const uint64_t i = blockIdx.x / (2 * A.L);
    const uint32_t c = (blockIdx.x / A.L) & 1u, l = blockIdx.x % A.L;
    const uint64_t LN = (uint64_t)A.L * kN4;
    const uint32_t q = A.q[l];
    const uint2 *T = tw_pairs(A.tw, l, kN4, TW_INV);
    bool has_odd;
    const uint64_t ce = even_ct(i, A.Rp, A.n, has_odd);
    const uint32_t *ev = A.in + ce * 2 * LN + c * LN + (uint64_t)l * kN4;
    const uint32_t *od = A.in + (ce + 1) * 2 * LN + c * LN + (uint64_t)l * kN4;
    const uint32_t t = threadIdx.x;
    uint32_t x[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const uint4 e = *reinterpret_cast<const uint4 *>(ev + 16 * t + k);
        const uint4 o = has_odd ? *reinterpret_cast<const uint4 *>(od + 16 * t + k) : make_uint4(0, 0, 0, 0);
        x[k] = o.x + q - e.x; x[k + 1] = o.y + q - e.y; x[k + 2] = o.z + q - e.z; x[k + 3] = o.w + q - e.w;
    }
    inv4096_rounds(x, sm, T, q, A.ninv[l], A.ninv_shoup[l], A.diff + i * 2 * LN + c * LN + (uint64_t)l * kN4);
}

struct MacArgs {
    const uint32_t *in;     // [G][n][2][L][N] (the even ciphertexts are added)
    const uint32_t *dn;     // [R][2 ell][L][N] NTT of the digits
    const uint32_t *C;      // tournament b's stage RGSW [2 ell][2][L][N] at C + b * c_stride
    uint32_t *out;          // [R][2][L][N]
    uint64_t R, Rp, n, c_stride;
    uint32_t N, L, ell;
    uint32_t q[PIR_MAX_RNS];
    uint64_t mu[PIR_MAX_RNS];
};

// out_i[c] = ct_2i[c] + sum_v D_i[v] . C[v][c]: both output polynomials from
// one read of the 2 ell digit values, four points per thread; the 2 ell <= 32
// products of residues below 2^29 sum below 2^63 without reduction.
__device__ __forceinline__ uint32_t mac_final(uint64_t acc, uint32_t e, uint32_t q, uint64_t mu) {
    const uint32_t r = barrett64(acc, q, mu) + e;
    return r >= q ? r - q : r;
}

// VC = 2 ell when known at compile time (ell = 5: the whole digit loop
// unrolled, all its loads in flight at once; 2.8% per tournament), else 0.
template <uint32_t VC>
__global__ void __launch_bounds__(CT_THREADS) coltor_mac_kernel(const MacArgs A) {
    pdl_wait();
    const uint64_t LN = (uint64_t)A.L * A.N;
    const uint64_t total4 = A.R * LN / 4;
    const uint32_t V = VC ? VC : 2 * A.ell;
    // the digit transforms are read exactly once: let them leave L2 first, so
    // that the RGSW rows and the next stage's inputs stay (2% per tournament)
    const uint64_t pol_first = policy_evict_first();
    for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total4;
         e += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t e0 = e * 4;
        const uint64_t i = e0 / LN, pt = e0 - i * LN;    // pt = l * N + j
        const uint32_t l = (uint32_t)(pt / A.N);
        bool has_odd;
        const uint64_t ce = even_ct(i, A.Rp, A.n, has_odd);
        const uint32_t *dp = A.dn + i * V * LN + pt;
        const uint32_t *cp = A.C + (uint64_t)((uint32_t)i / (uint32_t)A.Rp) * A.c_stride + pt;
        uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, b0 = 0, b1 = 0, b2 = 0, b3 = 0;
#pragma unroll (VC ? 10 : 4)
        for (uint32_t v = 0; v < V; ++v) {
            const uint4 d = ld_policy(dp + (uint64_t)v * LN, pol_first);
            const uint4 c0 = __ldg(reinterpret_cast<const uint4 *>(cp + (uint64_t)(2 * v) * LN));
            const uint4 c1 = __ldg(reinterpret_cast<const uint4 *>(cp + (uint64_t)(2 * v + 1) * LN));
            a0 += (uint64_t)d.x * c0.x; a1 += (uint64_t)d.y * c0.y; a2 += (uint64_t)d.z * c0.z; a3 += (uint64_t)d.w * c0.w;
            b0 += (uint64_t)d.x * c1.x; b1 += (uint64_t)d.y * c1.y; b2 += (uint64_t)d.z * c1.z; b3 += (uint64_t)d.w * c1.w;
        }
        const uint32_t q = pick(A.q, l);
        const uint64_t mu = pick(A.mu, l);
        const uint4 ev0 = ld_policy(A.in + ce * 2 * LN + pt, pol_first);
        const uint4 ev1 = ld_policy(A.in + ce * 2 * LN + LN + pt, pol_first);
        uint32_t *op = A.out + i * 2 * LN + pt;
        *reinterpret_cast<uint4 *>(op) = make_uint4(mac_final(a0, ev0.x, q, mu), mac_final(a1, ev0.y, q, mu),
                                                    mac_final(a2, ev0.z, q, mu), mac_final(a3, ev0.w, q, mu));
        *reinterpret_cast<uint4 *>(op + LN) = make_uint4(mac_final(b0, ev1.x, q, mu), mac_final(b1, ev1.y, q, mu),
                                                         mac_final(b2, ev1.z, q, mu), mac_final(b3, ev1.w, q, mu));
    }
}

uint64_t align64(uint64_t words) { return (words + 63) / 64 * 64; }

// Workspace regions (words) for the stages of G tournaments of n
// ciphertexts (G * ceil(n/2) pairs in the first stage).
struct CtLayout {
    uint64_t diff, dig, dn, ping, pong, total;   // offsets and total words
};

CtLayout ct_layout(const pir_ctx *ctx, uint64_t n, uint32_t ell, uint64_t G = 1) {
    const uint64_t Rp = (n + 1) / 2, R = G * Rp, LN = (uint64_t)ctx->L * ctx->N;
    CtLayout c;
    c.diff = 0;
    c.dig = c.diff + align64(R * 2 * LN);
    c.dn = c.dig + align64(R * 2 * ell * (uint64_t)ctx->N);
    c.ping = c.dn + align64(R * 2 * ell * LN);
    c.pong = c.ping + align64(R * 2 * LN);
    c.total = c.pong + align64(G * ((Rp + 1) / 2) * 2 * LN);
    return c;
}

// Pair indices stay below 2^31 (32-bit tournament division in the kernels).
int check_params(const pir_ctx *ctx, uint32_t ell, uint32_t w, uint64_t n, uint64_t G = 1) {
    if (!ctx || n == 0 || G == 0 || n > (1ull << 32) || G > (1ull << 31) || G * ((n + 1) / 2) >= (1ull << 31))
        return PIR_ERR_ARG;
    return gadget_params_ok(ctx, ell, w) ? PIR_OK : PIR_ERR_ARG;   // digits must cover [0, Q)
}

// Stages of a tournament of n ciphertexts: ceil(log2 n).
uint32_t stages_of(uint64_t n) {
    uint32_t s = 0;
    while ((1ull << s) < n) ++s;
    return s;
}

uint64_t grid_for(const pir_ctx *ctx, uint64_t work) { return gadget_grid(ctx, work); }

// One stage of G tournaments from `in` ([G][n] ciphertexts) to `out`
// ([G][ceil(n/2)]); tournament b's RGSW ciphertext is at C + b * c_stride.
// ws holds the diff, digit and digit-NTT regions of a layout for at least
// G tournaments of n ciphertexts.
int stage(pir_ctx *ctx, const uint32_t *C, uint64_t c_stride, uint32_t ell, uint32_t w, const uint32_t *in,
          uint64_t n, uint64_t G, uint32_t *out, uint32_t *ws, const CtLayout &lay, cudaStream_t st) {
    const uint64_t Rp = (n + 1) / 2, R = G * Rp, LN = (uint64_t)ctx->L * ctx->N;
    uint32_t *diff = ws + lay.diff, *dig = ws + lay.dig, *dn = ws + lay.dn;

    DiffArgs da;
    memset(&da, 0, sizeof(da));
    da.in = in;
    da.diff = diff;
    da.n = n;
    da.R = R;
    da.Rp = Rp;
    da.N = ctx->N;
    da.L = ctx->L;
    for (uint32_t l = 0; l < ctx->L; ++l) da.q[l] = ctx->q[l];
    int rc = PIR_OK;
    if (ctx->N == (uint32_t)kN4) {
        DiffInttArgs ia;
        memset(&ia, 0, sizeof(ia));
        ia.in = in;
        ia.diff = diff;
        ia.tw = ctx->d_tw;
        ia.n = n;
        ia.Rp = Rp;
        ia.L = ctx->L;
        for (uint32_t l = 0; l < ctx->L; ++l) {
            ia.q[l] = ctx->q[l];
            ia.ninv[l] = ctx->ninv[l];
            ia.ninv_shoup[l] = ctx->ninv_shoup[l];
        }
        if (R * 2 * ctx->L > 0x7fffffffull) return PIR_ERR_ARG;
        if (R * ctx->L >= (uint64_t)ctx->num_sms)
            pdl_launch(coltor_diff_intt4096_kernel, dim3((unsigned)(R * ctx->L)), dim3(kT4), 0, st, ia);
        else   // a small stage: one row per CTA
            pdl_launch(coltor_diff_intt4096_row_kernel, dim3((unsigned)(R * 2 * ctx->L)), dim3(kT4), 0, st, ia);
        if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;
    } else {
        pdl_launch(coltor_diff_kernel, dim3((unsigned)grid_for(ctx, R * 2 * LN / 4)), dim3(CT_THREADS), 0, st, da);
        if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;
        rc = pir_ntt_inv(ctx, diff, diff, R * 2, st);
        if (rc) return rc;
    }

    rc = gadget_dcp_launch(ctx, gadget_dcp_args(ctx, diff, LN, dig, R * 2, ell, w, 1), st);
    if (rc) return rc;

    rc = lift_ntt_digits(ctx, dig, dn, R * 2 * ell, w, st);
    if (rc) return rc;

    MacArgs ma;
    memset(&ma, 0, sizeof(ma));
    ma.in = in;
    ma.dn = dn;
    ma.C = C;
    ma.out = out;
    ma.R = R;
    ma.Rp = Rp;
    ma.n = n;
    ma.c_stride = c_stride;
    ma.N = ctx->N;
    ma.L = ctx->L;
    ma.ell = ell;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        ma.q[l] = ctx->q[l];
        ma.mu[l] = ctx->mu[l];
    }
    if (ell == 5)
        pdl_launch(coltor_mac_kernel<10>, dim3((unsigned)grid_for(ctx, R * LN / 4)), dim3(CT_THREADS), 0, st, ma);
    else
        pdl_launch(coltor_mac_kernel<0>, dim3((unsigned)grid_for(ctx, R * LN / 4)), dim3(CT_THREADS), 0, st, ma);
    return launch_status(cudaGetLastError());
}

bool overlaps(const void *a, uint64_t abytes, const void *b, uint64_t bbytes) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bbytes && y < x + abytes;
}

}  // namespace

extern "C" uint64_t pir_coltor_batch_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint64_t G, uint32_t ell) {
    if (!ctx || n == 0 || G == 0 || ell == 0 || ell > GD_MAX_ELL || n > (1ull << 32) || G > (1ull << 31) ||
        G * ((n + 1) / 2) >= (1ull << 31))
        return 0;
    return ct_layout(ctx, n, ell, G).total * 4;
}

extern "C" uint64_t pir_coltor_workspace_bytes(const pir_ctx *ctx, uint64_t n, uint32_t ell) {
    return pir_coltor_batch_workspace_bytes(ctx, n, 1, ell);
}

extern "C" int pir_coltor_stage(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w, const uint32_t *in,
                                uint64_t n, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                                void *stream) {
    int rc = check_params(ctx, ell, w, n);
    if (rc) return rc;
    if (!C || !in || !out || !workspace) return PIR_ERR_ARG;
    if (!aligned16(C) || !aligned16(in) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    const CtLayout lay = ct_layout(ctx, n, ell);
    if (workspace_bytes < lay.total * 4) return PIR_ERR_ARG;
    const uint64_t ctb = 2ull * ctx->L * ctx->N * 4;
    if (overlaps(in, n * ctb, out, ((n + 1) / 2) * ctb)) return PIR_ERR_ARG;
    // the stage writes its digits into the workspace while it reads in and writes out
    if (overlaps(workspace, lay.total * 4, in, n * ctb) || overlaps(workspace, lay.total * 4, out, ((n + 1) / 2) * ctb))
        return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    return stage(ctx, C, 0, ell, w, in, n, 1, out, static_cast<uint32_t *>(workspace), lay, (cudaStream_t)stream);
}

extern "C" int pir_coltor_batch(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w, const uint32_t *in,
                                uint64_t n, uint64_t G, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                                void *stream) {
    int rc = check_params(ctx, ell, w, n, G);
    if (rc) return rc;
    if (!C || !in || !out || !workspace) return PIR_ERR_ARG;
    if (!aligned16(C) || !aligned16(in) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    const CtLayout lay = ct_layout(ctx, n, ell, G);
    if (workspace_bytes < lay.total * 4) return PIR_ERR_ARG;
    const uint64_t ctw = 2ull * ctx->L * ctx->N;
    if (overlaps(in, G * n * ctw * 4, out, G * ctw * 4)) return PIR_ERR_ARG;
    // the stages ping-pong through the workspace while the first reads in and the last writes out
    if (overlaps(workspace, lay.total * 4, in, G * n * ctw * 4) || overlaps(workspace, lay.total * 4, out, G * ctw * 4))
        return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    if (n == 1)
        return cudaMemcpyAsync(out, in, G * ctw * 4, cudaMemcpyDeviceToDevice, st) == cudaSuccess ? PIR_OK
                                                                                                : PIR_ERR_CUDA;
    uint32_t *ws = static_cast<uint32_t *>(workspace);
    const uint64_t row = 2ull * ell * ctw;          // words of one stage's RGSW ciphertext
    const uint64_t c_stride = stages_of(n) * row;   // words of one tournament's RGSW ciphertexts
    const uint32_t *cur = in;
    uint64_t cnt = n;
    for (uint32_t s = 0; cnt > 1; ++s) {
        const uint64_t next = (cnt + 1) / 2;
        uint32_t *dst = next == 1 ? out : ws + ((s & 1) ? lay.pong : lay.ping);
        rc = stage(ctx, C + s * row, c_stride, ell, w, cur, cnt, G, dst, ws, lay, st);
        if (rc) return rc;
        cur = dst;
        cnt = next;
    }
    return PIR_OK;
}

extern "C" int pir_coltor(pir_ctx *ctx, const uint32_t *C, uint32_t ell, uint32_t w, const uint32_t *in, uint64_t n,
                          uint32_t *out, void *workspace, uint64_t workspace_bytes, void *stream) {
    return pir_coltor_batch(ctx, C, ell, w, in, n, 1, out, workspace, workspace_bytes, stream);
}
