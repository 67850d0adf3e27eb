// ntt.cu — batched RNS negacyclic NTT / INTT entry points.
//
// VIPIR sections 2.3 and 4.3: the per-row transform of an L x N residue
// matrix, one kernel per transform for N = 2^12 because the row fits on chip.
// Layout [cnt][L][N]: row r = poly*L + l uses prime l.  One CTA transforms
// RPC = max(1, 4096/N) rows staged in shared memory (16 KiB for N = 4096).
#include "common.cuh"
#include "ntt_core.cuh"

namespace {

// Loads that bypass L1: a row is read once, and L1 is better spent on the
// twiddle pairs that every CTA of a prime reads.
__device__ __forceinline__ uint32_t ld_na(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

constexpr int kNttThreads = 512;
constexpr uint32_t kMaxRowsPerCta = 4096 / 16;  // rows per CTA for the smallest ring (N = 16)

// LIFT: the input is [cnt][N] plain 32-bit coefficients; row r = poly*L + l
// reads polynomial poly and lifts each coefficient to its residue mod q_l.
template <bool FWD, bool LIFT>
__global__ void __launch_bounds__(kNttThreads) ntt_kernel(const uint32_t *__restrict__ in, uint32_t *out,
                                                          uint64_t rows, uint32_t rpc,
                                                          const __grid_constant__ RnsParams P) {
    pdl_wait();
    extern __shared__ __align__(16) uint32_t sm[];
    __shared__ uint8_t row_prime[kMaxRowsPerCta];
    const uint32_t N = P.N, L = P.L, logN = P.logN;
    const uint64_t row0 = (uint64_t)blockIdx.x * rpc;
    const uint32_t nrows = (uint32_t)((rows - row0) < rpc ? (rows - row0) : rpc);
    const uint32_t nwords = nrows * N;  // multiple of 16
    uint4 *s4 = reinterpret_cast<uint4 *>(sm);
    if (LIFT) {
        for (uint32_t i = threadIdx.x; i < nwords; i += blockDim.x) {
            const uint64_t row = row0 + (i >> logN);
            const uint32_t l = (uint32_t)(row % L), q = P.q[l];
            const uint32_t r = barrett32_lazy(in[(row / L) * N + (i & (N - 1))], q, (uint32_t)(P.mu[l] >> 32));
            sm[i] = r >= q ? r - q : r;
        }
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + row0 * N);
        for (uint32_t i = threadIdx.x; i < nwords / 4; i += blockDim.x) s4[i] = src[i];
    }
    if (threadIdx.x < nrows) row_prime[threadIdx.x] = (uint8_t)((row0 + threadIdx.x) % L);
    __syncthreads();

    auto prime_of = [&](uint32_t r) -> uint32_t { return row_prime[r]; };
    ntt_rows_smem<FWD>(sm, nrows, P, prime_of);

    uint4 *dst = reinterpret_cast<uint4 *>(out + row0 * N);
    for (uint32_t i = threadIdx.x; i < nwords / 4; i += blockDim.x) {
        const uint32_t l = row_prime[(i * 4) >> logN];
        const uint32_t q = P.q[l];
        uint4 v = s4[i];
        if (FWD) {
            v.x = fwd_final(v.x, q); v.y = fwd_final(v.y, q);
            v.z = fwd_final(v.z, q); v.w = fwd_final(v.w, q);
        } else {
            const uint32_t a = P.ninv[l], b = P.ninv_shoup[l];
            v.x = inv_final(v.x, a, b, q); v.y = inv_final(v.y, a, b, q);
            v.z = inv_final(v.z, a, b, q); v.w = inv_final(v.w, a, b, q);
        }
        dst[i] = v;
    }
}

template <bool FWD, bool LIFT>
__global__ void __launch_bounds__(kT4) ntt4096_kernel(const uint32_t *__restrict__ in, uint32_t *out,
                                                      const __grid_constant__ RnsParams P) {
    pdl_wait();
    static_assert(FWD || !LIFT, "the lift feeds the forward transform only");
    __shared__ __align__(16) uint32_t sm[kN4];
    const uint64_t row = blockIdx.x;
    const uint32_t l = (uint32_t)(row % P.L);
    const uint32_t q = P.q[l];
    const uint2 *T = tw_pairs(P.tw, l, kN4, FWD ? TW_FWD : TW_INV);
    const uint32_t mb = (uint32_t)(P.mu[l] >> 32);   // floor(2^32 / q) for the lift
    const uint32_t *src = in + (LIFT ? row / P.L : row) * kN4;
    uint32_t *dst = out + row * kN4;
    const uint32_t t = threadIdx.x;
    const Swz4096 z(t);       // shared-memory placement of the row
    uint32_t x[16];
    if (FWD) {
        // round 0: stages 0-3, distance 256, elements t + 256 i
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = LIFT ? barrett32_lazy(src[t + 256 * i], q, mb) : src[t + 256 * i];
        fwd_round16(x, 0, 0, T, q);
#pragma unroll
        for (int i = 0; i < 16; ++i) sm[z.col(i)] = x[i];
        __syncthreads();
        // round 1: stages 4-7, distance 16, elements (t>>4)*256 + (t&15) + 16 i
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = sm[z.mid(i)];
        fwd_round16(x, 4, t >> 4, T, q);
#pragma unroll
        for (int i = 0; i < 16; ++i) sm[z.mid(i)] = x[i];
        __syncthreads();
        // round 2: stages 8-11, distance 1, elements 16t .. 16t+15
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = sm[z.row(i)];
        fwd_round16(x, 8, t, T, q);
#pragma unroll
        for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<uint4 *>(dst + 16 * t + i) = make_uint4(fwd_final6(x[i], q), fwd_final6(x[i + 1], q),
                                                                      fwd_final6(x[i + 2], q), fwd_final6(x[i + 3], q));
    } else {
        // round 0: stages 11-8, distance 1, elements 16t .. 16t+15
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4 *>(src + 16 * t + i);
            x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
        }
        inv_round16(x, 11, t, T, q);
#pragma unroll
        for (int i = 0; i < 16; ++i) sm[z.row(i)] = x[i];
        __syncthreads();
        // round 1: stages 7-4, distance 16
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = sm[z.mid(i)];
        inv_round16(x, 7, t >> 4, T, q);
#pragma unroll
        for (int i = 0; i < 16; ++i) sm[z.mid(i)] = x[i];
        __syncthreads();
        // round 2: stages 3-0, distance 256, elements t + 256 i; then N^-1
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = sm[z.col(i)];
        inv_round16(x, 3, 0, T, q);
        const uint32_t ni = P.ninv[l], nis = P.ninv_shoup[l];
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[t + 256 * i] = inv_final(x[i], ni, nis, q);
    }
}

// Forward (and lift + forward) for N = 4096 on two rows of the same prime
// per CTA, rows 2pp*L + l and (2pp+1)*L + l: every twiddle load serves both
// rows and each thread carries two independent butterfly chains.  Rounds as
// in ntt4096_kernel; rows placed in shared memory by Swz4096.  (An exchange
// of the last round's inputs by warp shuffles -- a 16 x 16 transpose inside
// each half-warp by xor butterflies, 32 shuffles and 64 selects per row --
// measured slower than the swizzled shared-memory exchange.)
// SMALL (with LIFT): the caller guarantees every input word is below every
// q_l (gadget digits), so the lift is the identity.
template <bool LIFT, bool SMALL = false>
__global__ void __launch_bounds__(kT4, 4) ntt4096x2_fwd_kernel(const uint32_t *__restrict__ in, uint32_t *out,
                                                            uint64_t cnt, const __grid_constant__ RnsParams P) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sa[kN4];
    __shared__ __align__(16) uint32_t sb[kN4];
    // Prime-major CTA order: the CTAs resident on an SM at a time transform
    // rows of one prime, so one prime's 32 KiB of twiddle pairs stays in L1
    // (pair-major order kept all L tables live and missed L1 on a third of
    // the twiddle loads; the lift's raw rows are then re-read from L2 per prime).
    const uint32_t npairs = (uint32_t)((cnt + 1) / 2);   // the grid (npairs * L CTAs) is below 2^31
    const uint64_t pp = blockIdx.x % npairs;
    const uint32_t l = blockIdx.x / npairs;
    const uint64_t p0 = 2 * pp, p1 = p0 + 1;
    const bool two = p1 < cnt;
    const uint32_t q = P.q[l];
    const uint2 *T = tw_pairs(P.tw, l, kN4, TW_FWD);
    const uint32_t mb = (uint32_t)(P.mu[l] >> 32);   // floor(2^32 / q) for the lift
    const uint32_t *src0 = in + (LIFT ? p0 : p0 * P.L + l) * kN4;
    const uint32_t *src1 = in + (LIFT ? p1 : p1 * P.L + l) * kN4;
    uint32_t *dst0 = out + (p0 * P.L + l) * kN4, *dst1 = out + (p1 * P.L + l) * kN4;
    const uint32_t t = threadIdx.x;
    uint32_t x[16], y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t a = ld_na(src0 + t + 256 * i);
        const uint32_t b = two ? ld_na(src1 + t + 256 * i) : 0u;
        x[i] = (LIFT && !SMALL) ? barrett32_lazy(a, q, mb) : a;   // [0, 2q): the rounds' input range
        y[i] = (LIFT && !SMALL) ? barrett32_lazy(b, q, mb) : b;
    }
    const Swz4096 z(t);
    fwd_round16x2(x, y, 0, 0, T, q);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        sa[z.col(i)] = x[i];
        sb[z.col(i)] = y[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = sa[z.mid(i)];
        y[i] = sb[z.mid(i)];
    }
    fwd_round16x2(x, y, 4, t >> 4, T, q);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        sa[z.mid(i)] = x[i];
        sb[z.mid(i)] = y[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = sa[z.row(i)];
        y[i] = sb[z.row(i)];
    }
    fwd_round16x2(x, y, 8, t, T, q);
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        *reinterpret_cast<uint4 *>(dst0 + 16 * t + i) = make_uint4(fwd_final6(x[i], q), fwd_final6(x[i + 1], q),
                                                                   fwd_final6(x[i + 2], q), fwd_final6(x[i + 3], q));
        if (two)
            *reinterpret_cast<uint4 *>(dst1 + 16 * t + i) = make_uint4(fwd_final6(y[i], q), fwd_final6(y[i + 1], q),
                                                                       fwd_final6(y[i + 2], q), fwd_final6(y[i + 3], q));
    }
}

// Inverse for N = 4096 on two rows of one prime per CTA (as the forward).
__global__ void __launch_bounds__(kT4, 4) ntt4096x2_inv_kernel(const uint32_t *__restrict__ in, uint32_t *out,
                                                            uint64_t cnt, const __grid_constant__ RnsParams P) {
    pdl_wait();
    __shared__ __align__(16) uint32_t sa[kN4];
    __shared__ __align__(16) uint32_t sb[kN4];
    const uint64_t pp = blockIdx.x / P.L;
    const uint32_t l = blockIdx.x % P.L;
    const uint64_t r0 = (2 * pp) * P.L + l, r1 = (2 * pp + 1) * P.L + l;
    const bool two = 2 * pp + 1 < cnt;
    const uint32_t q = P.q[l];
    const uint2 *T = tw_pairs(P.tw, l, kN4, TW_INV);
    const uint32_t t = threadIdx.x;
    uint32_t x[16], y[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(in + r0 * kN4 + 16 * t + k);
        const uint4 v = two ? *reinterpret_cast<const uint4 *>(in + r1 * kN4 + 16 * t + k) : make_uint4(0, 0, 0, 0);
        x[k] = u.x; x[k + 1] = u.y; x[k + 2] = u.z; x[k + 3] = u.w;
        y[k] = v.x; y[k + 1] = v.y; y[k + 2] = v.z; y[k + 3] = v.w;
    }
    inv4096x2_rounds(x, y, sa, sb, T, q, P.ninv[l], P.ninv_shoup[l], out + r0 * kN4, out + r1 * kN4, two);
}

template <bool FWD, bool LIFT = false, bool SMALL = false>
int ntt_launch(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    if (!ctx) return PIR_ERR_ARG;
    if (cnt == 0) return PIR_OK;
    if (!in || !out || !aligned16(in) || !aligned16(out)) return PIR_ERR_ARG;
    const uint64_t rows = cnt * ctx->L;
    if (rows / ctx->L != cnt || rows > (1ull << 40)) return PIR_ERR_ARG;
    if (LIFT) {  // [cnt][N] in, [cnt][L][N] out: the two must not overlap at all
        const uint64_t ib = cnt * ctx->N * 4, ob = rows * ctx->N * 4;
        const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out;
        if (a < b + ob && b < a + ib) return PIR_ERR_ARG;
    }
    const uint32_t rpc = ctx->N >= 4096 ? 1 : 4096 / ctx->N;
    const uint64_t grid = (rows + rpc - 1) / rpc;
    if (grid > 0x7fffffffull) return PIR_ERR_ARG;
    const size_t smem = (size_t)rpc * ctx->N * sizeof(uint32_t);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    if (ctx->N == (uint32_t)kN4) {
        if (!LIFT && in != out && (uint64_t)((in < out ? out - in : in - out)) < rows * kN4)
            return PIR_ERR_ARG;  // partial overlap
        // two rows of one prime per CTA, unless that leaves SMs idle: a small
        // launch (the first stages of an expansion, the last of a tournament)
        // is latency-bound, and one row per CTA halves each CTA's chain
        if (cnt > 1 && (cnt + 1) / 2 * ctx->L >= (uint64_t)ctx->num_sms) {
            const uint64_t g2 = (cnt + 1) / 2 * ctx->L;
            if (g2 > 0x7fffffffull) return PIR_ERR_ARG;
            if (FWD)
                pdl_launch(ntt4096x2_fwd_kernel<LIFT, SMALL>, dim3((unsigned)g2), dim3(kT4), 0, (cudaStream_t)stream, in,
                           out, cnt, rns_params(ctx));
            else
                pdl_launch(ntt4096x2_inv_kernel, dim3((unsigned)g2), dim3(kT4), 0, (cudaStream_t)stream, in, out, cnt,
                           rns_params(ctx));
        } else {
            pdl_launch(ntt4096_kernel<FWD, LIFT>, dim3((unsigned)rows), dim3(kT4), 0, (cudaStream_t)stream, in, out,
                       rns_params(ctx));
        }
        return launch_status(cudaGetLastError());
    }
    pdl_launch(ntt_kernel<FWD, LIFT>, dim3((unsigned)grid), dim3(kNttThreads), smem, (cudaStream_t)stream, in, out,
               rows, rpc, rns_params(ctx));
    return launch_status(cudaGetLastError());
}

}  // namespace

extern "C" int pir_ntt_fwd(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    return ntt_launch<true>(ctx, in, out, cnt, stream);
}

extern "C" int pir_ntt_inv(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    return ntt_launch<false>(ctx, in, out, cnt, stream);
}

extern "C" int pir_lift_ntt(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, void *stream) {
    return ntt_launch<true, true>(ctx, raw, out, cnt, stream);
}

// The lift + forward NTT of gadget digits (ColTor, ExpandQuery, the RGSW
// conversion): when every digit is below every prime (2^w <= min q_l) the
// lift is the identity and is skipped; otherwise as pir_lift_ntt.
int lift_ntt_digits(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, uint32_t w, void *stream) {
    if (!ctx) return PIR_ERR_ARG;
    uint32_t qmin = ctx->q[0];
    for (uint32_t l = 1; l < ctx->L; ++l) qmin = ctx->q[l] < qmin ? ctx->q[l] : qmin;
    if (w < 32 && (1ull << w) <= qmin) return ntt_launch<true, true, true>(ctx, raw, out, cnt, stream);
    return ntt_launch<true, true>(ctx, raw, out, cnt, stream);
}
