// ntt.cu — batched RNS negacyclic NTT / INTT entry points.
//
// VIPIR sections 2.3 and 4.3: the per-row transform of an L x N residue
// matrix, one kernel per transform for N = 2^12 because the row fits on chip.
// Layout [cnt][L][N]: row r = poly*L + l uses prime l.  One CTA transforms
// RPC = max(1, 4096/N) rows staged in shared memory (16 KiB for N = 4096).
#include "common.cuh"
#include "ntt_core.cuh"

namespace {

constexpr int kNttThreads = 512;
constexpr uint32_t kMaxRowsPerCta = 4096 / 16;  // rows per CTA for the smallest ring (N = 16)

template <bool FWD>
__global__ void __launch_bounds__(kNttThreads) ntt_kernel(const uint32_t *__restrict__ in, uint32_t *out,
                                                          uint64_t rows, uint32_t rpc,
                                                          const __grid_constant__ RnsParams P) {
    extern __shared__ __align__(16) uint32_t sm[];
    __shared__ uint8_t row_prime[kMaxRowsPerCta];
    const uint32_t N = P.N, L = P.L, logN = P.logN;
    const uint64_t row0 = (uint64_t)blockIdx.x * rpc;
    const uint32_t nrows = (uint32_t)((rows - row0) < rpc ? (rows - row0) : rpc);
    const uint32_t nwords = nrows * N;  // multiple of 16
    const uint4 *src = reinterpret_cast<const uint4 *>(in + row0 * N);
    uint4 *s4 = reinterpret_cast<uint4 *>(sm);
    for (uint32_t i = threadIdx.x; i < nwords / 4; i += blockDim.x) s4[i] = src[i];
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

template <bool FWD>
int ntt_launch(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    if (!ctx) return PIR_ERR_ARG;
    if (cnt == 0) return PIR_OK;
    if (!in || !out || !aligned16(in) || !aligned16(out)) return PIR_ERR_ARG;
    const uint64_t rows = cnt * ctx->L;
    if (rows / ctx->L != cnt || rows > (1ull << 40)) return PIR_ERR_ARG;
    const uint32_t rpc = ctx->N >= 4096 ? 1 : 4096 / ctx->N;
    const uint64_t grid = (rows + rpc - 1) / rpc;
    if (grid > 0x7fffffffull) return PIR_ERR_ARG;
    const size_t smem = (size_t)rpc * ctx->N * sizeof(uint32_t);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    ntt_kernel<FWD><<<(unsigned)grid, kNttThreads, smem, (cudaStream_t)stream>>>(in, out, rows, rpc,
                                                                                  rns_params(ctx));
    return launch_status(cudaGetLastError());
}

}  // namespace

extern "C" int pir_ntt_fwd(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    return ntt_launch<true>(ctx, in, out, cnt, stream);
}

extern "C" int pir_ntt_inv(pir_ctx *ctx, const uint32_t *in, uint32_t *out, uint64_t cnt, void *stream) {
    return ntt_launch<false>(ctx, in, out, cnt, stream);
}
