// encode.cu — offline DB encoding for RowSel.
//
// VIPIR section 2.4: a plaintext record is lifted from R_p to R_q and
// transformed by the NTT before plaintext-ciphertext products (the ~4x
// "plaintext inflation").  GPIR section 2: RowSel wants data contiguous along
// k/n per evaluation point p rather than the p-major (NTT-friendly) layout,
// so the encoder writes the transposed layout directly:
//
//     db[p*D0*D1p + s*D0*128 + k*W_s + (n - 128*s)] = NTT(record(k,n))[l][j]
//
// with p = l*N + j, s = n/128 the column slab and W_s its width (128, or
// D1p - 128*(S-1) for the last slab).  Every (p, slab) is one contiguous
// D0 x W_s block that the scan streams with 1-D bulk copies.
//
// One CTA encodes 4 consecutive columns n0..n0+3 of DB row k for one prime l:
// 4 rows of N words in shared memory, forward NTT, then one 16-byte store per
// evaluation point.
#include "common.cuh"
#include "ntt_core.cuh"

namespace {

constexpr int kEncThreads = 512;
constexpr uint32_t kCols = 4;

struct EncodeArgs {
    const uint32_t *raw;  // [kcnt][D1][N]
    uint32_t *db;
    uint32_t k0, kcnt, D0, D1, D1p, S, Wlast;
    uint32_t groups;      // D1p / 4
};

__global__ void __launch_bounds__(kEncThreads) encode_kernel(const __grid_constant__ EncodeArgs A,
                                                             const __grid_constant__ RnsParams P) {
    extern __shared__ __align__(16) uint32_t sm[];  // [4][N]
    const uint32_t N = P.N;
    // blockIdx.x: column group, blockIdx.y: DB row within the chunk, blockIdx.z: prime
    const uint32_t grp = blockIdx.x, kk = blockIdx.y, l = blockIdx.z;
    const uint32_t n0 = grp * kCols;
    const uint32_t q = P.q[l];

    // lift: residue of each coefficient mod q_l (padding columns are zero)
    for (uint32_t i = threadIdx.x; i < kCols * N; i += blockDim.x) {
        const uint32_t c = i / N, t = i - c * N, n = n0 + c;
        uint32_t v = 0;
        if (n < A.D1) v = A.raw[((uint64_t)kk * A.D1 + n) * N + t] % q;
        sm[i] = v;
    }
    __syncthreads();
    ntt_rows_smem<true>(sm, kCols, P, [l](uint32_t) { return l; });

    const uint32_t k = A.k0 + kk;
    const uint32_t s = n0 / PIR_SLAB;
    const uint32_t Ws = (s == A.S - 1) ? A.Wlast : PIR_SLAB;
    const uint64_t pstride = (uint64_t)A.D0 * A.D1p;
    const uint64_t base = (uint64_t)s * A.D0 * PIR_SLAB + (uint64_t)k * Ws + (n0 - s * PIR_SLAB);
    for (uint32_t j = threadIdx.x; j < N; j += blockDim.x) {
        uint4 v;
        v.x = fwd_final(sm[0 * N + j], q);
        v.y = fwd_final(sm[1 * N + j], q);
        v.z = fwd_final(sm[2 * N + j], q);
        v.w = fwd_final(sm[3 * N + j], q);
        const uint64_t p = (uint64_t)l * N + j;
        *reinterpret_cast<uint4 *>(A.db + p * pstride + base) = v;
    }
}

}  // namespace

extern "C" uint64_t pir_db_bytes(const pir_ctx *ctx, uint32_t D0, uint32_t D1) {
    if (!ctx || D0 == 0 || D1 == 0) return 0;
    const uint64_t D1p = ((uint64_t)D1 + 3) / 4 * 4;
    return (uint64_t)ctx->L * ctx->N * D0 * D1p * 4;
}

extern "C" int pir_db_encode(pir_ctx *ctx, const uint32_t *raw, uint32_t k0, uint32_t kcnt, uint32_t D0,
                             uint32_t D1, uint32_t *db, void *stream) {
    if (!ctx || !raw || !db || !aligned16(raw) || !aligned16(db)) return PIR_ERR_ARG;
    if (D0 == 0 || D1 == 0 || kcnt == 0 || (uint64_t)k0 + kcnt > D0) return PIR_ERR_ARG;
    if (kcnt > 65535) return PIR_ERR_UNSUPPORTED;  // grid.y limit; encode in row chunks
    EncodeArgs A;
    A.raw = raw;
    A.db = db;
    A.k0 = k0;
    A.kcnt = kcnt;
    A.D0 = D0;
    A.D1 = D1;
    A.D1p = (D1 + 3) / 4 * 4;
    A.S = (D1 + PIR_SLAB - 1) / PIR_SLAB;
    A.Wlast = A.D1p - PIR_SLAB * (A.S - 1);
    A.groups = A.D1p / kCols;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    dim3 grid(A.groups, kcnt, ctx->L);
    const size_t smem = (size_t)kCols * ctx->N * sizeof(uint32_t);
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        cudaFuncSetAttribute(encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        attr_set[ctx->device] = true;
    }
    encode_kernel<<<grid, kEncThreads, smem, (cudaStream_t)stream>>>(A, rns_params(ctx));
    return launch_status(cudaGetLastError());
}
