// synth.cu — device half of the seeded input generator (see synth/__init__.py).
//
// Element idx of tensor `tid` under `seed`:
//     v = splitmix64((tid << 56) ^ (seed << 48) ^ idx)
// with splitmix64 the SplitMix64 output function (Steele, Lea, Flood,
// OOPSLA 2014) applied to x + 0x9E3779B97F4A7C15.  Holds no arithmetic of
// the PIR method; it only fills buffers with test and benchmark inputs.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t key(uint32_t seed, uint32_t tid, uint64_t idx) {
    return ((uint64_t)tid << 56) ^ ((uint64_t)seed << 48) ^ idx;
}

enum Kind { COEFF = 0, WORD = 1, RESIDUE = 2 };

struct Res { uint32_t N, L; uint64_t q[4]; };

__global__ void fill_u32(uint32_t *out, uint64_t count, uint64_t idx0, uint32_t seed, uint32_t tid, int kind,
                         Res R) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t idx = idx0 + i;
        const uint64_t v = sm64(key(seed, tid, idx));
        uint32_t o;
        if (kind == COEFF) o = (uint32_t)(v & 0xFFFFu);
        else if (kind == WORD) o = (uint32_t)(v >> 32);
        else o = (uint32_t)(v % R.q[(idx / R.N) % R.L]);
        out[i] = o;
    }
}

__global__ void fill_bytes(uint8_t *out, uint64_t count, uint64_t idx0, uint32_t seed, uint32_t tid) {
    // 16 bytes per thread-iteration; count must be a multiple of 16 (checked on the host)
    uint4 *o4 = reinterpret_cast<uint4 *>(out);
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count / 16;
         i += (uint64_t)gridDim.x * blockDim.x) {
        uint32_t w[4];
        for (int j = 0; j < 4; ++j) {
            uint32_t x = 0;
            for (int b = 0; b < 4; ++b) {
                const uint64_t idx = idx0 + i * 16 + j * 4 + b;
                x |= (uint32_t)(sm64(key(seed, tid, idx)) & 0xFFu) << (8 * b);
            }
            w[j] = x;
        }
        o4[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

int grid_for(uint64_t count) {
    uint64_t g = (count + 255) / 256;
    if (g > 152ull * 64) g = 152ull * 64;
    if (g == 0) g = 1;
    return (int)g;
}

}  // namespace

extern "C" int synth_fill(uint32_t *out, uint64_t count, uint64_t idx0, uint32_t seed, uint32_t tid, int kind,
                          uint32_t N, uint32_t L, const uint32_t *q, void *stream) {
    if (!out || count == 0) return count == 0 ? 0 : -1;
    Res R{};
    R.N = N ? N : 1;
    R.L = L ? L : 1;
    for (uint32_t l = 0; l < 4; ++l) R.q[l] = (q && l < L) ? q[l] : 1;
    if (kind == RESIDUE && (!q || L == 0 || L > 4 || N == 0)) return -1;
    fill_u32<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(out, count, idx0, seed, tid, kind, R);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

extern "C" int synth_fill_bytes(uint8_t *out, uint64_t count, uint64_t idx0, uint32_t seed, uint32_t tid,
                                void *stream) {
    if (!out || count % 16 || (reinterpret_cast<uintptr_t>(out) & 15)) return -1;
    if (count == 0) return 0;
    fill_bytes<<<grid_for(count / 16), 256, 0, (cudaStream_t)stream>>>(out, count, idx0, seed, tid);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
