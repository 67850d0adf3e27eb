// scalar.cu — scalar-HE DB scan (SimplePIR-family first fold) on tcgen05.
//
// VIPIR section 2.5: the online server work of SimplePIR with B batched
// queries is a D1 x B x D0 GEMM of a byte DB by 32-bit query words, mod 2^32
// (the reduction is free).  VIPIR section 4.1: run it on tensor cores by
// splitting each 32-bit word into four bytes, Q = sum_i 2^(8i) Q_i, so that
//     DB * Q = sum_i 2^(8i) (DB * Q_i)   mod 2^32.
//
// GB300 (sm_103a) has no integer tensor-core MMA (tcgen05 kind::i8 is not
// available on this target), so the byte products run on the fp16 path
// (kind::f16) where they are still exact:
//  * Q's bytes are re-expressed as balanced base-256 digits d_i in
//    [-128, 127] (Q = sum_i 256^i d_i mod 2^32), stored as fp16 (exact);
//  * DB bytes 0..255 are exact fp16 values;
//  * every product is an integer of magnitude <= 255*128 = 32640, so a sum
//    of 512 of them stays below 2^24 and is exact in the fp32 accumulator.
// The accumulator is therefore drained every 512 columns of the DB (a
// "chunk"): the four digit planes are converted to integers and folded into
// 32-bit running sums as  acc += S_0 + (S_1 << 8) + (S_2 << 16) + (S_3 << 24)
// with wrap-around, which is exactly the byte-split identity mod 2^32.
//
// Kernel structure (one CTA per SM, persistent over 128-row DB tiles):
//   warp 0      TMA producer: the 128 x 64-byte DB tile (tensor map) and the
//               matching 256 x 64 fp16 digit tile (1-D bulk copy of a block
//               pre-swizzled by the prep kernel) into a 4-stage ring;
//   warp 1      TMEM allocator and MMA issue (the warp runs the loop, so
//               its control flow and operands stay warp-uniform; one elected
//               lane issues):
//               4 x tcgen05.mma (M=128, N=256, K=16) per stage into one of
//               two 256-column fp32 accumulators (double buffered so that a
//               drain overlaps the next chunk's MMAs);
//   warps 2-9   converters: DB bytes -> fp16 in the 128B-swizzled K-major
//               layout the MMA reads; two groups of four warps take the even
//               and the odd stages, so two stages convert at once;
//   warps 10-13 epilogue: tcgen05.ld of a drained accumulator, integer
//               conversion and the shifted accumulation; one row per thread;
//               the 64 running sums per row are written at the end of a tile.
// All mbarrier waits are bounded (PIR_STATUS_TIMEOUT); TMEM is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"

namespace {

constexpr int SC_NS = 4;                      // pipeline stages (4 x 56 KiB)
constexpr int SC_KB = 64;                     // DB bytes (K elements) per stage
constexpr int SC_TM = 128;                    // DB rows per tile (MMA M)
constexpr int SC_BQ = 64;                     // queries per pass (digit planes hold 4 x 64 rows)
constexpr int SC_N = 4 * SC_BQ;               // MMA N = 256
constexpr int SC_CHUNK_STAGES = 8;            // stages per accumulator chunk: 512 K elements
constexpr uint32_t SC_A_BYTES = SC_TM * 128;  // fp16 A tile: 128 rows x 64 halves
constexpr uint32_t SC_B_BYTES = SC_N * 128;   // fp16 B tile: 256 rows x 64 halves
constexpr uint32_t SC_U8_BYTES = SC_TM * SC_KB;
constexpr uint32_t SC_STAGE_BYTES = SC_A_BYTES + SC_B_BYTES + SC_U8_BYTES;
constexpr int SC_THREADS = 448;
constexpr uint32_t SC_TMEM_COLS = 512;

// One lane of a fully active warp (the same one every time): true there.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n.reg .pred P;\n"
        "elect.sync _|P, 0xffffffff;\n"
        "selp.u32 %0, 1, 0, P;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// Byte offset of (row, 16-byte chunk j) in a K-major tile with the 128-byte
// swizzle: rows of 128 B, 8-row groups of 1 KiB, chunk index XOR (row % 8).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t j) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((j ^ (row & 7u)) << 4);
}

// ---------------------------------------------------------------- digit prep
// ws block kb (64 DB columns) = 256 rows (plane i, query b -> row 64 i + b)
// x 64 fp16 digits, 128B-swizzled, 32 KiB.
__global__ void __launch_bounds__(256) digits_kernel(const uint32_t *__restrict__ Q, uint32_t C, uint32_t B,
                                                     uint8_t *__restrict__ ws) {
    __shared__ uint32_t tile[64][SC_BQ + 1];
    pdl_wait();
    const uint32_t kb = blockIdx.x;
    for (uint32_t i = threadIdx.x; i < 64 * SC_BQ; i += blockDim.x) {
        const uint32_t k = i / SC_BQ, b = i % SC_BQ;
        tile[k][b] = b < B ? Q[(uint64_t)(kb * 64 + k) * B + b] : 0u;
    }
    __syncthreads();
    uint8_t *blk = ws + (uint64_t)kb * SC_B_BYTES;
    for (uint32_t t = threadIdx.x; t < SC_N * 8; t += blockDim.x) {
        const uint32_t n = t >> 3, j = t & 7;         // row n = 64*plane + b, chunk j = k 8j..8j+7
        const uint32_t plane = n / SC_BQ, b = n % SC_BQ;
        __align__(16) __half h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            uint64_t y = tile[8 * j + e][b];
            int d = 0;
            for (uint32_t i = 0; i <= plane; ++i) {   // balanced base-256 digits, low first
                const int lo = (int)(y & 0xFFu);
                d = lo >= 128 ? lo - 256 : lo;
                y = (y - (uint64_t)(int64_t)d) >> 8;
            }
            h[e] = __int2half_rn(d);
        }
        *reinterpret_cast<uint4 *>(blk + sw128_offset(n, j)) = *reinterpret_cast<const uint4 *>(h);
    }
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    // start>>4 | LBO (unused for swizzled K-major) | SBO 1024>>4 | version 1 | SWIZZLE_128B
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16, A = B = F16, D = F32, K-major A and B, N = 256, M = 128
constexpr uint32_t SC_IDESC = (1u << 4) | ((uint32_t)(SC_N >> 3) << 17) | ((uint32_t)(SC_TM >> 4) << 24);

// The four K = 16 MMAs of one stage; descriptors advance 32 bytes (2 units) per
// MMA inside the 128-byte swizzle atom.  acc = 0 starts the accumulator.
__device__ __forceinline__ void mma4(uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p, t;\nsetp.ne.b32 p, %3, 0;\nsetp.eq.b32 t, %3, %3;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %4, t;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %4, t;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %4, t;\n}\n" ::"r"(d),
        "l"(ad), "l"(bd), "r"(acc), "r"(SC_IDESC), "l"(ad + 2), "l"(bd + 2), "l"(ad + 4), "l"(bd + 4), "l"(ad + 6),
        "l"(bd + 6)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }


struct ScalarArgs {
    const uint8_t *ws;   // digit blocks
    uint32_t *out;
    uint32_t *status;
    uint64_t R;
    uint32_t C, B, ntiles, nkb;
};

__global__ void __launch_bounds__(SC_THREADS, 1)
    scalar_kernel(const __grid_constant__ CUtensorMap dbmap, const __grid_constant__ ScalarArgs A) {
    extern __shared__ uint8_t smraw[];
    // 1 KiB alignment for the swizzle atoms
    const uint32_t base_s = smem_u32(smraw);
    uint8_t *sm = smraw + (((base_s + 1023u) & ~1023u) - base_s);
    uint8_t *stA = sm;                                   // [NS][A]
    uint8_t *stB = stA + SC_NS * SC_A_BYTES;             // [NS][B]
    uint8_t *stU = stB + SC_NS * SC_B_BYTES;             // [NS][U8]
    uint64_t *bars = reinterpret_cast<uint64_t *>(stU + SC_NS * SC_U8_BYTES);
    uint64_t *full = bars, *conv = bars + SC_NS, *empty = bars + 2 * SC_NS;
    uint64_t *accf = bars + 3 * SC_NS, *acce = accf + 2, *done = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC_NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(conv + s, 4);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, 4);
        }
        mbar_init(done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(SC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the set-up above touches no global memory
    const uint32_t nchunks = (A.nkb + SC_CHUNK_STAGES - 1) / SC_CHUNK_STAGES;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_db = policy_evict_first(), pol_q = policy_evict_last();
            uint32_t it = 0;
            for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x) {
                for (uint32_t kb = 0; kb < A.nkb; ++kb, ++it) {
                    const uint32_t s = it % SC_NS, ph = (it / SC_NS) & 1;
                    if (abort_flag || !mbar_wait(empty + s, ph ^ 1, A.status)) {
                        abort_flag = 1;
                        continue;
                    }
                    mbar_arrive_expect_tx(full + s, SC_U8_BYTES + SC_B_BYTES);
                    tma_load_2d(stU + s * SC_U8_BYTES, &dbmap, (int)(kb * SC_KB), (int)(t * SC_TM), full + s, pol_db);
                    bulk_g2s(stB + s * SC_B_BYTES, A.ws + (uint64_t)kb * SC_B_BYTES, SC_B_BYTES, full + s, pol_q);
                }
            }
            // copies in flight land in this CTA's shared memory: wait for the last ones
            for (uint32_t i = 0; i < SC_NS && i < it; ++i) {
                const uint32_t j = it - 1 - i;
                mbar_wait(full + j % SC_NS, (j / SC_NS) & 1, A.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (control flow and operands warp-uniform);
        // one elected lane issues the MMAs and commits.
        bool ab = false;
        uint32_t g = 0, s = 0, ph = 0;
        const uint64_t ad0 = sdesc_sw128(smem_u32(stA)), bd0 = sdesc_sw128(smem_u32(stB));
        for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x) {
            ab = __any_sync(0xffffffffu, ab || abort_flag);
            for (uint32_t ch = 0; ch < nchunks; ++ch, ++g) {
                const uint32_t buf = g & 1, use = (g >> 1) & 1;
                ab = __any_sync(0xffffffffu, ab || !mbar_wait(acce + buf, use ^ 1, A.status));
                const uint32_t d = tmem + buf * SC_N;
                const uint32_t kb0 = ch * SC_CHUNK_STAGES, kb_end = min(A.nkb, kb0 + SC_CHUNK_STAGES);
                for (uint32_t kb = kb0; kb < kb_end; ++kb) {
                    ab = __any_sync(0xffffffffu, ab || !mbar_wait(conv + s, ph, A.status));
                    if (!ab) {
                        tc_fence_after();
                        if (elect_one()) {
                            mma4(d, ad0 + s * (SC_A_BYTES >> 4), bd0 + s * (SC_B_BYTES >> 4), kb > kb0);
                            mma_commit(empty + s);        // stage reusable once these MMAs finish
                        }
                        __syncwarp();
                    }
                    if (++s == SC_NS) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ab && elect_one()) mma_commit(accf + buf);  // chunk complete -> epilogue
                __syncwarp();
            }
        }
        if (lane == 0 && ab) abort_flag = 1;
        if (elect_one()) mma_commit(done);
        __syncwarp();
        mbar_wait(done, 0, A.status);

    } else if (warp < 10) {
        // ------------------------------------------------ converters: bytes -> fp16, swizzled
        // two groups of four warps on alternating stages: warps 2-5 the even
        // stages, warps 6-9 the odd ones (with SC_NS = 4 a ring slot always
        // belongs to the same group, so parity waits never skip a phase)
        const uint32_t grp = (uint32_t)(warp - 2) >> 2;
        const uint32_t ct = ((uint32_t)(warp - 2) & 3u) * 32u + lane;   // 0..127 within the group
        uint32_t it = 0;
        for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x) {
            for (uint32_t kb = 0; kb < A.nkb; ++kb, ++it) {
                if ((it & 1u) != grp) continue;
                const uint32_t s = it % SC_NS, ph = (it / SC_NS) & 1;
                if (!abort_flag && !mbar_wait(full + s, ph, A.status)) abort_flag = 1;
                if (!abort_flag) {
                    const uint8_t *u = stU + s * SC_U8_BYTES;
                    uint8_t *a = stA + s * SC_A_BYTES;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t q = ct + 128 * i;          // 16-byte piece: row q/4, part q%4
                        const uint32_t row = q >> 2, part = q & 3;
                        const uint4 w = *reinterpret_cast<const uint4 *>(u + row * SC_KB + part * 16);
                        const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
                        uint32_t h[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // 0x64xx is the fp16 value 1024 + x: subtract 1024 exactly
                            const uint32_t lo = __byte_perm(ws4[e], 0x64646464u, 0x5140);
                            const uint32_t hi = __byte_perm(ws4[e], 0x64646464u, 0x7362);
                            const __half2 c = __floats2half2_rn(1024.f, 1024.f);
                            __half2 l2 = __hsub2(*reinterpret_cast<const __half2 *>(&lo), c);
                            __half2 h2 = __hsub2(*reinterpret_cast<const __half2 *>(&hi), c);
                            h[2 * e] = *reinterpret_cast<uint32_t *>(&l2);
                            h[2 * e + 1] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(a + sw128_offset(row, 2 * part)) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4 *>(a + sw128_offset(row, 2 * part + 1)) =
                            make_uint4(h[4], h[5], h[6], h[7]);
                    }
                    fence_proxy_async();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(conv + s);
            }
        }
    } else {
        // ------------------------------------------------ epilogue: drain, convert, accumulate
        const uint32_t quad = warp & 3;               // TMEM lane quadrant of this warp
        const uint32_t row_in_tile = quad * 32 + lane;
        uint32_t g = 0;
        for (uint32_t t = blockIdx.x; t < A.ntiles; t += gridDim.x) {
            uint32_t acc[SC_BQ];
#pragma unroll
            for (int b = 0; b < SC_BQ; ++b) acc[b] = 0;
            for (uint32_t ch = 0; ch < nchunks; ++ch, ++g) {
                const uint32_t buf = g & 1, use = (g >> 1) & 1;
                if (!abort_flag && !mbar_wait(accf + buf, use, A.status)) abort_flag = 1;
                tc_fence_after();
                if (!abort_flag) {
                    const uint32_t taddr = tmem + ((quad * 32u) << 16) + buf * SC_N;
#pragma unroll
                    for (int plane = 0; plane < 4; ++plane) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t v[32];
                            tmem_ld32(taddr + plane * SC_BQ + half * 32, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int s = __float2int_rn(__uint_as_float(v[j]));
                                acc[half * 32 + j] += (uint32_t)s << (8 * plane);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + buf);
            }
            const uint64_t r = (uint64_t)t * SC_TM + row_in_tile;
            if (r < A.R && !abort_flag) {
                uint32_t *o = A.out + r * A.B;
                if (A.B == SC_BQ) {
#pragma unroll
                    for (int b = 0; b < SC_BQ; b += 4)
                        *reinterpret_cast<uint4 *>(o + b) = make_uint4(acc[b], acc[b + 1], acc[b + 2], acc[b + 3]);
                } else {
#pragma unroll
                    for (int b = 0; b < SC_BQ; ++b)
                        if ((uint32_t)b < A.B) o[b] = acc[b];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(SC_TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- small batches on CUDA cores
//
// For a handful of queries the tensor path wastes its 64-query width: one
// query costs as much as 64.  With B <= 4 the scan is a GEMV that the CUDA
// cores finish under the HBM time of the DB, using the same byte split with
// plain (unsigned) bytes of Q:
//     sum_c db[r][c] Q[c][b] = sum_i 2^(8i) sum_c db[r][c] Q_i[c][b]  mod 2^32,
// where each inner sum is a chain of 4-way byte dot products (dp4a).  An
// inner sum may wrap past 2^32: only its value mod 2^(32-8i) reaches the
// result, so the wrap is harmless.
//
// Query prep: for every 128 DB columns (a box) and query b, the 32 groups of
// 4 columns each become 4 "plane words" (byte j of plane word i = byte i of
// Q[4g + j][b]), 512 bytes per (box, query), stored box-major so that one
// bulk copy stages all B queries of a box.  The prep also zeroes the output,
// which the scan adds into.
//
// Scan: persistent CTAs, one per SM; the (256-row tile, 128-column box)
// units are split into equal contiguous ranges in tile-major order.  Warp 8
// (one thread) streams each unit's 256 x 128-byte DB box (TMA, 128-byte
// swizzle) and its plane words into a 6-stage ring; warps 0-7 own one DB row
// per thread and keep 4 x B running sums (the two column halves of a box in
// separate sums for instruction-level parallelism).  When the range moves to
// another row tile, or ends, each thread adds its combined sums into the
// output with a 32-bit atomic add (mod 2^32, so the order is irrelevant).
constexpr int GV_RT = 256;                     // DB rows per tile (one per consumer thread)
constexpr int GV_KB = 128;                     // DB columns per box (the 128-byte swizzle span)
constexpr int GV_NS = 6;                       // pipeline stages
constexpr int GV_THREADS = GV_RT + 32;
constexpr uint32_t GV_DB_BYTES = GV_RT * GV_KB;        // 32 KiB
constexpr uint32_t GV_QBOX_BYTES = GV_KB * 4;          // plane words of one query for one box: 512 B
constexpr uint32_t GV_MAX_B = 4;

__global__ void __launch_bounds__(256) gemv_prep_kernel(const uint32_t *__restrict__ Q, uint64_t C, uint32_t B,
                                                        uint32_t nkb, uint32_t *__restrict__ planes,
                                                        uint32_t *__restrict__ out, uint64_t out_words) {
    pdl_wait();
    const uint64_t tid = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t groups = (uint64_t)nkb * B * (GV_KB / 4);   // (box, query, group of 4 columns)
    for (uint64_t i = tid; i < groups; i += nthr) {
        const uint32_t g = (uint32_t)(i % (GV_KB / 4));
        const uint64_t kb_b = i / (GV_KB / 4);
        const uint32_t b = (uint32_t)(kb_b % B);
        const uint64_t c0 = (kb_b / B) * GV_KB + 4ull * g;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = (c0 + j < C) ? Q[(c0 + j) * B + b] : 0u;
        uint32_t pl[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            pl[p] = ((w[0] >> (8 * p)) & 0xFFu) | (((w[1] >> (8 * p)) & 0xFFu) << 8) |
                    (((w[2] >> (8 * p)) & 0xFFu) << 16) | (((w[3] >> (8 * p)) & 0xFFu) << 24);
        *reinterpret_cast<uint4 *>(planes + i * 4) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
    for (uint64_t i = tid; i < out_words; i += nthr) out[i] = 0u;
}

struct GemvArgs {
    const uint8_t *planes;   // [nkb][B][32 groups][4 planes] words
    uint32_t *out;           // [R][B], zeroed by the prep kernel
    uint32_t *status;
    uint64_t R;
    uint64_t units;          // ntiles * nkb
    uint32_t nkb;
};

template <int NB>
__global__ void __launch_bounds__(GV_THREADS, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap dbmap, const __grid_constant__ GemvArgs A) {
    constexpr uint32_t QB = NB * GV_QBOX_BYTES;
    extern __shared__ uint8_t smraw[];
    const uint32_t base_s = smem_u32(smraw);
    uint8_t *sm = smraw + (((base_s + 1023u) & ~1023u) - base_s);   // 1 KiB alignment for the swizzle
    uint8_t *stD = sm;                                                // [NS][256 rows x 128 B]
    uint8_t *stQ = stD + GV_NS * GV_DB_BYTES;                         // [NS][NB x 512 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(stQ + GV_NS * QB);
    uint64_t *empty = full + GV_NS;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < GV_NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, GV_RT / 32);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();   // the set-up above touches no global memory
    const uint64_t u0 = A.units * blockIdx.x / gridDim.x, u1 = A.units * (blockIdx.x + 1) / gridDim.x;

    if (warp == GV_RT / 32) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_db = policy_evict_first(), pol_q = policy_evict_last();
            uint32_t it = 0;
            for (uint64_t u = u0; u < u1; ++u, ++it) {
                const uint32_t s = it % GV_NS, ph = (it / GV_NS) & 1;
                if (abort_flag || !mbar_wait(empty + s, ph ^ 1, A.status)) {
                    abort_flag = 1;
                    continue;
                }
                const uint32_t kb = (uint32_t)(u % A.nkb);
                const uint32_t t = (uint32_t)(u / A.nkb);
                mbar_arrive_expect_tx(full + s, GV_DB_BYTES + QB);
                tma_load_2d(stD + s * GV_DB_BYTES, &dbmap, (int)(kb * GV_KB), (int)(t * GV_RT), full + s, pol_db);
                bulk_g2s(stQ + s * QB, A.planes + (uint64_t)kb * QB, QB, full + s, pol_q);
            }
            // copies in flight land in this CTA's shared memory: wait for the last ones
            for (uint32_t i = 0; i < GV_NS && i < it; ++i) {
                const uint32_t j = it - 1 - i;
                mbar_wait(full + j % GV_NS, (j / GV_NS) & 1, A.status);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers: one DB row per thread
    const uint32_t r = threadIdx.x;
    const uint32_t rsw = r & 7u;
    uint32_t acc[NB][4][2];
    auto clear = [&]() {
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[b][p][0] = acc[b][p][1] = 0u;
    };
    auto flush = [&](uint64_t tile) {
        const uint64_t row = tile * GV_RT + r;
        if (row < A.R && !abort_flag) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                uint32_t v = 0;
#pragma unroll
                for (int p = 0; p < 4; ++p) v += (acc[b][p][0] + acc[b][p][1]) << (8 * p);
                atomicAdd(A.out + row * NB + b, v);
            }
        }
    };
    clear();
    uint32_t it = 0;
    uint64_t cur = u0 < u1 ? u0 / A.nkb : 0;
    for (uint64_t u = u0; u < u1; ++u, ++it) {
        const uint64_t tile = u / A.nkb;
        if (tile != cur) {
            flush(cur);
            clear();
            cur = tile;
        }
        const uint32_t s = it % GV_NS, ph = (it / GV_NS) & 1;
        if (!abort_flag && !mbar_wait(full + s, ph, A.status)) abort_flag = 1;
        if (!abort_flag) {
            const uint8_t *rowp = stD + s * GV_DB_BYTES + (r >> 3) * 1024u + rsw * 128u;
            const uint4 *q4 = reinterpret_cast<const uint4 *>(stQ + s * QB);
#pragma unroll
            for (int j = 0; j < 8; ++j) {   // 16-byte chunk j: columns 16j .. 16j+15
                const uint4 d = *reinterpret_cast<const uint4 *>(rowp + ((j ^ rsw) << 4));
                const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int b = 0; b < NB; ++b) {
#pragma unroll
                    for (int gg = 0; gg < 4; ++gg) {   // group 4j + gg: its 4 plane words
                        const uint4 q = q4[b * (GV_KB / 4) + 4 * j + gg];
                        const int h = j >> 2;        // column half of the box: separate sums
                        acc[b][0][h] = __dp4a(dw[gg], q.x, acc[b][0][h]);
                        acc[b][1][h] = __dp4a(dw[gg], q.y, acc[b][1][h]);
                        acc[b][2][h] = __dp4a(dw[gg], q.z, acc[b][2][h]);
                        acc[b][3][h] = __dp4a(dw[gg], q.w, acc[b][3][h]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
    }
    if (u0 < u1) flush(cur);
}

size_t gemv_smem_bytes(uint32_t B) { return 1024 + (size_t)GV_NS * (GV_DB_BYTES + B * GV_QBOX_BYTES) + 256; }

PFN_cuTensorMapEncodeTiled_v12000 get_encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

size_t scalar_smem_bytes() { return 1024 + (size_t)SC_NS * SC_STAGE_BYTES + 256; }

template <int NB>
int gemv_launch(pir_ctx *ctx, const CUtensorMap &map, const GemvArgs &a, cudaStream_t st) {
    static bool attr_set[64] = {};
    const size_t smem = gemv_smem_bytes(NB);
    if (ctx->device >= 0 && ctx->device < 64 && !attr_set[ctx->device]) {
        if (cudaFuncSetAttribute(gemv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PIR_ERR_CUDA;
        attr_set[ctx->device] = true;
    }
    const uint64_t grid = a.units < (uint64_t)ctx->num_sms ? a.units : (uint64_t)ctx->num_sms;
    pdl_launch(gemv_kernel<NB>, dim3((unsigned)grid), dim3(GV_THREADS), smem, st, map, a);
    return launch_status(cudaGetLastError());
}

// B <= 4 queries: plane-word prep (also zeroes out) + the CUDA-core scan.
// The workspace holds nkb * B * 512 bytes, within pir_scalar_workspace_bytes.
int scalar_gemv(pir_ctx *ctx, PFN_cuTensorMapEncodeTiled_v12000 encode, const uint8_t *db, uint64_t R,
                uint64_t C, const uint32_t *Q, uint32_t B, uint32_t *out, void *workspace, cudaStream_t st) {
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    const cuuint64_t gdim[2] = {C, R};
    const cuuint64_t gstride[1] = {C};
    const cuuint32_t box[2] = {GV_KB, GV_RT};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(db), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PIR_ERR_ARG;
    const uint32_t nkb = (uint32_t)((C + GV_KB - 1) / GV_KB);
    const uint64_t ntiles = (R + GV_RT - 1) / GV_RT;
    uint32_t *planes = reinterpret_cast<uint32_t *>(workspace);
    const uint64_t work = (uint64_t)nkb * B * (GV_KB / 4);
    const uint64_t prep_blocks = (work + 255) / 256 < 4096 ? (work + 255) / 256 : 4096;
    pdl_launch(gemv_prep_kernel, dim3((unsigned)(prep_blocks ? prep_blocks : 1)), dim3(256), 0, st, Q, C, B, nkb, planes,
               out, R * B);
    if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;
    GemvArgs a;
    a.planes = reinterpret_cast<const uint8_t *>(workspace);
    a.out = out;
    a.status = ctx->d_status;
    a.R = R;
    a.units = ntiles * nkb;
    a.nkb = nkb;
    switch (B) {
        case 1: return gemv_launch<1>(ctx, map, a, st);
        case 2: return gemv_launch<2>(ctx, map, a, st);
        case 3: return gemv_launch<3>(ctx, map, a, st);
        default: return gemv_launch<4>(ctx, map, a, st);
    }
}

}  // namespace

extern "C" uint64_t pir_scalar_workspace_bytes(uint64_t C, uint32_t B) {
    if (C == 0 || B == 0 || C % SC_KB) return 0;
    return (C / SC_KB) * (uint64_t)SC_B_BYTES;
}

extern "C" int pir_scalar_scan(pir_ctx *ctx, const uint8_t *db, uint64_t R, uint64_t C, const uint32_t *Q,
                               uint32_t B, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                               void *stream) {
    if (!ctx || !db || !Q || !out || !workspace) return PIR_ERR_ARG;
    if (!aligned16(db) || !aligned16(Q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 127))
        return PIR_ERR_ARG;
    if (R == 0 || C == 0 || B == 0) return PIR_ERR_ARG;
    if (C % SC_KB || B > SC_BQ || C > (1ull << 31) || R > (1ull << 31)) return PIR_ERR_UNSUPPORTED;
    if (workspace_bytes < pir_scalar_workspace_bytes(C, B)) return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    auto encode = get_encode_tiled();
    if (!encode) return PIR_ERR_CUDA;
    if (B <= GV_MAX_B) return scalar_gemv(ctx, encode, db, R, C, Q, B, out, workspace, (cudaStream_t)stream);

    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    const cuuint64_t gdim[2] = {C, R};
    const cuuint64_t gstride[1] = {C};
    const cuuint32_t box[2] = {SC_KB, SC_TM};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(db), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PIR_ERR_ARG;

    cudaStream_t st = (cudaStream_t)stream;
    const uint32_t nkb = (uint32_t)(C / SC_KB);
    pdl_launch(digits_kernel, dim3(nkb), dim3(256), 0, st, Q, (uint32_t)C, B, reinterpret_cast<uint8_t *>(workspace));
    if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;

    const size_t smem = scalar_smem_bytes();
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        if (cudaFuncSetAttribute(scalar_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PIR_ERR_CUDA;
        attr_set[ctx->device] = true;
    }
    ScalarArgs a;
    a.ws = reinterpret_cast<const uint8_t *>(workspace);
    a.out = out;
    a.status = ctx->d_status;
    a.R = R;
    a.C = (uint32_t)C;
    a.B = B;
    a.ntiles = (uint32_t)((R + SC_TM - 1) / SC_TM);
    a.nkb = nkb;
    const uint32_t grid = a.ntiles < (uint32_t)ctx->num_sms ? a.ntiles : (uint32_t)ctx->num_sms;
    pdl_launch(scalar_kernel, grid, dim3(SC_THREADS), smem, st, map, a);
    return launch_status(cudaGetLastError());
}

// ---------------------------------------------------------------- allocation-free variant
//
// Some callers cannot allocate device memory when they run the scan: code
// that runs while a framework's caching allocator owns the whole device pool,
// plugin or serving paths that are handed only the input and output buffers,
// and latency-critical loops where a cudaMalloc (which may synchronise the
// device) is not acceptable.  For them the split-query scratch lives in a
// fixed static device array instead of a caller-provided workspace.
//
// Limit: the array holds the digit blocks for at most kNoAllocMaxC DB
// columns (C * 512 bytes; 8 MiB for 16384 columns).  Every GPU on which the
// library is loaded keeps this array until the process exits.
#include <atomic>

namespace {

constexpr uint64_t kNoAllocMaxC = 16384;
constexpr uint64_t kNoAllocScratchBytes = kNoAllocMaxC / SC_KB * SC_B_BYTES;  // 8 MiB

static __device__ __align__(256) uint8_t g_scalar_scratch[kNoAllocScratchBytes];

// Device address of g_scalar_scratch, looked up once per device.
std::atomic<void *> g_scratch_addr[64];

}  // namespace

extern "C" int pir_scalar_scan_noalloc(pir_ctx *ctx, const uint8_t *db, uint64_t R, uint64_t C, const uint32_t *Q,
                                       uint32_t B, uint32_t *out, void *stream) {
    if (!ctx || ctx->device < 0 || ctx->device >= 64) return PIR_ERR_ARG;
    if (C > kNoAllocMaxC) return PIR_ERR_UNSUPPORTED;  // beyond the static scratch
    // Make the context's device current before touching its copy of the array.
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    void *scratch = g_scratch_addr[ctx->device].load(std::memory_order_acquire);
    if (!scratch) {
        // One-time set-up per device: the symbol's host-side name is only a
        // stand-in, so ask the runtime for the device address.
        if (cudaGetSymbolAddress(&scratch, g_scalar_scratch) != cudaSuccess || !scratch) return PIR_ERR_CUDA;
        g_scratch_addr[ctx->device].store(scratch, std::memory_order_release);
    }
    // The digit kernel rewrites every scratch block the scan reads, so stale
    // contents from an earlier call never leak into this one.
    return pir_scalar_scan(ctx, db, R, C, Q, B, out, scratch, kNoAllocScratchBytes, stream);
}
