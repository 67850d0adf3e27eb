// rowsel_tc.cu — RowSel on the tensor cores for query batches (2B > 16 polynomials).
//
// GPIR section 2: RowSel is L*N point-wise GEMMs
//     M_out[p,m,n] = sum_k M_in0[p,m,k] * M_in1[p,k,n]  mod q_l.
// With a batch of queries every DB word meets 2B query words, and the
// 32x32->64-bit multiply-adds of the CUDA-core scan become the bound.  This
// path computes the same sums exactly on the fp16 tensor cores (tcgen05
// kind::f16, fp32 accumulation in TMEM), using the byte-split idea of VIPIR
// section 4.1 on both operands:
//   * query residues a < 2^29 as balanced base-256 digits a_i in [-128, 128]
//     (a = sum_i 256^i a_i exactly; a_3 <= 32),
//   * DB residues b < 2^29 as their plain bytes b_j in [0, 255],
// so a*b = sum_{i,j} 256^(i+j) a_i b_j.  Every digit product is an integer of
// magnitude <= 128*255, and 512 of them sum below 2^24: exact in fp32.  The
// rows of a point are therefore taken in K segments of at most 512 rows.
//
// MMA tile (one per 32 DB columns of a point and segment): M = 128 rows
// (i, m) = 4 query digit planes x 32 polynomials, N = 128 columns (j, n) =
// 4 DB byte planes x 32 columns, K = the segment's rows.  The A operand
// (query digits of the segment) sits in TMEM for all tiles of the segment;
// the accumulator (128 columns, double buffered) then holds S_ij[m][n].
// The epilogue forms
//     out[m][n] = sum_i 2^(8i) (sum_j 2^(8j) S_ij[m][n])  mod q
// with one reduction per (i, m, n) (32-bit arithmetic and an fp32 quotient
// estimate, valid for q >= 2^26) and a cross-plane sum; segments after the
// first add their residue to the stored one.
//
// Warp roles (512 threads, one CTA per SM, persistent over a range of points).
// A warp's scheduler is fixed by warp % 4, and the MMA-issuing thread loses
// most of its issue rate to any ALU-busy warp on its scheduler, so scheduler 1
// carries only light roles besides the plane-1 epilogue:
//   warps 0-3   query digits of the next segment -> TMEM (tcgen05.st), warp w
//               writes digit plane w into TMEM lanes 32w..32w+31, from the
//               segment's query slice that the producer bulk-copies into
//               shared memory while the previous segment is still in flight
//               (warps 0, 2, 3 also convert; warp 1 only writes digits);
//   warps 4-7   epilogue: tcgen05.ld of a finished accumulator, reduction,
//               cross-plane sum through shared memory, output stores;
//   converters  three groups of three warps, {0, 2, 3}, {8, 10, 11} and
//               {12, 14, 15}, each converting every third stage: 64 x 32 DB
//               words (TMA-staged) -> 4 byte planes of fp16 in the
//               128B-swizzled K-major layout of the B operand;
//   warp 9      TMEM allocation and the TMA producer of query slices and DB
//               word tiles;
//   warp 13     MMA issue (one thread).
// DB word stages (TMA -> converters) and fp16 operand stages (converters ->
// MMA) are separate rings, so a word stage is refilled as soon as it has
// been read.  The MMA thread keeps its loop short: any shared-memory access
// of the issuing thread (a barrier wait included) stalls until the tensor
// core has taken its previous MMAs, so bookkeeping between MMAs leaves the
// tensor pipe idle.
// All mbarrier waits are bounded; TMEM is always released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"

namespace {

constexpr int TC_NR = 6;                      // DB word stages (TMA -> converters)
constexpr int TC_NB = 6;                       // fp16 operand stages (converters -> MMA)
constexpr int TC_KS = 64;                      // DB rows (K) per stage
constexpr int TC_NT = 32;                      // DB columns per MMA tile
constexpr uint32_t TC_RAW_BYTES = TC_KS * TC_NT * 4;   // 8 KiB of DB words
constexpr uint32_t TC_B_BYTES = 128 * 128;             // 128 rows x 64 fp16
constexpr int TC_THREADS = 16 * 32;
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr uint32_t TC_ACC_COL = 256;           // accumulators at columns 256 and 384
constexpr uint32_t TC_SEG = 512;               // rows per K segment: the exactness bound of one fp32 accumulation
constexpr uint32_t TC_MIN_Q = 1u << 26;        // smallest prime the epilogue's reduction supports
constexpr uint32_t TC_Q_BYTES = TC_SEG * 32 * 4;        // one segment's query slice (64 KiB)
constexpr uint32_t TC_RED_PITCH = 33;          // words per row of the epilogue's plane sums (no bank conflicts)
constexpr uint32_t TC_PREFETCH_PIECE = 64 * 1024;
constexpr float TC_MAGIC = 12582912.0f;        // 1.5 * 2^23
constexpr uint32_t TC_MAGIC_BITS = 0x4B400000u;

struct TcArgs {
    const uint32_t *qT;     // point-major query, [P][PS], 32 polynomials per k
    uint32_t *outT;         // point-major results [P][Mv][D1p]
    uint32_t *status;
    uint32_t N, D0, D1, D1p, S, Wlast, PS, Mv;
    uint32_t H, Dlast;      // K segments of TC_SEG rows per point (the last has Dlast rows)
    uint64_t P;
    uint32_t q[PIR_MAX_RNS];
    float qinv[PIR_MAX_RNS];          // 1/q rounded to fp32 (quotient estimate of the epilogue)
    uint32_t c[PIR_MAX_RNS][4];       // 2^(8i) mod q
    uint32_t cs[PIR_MAX_RNS][4];      // Shoup companions of c
    uint64_t wait_ns;                 // limit of the ordinary waits (drains keep PIR_WAIT_LIMIT_NS)
    uint32_t hook;                    // PIR_HOOK_* of the context
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t j) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((j ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16, A = B = F16, D = F32, K-major, N = 128, M = 128
constexpr uint32_t TC_IDESC = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// The four K = 16 MMAs of one 64-row stage: A (query digits) from TMEM
// columns a_tmem + 8*kk, B (DB byte planes) from the stage's swizzled tile,
// whose descriptor start address advances 32 bytes (2 units) per kk.  The
// first stage of a tile (ks == 0) starts the accumulator from zero.
__device__ __forceinline__ void mma_stage(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t ks) {
    asm volatile(
        "{\n.reg .pred p, t;\n"
        "setp.ne.b32 p, %3, 0;\n"
        "setp.eq.b32 t, %3, %3;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %4, t;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %4, t;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %4, t;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(bdesc), "r"(ks), "r"(TC_IDESC), "r"(a_tmem + 8), "l"(bdesc + 2), "r"(a_tmem + 16),
        "l"(bdesc + 4), "r"(a_tmem + 24), "l"(bdesc + 6)
        : "memory");
}

__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Balanced base-256 digit `plane` of two residues a0, a1 < 2^29, packed as
// two fp16 values (a0 in the low half).  a + 0x808080 has the bytes d_i + 128
// (i < 3) and d_3 on top, because balanced digits never carry; 0x64xx is the
// fp16 value 1024 + xx, so subtracting 1152 (1024 for the top digit) leaves d.
__device__ __forceinline__ uint32_t digit_pair(uint32_t a0, uint32_t a1, uint32_t plane) {
    const uint32_t x0 = a0 + 0x808080u, x1 = a1 + 0x808080u;
    const uint32_t hh = (__byte_perm(x0, x1, plane | ((4 + plane) << 8)) & 0x00FF00FFu) | 0x64006400u;
    const float off = plane < 3 ? 1152.f : 1024.f;
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&hh), __floats2half2_rn(off, off));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Rows of K segment h and its 64-row stage count.
__device__ __forceinline__ uint32_t seg_rows(const TcArgs &A, uint32_t h) { return h + 1 < A.H ? TC_SEG : A.Dlast; }
__device__ __forceinline__ uint32_t seg_stages(const TcArgs &A, uint32_t h) {
    return (seg_rows(A, h) + TC_KS - 1) / TC_KS;
}

// Number of 32-column tiles of slab s.
__device__ __forceinline__ uint32_t tiles_of(const TcArgs &A, uint32_t s) {
    const uint32_t w = (s == A.S - 1) ? A.Wlast : PIR_SLAB;
    return (w + TC_NT - 1) / TC_NT;
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned address,
// in pieces of at most 64 KiB.
__device__ __forceinline__ void l2_prefetch(const void *src, uint64_t bytes) {
    const char *s = static_cast<const char *>(src);
    for (uint64_t off = 0; off < bytes; off += TC_PREFETCH_PIECE) {
        const uint32_t n = (uint32_t)(bytes - off < TC_PREFETCH_PIECE ? bytes - off : TC_PREFETCH_PIECE);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s + off), "r"(n) : "memory");
    }
}

// A stage holds 64 DB rows x 32 columns of words (row-major).  Converting it
// writes the 4 byte planes as fp16 in the 128B-swizzled K-major B layout
// (row j*32 + n, K = DB row).  The work is cut into 8 chunks of 8 rows; lane
// n of a converter warp handles column n of chunks kc = gw, gw + 3, gw + 6
// (gw = the warp's position 0..2 in its group of three).
__device__ __forceinline__ void load_chunks(const uint32_t *raw, uint32_t gw, uint32_t n, uint32_t (&w)[3][8]) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const uint32_t kc = gw + 3 * c;
        if (kc < 8) {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[c][e] = raw[(kc * 8 + e) * TC_NT + n];
        }
    }
}

__device__ __forceinline__ void store_chunks(uint8_t *bt, uint32_t gw, uint32_t n, const uint32_t (&w)[3][8]) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const uint32_t kc = gw + 3 * c;
        if (kc < 8) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t hv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // bytes j of two words -> halves 0x64xx = 1024 + byte
                    const uint32_t x = __byte_perm(w[c][2 * e], w[c][2 * e + 1], j | ((4 + j) << 8));
                    const uint32_t hh = (x & 0x00FF00FFu) | 0x64006400u;
                    const __half2 r =
                        __hsub2(*reinterpret_cast<const __half2 *>(&hh), __floats2half2_rn(1024.f, 1024.f));
                    hv[e] = *reinterpret_cast<const uint32_t *>(&r);
                }
                *reinterpret_cast<uint4 *>(bt + sw128(j * 32 + n, kc)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    rowsel_tc_kernel(const __grid_constant__ CUtensorMap full_map, const __grid_constant__ CUtensorMap last_map,
                     const __grid_constant__ TcArgs A) {
    extern __shared__ uint8_t smraw[];
    const uint32_t base_s = smem_u32(smraw);
    uint8_t *sm = smraw + (((base_s + 1023u) & ~1023u) - base_s);
    uint8_t *stB = sm;                                   // [NS][16 KiB] fp16 digit tiles
    uint8_t *stR = stB + TC_NB * TC_B_BYTES;             // [NR][8 KiB] DB words
    uint32_t *qsm = reinterpret_cast<uint32_t *>(stR + TC_NR * TC_RAW_BYTES);   // [D0][32] query slice
    uint32_t *red = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(qsm) + TC_Q_BYTES);  // [128][33]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + 128 * TC_RED_PITCH);
    uint64_t *rfull = bars, *rempty = rfull + TC_NR, *bfull = rempty + TC_NR, *bempty = bfull + TC_NB;
    uint64_t *accf = bempty + TC_NB, *acce = accf + 2, *afull = acce + 2, *aempty = afull + 1, *done = aempty + 1;
    uint64_t *qfull = done + 1, *qempty = qfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(qempty + 1);
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t p_begin = (uint64_t)blockIdx.x * A.P / gridDim.x;
    const uint64_t p_end = (uint64_t)(blockIdx.x + 1) * A.P / gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_NR; ++s) {
            mbar_init(rfull + s, 1);
            mbar_init(rempty + s, 3);
        }
        for (int s = 0; s < TC_NB; ++s) {
            mbar_init(bfull + s, 3);
            mbar_init(bempty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, 4);
        }
        mbar_init(afull, 4);
        mbar_init(aempty, 1);
        mbar_init(done, 1);
        mbar_init(qfull, 1);
        mbar_init(qempty, 4);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 9 && lane == 0) {
        // ------------------------------------------------ TMA producer: query slices and DB word tiles
        // The next segment's query slice is prefetched into L2 a segment ahead.
        // (Prefetching whole DB slab blocks ahead was measured too: 152 SMs x
        // two 256 KiB slabs crowd the L2 next to the streaming result writes,
        // and 40% of the DB was read twice.)
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0, pc = 0;
        bool withheld = false;

        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h, ++pc) {
            // the segment's query slice (the query warps release the buffer once digitised)
            const uint32_t nks = seg_stages(A, h), qbytes = seg_rows(A, h) * 32 * 4;
            const uint32_t *qsrc = A.qT + p * A.PS + (uint64_t)h * TC_SEG * 32;
            if (abort_flag || !mbar_wait(qempty, (pc & 1) ^ 1, A.status, A.wait_ns)) {
                abort_flag = 1;
            } else {
                mbar_arrive_expect_tx(qfull, qbytes);
                bulk_g2s(qsm, qsrc, qbytes, qfull, pol);
            }
            if (h + 1 < A.H)
                l2_prefetch(qsrc + TC_SEG * 32, seg_rows(A, h + 1) * 32 * 4);
            else if (p + 1 < p_end)
                l2_prefetch(A.qT + (p + 1) * A.PS, seg_rows(A, 0) * 32 * 4);
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                for (uint32_t t = 0; t < nt; ++t)
                    for (uint32_t ks = 0; ks < nks; ++ks, ++it) {
                        const uint32_t st = it % TC_NR, ph = (it / TC_NR) & 1;
                        if (abort_flag || !mbar_wait(rempty + st, ph ^ 1, A.status, A.wait_ns)) {
                            abort_flag = 1;
                            continue;
                        }
                        if (A.hook == PIR_HOOK_WITHHOLD_LAST_COPY && blockIdx.x == 0 && p + 1 == p_end &&
                            h + 1 == A.H && s + 1 == A.S && t + 1 == nt && ks + 1 == nks) {
                            // failure-path test: the CTA's last DB tile is never copied, so
                            // its converters' wait runs out; nothing reuses this stage
                            withheld = true;
                            continue;
                        }
                        mbar_arrive_expect_tx(rfull + st, TC_RAW_BYTES);
                        const int y = (int)(h * TC_SEG + ks * TC_KS);   // DB row; rows >= D0 read as zero
                        if (s + 1 < A.S)
                            tma_load_4d(stR + st * TC_RAW_BYTES, &full_map, (int)(t * TC_NT), y, (int)s, (int)p,
                                        rfull + st, pol);
                        else
                            tma_load_4d(stR + st * TC_RAW_BYTES, &last_map, (int)(t * TC_NT), y, 0, (int)p,
                                        rfull + st, pol);
                    }
            }
          }
        // copies in flight land first (full limit); a withheld copy was the last stage
        for (uint32_t i = withheld ? 1u : 0u; i < TC_NR && i < it; ++i) {
            const uint32_t j = it - 1 - i;
            mbar_wait(rfull + j % TC_NR, (j / TC_NR) & 1, A.status);
        }
        if (pc) mbar_wait(qfull, (pc - 1) & 1, A.status);
    } else if (warp == 13 && lane == 0) {
        // ------------------------------------------------ MMA issue
        // One thread whose warp shares its scheduler with three busy warps:
        // the per-stage path is kept short (a local abort flag, descriptors
        // advanced by addition, the stage's four MMAs in one asm block).
        bool ab = false;
        uint32_t it = 0, g = 0, pc = 0, st = 0, ph = 0;
        const uint64_t bdesc0 = sdesc(smem_u32(stB));
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h) {
            ab = ab || abort_flag;
            bool first = true;
            const uint32_t nks = seg_stages(A, h);
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                for (uint32_t t = 0; t < nt; ++t, ++g) {
                    const uint32_t buf = g & 1, use = (g >> 1) & 1;
                    if (!ab && !mbar_wait(acce + buf, use ^ 1, A.status, A.wait_ns)) ab = true;
                    if (first) {
                        if (!ab && !mbar_wait(afull, pc & 1, A.status, A.wait_ns)) ab = true;
                        first = false;
                    }
                    const uint32_t d = tmem + TC_ACC_COL + buf * 128;
                    for (uint32_t ks = 0; ks < nks; ++ks, ++it) {
                        if (!ab && !mbar_wait(bfull + st, ph, A.status, A.wait_ns)) ab = true;
                        if (!ab) {
                            fence_after();
                            mma_stage(d, tmem + ks * 32, bdesc0 + st * (TC_B_BYTES >> 4), ks);
                            commit(bempty + st);
                        }
                        if (++st == TC_NB) {
                            st = 0;
                            ph ^= 1;
                        }
                    }
                    if (!ab) commit(accf + buf);
                }
            }
            commit(aempty);  // A (query digits) reusable once this segment's MMAs finish
            ++pc;
          }
        if (ab) abort_flag = 1;
        commit(done);
        mbar_wait(done, 0, A.status);
    } else if (warp < 4 || (warp >= 8 && (warp & 3) != 1)) {
        // ------------------------------------------------ query digits and converters
        // Warps 0-3 write the query digits of each segment into TMEM (plane =
        // warp) before that segment's stages.  Three groups of three converter
        // warps -- {0, 2, 3}, {8, 10, 11}, {12, 14, 15} -- take every third
        // stage each; none of them shares a scheduler with the MMA warp (13).
        const bool digitizer = warp < 4, converter = warp != 1;
        const uint32_t gi = warp < 4 ? 0u : (uint32_t)(warp >> 2) - 1u;          // group 0..2
        const uint32_t gw = (warp & 3) == 0 ? 0u : (uint32_t)(warp & 3) - 1u;     // position 0..2
        uint32_t it = 0, pc = 0, sel = 0;                                         // sel = it % 3
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h, ++pc) {
            const uint32_t nks = seg_stages(A, h);
            if (digitizer) {
                // query digits of the segment -> TMEM (plane = warp, polynomial m = lane)
                const uint32_t plane = warp, m = lane, rows = seg_rows(A, h);
                if (!abort_flag && !mbar_wait(qfull, pc & 1, A.status, A.wait_ns)) abort_flag = 1;
                if (!abort_flag && !mbar_wait(aempty, (pc & 1) ^ 1, A.status, A.wait_ns)) abort_flag = 1;
                fence_after();
                if (!abort_flag) {
                    const bool live = m < A.Mv;
                    for (uint32_t kc = 0; kc < nks; ++kc) {
                        uint32_t v[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const uint32_t k0 = kc * 64 + 2 * e;
                            const uint32_t a0 = (live && k0 < rows) ? qsm[k0 * 32 + m] : 0u;
                            const uint32_t a1 = (live && k0 + 1 < rows) ? qsm[(k0 + 1) * 32 + m] : 0u;
                            v[e] = digit_pair(a0, a1, plane);
                        }
                        tmem_st32(tmem + ((plane * 32u) << 16) + kc * 32, v);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
                fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(afull);
                    mbar_arrive(qempty);
                }
            }
            if (!converter) continue;
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                for (uint32_t t = 0; t < nt; ++t)
                    for (uint32_t ks = 0; ks < nks; ++ks, ++it) {
                        const bool my_stage = sel == gi;
                        sel = sel == 2 ? 0u : sel + 1;
                        if (!my_stage) continue;
                        const uint32_t rs = it % TC_NR, rph = (it / TC_NR) & 1;
                        const uint32_t bs = it % TC_NB, bph = (it / TC_NB) & 1;
                        uint32_t w[3][8];
                        if (!abort_flag && !mbar_wait(rfull + rs, rph, A.status, A.wait_ns)) abort_flag = 1;
                        if (!abort_flag)
                            load_chunks(reinterpret_cast<const uint32_t *>(stR + rs * TC_RAW_BYTES), gw, lane, w);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rempty + rs);     // the words are in registers
                        if (!abort_flag && !mbar_wait(bempty + bs, bph ^ 1, A.status, A.wait_ns)) abort_flag = 1;
                        if (!abort_flag) store_chunks(stB + bs * TC_B_BYTES, gw, lane, w);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bfull + bs);
                    }
            }
          }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ epilogue
        const uint32_t plane = warp & 3, m = lane;
        const uint32_t etid = threadIdx.x - 128;  // 0..127
        uint32_t g = 0;
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h) {
            const uint32_t l = (uint32_t)(p / A.N);
            const uint32_t q = A.q[l];
            const float qinv = A.qinv[l];
            const uint32_t ci = A.c[l][plane], cis = A.cs[l][plane];
            // + q, + 0x4B400000 * q for the quotient's magic bits, - the magic offsets in lo
            const uint32_t lo_off = plane == 3 ? TC_MAGIC_BITS + (TC_MAGIC_BITS << 8) : TC_MAGIC_BITS << 24;
            const uint32_t rc = q + TC_MAGIC_BITS * q - lo_off;
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                const uint32_t Ws = (s == A.S - 1) ? A.Wlast : PIR_SLAB;
                for (uint32_t t = 0; t < nt; ++t, ++g) {
                    const uint32_t buf = g & 1, use = (g >> 1) & 1;
                    if (!abort_flag && !mbar_wait(accf + buf, use, A.status, A.wait_ns)) abort_flag = 1;
                    fence_after();
                    // W[n] = sum_j 2^(8j) S_j[n] = sum_k d_i(query) * DB word is reduced
                    // mod q without 64-bit arithmetic.  Its low 32 bits come exactly
                    // from wrapping 32-bit sums of the integer plane sums S_j; the
                    // quotient k = round(W / q) comes from an fp32 estimate of W.
                    // Every partial sum of the estimate is below 128 * 512 * (2^24 + q)
                    // <= 2^46 (a segment has at most 512 rows), so its three roundings
                    // add at most 3 * 2^22, and |W| / q <= 128 * 512 = 2^16; with
                    // q >= 2^26 the estimate of W / q is off by less than 0.2 and
                    // W - k*q lies in (-0.7q, 1.7q).
                    // Integer conversions: an fp32 integer x with |x| < 2^22 gives
                    // x + 1.5 * 2^23 exactly, whose bits are 0x4B400000 + x (an FADD
                    // instead of a conversion).  That holds for S_3 (top DB byte
                    // <= 31: |S| <= 128 * 31 * 512), for every S of plane 3 (top
                    // query digit <= 32: |S| <= 32 * 255 * 512 < 2^22) and for the
                    // quotient k; the other sums reach 2^24 and are converted.  The
                    // offsets the magic bits leave in lo and in k*q are folded into rc.
                    uint32_t lo[32];
                    float wf[32];
#pragma unroll
                    for (int n = 0; n < 32; ++n) {
                        lo[n] = 0;
                        wf[n] = 0.f;
                    }
                    if (!abort_flag) {
                        const uint32_t taddr = tmem + ((plane * 32u) << 16) + TC_ACC_COL + buf * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t v[32];
                            tmem_ld32(taddr + j * 32, v);
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                            const float scale = (float)(1u << (8 * j));
                            if (j == 3 || plane == 3) {
#pragma unroll
                                for (int n = 0; n < 32; ++n) {
                                    const float x = __uint_as_float(v[n]);
                                    lo[n] += __float_as_uint(x + TC_MAGIC) << (8 * j);
                                    wf[n] = fmaf(x, scale, wf[n]);
                                }
                            } else {
#pragma unroll
                                for (int n = 0; n < 32; ++n) {
                                    const float x = __uint_as_float(v[n]);
                                    lo[n] += (uint32_t)__float2int_rn(x) << (8 * j);
                                    wf[n] = fmaf(x, scale, wf[n]);
                                }
                            }
                        }
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce + buf);  // accumulator drained
                    named_barrier(2, 128);                    // previous tile's readers of red are done
#pragma unroll
                    for (int n = 0; n < 32; ++n) {
                        // W - k*q lies in (-0.7q, 1.7q); + q makes it a positive 32-bit value
                        // congruent to W, which the Shoup product accepts as is: 2^(8i) * W
                        // mod q lands in [0, 2q)
                        const uint32_t kb = __float_as_uint(fmaf(wf[n], qinv, TC_MAGIC));   // 0x4B400000 + k
                        const uint32_t r = lo[n] - kb * q + rc;
                        red[(plane * 32 + m) * TC_RED_PITCH + n] = shoup_mul(r, ci, cis, q);
                    }
                    named_barrier(2, 128);
                    {
                        // this thread's outputs: column nn, rows m0, m0 + 4, ..., m0 + 28
                        const uint32_t nn = etid & 31, m0 = etid >> 5;
                        const uint32_t col = t * TC_NT + nn;
                        if (col < Ws) {
                            uint32_t v[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint32_t *rr = red + (m0 + 4 * i) * TC_RED_PITCH + nn;
                                // four plane terms, each in [0, 2q): the sum is below 8q < 2^32
                                v[i] = rr[0] + rr[32 * TC_RED_PITCH] + rr[64 * TC_RED_PITCH] + rr[96 * TC_RED_PITCH];
                            }
                            uint32_t *o = A.outT + (p * A.Mv + m0) * A.D1p + s * PIR_SLAB + col;
                            const size_t ostep = (size_t)4 * A.D1p;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (m0 + 4 * i < A.Mv) {
                                    uint32_t x = v[i];
                                    x = min(x, x - 4 * q);   // x - cq wraps above x when x < cq
                                    x = min(x, x - 2 * q);
                                    x = min(x, x - q);
                                    if (h) {   // later segments add to the sum this thread stored for the earlier ones
                                        x += o[i * ostep];
                                        x = min(x, x - q);
                                    }
                                    o[i * ostep] = x;
                                }
                            }
                        }
                    }
                }
            }
          }
    }

    fence_before();
    __syncthreads();
    if (warp == 9) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

size_t tc_smem_bytes() {
    return 1024 + (size_t)TC_NB * TC_B_BYTES + (size_t)TC_NR * TC_RAW_BYTES + TC_Q_BYTES + 128 * TC_RED_PITCH * 4 +
           (2 * TC_NR + 2 * TC_NB + 11) * 8 + 16;
}

uint64_t powmod_host(uint64_t b, uint64_t e, uint64_t m) {
    uint64_t r = 1 % m;
    b %= m;
    for (; e; e >>= 1) {
        if (e & 1) r = (uint64_t)((unsigned __int128)r * b % m);
        b = (uint64_t)((unsigned __int128)b * b % m);
    }
    return r;
}

}  // namespace

// Whether the context's primes allow this path (passes of 17..32 polynomials).
bool rowsel_tc_primes_ok(const pir_ctx *ctx) {
    for (uint32_t l = 0; l < ctx->L; ++l)
        if (ctx->q[l] < TC_MIN_Q) return false;   // the epilogue's quotient estimate needs q >= 2^26
    return true;
}

// One RowSel pass on the tensor cores.  qT holds the pass's query slices
// (32 polynomials per k, PS words per point); db is the slab-encoded DB.
int rowsel_tc_pass(pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1, const uint32_t *qT, uint32_t PS,
                   uint32_t Mv, uint32_t *outT, cudaStream_t st) {
    auto encode = encode_fn();
    if (!encode) return PIR_ERR_CUDA;
    const uint64_t P = (uint64_t)ctx->L * ctx->N;
    const uint32_t D1p = (D1 + 3) / 4 * 4;
    const uint32_t S = (D1 + PIR_SLAB - 1) / PIR_SLAB;
    const uint32_t Wlast = D1p - PIR_SLAB * (S - 1);

    // Full slabs: 4-D view (column, row k, slab, point) of the first S-1 slabs of every point.
    // L2 promotion stays at 128 B: a tile reads one 128-byte line of each
    // 512-byte slab row, and 256-byte promotion fetched the neighbouring
    // tile's line too, which was evicted before use (30% more DRAM reads).
    CUtensorMap full_map, last_map;
    memset(&full_map, 0, sizeof(full_map));
    memset(&last_map, 0, sizeof(last_map));
    const cuuint32_t box[4] = {TC_NT, TC_KS, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    void *dbp = const_cast<uint32_t *>(db);
    if (S > 1) {
        const cuuint64_t dim[4] = {PIR_SLAB, D0, S - 1, P};
        const cuuint64_t str[3] = {(cuuint64_t)PIR_SLAB * 4, (cuuint64_t)D0 * PIR_SLAB * 4, (cuuint64_t)D0 * D1p * 4};
        if (encode(&full_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, dbp, dim, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PIR_ERR_ARG;
    }
    {
        // Last slab of every point: (column, row k, 1, point), base at slab S-1.
        const cuuint64_t dim[4] = {Wlast, D0, 1, P};
        const cuuint64_t str[3] = {(cuuint64_t)Wlast * 4, (cuuint64_t)D0 * Wlast * 4, (cuuint64_t)D0 * D1p * 4};
        void *lastp = const_cast<uint32_t *>(db + (uint64_t)(S - 1) * D0 * PIR_SLAB);
        if (encode(&last_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, lastp, dim, str, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PIR_ERR_ARG;
    }
    if (S == 1) full_map = last_map;  // never used

    TcArgs a;
    memset(&a, 0, sizeof(a));
    a.qT = qT;
    a.outT = outT;
    a.status = ctx->d_status;
    a.wait_ns = ctx->wait_limit_ns;
    a.hook = ctx->test_hook;
    a.N = ctx->N;
    a.D0 = D0;
    a.D1 = D1;
    a.D1p = D1p;
    a.S = S;
    a.Wlast = Wlast;
    a.PS = PS;
    a.H = (D0 + TC_SEG - 1) / TC_SEG;
    a.Dlast = D0 - TC_SEG * (a.H - 1);
    a.Mv = Mv;
    a.P = P;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        const uint64_t q = ctx->q[l];
        a.q[l] = (uint32_t)q;
        a.qinv[l] = 1.0f / (float)q;
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = (uint32_t)powmod_host(2, 8 * i, q);
            a.c[l][i] = c;
            a.cs[l][i] = (uint32_t)(((uint64_t)c << 32) / q);
        }
    }
    const size_t smem = tc_smem_bytes();
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        if (cudaFuncSetAttribute(rowsel_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PIR_ERR_CUDA;
        attr_set[ctx->device] = true;
    }
    const uint64_t grid = P < (uint64_t)ctx->num_sms ? P : (uint64_t)ctx->num_sms;
    rowsel_tc_kernel<<<(unsigned)grid, TC_THREADS, smem, st>>>(full_map, last_map, a);
    return launch_status(cudaGetLastError());
}
