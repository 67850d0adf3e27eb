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
//   * DB residues b < 2^29 as their plain bytes b_j in [0, 255], each taken
//     as the fp16 subnormal b_j * 2^-24 (the halfword 0x00bb: a zero
//     extension, two byte permutes per DB word),
// so a*b = sum_{i,j} 256^(i+j) a_i b_j.  Every digit product is an integer of
// magnitude <= 128*255 (times 2^-24), and 512 of them sum below 2^24 (times
// 2^-24): exact in fp32.  The rows of a point are therefore taken in K
// segments of at most 512 rows.
//
// MMA (M = 128, N = 256 as two N = 128 halves, K = 16): M rows = 32
// polynomials x 4 query digit planes (row 4m + i), N columns = 64 DB columns x
// 4 byte planes, K = DB rows.  The A operand (query digits of the segment,
// 256 TMEM columns) sits in TMEM for all tiles of the segment; the B operand
// is MN-major (a DB row's bytes are contiguous along N, so a word's four
// bytes land side by side); one accumulator (the other 256 TMEM columns)
// holds S_ij[m][n] * 2^-24 for one 64-column tile.  A stage's 64 rows are 4
// K steps x 2 halves = 8 MMAs (1.4% faster than 4 of N = 256 on the
// 24 GiB x 16 and 64 GiB x 16 cases).
//
// The epilogue forms
//     out[m][n] = sum_i 2^(8i) (sum_j 2^(8j) S_ij[m][n])  mod q
// with one reduction per (i, m, n) (32-bit arithmetic and an fp32 quotient
// estimate, valid for q >= 2^26) and a cross-plane sum over the four lanes
// 4m .. 4m+3 by warp shuffles; segments after the first add their residue to
// the stored one.
//
// Warp roles (22 warps, one CTA per SM, persistent over a range of points).
// A warp's scheduler is warp % 4 and a warp reaches only the TMEM lane
// quarter warp % 4:
//   warp 0        TMEM allocation; lane 0 is the TMA producer of query
//                 slices and DB word tiles;
//   warps 1-16    epilogue, four per lane quarter, each draining 64 of the
//                 256 accumulator columns right after the tile's MMAs (so
//                 the single accumulator is free again within a TMEM load),
//                 then reducing them; they also write the query digits of
//                 each segment into TMEM (lane quarter x a quarter of the rows);
//   warp 17       MMA issue: the warp runs the loop (control flow and
//                 operands warp-uniform), one elected lane issues;
//   warps 18-21   converters: 64 x 64 DB words (TMA-staged) -> their bytes
//                 as fp16 subnormals in the 128B-swizzled MN-major layout of
//                 the B operand, a quarter of every stage each.
// Registers: the 16 epilogue warps hold a drained tile (64 values a thread),
// which caps the CTA at 22 warps; two converter warps measured 9.9 ms on the
// 24 GiB x 16 case, four 7.3 ms, six the same, eight slower (spills).
// DB word stages (TMA -> converters) and fp16 operand stages (converters ->
// MMA) are separate rings, so a word stage is refilled as soon as it has
// been read.  All mbarrier waits are bounded; TMEM is always released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"

namespace {

constexpr int TC_NR = 4;                       // DB word stages (TMA -> converters)
constexpr int TC_NB = 3;                       // fp16 operand stages (converters -> MMA)
constexpr int TC_KS = 64;                      // DB rows (K) per stage
constexpr int TC_NT = 64;                      // DB columns per tile (N = 256)
constexpr uint32_t TC_RAW_BYTES = TC_KS * TC_NT * 4;   // 16 KiB of DB words
constexpr uint32_t TC_B_GROUP = 4096;                  // 8 rows x 256 halves
constexpr uint32_t TC_B_BYTES = (TC_KS / 8) * TC_B_GROUP;   // 32 KiB
constexpr int TC_EPI_WARPS = 16;
constexpr int TC_CONV_WARPS = 4;
constexpr int TC_W_MMA = 17;
constexpr int TC_W_CONV = 18;
constexpr int TC_THREADS = 22 * 32;
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr uint32_t TC_ACC_COL = 256;           // the accumulator: columns 256..511
constexpr uint32_t TC_SEG = 512;               // rows per K segment: the exactness bound of one fp32 accumulation
constexpr uint32_t TC_MIN_Q = 1u << 26;        // smallest prime the epilogue's reduction supports
constexpr uint32_t TC_Q_BYTES = TC_SEG * 32 * 4;        // one segment's query slice (64 KiB)
constexpr uint32_t TC_PREFETCH_PIECE = 64 * 1024;
constexpr float TC_MAGIC = 12582912.0f;        // 1.5 * 2^23
constexpr uint32_t TC_MAGIC_BITS = 0x4B400000u;
constexpr float TC_SMAGIC = 0.75f;             // 1.5 * 2^-1: x + 0.75 has ulp 2^-24 for |x| <= 1/4
constexpr uint32_t TC_SMAGIC_BITS = 0x3F400000u;
constexpr float TC_UNSCALE = 16777216.0f;      // 2^24: accumulators hold S * 2^-24

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

// B operand of a stage (64 DB rows = K, 256 columns = N), MN-major with the
// 128-byte swizzle: atoms of 8 K rows x 64 N halves (1 KiB), the four N
// atoms of a group of 8 rows side by side (leading byte offset 1 KiB), groups
// of 8 rows 4 KiB apart (stride byte offset); inside an atom, 16-byte chunk c
// of row r sits at chunk position c ^ r.  One K = 16 MMA reads 8 KiB.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(1024 >> 4) << 16) | ((uint64_t)(TC_B_GROUP >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// kind::f16, A = B = F16, D = F32, A K-major (TMEM), B MN-major, N = 128, M = 128
constexpr uint32_t TC_IDESC = (1u << 4) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// One MMA; acc == 0 starts the accumulator from zero.
__device__ __forceinline__ void mma1(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(TC_IDESC), "r"(acc)
        : "memory");
}

// The MMAs of one 64-row stage: for each K = 16 step kk, A (query digits)
// from TMEM columns a_tmem + 8*kk and B (DB bytes) from the stage's swizzled
// tile, whose descriptor start advances two row groups (8 KiB = 512 units)
// per kk; N columns 0..127 (N atoms 0, 1) go to accumulator columns d .. d+127,
// N columns 128..255 (atoms 2, 3: 2 KiB further) to d+128 .. d+255.  The
// first stage of a tile (ks == 0) starts the accumulator from zero.
__device__ __forceinline__ void mma_stage(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t ks) {
    constexpr uint64_t kstep = (2 * TC_B_GROUP) >> 4;
    constexpr uint64_t half = 2048 >> 4;
#pragma unroll
    for (uint32_t kk = 0; kk < 4; ++kk) {
        mma1(d, a_tmem + 8 * kk, bdesc + kk * kstep, ks | kk);
        mma1(d + 128, a_tmem + 8 * kk, bdesc + kk * kstep + half, ks | kk);
    }
}

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

// Bounded wait that lets the thread sleep in the hardware until the phase
// completes (suspend-time hint) instead of spinning: for warps that wait most
// of the time, so their issue slots go to the warps sharing their scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t *status, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_sleep(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(a, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, PIR_STATUS_TIMEOUT);
            return false;
        }
    }
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

// Number of 64-column tiles of slab s.
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

// A stage holds 64 DB rows x 64 columns of words (row-major, 256 bytes a
// row).  Converting it writes every byte as an fp16 subnormal (the halfword
// 0x00bb = bb * 2^-24) into the MN-major B tile; byte j of column
// n = 32 hr + 4 q4 + e (hr = 0, 1; q4 = 0..7; e = 0..3) goes to
//     N = 128 hr + 64 (e / 2) + 8 q4 + 4 (e % 2) + j,
// i.e. N atom 2 hr + e / 2, chunk q4.  A lane's task is one row and four
// columns (one 16-byte load): columns 4 q4 + 0, 1 fill chunk q4 of atom 2 hr,
// columns 4 q4 + 2, 3 chunk q4 of atom 2 hr + 1, so the eight lanes of a
// quarter-warp (one half row) load 128 contiguous bytes and store to eight
// distinct chunk positions.  Converter warp cw takes rows 8c + 2cw + (0, 1),
// c = 0..7: a quarter of every stage.
constexpr int TC_CTASKS = 8;

__device__ __forceinline__ void load_tasks(const uint32_t *raw, uint32_t cw, uint32_t lane, uint4 (&w)[TC_CTASKS]) {
    const uint32_t *base = raw + (2 * cw + (lane >> 4)) * TC_NT + 4 * (lane & 15);
#pragma unroll
    for (int c = 0; c < TC_CTASKS; ++c) w[c] = *reinterpret_cast<const uint4 *>(base + 8 * c * TC_NT);
}

// bytes 0, 1 (sel 0x4140) or 2, 3 (sel 0x4342) of x, each zero-extended to a halfword
__device__ __forceinline__ uint32_t zx_pair(uint32_t x, uint32_t sel) { return __byte_perm(x, 0u, sel); }

__device__ __forceinline__ void store_tasks(uint8_t *bt, uint32_t cw, uint32_t lane, const uint4 (&w)[TC_CTASKS]) {
    const uint32_t q16 = lane & 15, hr = q16 >> 3, q4 = q16 & 7;
    const uint32_t re = 2 * cw + (lane >> 4);   // row in its group of 8
    uint8_t *pe = bt + hr * 2048 + re * 128 + ((q4 ^ re) << 4);
#pragma unroll
    for (int c = 0; c < TC_CTASKS; ++c) {
        uint8_t *d = pe + c * TC_B_GROUP;
        *reinterpret_cast<uint4 *>(d) = make_uint4(zx_pair(w[c].x, 0x4140), zx_pair(w[c].x, 0x4342),
                                                   zx_pair(w[c].y, 0x4140), zx_pair(w[c].y, 0x4342));
        *reinterpret_cast<uint4 *>(d + 1024) = make_uint4(zx_pair(w[c].z, 0x4140), zx_pair(w[c].z, 0x4342),
                                                          zx_pair(w[c].w, 0x4140), zx_pair(w[c].w, 0x4342));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    rowsel_tc_kernel(const __grid_constant__ CUtensorMap full_map, const __grid_constant__ CUtensorMap last_map,
                     const __grid_constant__ TcArgs A) {
    extern __shared__ uint8_t smraw[];
    const uint32_t base_s = smem_u32(smraw);
    uint8_t *sm = smraw + (((base_s + 1023u) & ~1023u) - base_s);
    uint8_t *stB = sm;                                   // [NB][32 KiB] fp16 operand tiles
    uint8_t *stR = stB + TC_NB * TC_B_BYTES;             // [NR][16 KiB] DB words
    uint32_t *qsm = reinterpret_cast<uint32_t *>(stR + TC_NR * TC_RAW_BYTES);   // [512][32] query slice
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(qsm) + TC_Q_BYTES);
    uint64_t *rfull = bars, *rempty = rfull + TC_NR, *bfull = rempty + TC_NR, *bempty = bfull + TC_NB;
    uint64_t *accf = bempty + TC_NB, *acce = accf + 1, *afull = acce + 1, *qfull = afull + 1, *qempty = qfull + 1;
    uint64_t *done = qempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t p_begin = (uint64_t)blockIdx.x * A.P / gridDim.x;
    const uint64_t p_end = (uint64_t)(blockIdx.x + 1) * A.P / gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_NR; ++s) {
            mbar_init(rfull + s, 1);
            mbar_init(rempty + s, TC_CONV_WARPS);
        }
        for (int s = 0; s < TC_NB; ++s) {
            mbar_init(bfull + s, TC_CONV_WARPS);
            mbar_init(bempty + s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(acce, TC_EPI_WARPS);
        mbar_init(afull, TC_EPI_WARPS);
        mbar_init(qfull, 1);
        mbar_init(qempty, TC_EPI_WARPS);
        mbar_init(done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the set-up above touches no global memory

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer: query slices and DB word tiles
        // The next segment's query slice is prefetched into L2 a segment ahead.
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0, pc = 0;
        bool withheld = false;

        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h, ++pc) {
            // the segment's query slice (the digit writers release the buffer once digitised)
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
                        if (abort_flag || !mbar_wait_sleep(rempty + st, ph ^ 1, A.status, A.wait_ns)) {
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
    } else if (warp == TC_W_MMA) {
        // ------------------------------------------------ MMA issue
        // The whole warp runs the loop (its control flow and operands stay
        // warp-uniform); one elected lane issues the MMAs and commits.
        bool ab = false;
        uint32_t g = 0, pc = 0, st = 0, ph = 0;
        const uint64_t bdesc0 = sdesc_mn(smem_u32(stB));
        const uint32_t d = tmem + TC_ACC_COL;
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h, ++pc) {
            ab = __any_sync(0xffffffffu, ab || abort_flag);
            bool first = true;
            const uint32_t nks = seg_stages(A, h);
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                for (uint32_t t = 0; t < nt; ++t, ++g) {
                    // the previous tile's accumulator has been drained; the segment's digits are in TMEM
                    bool bad = !ab && !mbar_wait(acce, (g & 1) ^ 1, A.status, A.wait_ns);
                    if (first) {
                        bad = bad || (!ab && !mbar_wait(afull, pc & 1, A.status, A.wait_ns));
                        first = false;
                    }
                    ab = __any_sync(0xffffffffu, ab || bad);
                    for (uint32_t ks = 0; ks < nks; ++ks) {
                        ab = __any_sync(0xffffffffu, ab || !mbar_wait(bfull + st, ph, A.status, A.wait_ns));
                        if (!ab) {
                            fence_after();
                            if (elect_one()) {
                                mma_stage(d, tmem + ks * 32, bdesc0 + st * (TC_B_BYTES >> 4), ks);
                                commit(bempty + st);
                            }
                            __syncwarp();
                        }
                        if (++st == TC_NB) {
                            st = 0;
                            ph ^= 1;
                        }
                    }
                    if (!ab && elect_one()) commit(accf);
                    __syncwarp();
                }
            }
          }
        if (lane == 0 && ab) abort_flag = 1;
        if (elect_one()) commit(done);
        __syncwarp();
        mbar_wait(done, 0, A.status);
    } else if (warp >= TC_W_CONV) {
        // ------------------------------------------------ converters
        const uint32_t cw = (uint32_t)(warp - TC_W_CONV);
        uint32_t it = 0;
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h) {
            const uint32_t nks = seg_stages(A, h);
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                for (uint32_t t = 0; t < nt; ++t)
                    for (uint32_t ks = 0; ks < nks; ++ks, ++it) {
                        const uint32_t rs = it % TC_NR, rph = (it / TC_NR) & 1;
                        const uint32_t bs = it % TC_NB, bph = (it / TC_NB) & 1;
                        uint4 w[TC_CTASKS];
                        if (!abort_flag && !mbar_wait(rfull + rs, rph, A.status, A.wait_ns)) abort_flag = 1;
                        if (!abort_flag)
                            load_tasks(reinterpret_cast<const uint32_t *>(stR + rs * TC_RAW_BYTES), cw, lane, w);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rempty + rs);     // the words are in registers
                        if (!abort_flag && !mbar_wait(bempty + bs, bph ^ 1, A.status, A.wait_ns)) abort_flag = 1;
                        if (!abort_flag) store_tasks(stB + bs * TC_B_BYTES, cw, lane, w);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bfull + bs);
                    }
            }
          }
    } else if (warp >= 1 && warp <= TC_EPI_WARPS) {
        // ------------------------------------------------ epilogue and query digits (warps 1-16)
        // Lane quarter qq = warp % 4 (TMEM lanes 32 qq .. 32 qq + 31 = polynomials
        // 8 qq .. 8 qq + 7, lane = 4 (m - 8 qq) + i), accumulator columns
        // 64 cq .. 64 cq + 63 (cq = (warp - 1) / 4): DB columns
        // n = 32 hr + 4 q4 + 2 (cq % 2) + e1 with hr = cq / 2, q4 = 0..7, e1 = 0, 1.
        const uint32_t qq = (uint32_t)warp & 3u, cq = (uint32_t)(warp - 1) >> 2;
        const uint32_t i = (uint32_t)lane & 3u, m = 8 * qq + ((uint32_t)lane >> 2);
        const uint32_t b0 = i & 1u, b1 = i >> 1;
        const bool live = m < A.Mv;
        uint32_t g = 0, pc = 0;
        for (uint64_t p = p_begin; p < p_end; ++p)
          for (uint32_t h = 0; h < A.H; ++h, ++pc) {
            const uint32_t l = (uint32_t)(p / A.N);
            const uint32_t q = A.q[l];
            const float qinv = A.qinv[l];
            const uint32_t ci = A.c[l][i], cis = A.cs[l][i];
            // + q, + 0x4B400000 * q for the quotient's magic bits, - the magic offset of S_3 in lo
            const uint32_t rc = q + TC_MAGIC_BITS * q - (TC_SMAGIC_BITS << 24);
            const uint32_t nks = seg_stages(A, h), rows = seg_rows(A, h);
            // query digits of the segment -> TMEM.  The A operand is free: every
            // MMA of the previous segment completed before its last accumulator
            // was handed to this warp.
            // (every TMEM access below is taken or skipped by the whole warp)
            bool ok = __all_sync(0xffffffffu, !abort_flag && mbar_wait_sleep(qfull, pc & 1, A.status, A.wait_ns));
            if (!ok) abort_flag = 1;
            fence_after();
            if (ok) {
                for (uint32_t kc = cq; kc < nks; kc += 4) {
                    uint32_t v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const uint32_t k0 = kc * 64 + 2 * e;
                        const uint32_t a0 = (live && k0 < rows) ? qsm[k0 * 32 + m] : 0u;
                        const uint32_t a1 = (live && k0 + 1 < rows) ? qsm[(k0 + 1) * 32 + m] : 0u;
                        v[e] = digit_pair(a0, a1, i);
                    }
                    tmem_st32(tmem + ((qq * 32u) << 16) + kc * 32, v);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull);
                mbar_arrive(qempty);
            }
            for (uint32_t s = 0; s < A.S; ++s) {
                const uint32_t nt = tiles_of(A, s);
                const uint32_t Ws = (s == A.S - 1) ? A.Wlast : PIR_SLAB;
                for (uint32_t t = 0; t < nt; ++t, ++g) {
                    ok = __all_sync(0xffffffffu, !abort_flag && mbar_wait_sleep(accf, g & 1, A.status, A.wait_ns));
                    if (!ok) abort_flag = 1;
                    fence_after();
                    uint32_t v0[32], v1[32];
                    if (ok) {
                        const uint32_t taddr = tmem + ((qq * 32u) << 16) + TC_ACC_COL + 64 * cq;
                        tmem_ld32(taddr, v0);
                        tmem_ld32(taddr + 32, v1);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) v0[x] = v1[x] = 0u;
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce);  // accumulator drained: the next tile's MMAs may start
                    // W = sum_j 2^(8j) S_j = sum_k d_i(query) * DB word is reduced mod q
                    // without 64-bit arithmetic.  Its low 32 bits come exactly from
                    // wrapping 32-bit sums of the integer plane sums S_j; the quotient
                    // k = round(W / q) comes from an fp32 estimate of W.  Every partial
                    // sum of the estimate is below 128 * 512 * (2^24 + q) <= 2^46 (a
                    // segment has at most 512 rows), so its three roundings add at most
                    // 3 * 2^22, and |W| / q <= 128 * 512 = 2^16; with q >= 2^26 the
                    // estimate of W / q is off by less than 0.2 and W - k*q lies in
                    // (-0.7q, 1.7q).  The accumulators hold x = S * 2^-24: S_3 (top DB
                    // byte <= 31: |S| <= 128 * 31 * 512 < 2^22) comes from the bits of
                    // x + 0.75 (exact, ulp 2^-24: 0x3F400000 + S), the other sums
                    // (up to 2^24) from converting x * 2^24 (exact).
                    uint32_t y[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        // local column u = 8 t' + 2 q4' + e1: load t', q4 = 4 t' + q4'
                        const int tp = u >> 3, q4p = (u >> 1) & 3, e1 = u & 1;
                        uint32_t lo = 0;
                        float wf = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int idx = 8 * q4p + 4 * e1 + j;
                            const float x = __uint_as_float(tp ? v1[idx] : v0[idx]);
                            const uint32_t si = j == 3 ? __float_as_uint(x + TC_SMAGIC)
                                                       : (uint32_t)__float2int_rn(x * TC_UNSCALE);
                            lo += si << (8 * j);
                            wf = fmaf(x, TC_UNSCALE * (float)(1u << (8 * j)), wf);
                        }
                        // W - k*q lies in (-0.7q, 1.7q); + q makes it a positive 32-bit value
                        // congruent to W, which the Shoup product accepts as is: 2^(8i) * W
                        // mod q lands in [0, 2q)
                        const uint32_t kb = __float_as_uint(fmaf(wf, qinv, TC_MAGIC));   // 0x4B400000 + k
                        const uint32_t r = lo - kb * q + rc;
                        y[u] = shoup_mul(r, ci, cis, q);
                    }
                    // Sum over the four planes (lanes 4m' .. 4m'+3) as a reduce-scatter:
                    // after the xor-1 step a lane keeps the columns u with u % 2 == i % 2,
                    // after the xor-2 step those with u % 4 == i (four terms in [0, 2q):
                    // below 8q < 2^32).
                    uint32_t z[8];
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        const uint32_t keep = b0 ? y[2 * a + 1] : y[2 * a];
                        const uint32_t send = b0 ? y[2 * a] : y[2 * a + 1];
                        z[a] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                    }
                    uint32_t wsum[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t keep = b1 ? z[2 * c + 1] : z[2 * c];
                        const uint32_t send = b1 ? z[2 * c] : z[2 * c + 1];
                        wsum[c] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                    }
                    if (live && ok) {
                        uint32_t *orow = A.outT + (p * A.Mv + m) * A.D1p + s * PIR_SLAB + t * TC_NT;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            // column u = 4c + i: t' = c / 2, q4 = 4 t' + 2 (c % 2) + b1, e1 = b0
                            const uint32_t q4 = 4 * (c >> 1) + 2 * (c & 1) + b1;
                            const uint32_t n = 32 * (cq >> 1) + 4 * q4 + 2 * (cq & 1) + b0;
                            if (t * TC_NT + n < Ws) {
                                uint32_t x = wsum[c];
                                x = min(x, x - 4 * q);   // x - cq wraps above x when x < cq
                                x = min(x, x - 2 * q);
                                x = min(x, x - q);
                                if (h) {   // later segments add to the sum this thread stored for the earlier ones
                                    x += orow[n];
                                    x = min(x, x - q);
                                }
                                orow[n] = x;
                            }
                        }
                    }
                }
            }
          }
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
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
    return 1024 + (size_t)TC_NB * TC_B_BYTES + (size_t)TC_NR * TC_RAW_BYTES + TC_Q_BYTES +
           (2 * TC_NR + 2 * TC_NB + 6) * 8 + 16;
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
    // A tile reads one 256-byte half of each 512-byte slab row (L2 promotion 256 B).
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
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PIR_ERR_ARG;
    }
    {
        // Last slab of every point: (column, row k, 1, point), base at slab S-1.
        const cuuint64_t dim[4] = {Wlast, D0, 1, P};
        const cuuint64_t str[3] = {(cuuint64_t)Wlast * 4, (cuuint64_t)D0 * Wlast * 4, (cuuint64_t)D0 * D1p * 4};
        void *lastp = const_cast<uint32_t *>(db + (uint64_t)(S - 1) * D0 * PIR_SLAB);
        if (encode(&last_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, lastp, dim, str, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
    pdl_launch(rowsel_tc_kernel, dim3((unsigned)grid), dim3(TC_THREADS), smem, st, full_map, last_map, a);
    return launch_status(cudaGetLastError());
}
