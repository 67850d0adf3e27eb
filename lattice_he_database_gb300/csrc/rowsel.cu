// rowsel.cu — the RowSel scan of the OnionPIR family on GB300.
//
// GPIR (arXiv 2604.04696) section 2: RowSel is L*N independent point-wise
// GEMMs  M_out[p,m,n] = sum_k M_in0[p,m,k] * M_in1[p,k,n]  (p: evaluation
// point, m: ciphertext polynomial, k < D0 DB row, n < D1 DB column), and GEMM
// kernels want the DB contiguous along k/n per point rather than p-major.
// VIPIR section 4.2: with primes below 2^29 and 64-bit accumulators the
// modular reduction can be deferred across many multiply-adds.
//
// Design (one GPU, HBM-bound for small B):
//  * The DB is pre-encoded (encode.cu) so that every (p, column slab) is one
//    contiguous D0 x W_s block, W_s <= 128 words.  A unit of work is one such
//    block; units are split into equal contiguous ranges, one per CTA of a
//    persistent grid, so each CTA streams its own region of HBM exactly once.
//  * A producer warp moves the block through a 3-stage shared-memory ring
//    with 1-D bulk async copies (cp.async.bulk, L2 evict-first) of 64 rows
//    (32 KiB) each, signalling mbarriers; 8 consumer warps compute from
//    shared memory.
//  * The query is first transposed (GPIR's NTT-to-GEMM layout change) into
//    a workspace qT[p][k][m], so that the slice M_in0[p, :, :] of a point
//    is one contiguous block; the producer bulk-copies it into shared
//    memory ahead of the point's DB chunks (double-buffered when it fits).
//  * Thread tile: 4 consecutive columns x MT ciphertext polynomials; warps
//    split the polynomials (msplit) and the rows of each chunk (ksplit).
//    Products of residues < 2^29 are accumulated with 32x32->64-bit
//    multiply-adds; at least every 48 products the accumulator is folded
//    (lo + hi * (2^32 mod q)); one Barrett reduction per output at the end,
//    plus a sum of the ksplit partial residues.
//  * Device waits are bounded; on a timeout the kernel raises
//    PIR_STATUS_TIMEOUT, stops issuing copies, drains those in flight and
//    runs the remaining control flow without waiting, so it always ends.
#include <cstring>

#include "common.cuh"

namespace {

constexpr int KC = 64;                         // DB rows per ring stage
constexpr int NST = 3;                         // ring stages
constexpr int NWC = 8;                         // consumer warps
constexpr int NTHREADS = (NWC + 1) * 32;       // + one producer warp
constexpr uint32_t STAGE_WORDS = KC * PIR_SLAB;  // 32 KiB
constexpr uint32_t IN0_MAX_BYTES = 112 * 1024;  // one query slice; the ring takes 96 KiB
constexpr uint32_t FOLD_LIMIT = 48;            // products between folds
static_assert(KC / 2 <= 32, "a chunk must add at most 32 products per accumulator (ksplit >= 2)");

struct RowselArgs {
    const uint32_t *db;
    const uint32_t *qT;      // transposed query [P][PS] (PS >= D0*Mp, multiple of 4)
    uint32_t *out;
    uint32_t *status;
    uint32_t N, L, D0, D1, D1p, S, Wlast;
    uint32_t B, b0, Mv, Mp, msplit, ksplit, nchunks;
    uint32_t PS, nb;         // query slice stride (words) and number of slice buffers (1 or 2)
    uint32_t *outT;          // point-major results [P][Mv][D1p] of the pass
    uint64_t P, units;
    uint32_t q[PIR_MAX_RNS], r32[PIR_MAX_RNS];
    uint64_t mu[PIR_MAX_RNS];
    uint64_t wait_ns;        // limit of the ordinary waits (drains keep PIR_WAIT_LIMIT_NS)
    uint32_t hook;           // PIR_HOOK_* of the context
};

__device__ __forceinline__ uint32_t slab_width(const RowselArgs &A, uint32_t s) {
    return s == A.S - 1 ? A.Wlast : PIR_SLAB;
}

// Both transposes move 64 x 64-word tiles through shared memory (row pitch
// 65 words) with 16-byte global accesses on both sides: 256 threads, each
// loading four 16-byte pieces along one side and storing four along the
// other.  P = L*N is a multiple of 16, PS and the outT row length Mv*D1p are
// multiples of 4, so a 16-byte piece is either wholly inside or wholly out.
constexpr int TT = 64;
constexpr int TPITCH = TT + 1;

// Transpose of the query into qT[p][k][m] (m = 2b + c relative to the pass's
// first query b0; polynomials m >= Mv of the padded count are zero).  Column
// r = k*Mp + m of qT is row ((b0 + m/2)*D0 + k)*2 + (m&1) of the query.
__global__ void __launch_bounds__(256) transpose_query_kernel(const uint32_t *__restrict__ query,
                                                              uint32_t *__restrict__ qT, uint64_t P,
                                                              uint32_t D0, uint32_t Mp, uint32_t Mv,
                                                              uint32_t b0, uint32_t PS) {
    __shared__ uint32_t tile[TT][TPITCH];   // [r][p]
    pdl_wait();
    const uint64_t p0 = (uint64_t)blockIdx.x * TT;
    const uint32_t r0 = blockIdx.y * TT;
    const uint32_t rows = D0 * Mp;
    const uint32_t lo = threadIdx.x & 15, hi = threadIdx.x >> 4;   // 16 x 16
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t rr = hi + 16 * i, r = r0 + rr;
        const uint64_t p = p0 + 4 * lo;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && p < P) {
            const uint32_t k = r / Mp, m = r - k * Mp;
            if (m < Mv)
                v = *reinterpret_cast<const uint4 *>(query + (((uint64_t)(b0 + (m >> 1)) * D0 + k) * 2 + (m & 1)) * P + p);
        }
        uint32_t *t = &tile[rr][4 * lo];
        t[0] = v.x; t[1] = v.y; t[2] = v.z; t[3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t pp = hi + 16 * i;
        const uint64_t p = p0 + pp;
        const uint32_t r = r0 + 4 * lo;
        if (p < P && r < PS)
            *reinterpret_cast<uint4 *>(qT + p * PS + r) =
                make_uint4(tile[4 * lo][pp], tile[4 * lo + 1][pp], tile[4 * lo + 2][pp], tile[4 * lo + 3][pp]);
    }
}

// Results of a pass from the point-major block outT[p][w] (w = m*D1p + n,
// row length W = Mv*D1p) to out[b][n][c][p] (m = 2(b - b0) + c); padding
// columns n >= D1 are dropped.  With an addend G (ring packing), G[b][n]
// joins polynomial c = 1 of every ciphertext.
struct AddendArgs {
    const uint32_t *G;       // [B][D1][L][N] residues added to polynomial c = 1, or null
    uint32_t N;
    uint32_t q[PIR_MAX_RNS];
};

__global__ void __launch_bounds__(256) transpose_out_kernel(const uint32_t *__restrict__ outT,
                                                            uint32_t *__restrict__ out, uint64_t P, uint32_t D1,
                                                            uint32_t D1p, uint32_t Mv, uint32_t b0,
                                                            const __grid_constant__ AddendArgs add) {
    __shared__ uint32_t tile[TT][TPITCH];   // [w][p]
    pdl_wait();
    const uint64_t p0 = (uint64_t)blockIdx.x * TT;
    const uint32_t w0 = blockIdx.y * TT;
    const uint32_t W = Mv * D1p;
    const uint32_t lo = threadIdx.x & 15, hi = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t pp = hi + 16 * i;
        const uint64_t p = p0 + pp;
        const uint32_t w = w0 + 4 * lo;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (p < P && w < W) v = *reinterpret_cast<const uint4 *>(outT + p * W + w);
        tile[4 * lo][pp] = v.x;
        tile[4 * lo + 1][pp] = v.y;
        tile[4 * lo + 2][pp] = v.z;
        tile[4 * lo + 3][pp] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ww = hi + 16 * i, w = w0 + ww;
        const uint64_t p = p0 + 4 * lo;
        if (w >= W || p >= P) continue;
        const uint32_t m = w / D1p, n = w - m * D1p;
        if (n >= D1) continue;
        const uint64_t b = b0 + (m >> 1);
        const uint32_t *t = &tile[ww][4 * lo];
        uint4 v = make_uint4(t[0], t[1], t[2], t[3]);
        if (add.G && (m & 1)) {  // (0 | G): the second polynomial of each ciphertext
            const uint32_t q = add.q[p / add.N];   // 4 consecutive points share a prime (N >= 16)
            const uint4 g = *reinterpret_cast<const uint4 *>(add.G + (b * D1 + n) * P + p);
            v.x += g.x; v.x = v.x >= q ? v.x - q : v.x;
            v.y += g.y; v.y = v.y >= q ? v.y - q : v.y;
            v.z += g.z; v.z = v.z >= q ? v.z - q : v.z;
            v.w += g.w; v.w = v.w >= q ? v.w - q : v.w;
        }
        *reinterpret_cast<uint4 *>(out + ((b * D1 + n) * 2 + (m & 1)) * P + p) = v;
    }
}

template <int MT>
__global__ void __launch_bounds__(NTHREADS) rowsel_kernel(const __grid_constant__ RowselArgs A) {
    extern __shared__ __align__(128) uint32_t smw[];
    uint32_t *ring = smw;                                    // NST * STAGE_WORDS
    uint32_t *in0s = ring + NST * STAGE_WORDS;               // nb * PS   (k-major query slices)
    uint32_t *red = in0s + (size_t)A.nb * A.PS;              // Mp * 128 sums of the ksplit partials
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + (A.ksplit > 1 ? A.Mp * PIR_SLAB : 0));
    uint64_t *full = bars, *empty = bars + NST, *qfull = bars + 2 * NST, *qempty = qfull + 2;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t u0 = (uint64_t)blockIdx.x * A.units / gridDim.x;
    const uint64_t u1 = (uint64_t)(blockIdx.x + 1) * A.units / gridDim.x;
    const uint32_t qbytes = A.PS * 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, NWC);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull + i, 1);
            mbar_init(qempty + i, NWC);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (A.ksplit > 1)   // the partial-sum rows start at zero; each unit's reader clears what it read
        for (uint32_t i = threadIdx.x; i < A.Mp * PIR_SLAB; i += blockDim.x) red[i] = 0;
    __syncthreads();
    pdl_wait();   // the set-up above touches no global memory

    // ------------------------------------------------------------ producer
    if (warp == NWC) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t stage = 0, phase = 0, pc = 0;
            uint64_t issued = 0, cur_p = ~0ull;
            bool withheld = false;
            for (uint64_t u = u0; u < u1 && !abort_flag; ++u) {
                const uint64_t p = u / A.S;
                const uint32_t s = (uint32_t)(u - p * A.S);
                if (p != cur_p) {  // the point's query slice goes first (consumers need it first)
                    const uint32_t slot = pc % A.nb, use = (pc / A.nb) & 1;
                    if (!mbar_wait(qempty + slot, use ^ 1, A.status, A.wait_ns)) {
                        abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(qfull + slot, qbytes);
                    bulk_g2s(in0s + (size_t)slot * A.PS, A.qT + p * A.PS, qbytes, qfull + slot, pol);
                    ++pc;
                    cur_p = p;
                }
                const uint32_t Ws = slab_width(A, s);
                const uint32_t *src = A.db + p * A.D0 * A.D1p + (uint64_t)s * A.D0 * PIR_SLAB;
                for (uint32_t c = 0; c < A.nchunks; ++c) {
                    const uint32_t rows = min((uint32_t)KC, A.D0 - c * KC);
                    const uint32_t bytes = rows * Ws * 4;
                    if (!mbar_wait(empty + stage, phase ^ 1, A.status, A.wait_ns)) {
                        abort_flag = 1;
                        break;
                    }
                    if (A.hook == PIR_HOOK_WITHHOLD_LAST_COPY && blockIdx.x == 0 && u + 1 == u1 &&
                        c + 1 == A.nchunks) {
                        // failure-path test: the CTA's last chunk is never copied, so its
                        // consumers' wait runs out; nothing reuses this stage afterwards
                        withheld = true;
                    } else {
                        mbar_arrive_expect_tx(full + stage, bytes);
                        bulk_g2s(ring + stage * STAGE_WORDS, src + (uint64_t)c * KC * Ws, bytes, full + stage, pol);
                        ++issued;
                    }
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            // The copies still in flight target this CTA's shared memory:
            // wait (bounded, full limit) for the last ring copies and query
            // slices to land.  A withheld copy was the CTA's last chunk: step
            // back over its stage, and only NST - 1 stages before it can hold
            // copies still in flight.
            if (withheld) {
                if (stage == 0) { stage = NST - 1; phase ^= 1; } else { --stage; }
            }
            const uint32_t cap = withheld ? NST - 1 : NST;
            const uint32_t pend = issued < (uint64_t)cap ? (uint32_t)issued : cap;
            for (uint32_t i = 0; i < pend; ++i) {
                if (stage == 0) { stage = NST - 1; phase ^= 1; } else { --stage; }
                mbar_wait(full + stage, phase, A.status);
            }
            const uint32_t qpend = pc < A.nb ? pc : A.nb;
            for (uint32_t i = 0; i < qpend; ++i) {
                const uint32_t j = pc - 1 - i;
                mbar_wait(qfull + j % A.nb, (j / A.nb) & 1, A.status);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const uint32_t ctid = threadIdx.x;  // 0 .. NWC*32-1
    const uint32_t ms = warp % A.msplit, ks = warp / A.msplit;
    uint32_t stage = 0, phase = 0, pc = 0, qslot = 0;
    uint64_t cur_p = ~0ull;

    for (uint64_t u = u0; u < u1; ++u) {
        const uint64_t p = u / A.S;
        const uint32_t s = (uint32_t)(u - p * A.S);
        const uint32_t Ws = slab_width(A, s);
        const uint32_t l = (uint32_t)(p / A.N);
        const uint32_t q = A.q[l], r32 = A.r32[l];
        const uint64_t mu = A.mu[l];

        if (p != cur_p) {  // release the previous point's slice, wait for this one
            if (cur_p != ~0ull) {
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty + qslot);
            }
            qslot = pc % A.nb;
            if (!abort_flag && !mbar_wait(qfull + qslot, (pc / A.nb) & 1, A.status, A.wait_ns)) abort_flag = 1;
            ++pc;
            cur_p = p;
        }

        uint64_t acc[MT][4];
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0;
        uint32_t cnt = 0;
        const bool active = 4u * lane < Ws;
        const uint32_t *a_base = in0s + (size_t)qslot * A.PS + ms * MT;

        for (uint32_t c = 0; c < A.nchunks; ++c) {
            const uint32_t rows = min((uint32_t)KC, A.D0 - c * KC);
            bool ok = !abort_flag;
            if (ok && !mbar_wait(full + stage, phase, A.status, A.wait_ns)) {
                abort_flag = 1;
                ok = false;
            }
            // KC / ksplit <= 32 (host guarantees ksplit >= 2), so a fold is
            // never more than FOLD_LIMIT (48) products away
            const uint32_t per = rows > ks ? (rows - ks + A.ksplit - 1) / A.ksplit : 0;
            if (cnt + per > FOLD_LIMIT) {
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fold64(acc[i][j], r32);
                cnt = 0;
            }
            cnt += per;
            if (ok && active) {
                const uint32_t *st = ring + stage * STAGE_WORDS + 4 * lane;
                const uint32_t *ak = a_base + (size_t)c * KC * A.Mp;
#pragma unroll(MT == 8 ? 1 : (MT == 2 ? 4 : 2))
                for (uint32_t r = ks; r < rows; r += A.ksplit) {
                    const uint4 d = *reinterpret_cast<const uint4 *>(st + r * Ws);
                    uint32_t a[MT];
                    if constexpr (MT == 2) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(ak + r * A.Mp);
                        a[0] = v.x;
                        a[1] = v.y;
                    } else {
#pragma unroll
                        for (int i = 0; i < MT; i += 4) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(ak + r * A.Mp + i);
                            a[i] = v.x;
                            a[i + 1] = v.y;
                            a[i + 2] = v.z;
                            a[i + 3] = v.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        acc[i][0] += (uint64_t)a[i] * d.x;
                        acc[i][1] += (uint64_t)a[i] * d.y;
                        acc[i][2] += (uint64_t)a[i] * d.z;
                        acc[i][3] += (uint64_t)a[i] * d.w;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + stage);
            if (++stage == NST) { stage = 0; phase ^= 1; }
        }

        // ---- unit epilogue: one reduction per output, then the write
        const uint32_t nbase = s * PIR_SLAB;
        // results go to the point-major block outT[p][m][n] (coalesced); a
        // transpose kernel then lays them out as [b][n][c][p]
        uint32_t *ot = A.outT + p * (uint64_t)A.Mv * A.D1p + nbase;
        if (A.ksplit == 1) {
            if (active) {
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const uint32_t m = ms * MT + i;
                    if (m >= A.Mv) continue;
                    *reinterpret_cast<uint4 *>(ot + (uint64_t)m * A.D1p + 4 * lane) =
                        make_uint4(barrett64(acc[i][0], q, mu), barrett64(acc[i][1], q, mu),
                                   barrett64(acc[i][2], q, mu), barrett64(acc[i][3], q, mu));
                }
            }
        } else {
            // the ksplit partial residues of an output are summed with shared-
            // memory atomics (at most 8 residues < 2^29: the sum fits 32 bits)
            named_barrier(1, NWC * 32);  // previous unit's readers have read and cleared `red`
            if (active) {
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        atomicAdd(red + (ms * MT + i) * PIR_SLAB + 4 * lane + j, barrett64(acc[i][j], q, mu));
            }
            named_barrier(1, NWC * 32);
            const uint32_t tot = A.Mv * Ws;
            for (uint32_t idx = ctid; idx < tot; idx += NWC * 32) {
                const uint32_t m = idx / Ws, col = idx - m * Ws;
                const uint32_t sum = red[m * PIR_SLAB + col];
                red[m * PIR_SLAB + col] = 0;
                ot[(uint64_t)m * A.D1p + col] = sum % q;
            }
        }
    }
}

size_t rowsel_smem(const RowselArgs &A, uint32_t nb) {
    return (size_t)NST * STAGE_WORDS * 4 + (size_t)nb * A.PS * 4 +
           (A.ksplit > 1 ? (size_t)A.Mp * PIR_SLAB * 4 : 0) + (2 * NST + 4) * sizeof(uint64_t);
}

template <int MT>
int launch_pass(pir_ctx *ctx, RowselArgs &A, cudaStream_t st) {
    // Double-buffer the query slices when that still leaves room for two
    // CTAs per SM, or when one CTA per SM is the outcome either way.
    constexpr size_t kTwoPerSm = 113 * 1024, kMax = 220 * 1024;  // 228 KiB per SM, 1 KiB reserved per CTA
    const size_t s1 = rowsel_smem(A, 1), s2 = rowsel_smem(A, 2);
    A.nb = (s2 <= kTwoPerSm || (s1 > kTwoPerSm && s2 <= kMax)) ? 2 : 1;
    const size_t smem = rowsel_smem(A, A.nb);
    if (smem > kMax) return PIR_ERR_UNSUPPORTED;
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        if (cudaFuncSetAttribute(rowsel_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMax) !=
            cudaSuccess)
            return PIR_ERR_CUDA;
        attr_set[ctx->device] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rowsel_kernel<MT>, NTHREADS, smem) != cudaSuccess ||
        per_sm < 1)
        return PIR_ERR_CUDA;
    const uint64_t cap = (uint64_t)ctx->num_sms * per_sm;
    const uint64_t grid = A.units < cap ? A.units : cap;
    pdl_launch(rowsel_kernel<MT>, dim3((unsigned)grid), dim3(NTHREADS), smem, st, A);
    return launch_status(cudaGetLastError());
}

// Polynomials per pass: the padded count Mp must be MT * msplit with
// msplit | NWC, and one query slice D0 * Mp words must fit on chip.
uint32_t mp_capacity(uint32_t D0) {
    uint32_t cap = 32;
    while (cap > 2 && (uint64_t)D0 * cap * 4 > IN0_MAX_BYTES) cap >>= 1;
    return (uint64_t)D0 * cap * 4 > IN0_MAX_BYTES ? 0 : cap;
}

uint32_t padded_mp(uint32_t Mv) {
    if (Mv <= 2) return 2;
    uint32_t mp = 4;
    while (mp < Mv) mp <<= 1;
    return mp;
}

}  // namespace

// Tensor-core path for large batches (rowsel_tc.cu).
bool rowsel_tc_primes_ok(const pir_ctx *ctx);
int rowsel_tc_pass(pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1, const uint32_t *qT, uint32_t PS,
                   uint32_t Mv, uint32_t *outT, cudaStream_t st);

namespace {

// Queries in the next pass when `left` remain: 16 on the tensor cores while
// more than 8 remain (passes of 17..32 polynomials, any D0), otherwise as
// many as one on-chip query slice of the CUDA-core kernel holds (cap
// polynomials).  The pass runs on the tensor cores iff it has more than 8.
uint32_t pass_queries(bool tc, uint32_t cap, uint32_t left) {
    if (tc && left > 8) return left < 16 ? left : 16;
    return left < cap / 2 ? left : cap / 2;
}

// Workspace: the pass's query slices (point-major) followed by the pass's
// results (point-major, 256-byte aligned).
struct WsLayout {
    uint64_t qT_words, outT_offset_words, total_bytes;
};

WsLayout ws_layout(const pir_ctx *ctx, uint32_t D0, uint32_t D1, uint32_t B) {
    WsLayout w{0, 0, 0};
    const uint32_t cap = mp_capacity(D0);
    if (!cap) return w;
    const bool tc = rowsel_tc_primes_ok(ctx);
    uint32_t nb = 0;   // queries in the largest pass
    for (uint32_t left = B; left;) {
        const uint32_t n = pass_queries(tc, cap, left);
        nb = n > nb ? n : nb;
        left -= n;
    }
    const uint32_t mp = padded_mp(2 * nb);
    const uint64_t P = (uint64_t)ctx->L * ctx->N;
    const uint64_t ps = ((uint64_t)D0 * mp + 3) / 4 * 4;
    const uint64_t D1p = ((uint64_t)D1 + 3) / 4 * 4;
    w.qT_words = P * ps;
    w.outT_offset_words = (w.qT_words + 63) / 64 * 64;
    w.total_bytes = (w.outT_offset_words + P * 2 * nb * D1p) * 4;
    return w;
}

}  // namespace

extern "C" uint64_t pir_rowsel_workspace_bytes(const pir_ctx *ctx, uint32_t D0, uint32_t D1, uint32_t B) {
    if (!ctx || D0 == 0 || D1 == 0 || B == 0 || D0 > 14336) return 0;
    return ws_layout(ctx, D0, D1, B).total_bytes;
}

namespace {

// RowSel passes over an encoded DB, with an optional addend G on the second
// polynomial of every result ciphertext (the ExpPack GEMM H*C + (0 | G)).
int rowsel_impl(pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1, const uint32_t *query, uint32_t B,
                const uint32_t *G, uint32_t *out, void *workspace, uint64_t workspace_bytes, void *stream) {
    if (!ctx || !db || !query || !out || !workspace) return PIR_ERR_ARG;
    if (G && !aligned16(G)) return PIR_ERR_ARG;
    if (!aligned16(db) || !aligned16(query) || !aligned16(out) || !aligned16(workspace)) return PIR_ERR_ARG;
    if (D0 == 0 || D1 == 0 || B == 0) return PIR_ERR_ARG;
    if (D0 > 14336) return PIR_ERR_UNSUPPORTED;
    const WsLayout wl = ws_layout(ctx, D0, D1, B);
    if (workspace_bytes < wl.total_bytes) return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;

    RowselArgs A;
    memset(&A, 0, sizeof(A));
    A.db = db;
    A.qT = reinterpret_cast<const uint32_t *>(workspace);
    A.outT = reinterpret_cast<uint32_t *>(workspace) + wl.outT_offset_words;
    A.out = out;
    A.status = ctx->d_status;
    A.wait_ns = ctx->wait_limit_ns;
    A.hook = ctx->test_hook;
    A.N = ctx->N;
    A.L = ctx->L;
    A.D0 = D0;
    A.D1 = D1;
    A.D1p = (D1 + 3) / 4 * 4;
    A.S = (D1 + PIR_SLAB - 1) / PIR_SLAB;
    A.Wlast = A.D1p - PIR_SLAB * (A.S - 1);
    A.B = B;
    A.P = (uint64_t)ctx->L * ctx->N;
    A.units = A.P * A.S;
    A.nchunks = (D0 + KC - 1) / KC;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        A.q[l] = ctx->q[l];
        A.r32[l] = ctx->r32[l];
        A.mu[l] = ctx->mu[l];
    }
    const uint32_t cap = mp_capacity(D0);
    if (!cap) return PIR_ERR_UNSUPPORTED;
    const bool tc = rowsel_tc_primes_ok(ctx);
    cudaStream_t st = (cudaStream_t)stream;
    for (uint32_t b0 = 0, nb = 0; b0 < B; b0 += nb) {
        nb = pass_queries(tc, cap, B - b0);
        A.b0 = b0;
        A.Mv = 2 * nb;
        A.Mp = padded_mp(A.Mv);
        A.PS = (D0 * A.Mp + 3) / 4 * 4;
        // the pass's query slices, point-major
        const dim3 tgrid((unsigned)((A.P + TT - 1) / TT), (A.PS + TT - 1) / TT);
        uint32_t *qT = reinterpret_cast<uint32_t *>(workspace);
        pdl_launch(transpose_query_kernel, tgrid, dim3(256), 0, st, query, qT, A.P, D0, A.Mp, A.Mv, b0, A.PS);
        if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;
        int rc = PIR_OK;
        if (tc && nb > 8) {  // 17..32 polynomials, q >= 2^26: exact fp16 tensor-core GEMMs
            rc = rowsel_tc_pass(ctx, db, D0, D1, qT, A.PS, A.Mv, A.outT, st);
        // thread tile MT polynomials x 4 columns; warps split the padded
        // polynomials (msplit) and the rows of a chunk (ksplit >= 2)
        } else if (A.Mp == 2) {
            A.msplit = 1;
            A.ksplit = NWC;
            rc = launch_pass<2>(ctx, A, st);
        } else if (A.Mp == 4) {
            A.msplit = 1;
            A.ksplit = NWC;
            rc = launch_pass<4>(ctx, A, st);
        } else {
            A.msplit = A.Mp / 8;
            A.ksplit = NWC / A.msplit;
            rc = launch_pass<8>(ctx, A, st);
        }
        if (rc) return rc;
        // the pass's results into the caller's [B][D1][2][L][N] layout
        AddendArgs add;
        memset(&add, 0, sizeof(add));
        add.G = G;
        add.N = ctx->N;
        for (uint32_t l = 0; l < ctx->L; ++l) add.q[l] = ctx->q[l];
        const dim3 ogrid((unsigned)((A.P + TT - 1) / TT), (A.Mv * A.D1p + TT - 1) / TT);
        pdl_launch(transpose_out_kernel, ogrid, dim3(256), 0, st, (const uint32_t *)A.outT, out, A.P, D1, A.D1p, A.Mv, b0,
                   add);
        if (cudaGetLastError() != cudaSuccess) return PIR_ERR_CUDA;
    }
    return PIR_OK;
}

}  // namespace

extern "C" int pir_rowsel(pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1, const uint32_t *query,
                          uint32_t B, uint32_t *out, void *workspace, uint64_t workspace_bytes, void *stream) {
    return rowsel_impl(ctx, db, D0, D1, query, B, nullptr, out, workspace, workspace_bytes, stream);
}

extern "C" int pir_exppack(pir_ctx *ctx, const uint32_t *h_db, uint32_t n, uint32_t Dr, const uint32_t *C,
                           const uint32_t *G, uint32_t B, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                           void *stream) {
    if (!G) return PIR_ERR_ARG;
    return rowsel_impl(ctx, h_db, n, Dr, C, B, G, out, workspace, workspace_bytes, stream);
}
