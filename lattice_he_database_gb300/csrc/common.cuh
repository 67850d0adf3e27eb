// common.cuh — internal definitions shared by the library's translation units.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "pir.h"

// ---------------------------------------------------------------- context
struct pir_ctx {
    int device;
    int num_sms;
    uint32_t N, logN, L;
    uint32_t q[PIR_MAX_RNS];
    uint32_t psi[PIR_MAX_RNS];
    uint32_t ninv[PIR_MAX_RNS];        // N^-1 mod q
    uint32_t ninv_shoup[PIR_MAX_RNS];  // floor(ninv * 2^32 / q)
    uint32_t r32[PIR_MAX_RNS];         // 2^32 mod q
    uint64_t mu[PIR_MAX_RNS];          // floor(2^64 / q)
    uint32_t *d_tw;                    // device twiddles [L][4][N]
    uint32_t *d_xpow;                  // device [logN][L][N]: NTT(X^(-2^j)) mod q_l, slot order (ExpandQuery)
    uint32_t *d_status;                // device status word
    uint64_t wait_limit_ns;            // limit of the kernels' ordinary waits (pir_ctx_set_wait_limit)
    uint32_t test_hook;                // PIR_HOOK_* (pir_ctx_set_test_hook); PIR_HOOK_NONE in normal use
};

// Parameters of the RNS ring passed by value to kernels.
struct RnsParams {
    uint32_t N, logN, L;
    uint32_t q[PIR_MAX_RNS];
    uint32_t ninv[PIR_MAX_RNS];
    uint32_t ninv_shoup[PIR_MAX_RNS];
    uint32_t r32[PIR_MAX_RNS];
    uint64_t mu[PIR_MAX_RNS];
    const uint32_t *tw;  // [L][2][N] pairs {w, floor(w 2^32 / q)}: w = psi^brv(i), then psi^-brv(i)
    uint32_t *status;    // the context's device status word (bounded waits report here)
};

RnsParams rns_params(const pir_ctx *ctx);

// Twiddle pairs {w, Shoup companion} of prime l in direction TW_FWD
// (psi^brv(i)) or TW_INV (psi^-brv(i)): one 8-byte load per butterfly.
enum { TW_FWD = 0, TW_INV = 1 };
__host__ __device__ __forceinline__ const uint2 *tw_pairs(const uint32_t *tw, uint32_t l, uint32_t N, int dir) {
    return reinterpret_cast<const uint2 *>(tw) + ((size_t)l * 2 + (size_t)dir) * N;
}

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch_status(cudaError_t e);  // maps a CUDA error to PIR_OK / PIR_ERR_CUDA

// Lift + forward NTT of cnt rows of gadget digits below 2^w (ntt.cu).
int lift_ntt_digits(pir_ctx *ctx, const uint32_t *raw, uint32_t *out, uint64_t cnt, uint32_t w, void *stream);

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel started by pdl_launch may be launched before the previous kernel
// of its stream has finished flushing its memory: the next grid's launch
// overlaps the previous grid's completion, which shortens chains of
// dependent kernels (ColTor and ExpandQuery run ~40 a call).  Such kernels
// call pdl_wait() before touching global memory; it returns once the
// previous kernel has completed and its memory operations are visible (and
// at once for an ordinary launch).  The kernels do not trigger their
// dependents early (griddepcontrol.launch_dependents at entry let waiting
// CTAs take SM slots from the previous kernel's last waves: slower in CUDA
// graphs), so the trigger is the implicit one at completion.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- modular helpers
// Shoup product: w * y mod q in [0, 2q) for y < 2^32, w < q < 2^31,
// wp = floor(w * 2^32 / q).
__device__ __forceinline__ uint32_t shoup_mul(uint32_t y, uint32_t w, uint32_t wp, uint32_t q) {
    uint32_t qh = __umulhi(y, wp);
    return y * w - qh * q;
}

// x mod q up to one subtraction for a 32-bit x: with m = floor(2^32 / q)
// (= mu >> 32), x - floor(x m / 2^32) q lies in [0, 2q) (Barrett).
__device__ __forceinline__ uint32_t barrett32_lazy(uint32_t x, uint32_t q, uint32_t m) {
    return x - __umulhi(x, m) * q;
}

// Barrett reduction of a 64-bit value: x mod q with mu = floor(2^64 / q).
__device__ __forceinline__ uint32_t barrett64(uint64_t x, uint32_t q, uint64_t mu) {
    uint64_t qh = __umul64hi(x, mu);
    uint64_t r = x - qh * q;  // in [0, 2q)
    return (uint32_t)(r >= q ? r - q : r);
}

// One lazy fold of a 64-bit accumulator: lo + hi * (2^32 mod q).  Keeps the
// value congruent mod q and brings it below 2^61 + 2^32 for q < 2^29.
__device__ __forceinline__ uint64_t fold64(uint64_t acc, uint32_t r32) {
    return (acc & 0xffffffffull) + (acc >> 32) * (uint64_t)r32;
}

// ---------------------------------------------------------------- async-copy / mbarrier PTX
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wall-clock limit of one device-side wait.  A correct launch never waits
// more than milliseconds; the limit only turns a lost arrival into an error.
// Kernels that take a context's limit (pir_ctx_set_wait_limit) use it for
// their ordinary waits; the waits that drain a kernel's own copies in flight
// before it exits always keep this full limit.
#define PIR_WAIT_LIMIT_NS 2000000000ull

// Bounded wait for the phase with parity `parity` of an mbarrier.  Returns
// false (and sets PIR_STATUS_TIMEOUT in *status) if `limit_ns` runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          uint64_t limit_ns = PIR_WAIT_LIMIT_NS) {
    uint32_t a = smem_u32(bar);
    for (int i = 0; i < 128; ++i)
        if (mbar_try_wait(a, parity)) return true;
    uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, PIR_STATUS_TIMEOUT);
            return false;
        }
    }
}

// L2 policy for data read exactly once (let it leave L2 first).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16-byte global load with an L2 eviction-priority policy (createpolicy);
// for data the kernel only reads.
__device__ __forceinline__ uint4 ld_policy(const void *p, uint64_t policy) {
    uint4 v;
    asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(policy));
    return v;
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy / TMA) accesses of the same locations.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Barrier among `nthreads` threads (a multiple of 32) with hardware id `id`.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
