// ctx.cu — context creation, parameter validation, twiddle tables, status word.
//
// Ring parameters follow VIPIR (sections 2.2, 2.3, 4.2): N = 2^12, q split
// into #RNS primes q_i < 2^29, each q_i = 1 mod 2N so that the negacyclic
// NTT of length N exists mod q_i.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "common.cuh"

namespace {

uint64_t mulmod64(uint64_t a, uint64_t b, uint64_t m) { return (uint64_t)((unsigned __int128)a * b % m); }

uint64_t powmod64(uint64_t b, uint64_t e, uint64_t m) {
    uint64_t r = 1 % m;
    b %= m;
    for (; e; e >>= 1) {
        if (e & 1) r = mulmod64(r, b, m);
        b = mulmod64(b, b, m);
    }
    return r;
}

// Deterministic Miller-Rabin for 32-bit n (bases 2, 7, 61 suffice below 4.7e9).
bool is_prime32(uint32_t n) {
    if (n < 2) return false;
    for (uint32_t p : {2u, 3u, 5u, 7u, 11u, 13u, 61u})
        if (n % p == 0) return n == p;
    uint32_t d = n - 1, s = 0;
    while ((d & 1) == 0) { d >>= 1; ++s; }
    for (uint32_t a : {2u, 7u, 61u}) {
        uint64_t x = powmod64(a, d, n);
        if (x == 1 || x == n - 1) continue;
        bool comp = true;
        for (uint32_t r = 1; r < s; ++r) {
            x = mulmod64(x, x, n);
            if (x == n - 1) { comp = false; break; }
        }
        if (comp) return false;
    }
    return true;
}

uint32_t bit_reverse(uint32_t x, uint32_t bits) {
    uint32_t r = 0;
    for (uint32_t i = 0; i < bits; ++i) { r = (r << 1) | (x & 1); x >>= 1; }
    return r;
}

// Smallest primitive 2N-th root of unity mod q: take any element of order
// 2N (c = x^((q-1)/2N) with c^N = -1) and scan its odd powers, which are
// exactly the primitive 2N-th roots.
uint32_t smallest_psi(uint32_t q, uint32_t N) {
    uint64_t c = 0;
    for (uint64_t x = 2; x < q; ++x) {
        uint64_t cand = powmod64(x, (q - 1) / (2ull * N), q);
        if (powmod64(cand, N, q) == q - 1ull) { c = cand; break; }
    }
    if (!c) return 0;
    uint64_t c2 = mulmod64(c, c, q), cur = c, best = c;
    for (uint32_t e = 1; e < 2 * N; e += 2) {
        if (cur < best) best = cur;
        cur = mulmod64(cur, c2, q);
    }
    return (uint32_t)best;
}

uint32_t shoup_of(uint32_t w, uint32_t q) { return (uint32_t)(((uint64_t)w << 32) / q); }

}  // namespace

extern "C" int pir_params_check(uint32_t N, uint32_t L, const uint32_t *q) {
    if (N < 16 || N > 4096 || (N & (N - 1))) return PIR_ERR_ARG;
    if (L < 1 || L > PIR_MAX_RNS || !q) return PIR_ERR_ARG;
    for (uint32_t i = 0; i < L; ++i) {
        if (q[i] >= (1u << 29) || q[i] % (2 * N) != 1 || !is_prime32(q[i])) return PIR_ERR_ARG;
        for (uint32_t j = 0; j < i; ++j)
            if (q[j] == q[i]) return PIR_ERR_ARG;
    }
    return PIR_OK;
}

extern "C" int pir_primes(uint32_t N, uint32_t L, uint32_t *q) {
    if (N < 16 || N > 4096 || (N & (N - 1)) || L < 1 || L > PIR_MAX_RNS || !q) return PIR_ERR_ARG;
    const uint32_t step = 2 * N;
    uint32_t found = 0;
    // candidates 1 + t*2N below 2^29, from the top down
    for (uint64_t x = ((1ull << 29) - 1) / step * step + 1; x > step && found < L; x -= step)
        if (x < (1ull << 29) && is_prime32((uint32_t)x)) q[found++] = (uint32_t)x;
    return found == L ? PIR_OK : PIR_ERR_ARG;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? PIR_OK : PIR_ERR_CUDA; }

RnsParams rns_params(const pir_ctx *ctx) {
    RnsParams P;
    memset(&P, 0, sizeof(P));
    P.N = ctx->N;
    P.logN = ctx->logN;
    P.L = ctx->L;
    for (uint32_t l = 0; l < ctx->L; ++l) {
        P.q[l] = ctx->q[l];
        P.ninv[l] = ctx->ninv[l];
        P.ninv_shoup[l] = ctx->ninv_shoup[l];
        P.r32[l] = ctx->r32[l];
        P.mu[l] = ctx->mu[l];
    }
    P.tw = ctx->d_tw;
    P.status = ctx->d_status;
    return P;
}

extern "C" int pir_ctx_create(pir_ctx **out, uint32_t N, uint32_t L, const uint32_t *q, int device) {
    if (!out) return PIR_ERR_ARG;
    *out = nullptr;
    int rc = pir_params_check(N, L, q);
    if (rc) return rc;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return PIR_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return PIR_ERR_CUDA;

    pir_ctx *c = (pir_ctx *)calloc(1, sizeof(pir_ctx));
    if (!c) return PIR_ERR_ALLOC;
    c->device = device;
    c->wait_limit_ns = PIR_WAIT_LIMIT_NS;
    c->test_hook = PIR_HOOK_NONE;
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
    c->N = N;
    c->L = L;
    while ((1u << c->logN) < N) ++c->logN;

    std::vector<uint32_t> tw((size_t)L * 4 * N);   // [L][2][N] pairs {w, shoup(w)}
    // NTT(X^(-2^j)) for every expansion stage j < logN: slot s holds the value
    // at psi^(2 brv(s) + 1), i.e. psi^(-E) with E = 2^j (2 brv(s) + 1) mod 2N.
    std::vector<uint32_t> xpow((size_t)c->logN * L * N);
    std::vector<uint32_t> pinv((size_t)2 * N);
    for (uint32_t l = 0; l < L; ++l) {
        uint32_t ql = q[l];
        c->q[l] = ql;
        c->psi[l] = smallest_psi(ql, N);
        if (!c->psi[l]) { free(c); return PIR_ERR_ARG; }
        c->ninv[l] = (uint32_t)powmod64(N, ql - 2, ql);
        c->ninv_shoup[l] = shoup_of(c->ninv[l], ql);
        c->r32[l] = (uint32_t)((1ull << 32) % ql);
        c->mu[l] = (uint64_t)(((unsigned __int128)1 << 64) / ql);
        uint64_t psi_inv = powmod64(c->psi[l], ql - 2, ql);
        uint32_t *F = tw.data() + ((size_t)l * 2 + TW_FWD) * 2 * N;
        uint32_t *I = tw.data() + ((size_t)l * 2 + TW_INV) * 2 * N;
        for (uint32_t i = 0; i < N; ++i) {
            uint32_t e = bit_reverse(i, c->logN);
            uint32_t wf = (uint32_t)powmod64(c->psi[l], e, ql);
            uint32_t wi = (uint32_t)powmod64(psi_inv, e, ql);
            F[2 * i] = wf;
            F[2 * i + 1] = shoup_of(wf, ql);
            I[2 * i] = wi;
            I[2 * i + 1] = shoup_of(wi, ql);
        }
        pinv[0] = 1;
        for (uint32_t e = 1; e < 2 * N; ++e) pinv[e] = (uint32_t)((uint64_t)pinv[e - 1] * psi_inv % ql);
        for (uint32_t j = 0; j < c->logN; ++j)
            for (uint32_t s = 0; s < N; ++s) {
                const uint32_t E = (uint32_t)(((uint64_t)(2 * bit_reverse(s, c->logN) + 1) << j) & (2 * N - 1));
                xpow[((size_t)j * L + l) * N + s] = pinv[E];
            }
    }
    if (cudaMalloc(&c->d_tw, tw.size() * sizeof(uint32_t)) != cudaSuccess) { free(c); return PIR_ERR_ALLOC; }
    if (cudaMalloc(&c->d_xpow, xpow.size() * sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(c->d_tw);
        free(c);
        return PIR_ERR_ALLOC;
    }
    if (cudaMalloc(&c->d_status, 256) != cudaSuccess) {
        cudaFree(c->d_tw);
        cudaFree(c->d_xpow);
        free(c);
        return PIR_ERR_ALLOC;
    }
    if (cudaMemcpy(c->d_tw, tw.data(), tw.size() * sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(c->d_xpow, xpow.data(), xpow.size() * sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(c->d_status, 0, 256) != cudaSuccess) {
        cudaFree(c->d_tw);
        cudaFree(c->d_xpow);
        cudaFree(c->d_status);
        free(c);
        return PIR_ERR_CUDA;
    }
    *out = c;
    return PIR_OK;
}

extern "C" void pir_ctx_destroy(pir_ctx *ctx) {
    if (!ctx) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    cudaDeviceSynchronize();
    cudaFree(ctx->d_tw);
    cudaFree(ctx->d_xpow);
    cudaFree(ctx->d_status);
    cudaSetDevice(prev);
    free(ctx);
}

extern "C" int pir_ctx_psi(const pir_ctx *ctx, uint32_t *psi) {
    if (!ctx || !psi) return PIR_ERR_ARG;
    for (uint32_t l = 0; l < ctx->L; ++l) psi[l] = ctx->psi[l];
    return PIR_OK;
}

extern "C" int pir_status(pir_ctx *ctx, uint32_t *flags, int clear) {
    if (!ctx || !flags) return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PIR_ERR_CUDA;
    if (cudaMemcpy(flags, ctx->d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return PIR_ERR_CUDA;
    if (clear && cudaMemset(ctx->d_status, 0, sizeof(uint32_t)) != cudaSuccess) return PIR_ERR_CUDA;
    return PIR_OK;
}

extern "C" int pir_ctx_set_wait_limit(pir_ctx *ctx, uint64_t ns) {
    if (!ctx || ns > PIR_WAIT_LIMIT_NS) return PIR_ERR_ARG;
    ctx->wait_limit_ns = ns ? ns : PIR_WAIT_LIMIT_NS;
    return PIR_OK;
}

extern "C" int pir_ctx_set_test_hook(pir_ctx *ctx, uint32_t hook) {
    if (!ctx || hook > PIR_HOOK_WITHHOLD_LAST_COPY) return PIR_ERR_ARG;
    ctx->test_hook = hook;
    return PIR_OK;
}

extern "C" const char *pir_strerror(int code) {
    switch (code) {
        case PIR_OK: return "ok";
        case PIR_ERR_ARG: return "invalid argument";
        case PIR_ERR_CUDA: return "CUDA error";
        case PIR_ERR_UNSUPPORTED: return "unsupported configuration";
        case PIR_ERR_ALLOC: return "allocation failed";
        default: return "unknown error";
    }
}
