// server.cu — pipelined query server over a resident RowSel DB (host runtime).
//
// GPIR section 2 (OnionPIRv2 online phase): for every query the server runs
// NTT(query) -> RowSel -> INTT(result).  Serving a stream of queries from
// host memory adds two copies per query (query in, result out).  They use
// the copy engines, not the SMs, so this object overlaps them with the scan
// of the neighbouring queries: query i+1 is copied in and the result of
// query i-1 is copied out while query i is scanned.
//
// Three streams and two buffer slots:
//   h2d      : wait until slot s's query buffer is free, copy query i in;
//   compute  : NTT(q_coef[s]) -> q_ntt, RowSel -> o_ntt, INTT -> o_coef[s]
//              (after slot s's previous result has left), in order;
//   d2h      : copy o_coef[s] out; the host waits on this copy's event.
// The NTT-domain buffers and the RowSel workspace are shared by the slots
// because the compute stream runs one query at a time.
#include <cuda_runtime.h>

#include <new>

#include "common.cuh"

struct pir_server {
    pir_ctx *ctx = nullptr;
    const uint32_t *db = nullptr;
    uint32_t D0 = 0, D1 = 0, B = 0;
    uint64_t q_words = 0, o_words = 0, ws_bytes = 0;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    uint32_t *q_coef[2] = {nullptr, nullptr}, *o_coef[2] = {nullptr, nullptr};
    uint32_t *q_ntt = nullptr, *o_ntt = nullptr;
    void *ws = nullptr;
    uint32_t *status_h = nullptr;               // pinned: the status word after each slot's query
    cudaEvent_t in_done[2] = {}, q_free[2] = {}, comp_done[2] = {}, out_done[2] = {};
    cudaEvent_t mark[2] = {};
    uint64_t next_ticket = 0;
    uint64_t done_ticket[2] = {~0ull, ~0ull};   // ticket whose copy-out out_done[s] tracks
};

namespace {

void release(pir_server *s) {
    for (int i = 0; i < 2; ++i) {
        if (s->q_coef[i]) cudaFree(s->q_coef[i]);
        if (s->o_coef[i]) cudaFree(s->o_coef[i]);
        for (cudaEvent_t e : {s->in_done[i], s->q_free[i], s->comp_done[i], s->out_done[i], s->mark[i]})
            if (e) cudaEventDestroy(e);
    }
    if (s->q_ntt) cudaFree(s->q_ntt);
    if (s->o_ntt) cudaFree(s->o_ntt);
    if (s->ws) cudaFree(s->ws);
    if (s->status_h) cudaFreeHost(s->status_h);
    for (cudaStream_t st : {s->h2d, s->comp, s->d2h})
        if (st) cudaStreamDestroy(st);
    delete s;
}

}  // namespace

extern "C" int pir_server_create(pir_server **out, pir_ctx *ctx, const uint32_t *db, uint32_t D0, uint32_t D1,
                                 uint32_t B) {
    if (!out) return PIR_ERR_ARG;
    *out = nullptr;
    if (!ctx || !db || D0 == 0 || D1 == 0 || B == 0) return PIR_ERR_ARG;
    const uint64_t P = (uint64_t)ctx->L * ctx->N;
    const uint64_t ws = pir_rowsel_workspace_bytes(ctx, D0, D1, B);
    if (ws == 0) return PIR_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    pir_server *s = new (std::nothrow) pir_server;
    if (!s) return PIR_ERR_ALLOC;
    s->ctx = ctx;
    s->db = db;
    s->D0 = D0;
    s->D1 = D1;
    s->B = B;
    s->q_words = (uint64_t)B * D0 * 2 * P;
    s->o_words = (uint64_t)B * D1 * 2 * P;
    s->ws_bytes = ws;
    bool ok = true;
    for (cudaStream_t *st : {&s->h2d, &s->comp, &s->d2h})
        ok = ok && cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i) {
        ok = ok && cudaMalloc(&s->q_coef[i], s->q_words * 4) == cudaSuccess;
        ok = ok && cudaMalloc(&s->o_coef[i], s->o_words * 4) == cudaSuccess;
        for (cudaEvent_t *e : {&s->in_done[i], &s->q_free[i], &s->comp_done[i], &s->out_done[i]})
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreate(&s->mark[i]) == cudaSuccess;
    }
    ok = ok && cudaMalloc(&s->q_ntt, s->q_words * 4) == cudaSuccess;
    ok = ok && cudaMalloc(&s->o_ntt, s->o_words * 4) == cudaSuccess;
    ok = ok && cudaMalloc(&s->ws, ws) == cudaSuccess;
    ok = ok && cudaHostAlloc(reinterpret_cast<void **>(&s->status_h), 2 * sizeof(uint32_t), cudaHostAllocDefault) ==
                   cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        release(s);
        return PIR_ERR_ALLOC;
    }
    *out = s;
    return PIR_OK;
}

extern "C" void pir_server_destroy(pir_server *s) {
    if (!s) return;
    cudaSetDevice(s->ctx->device);
    for (cudaStream_t st : {s->h2d, s->comp, s->d2h})
        if (st) cudaStreamSynchronize(st);
    release(s);
}

extern "C" int pir_server_submit(pir_server *s, const uint32_t *host_query, uint32_t *host_result,
                                 uint64_t *ticket) {
    if (!s || !host_query || !host_result) return PIR_ERR_ARG;
    if (cudaSetDevice(s->ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    const uint64_t t = s->next_ticket;
    const int k = (int)(t & 1);
    // query in: once the NTT of this slot's previous query has read q_coef[k]
    if (cudaStreamWaitEvent(s->h2d, s->q_free[k], 0) != cudaSuccess) return PIR_ERR_CUDA;
    if (cudaMemcpyAsync(s->q_coef[k], host_query, s->q_words * 4, cudaMemcpyHostToDevice, s->h2d) != cudaSuccess)
        return PIR_ERR_CUDA;
    if (cudaEventRecord(s->in_done[k], s->h2d) != cudaSuccess) return PIR_ERR_CUDA;
    // compute: NTT -> RowSel -> INTT, the INTT after this slot's previous copy-out
    if (cudaStreamWaitEvent(s->comp, s->in_done[k], 0) != cudaSuccess) return PIR_ERR_CUDA;
    int rc = pir_ntt_fwd(s->ctx, s->q_coef[k], s->q_ntt, (uint64_t)s->B * s->D0 * 2, s->comp);
    if (rc) return rc;
    if (cudaEventRecord(s->q_free[k], s->comp) != cudaSuccess) return PIR_ERR_CUDA;
    rc = pir_rowsel(s->ctx, s->db, s->D0, s->D1, s->q_ntt, s->B, s->o_ntt, s->ws, s->ws_bytes, s->comp);
    if (rc) return rc;
    if (cudaStreamWaitEvent(s->comp, s->out_done[k], 0) != cudaSuccess) return PIR_ERR_CUDA;
    rc = pir_ntt_inv(s->ctx, s->o_ntt, s->o_coef[k], (uint64_t)s->B * s->D1 * 2, s->comp);
    if (rc) return rc;
    if (cudaEventRecord(s->comp_done[k], s->comp) != cudaSuccess) return PIR_ERR_CUDA;
    // result out
    if (cudaStreamWaitEvent(s->d2h, s->comp_done[k], 0) != cudaSuccess) return PIR_ERR_CUDA;
    if (cudaMemcpyAsync(host_result, s->o_coef[k], s->o_words * 4, cudaMemcpyDeviceToHost, s->d2h) != cudaSuccess)
        return PIR_ERR_CUDA;
    // the context's status word as of this query, read without a device-wide sync
    if (cudaMemcpyAsync(s->status_h + k, s->ctx->d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s->d2h) !=
        cudaSuccess)
        return PIR_ERR_CUDA;
    if (cudaEventRecord(s->out_done[k], s->d2h) != cudaSuccess) return PIR_ERR_CUDA;
    s->done_ticket[k] = t;
    s->next_ticket = t + 1;
    if (ticket) *ticket = t;
    return PIR_OK;
}

extern "C" int pir_server_wait(pir_server *s, uint64_t ticket) {
    if (!s || ticket >= s->next_ticket) return PIR_ERR_ARG;
    if (cudaSetDevice(s->ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    const int k = (int)(ticket & 1);
    // the slot's event tracks `ticket` or a later query of the same slot,
    // which finishes after it (copy-outs leave in submission order)
    if (s->done_ticket[k] < ticket) return PIR_ERR_ARG;
    if (cudaEventSynchronize(s->out_done[k]) != cudaSuccess) return PIR_ERR_CUDA;
    // status of the slot's latest query (no device-wide synchronisation,
    // which would stall the pipeline): a device-side timeout is sticky, so
    // it shows up in every later query's copy too
    return s->status_h[k] ? PIR_ERR_CUDA : PIR_OK;
}

extern "C" int pir_server_mark(pir_server *s, int which) {
    if (!s || (which != 0 && which != 1)) return PIR_ERR_ARG;
    if (cudaSetDevice(s->ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    // begin: on the copy-in stream, before the next query's copy;
    // end: on the copy-out stream, after the last submitted result's copy
    return cudaEventRecord(s->mark[which], which == 0 ? s->h2d : s->d2h) == cudaSuccess ? PIR_OK : PIR_ERR_CUDA;
}

extern "C" int pir_server_elapsed_ms(pir_server *s, float *ms) {
    if (!s || !ms) return PIR_ERR_ARG;
    if (cudaSetDevice(s->ctx->device) != cudaSuccess) return PIR_ERR_CUDA;
    if (cudaEventSynchronize(s->mark[1]) != cudaSuccess) return PIR_ERR_CUDA;
    return cudaEventElapsedTime(ms, s->mark[0], s->mark[1]) == cudaSuccess ? PIR_OK : PIR_ERR_CUDA;
}
