// scalar.cu — scalar-HE scan (placeholder until the tensor-core kernel lands).
#include "common.cuh"

extern "C" uint64_t pir_scalar_workspace_bytes(uint64_t C, uint32_t B) {
    if (C == 0 || B == 0) return 0;
    return C * (uint64_t)B * 4 * 2;
}

extern "C" int pir_scalar_scan(pir_ctx *ctx, const uint8_t *db, uint64_t R, uint64_t C, const uint32_t *Q,
                               uint32_t B, uint32_t *out, void *workspace, uint64_t workspace_bytes,
                               void *stream) {
    (void)ctx; (void)db; (void)R; (void)C; (void)Q; (void)B; (void)out; (void)workspace;
    (void)workspace_bytes; (void)stream;
    return PIR_ERR_UNSUPPORTED;
}
