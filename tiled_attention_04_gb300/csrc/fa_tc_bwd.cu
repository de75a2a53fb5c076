// tcgen05 backward kernels (placeholder until the tensor-core path lands).
#include "fa_internal.h"

__device__ unsigned g_fa_bwd_status;

bool tc_bwd_supported(const FaProblem &) { return false; }
cudaError_t tc_bwd_preprocess(const FaProblem &, const void *, const void *, float *, float *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_bwd_dkdv(const FaProblem &, const void *, const void *, const void *, const void *, const float *,
                        const float *, float *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_bwd_dq(const FaProblem &, const float *, void *, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t tc_bwd_read_status(unsigned *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_bwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}
cudaError_t tc_bwd_reset_status(cudaStream_t st) {
    static const unsigned zero = 0;
    return cudaMemcpyToSymbolAsync(g_fa_bwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
}
