// tcgen05 forward kernel (placeholder until the tensor-core path lands).
#include "fa_internal.h"

__device__ unsigned g_fa_fwd_status;

bool tc_fwd_supported(const FaProblem &) { return false; }
cudaError_t tc_fwd(const FaProblem &, const void *, const void *, const void *, void *, float *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_fwd_read_status(unsigned *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_fwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}
cudaError_t tc_fwd_reset_status(cudaStream_t st) {
    static const unsigned zero = 0;
    return cudaMemcpyToSymbolAsync(g_fa_fwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
}
