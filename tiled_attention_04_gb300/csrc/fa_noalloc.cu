// fa_bwd_noalloc: the backward pass with its scratch memory inside the library.
//
// fa_bwd needs a caller-owned device workspace (per query row: D = rowsum(dO*O)
// and, on the tensor-core path, a copy of L).  Some callers cannot provide
// one: code that only receives raw pointers from a host framework and has no
// allocator of its own, or code that must not call cudaMalloc/cudaFree because
// those calls can synchronise the whole device and stall unrelated streams.
// For them this entry point uses a fixed-size array in device global memory
// that lives in this translation unit.  The array exists on every GPU that
// loads the library and stays allocated until the process exits.
//
// Rules for callers:
//  * the scratch is shared by every call: calls whose GPU work overlaps (two
//    streams, or two host threads) race on it and give wrong results; order
//    them on one stream or serialise them;
//  * nothing in the scratch needs to start at zero: each call writes every
//    scratch word it later reads, so the previous call's leftovers are harmless;
//  * the first call on a device looks up the array's device address (with that
//    device current) and caches it; make that first call before any stream
//    capture begins.  The cache lives as long as the process: cudaDeviceReset
//    reloads the module (and the array) elsewhere, so no call may follow a reset;
//  * where the library would form dQ by reduction (an fp32 dQ accumulator in the
//    workspace) and that does not fit, the call forms dQ by the separate pass;
//    fp32 inputs whose split bf16 copies do not fit run the CUDA-core kernels;
//    shapes whose workspace exceeds FA_NOALLOC_SCRATCH_BYTES even so are refused
//    with FA_ERR_WORKSPACE before anything is launched.
#include <cuda_runtime.h>


#include "fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// device address of the scratch array on the current device, looked up on every
// call (a cached address would not survive a cudaDeviceReset, which reloads the module)
fa_status scratch_for_current_device(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? FA_ERR_NO_DEVICE : FA_ERR_LAUNCH;
    }
    *out = p;
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_noalloc_scratch_bytes(void) { return FA_NOALLOC_SCRATCH_BYTES; }

fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *L,
                         void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale,
                         int is_causal, fa_dtype dtype, fa_stream_t stream) {
    size_t need = fa_bwd_workspace_size(B, H, Nq, Nk, d, is_causal, dtype);
    if (need == 0) {
        // unsupported arguments: let fa_bwd name the problem (it launches nothing)
        return fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, nullptr, 0, stream);
    }
    // dQ formed by reduction keeps an fp32 dQ accumulator in the workspace; where that
    // does not fit the array, this call forms dQ by the separate pass, which needs
    // only the two per-row constants
    DqStrategy forced = DqStrategy::kAuto;
    bool x3_off = false;
    if (need > FA_NOALLOC_SCRATCH_BYTES && dtype == FA_DTYPE_F32) {
        // fp32 inputs: the split bf16 copies of the tensor-core path (256 or 512 bytes
        // per row of each of Q, dO, K, V) do not fit; the CUDA-core kernels need only D
        tc_disable_x3(true);
        need = fa_bwd_workspace_size(B, H, Nq, Nk, d, is_causal, dtype);
        tc_disable_x3(false);
        if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
        x3_off = true;
    } else if (need > FA_NOALLOC_SCRATCH_BYTES) {
        tc_override_dq_strategy(DqStrategy::kSeparatePass);
        need = fa_bwd_workspace_size(B, H, Nq, Nk, d, is_causal, dtype);
        tc_override_dq_strategy(DqStrategy::kAuto);
        if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
        forced = DqStrategy::kSeparatePass;
    }
    void *scratch = nullptr;
    fa_status s = scratch_for_current_device(&scratch);
    if (s != FA_OK) return s;
    tc_override_dq_strategy(forced);
    tc_disable_x3(x3_off);
    s = fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, scratch,
               FA_NOALLOC_SCRATCH_BYTES, stream);
    tc_disable_x3(false);
    tc_override_dq_strategy(DqStrategy::kAuto);
    return s;
}

}  // extern "C"
