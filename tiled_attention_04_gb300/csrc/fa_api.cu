// The C ABI (include/fa.h): argument checks, kernel-family choice, launches.
//
// The interface mirrors the autograd Function of CS336 A2 "Systems and
// Parallelism", problem flash_forward: forward(Q, K, V, is_causal) -> O with L
// kept for the backward, and backward -> dQ, dK, dV (problem flash_backward).
// Nothing here computes attention; every step runs in the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "fa.h"
#include "fa_internal.h"

namespace {

std::atomic<uint32_t> g_wait_limit{0};
std::atomic<uint32_t> g_force_stall{0};
constexpr uint32_t kDefaultWaitLimit = 1u << 26;   // polls; far above any legitimate wait

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

fa_status check_common(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype, float scale,
                       bool check_scale, FaProblem *out) {
    if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED_DTYPE;
    if (d != 16 && d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED_HEAD_DIM;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_BAD_SHAPE;
    const long long BH = (long long)B * H;
    if (BH > INT32_MAX) return FA_ERR_BAD_SHAPE;
    if (BH > 0 && Nq > 0 && Nk == 0) return FA_ERR_BAD_SHAPE;   // softmax over no keys
    if (BH * (long long)(Nq > Nk ? Nq : Nk) > INT32_MAX) return FA_ERR_BAD_SHAPE;
    if (is_causal != 0 && is_causal != 1) return FA_ERR_BAD_ARG;
    if (check_scale && !isfinite(scale)) return FA_ERR_BAD_ARG;
    out->BH = (int)BH;
    out->Nq = Nq;
    out->Nk = Nk;
    out->d = d;
    out->scale = scale;
    out->causal = is_causal;
    out->dtype = dtype;
    const uint32_t w = g_wait_limit.load(std::memory_order_relaxed);
    out->wait_limit = w ? w : kDefaultWaitLimit;
    out->force_stall = g_force_stall.load(std::memory_order_relaxed);
    return FA_OK;
}

fa_status check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (!p) return FA_ERR_NULL_PTR;
    for (const void *p : ptrs)
        if (!aligned16(p)) return FA_ERR_MISALIGNED;
    return FA_OK;
}

fa_status map_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FA_OK;
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return FA_ERR_NO_DEVICE;
    return FA_ERR_LAUNCH;
}

fa_status device_ok() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    return FA_OK;
}

size_t elem_bytes(fa_dtype t) { return t == FA_DTYPE_F32 ? 4 : 2; }

// Backward workspace.  CUDA-core path: D (BH*Nq fp32).  Tensor-core path:
// D then L*log2(e), each BH * padded_rows(Nq) fp32 (see fa_tc_bwd.cu).
struct Workspace {
    bool tc;
    size_t d_off, l_off, total;
};
Workspace workspace_layout(const FaProblem &p) {
    Workspace w{};
    w.tc = tc_bwd_supported(p);
    const size_t rows = w.tc ? tc_bwd_ld_rows(p) : (size_t)p.BH * p.Nq;
    const size_t bytes = align_up(rows * sizeof(float), 256);
    w.d_off = 0;
    w.l_off = bytes;
    w.total = w.tc ? 2 * bytes : bytes;
    if (w.total == 0) w.total = 256;
    return w;
}

fa_status bwd_args(const void *Q, const void *K, const void *V, const void *dO, const float *L, const void *dQ,
                   const void *dK, const void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                   fa_dtype dtype, void *workspace, size_t workspace_bytes, FaProblem *p, Workspace *w,
                   bool need_q_side) {
    fa_status s = check_common(B, H, Nq, Nk, d, is_causal, dtype, scale, true, p);
    if (s != FA_OK) return s;
    if (need_q_side) {
        if ((s = check_ptrs({Q, K, V, dO, L, dQ, dK, dV})) != FA_OK) return s;
    }
    if (!workspace) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_MISALIGNED;
    *w = workspace_layout(*p);
    if (workspace_bytes < w->total) return FA_ERR_WORKSPACE;
    return FA_OK;
}

}  // namespace

extern "C" {

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_NULL_PTR: return "null pointer";
        case FA_ERR_BAD_SHAPE: return "bad shape";
        case FA_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dim (need 16, 32, 64 or 128)";
        case FA_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case FA_ERR_WORKSPACE: return "workspace missing or too small";
        case FA_ERR_LAUNCH: return "CUDA launch error";
        case FA_ERR_TIMEOUT: return "device-side wait timed out";
        case FA_ERR_NO_DEVICE: return "no CUDA device";
        case FA_ERR_BAD_ARG: return "bad argument";
    }
    return "unknown status";
}

void fa_set_wait_limit(uint32_t spins) { g_wait_limit.store(spins, std::memory_order_relaxed); }

void fa_debug_force_stall(int on) { g_force_stall.store(on ? 1u : 0u, std::memory_order_relaxed); }

const char *fa_path_name(int Nq, int Nk, int d, int is_causal, fa_dtype dtype) {
    FaProblem p{};
    if (check_common(1, 1, Nq, Nk, d, is_causal, dtype, 1.f, false, &p) != FA_OK) return nullptr;
    return tc_fwd_supported(p) ? "tc" : "simt";
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H, int Nq, int Nk,
                 int d, float scale, int is_causal, fa_dtype dtype, fa_stream_t stream) {
    FaProblem p{};
    fa_status s = check_common(B, H, Nq, Nk, d, is_causal, dtype, scale, true, &p);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    if ((s = check_ptrs({Q, K, V, O, L})) != FA_OK) return s;
    if ((s = device_ok()) != FA_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = tc_fwd_supported(p) ? tc_fwd(p, Q, K, V, O, L, st) : simt_fwd(p, Q, K, V, O, L, st);
    return map_cuda(e);
}

size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype) {
    FaProblem p{};
    if (check_common(B, H, Nq, Nk, d, is_causal, dtype, 1.f, false, &p) != FA_OK) return 0;
    return workspace_layout(p).total;
}

fa_status fa_bwd_preprocess(const void *O, const void *dO, const float *L, int B, int H, int Nq, int Nk, int d,
                            int is_causal, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                            fa_stream_t stream) {
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(nullptr, nullptr, nullptr, dO, nullptr, nullptr, nullptr, nullptr, B, H, Nq, Nk, d, 1.f,
                           is_causal, dtype, workspace, workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    if ((s = check_ptrs({O, dO, L})) != FA_OK) return s;
    if ((s = device_ok()) != FA_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    float *Dv = reinterpret_cast<float *>(ws + w.d_off);
    cudaError_t e = w.tc ? tc_bwd_preprocess(p, O, dO, L, Dv, reinterpret_cast<float *>(ws + w.l_off), st)
                         : simt_bwd_preprocess(p, O, dO, Dv, st);
    return map_cuda(e);
}

fa_status fa_bwd_dkdv(const void *Q, const void *K, const void *V, const void *dO, const float *L, void *dQ,
                      void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                      fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                           workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nk == 0) return FA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = check_ptrs({dK, dV})) != FA_OK) return s;
    if ((s = device_ok()) != FA_OK) return s;
    if (p.Nq == 0) {   // no query sees any key: the gradients are zero
        const size_t bytes = (size_t)p.BH * p.Nk * p.d * elem_bytes(dtype);
        cudaError_t e = cudaMemsetAsync(dK, 0, bytes, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dV, 0, bytes, st);
        return map_cuda(e);
    }
    if ((s = check_ptrs({Q, K, V, dO, L, dQ})) != FA_OK) return s;
    char *ws = static_cast<char *>(workspace);
    const float *Dv = reinterpret_cast<const float *>(ws + w.d_off);
    cudaError_t e = w.tc ? tc_bwd_dkdv(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off), Dv, dK, dV, st)
                         : simt_bwd_dkdv(p, Q, K, V, dO, L, Dv, dK, dV, st);
    return map_cuda(e);
}

fa_status fa_bwd_dq(const void *Q, const void *K, const void *V, const void *dO, const float *L, void *dQ, int B,
                    int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype, void *workspace,
                    size_t workspace_bytes, fa_stream_t stream) {
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, nullptr, nullptr, B, H, Nq, Nk, d, scale, is_causal, dtype,
                           workspace, workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    if ((s = check_ptrs({Q, K, V, dO, L, dQ})) != FA_OK) return s;
    if ((s = device_ok()) != FA_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const float *Dv = reinterpret_cast<const float *>(ws + w.d_off);
    cudaError_t e = w.tc ? tc_bwd_dq(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off), Dv, dQ, st)
                         : simt_bwd_dq(p, Q, K, V, dO, L, Dv, dQ, st);
    return map_cuda(e);
}

fa_status fa_bwd_grads(const void *Q, const void *K, const void *V, const void *dO, const float *L, void *dQ,
                       void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                       fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                           workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    const bool any_q = (long long)p.BH * p.Nq > 0, any_k = (long long)p.BH * p.Nk > 0;
    if (!any_q && !any_k) return FA_OK;
    if (any_q && (s = check_ptrs({Q, K, V, dO, L, dQ})) != FA_OK) return s;
    if (any_k && (s = check_ptrs({dK, dV})) != FA_OK) return s;
    if (!w.tc || !any_q) {   // CUDA-core kernels, or no queries (then dK = dV = 0)
        if ((s = fa_bwd_dkdv(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                             workspace_bytes, stream)) != FA_OK)
            return s;
        return fa_bwd_dq(Q, K, V, dO, L, dQ, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace, workspace_bytes,
                         stream);
    }
    if ((s = device_ok()) != FA_OK) return s;
    char *ws = static_cast<char *>(workspace);
    return map_cuda(tc_bwd_grads(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off),
                                 reinterpret_cast<const float *>(ws + w.d_off), dQ, dK, dV, true, true,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *L,
                 void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                 fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    // validate everything up front so that a bad argument launches nothing at all
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                           workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    const bool any_q = (long long)p.BH * p.Nq > 0, any_k = (long long)p.BH * p.Nk > 0;
    if (!any_q && !any_k) return FA_OK;
    if (any_q && (s = check_ptrs({Q, K, V, O, dO, L, dQ})) != FA_OK) return s;
    if (any_k && (s = check_ptrs({dK, dV})) != FA_OK) return s;
    if ((s = fa_bwd_preprocess(O, dO, L, B, H, Nq, Nk, d, is_causal, dtype, workspace, workspace_bytes, stream)) !=
        FA_OK)
        return s;
    return fa_bwd_grads(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                        workspace_bytes, stream);
}

fa_status fa_get_device_status(fa_stream_t stream) {
    if (device_ok() != FA_OK) return FA_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return FA_ERR_LAUNCH;
    unsigned a = 0, b = 0;
    if (tc_fwd_read_status(&a, st) != cudaSuccess || tc_bwd_read_status(&b, st) != cudaSuccess) return FA_ERR_LAUNCH;
    return (a | b) ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status fa_reset_device_status(fa_stream_t stream) {
    if (device_ok() != FA_OK) return FA_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = tc_fwd_reset_status(st);
    if (e == cudaSuccess) e = tc_bwd_reset_status(st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return map_cuda(e);
}

}  // extern "C"
