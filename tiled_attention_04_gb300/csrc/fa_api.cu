// The C ABI (include/fa.h): argument checks, kernel-family choice, launches.
//
// The interface mirrors the autograd Function of CS336 A2 "Systems and
// Parallelism", problem flash_forward: forward(Q, K, V, is_causal) -> O with L
// kept for the backward, and backward -> dQ, dK, dV (problem flash_backward).
// Nothing here computes attention; every step runs in the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

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
    out->B = B;
    out->H = H;
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
    const FaStrides q{(long long)H * Nq * d, (long long)Nq * d, d}, k{(long long)H * Nk * d, (long long)Nk * d, d};
    out->sQ = out->sO = out->sdO = out->sdQ = q;
    out->sK = out->sV = out->sdK = out->sdV = k;
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

// Takes the strides of one (B, H, N, d) view (NULL: keep the contiguous ones
// already in *s).  A dimension of extent 1 keeps its contiguous stride, whatever
// the caller passed: its index is always 0.  The others must be positive
// multiples of 16 bytes below 2^40 bytes (the limits of a TMA descriptor).  An
// output view must not overlap itself.
fa_status take_strides(const fa_strides *in, int B, int H, int N, int d, fa_dtype dt, bool output, FaStrides *s) {
    if (!in) return FA_OK;
    const long long eb = (long long)elem_bytes(dt);
    const long long ext[3] = {B, H, N};
    const long long given[3] = {in->b, in->h, in->n};
    long long *dst[3] = {&s->b, &s->h, &s->n};
    long long span = d - 1;   // largest element index the view reaches
    for (int i = 0; i < 3; ++i) {
        if (ext[i] <= 1) continue;
        const long long v = given[i];
        if (v <= 0 || v >= (1LL << 40) / eb) return FA_ERR_BAD_SHAPE;
        if ((v * eb) % 16 != 0) return FA_ERR_MISALIGNED;
        if (v > ((1LL << 48) / eb) / (ext[i] - 1)) return FA_ERR_BAD_SHAPE;
        span += v * (ext[i] - 1);
        if (span >= (1LL << 48) / eb) return FA_ERR_BAD_SHAPE;
        *dst[i] = v;
    }
    if (output) {
        // sorted by stride, every dimension must step past the whole span of the ones below it
        long long st[4] = {1, 0, 0, 0}, ex[4] = {d, 0, 0, 0};
        int n = 1;
        for (int i = 0; i < 3; ++i)
            if (ext[i] > 1) {
                st[n] = *dst[i];
                ex[n] = ext[i];
                ++n;
            }
        for (int i = 1; i < n; ++i)   // insertion sort of at most four entries
            for (int j = i; j > 0 && st[j] < st[j - 1]; --j) {
                std::swap(st[j], st[j - 1]);
                std::swap(ex[j], ex[j - 1]);
            }
        for (int i = 1; i < n; ++i)
            if (st[i] / ex[i - 1] < st[i - 1]) return FA_ERR_BAD_SHAPE;
    }
    return FA_OK;
}

// Backward workspace.  CUDA-core path: D (BH*Nq fp32) at sd_off.  Tensor-core
// path: -D then -L*log2(e), each BH * padded_rows(Nq) fp32, then (dQ by
// reduction) the fp32 dQ accumulator (see fa_tc_bwd.cu).  fp32 inputs that may
// take the split pairs (for some scale: the preprocessing phase has no scale
// argument) get both layouts: the tensor-core rows, the split bf16 copies of Q,
// dO, K and V (256 or 512 bytes per row each), and the CUDA-core D at sd_off.
struct Workspace {
    bool tc;
    size_t d_off, l_off, dqa_off, total;
    bool red;           // dQ by fp32 reduction into the accumulator at dqa_off
    bool x3;            // this call runs on split bf16 copies at q2_off, do2_off, k2_off, v2_off
    bool x3_possible;   // some scale would (the layout then holds both paths' data)
    size_t q2_off, do2_off, k2_off, v2_off;
    size_t sd_off;      // D of the CUDA-core kernels
};
size_t x3_bytes(const FaProblem &p, int N) { return align_up((size_t)p.BH * N * tc_x3_row_bytes(p), 256); }
Workspace workspace_layout(const FaProblem &p) {
    Workspace w{};
    w.tc = tc_bwd_supported(p);
    w.x3_possible = tc_x3_possible(p);
    w.x3 = w.x3_possible && tc_x3(p);
    const bool tc_rows = w.tc || w.x3_possible;
    const size_t rows = tc_rows ? tc_bwd_ld_rows(p) : (size_t)p.BH * p.Nq;
    const size_t bytes = align_up(rows * sizeof(float), 256);
    const size_t dqa = w.tc ? tc_bwd_dqa_floats(p) * sizeof(float) : 0;
    w.red = dqa > 0;
    w.d_off = 0;
    w.l_off = bytes;
    w.dqa_off = 2 * bytes;
    w.sd_off = 0;
    w.total = tc_rows ? 2 * bytes + align_up(dqa, 256) : bytes;
    if (w.x3_possible) {
        w.q2_off = w.total;
        w.do2_off = w.q2_off + x3_bytes(p, p.Nq);
        w.k2_off = w.do2_off + x3_bytes(p, p.Nq);
        w.v2_off = w.k2_off + x3_bytes(p, p.Nk);
        w.sd_off = w.v2_off + x3_bytes(p, p.Nk);
        w.total = w.sd_off + align_up((size_t)p.BH * p.Nq * sizeof(float), 256);
    }
    if (w.total == 0) w.total = 256;
    return w;
}

// fp32 inputs on the tensor cores: Q, K, V split into the bf16 pair copies at q2, k2, v2
cudaError_t split_qkv(const FaProblem &p, const void *Q, const void *K, const void *V, void *q2, void *k2, void *v2,
                      cudaStream_t st) {
    const void *X[3] = {Q, K, V};
    const FaStrides s[3] = {p.sQ, p.sK, p.sV};
    const int N[3] = {p.Nq, p.Nk, p.Nk};
    void *X2[3] = {q2, k2, v2};
    return tc_split_x3(p, 3, X, s, N, X2, st);
}

// The forward alone has no workspace argument, so fp32 inputs take their split
// copies from a stream-ordered pool of the library's own, one per device, that
// keeps its memory between calls: the first call (or the first larger one)
// allocates, later ones reuse the memory without synchronising anything.
cudaError_t x3_pool(cudaMemPool_t *out) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxDevices] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;   // never hand memory back between calls
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        pools[dev] = pool;
    }
    *out = pools[dev];
    return cudaSuccess;
}

cudaError_t fwd_x3_pooled(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                          cudaStream_t st) {
    const size_t qb = x3_bytes(p, p.Nq), kb = x3_bytes(p, p.Nk);
    cudaMemPool_t pool = nullptr;
    cudaError_t e = x3_pool(&pool);
    if (e != cudaSuccess) return e;
    void *buf = nullptr;
    if ((e = cudaMallocFromPoolAsync(&buf, qb + 2 * kb, pool, st)) != cudaSuccess) return e;
    char *b = static_cast<char *>(buf);
    e = split_qkv(p, Q, K, V, b, b + qb, b + qb + kb, st);
    if (e == cudaSuccess) e = tc_fwd_x3(p, b, b + qb, b + qb + kb, O, L, st);
    const cudaError_t f = cudaFreeAsync(buf, st);   // stream-ordered: after the forward's reads
    return e != cudaSuccess ? e : f;
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


// ---- runners: arguments already checked (shape, strides, pointers, workspace)

cudaStream_t as_stream(fa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

fa_status run_fwd(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                  fa_stream_t stream) {
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    fa_status s = device_ok();
    if (s != FA_OK) return s;
    const cudaStream_t st = as_stream(stream);
    if (tc_x3(p)) return map_cuda(fwd_x3_pooled(p, Q, K, V, O, L, st));
    return map_cuda(tc_fwd_supported(p) ? tc_fwd(p, Q, K, V, O, L, st) : simt_fwd(p, Q, K, V, O, L, st));
}

// scale_known: false for the exported preprocessing phase, whose fp32 inputs may
// go either way afterwards; it then prepares both paths' data
fa_status run_preprocess(const FaProblem &p, const Workspace &w, const void *O, const void *dO, const float *L,
                         void *workspace, fa_stream_t stream, bool scale_known = true) {
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    fa_status s = device_ok();
    if (s != FA_OK) return s;
    char *ws = static_cast<char *>(workspace);
    float *Dv = reinterpret_cast<float *>(ws + w.d_off);
    const cudaStream_t st = as_stream(stream);
    float *dqa = w.red ? reinterpret_cast<float *>(ws + w.dqa_off) : nullptr;
    if (w.x3 || (w.x3_possible && !scale_known)) {
        // the row constants and dO's split copy; without the scale, the CUDA-core
        // kernels' D as well (their own preprocessing: the same bits as fa_bwd's)
        cudaError_t e =
            tc_bwd_preprocess_x3(p, O, dO, L, Dv, reinterpret_cast<float *>(ws + w.l_off), ws + w.do2_off, st);
        if (e == cudaSuccess && !scale_known)
            e = simt_bwd_preprocess(p, O, dO, reinterpret_cast<float *>(ws + w.sd_off), st);
        return map_cuda(e);
    }
    if (!w.tc) return map_cuda(simt_bwd_preprocess(p, O, dO, reinterpret_cast<float *>(ws + w.sd_off), st));
    return map_cuda(tc_bwd_preprocess(p, O, dO, L, Dv, reinterpret_cast<float *>(ws + w.l_off), dqa, st));
}

// fp32 inputs on the tensor cores: Q, K, V split into the workspace, then the gradient
// items on the copies (dO's copy was made by the preprocessing)
fa_status run_grads_x3(const FaProblem &p, const Workspace &w, const void *Q, const void *K, const void *V,
                       void *dQ, void *dK, void *dV, bool do_kv, bool do_q, void *workspace, cudaStream_t st) {
    char *ws = static_cast<char *>(workspace);
    cudaError_t e = split_qkv(p, Q, K, V, ws + w.q2_off, ws + w.k2_off, ws + w.v2_off, st);
    if (e == cudaSuccess)
        e = tc_bwd_grads_x3(p, ws + w.q2_off, ws + w.k2_off, ws + w.v2_off, ws + w.do2_off,
                            reinterpret_cast<const float *>(ws + w.l_off), reinterpret_cast<const float *>(ws + w.d_off),
                            dQ, dK, dV, do_kv, do_q, st);
    return map_cuda(e);
}

fa_status run_dkdv(const FaProblem &p, const Workspace &w, const void *Q, const void *K, const void *V,
                   const void *dO, const float *L, void *dK, void *dV, void *workspace, fa_stream_t stream) {
    if ((long long)p.BH * p.Nk == 0) return FA_OK;
    fa_status s = device_ok();
    if (s != FA_OK) return s;
    const cudaStream_t st = as_stream(stream);
    if (p.Nq == 0) {   // no query sees any key: the gradients are zero
        cudaError_t e = simt_zero_rows(p, dK, p.sdK, p.Nk, st);
        if (e == cudaSuccess) e = simt_zero_rows(p, dV, p.sdV, p.Nk, st);
        return map_cuda(e);
    }
    if (w.x3) return run_grads_x3(p, w, Q, K, V, nullptr, dK, dV, true, false, workspace, st);
    char *ws = static_cast<char *>(workspace);
    const float *Dv = reinterpret_cast<const float *>(ws + w.d_off);
    return map_cuda(w.tc ? tc_bwd_dkdv(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off), Dv, dK, dV, st)
                         : simt_bwd_dkdv(p, Q, K, V, dO, L, reinterpret_cast<const float *>(ws + w.sd_off), dK, dV,
                                         st));
}

fa_status run_dq(const FaProblem &p, const Workspace &w, const void *Q, const void *K, const void *V,
                 const void *dO, const float *L, void *dQ, void *workspace, fa_stream_t stream) {
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    fa_status s = device_ok();
    if (s != FA_OK) return s;
    char *ws = static_cast<char *>(workspace);
    const float *Dv = reinterpret_cast<const float *>(ws + w.d_off);
    const cudaStream_t st = as_stream(stream);
    if (w.x3) return run_grads_x3(p, w, Q, K, V, dQ, nullptr, nullptr, false, true, workspace, st);
    return map_cuda(w.tc ? tc_bwd_dq(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off), Dv, dQ, st)
                         : simt_bwd_dq(p, Q, K, V, dO, L, reinterpret_cast<const float *>(ws + w.sd_off), dQ, st));
}

fa_status run_grads(const FaProblem &p, const Workspace &w, const void *Q, const void *K, const void *V,
                    const void *dO, const float *L, void *dQ, void *dK, void *dV, void *workspace,
                    fa_stream_t stream) {
    const bool any_q = (long long)p.BH * p.Nq > 0;
    if (!w.tc || !any_q) {   // CUDA-core kernels, or no queries (then dK = dV = 0)
        fa_status s = run_dkdv(p, w, Q, K, V, dO, L, dK, dV, workspace, stream);
        if (s != FA_OK) return s;
        return run_dq(p, w, Q, K, V, dO, L, dQ, workspace, stream);
    }
    fa_status s = device_ok();
    if (s != FA_OK) return s;
    if (w.x3) return run_grads_x3(p, w, Q, K, V, dQ, dK, dV, true, true, workspace, as_stream(stream));
    char *ws = static_cast<char *>(workspace);
    float *dqa = w.red ? reinterpret_cast<float *>(ws + w.dqa_off) : nullptr;
    return map_cuda(tc_bwd_grads(p, Q, K, V, dO, reinterpret_cast<const float *>(ws + w.l_off),
                                 reinterpret_cast<const float *>(ws + w.d_off), dqa, dQ, dK, dV, as_stream(stream)));
}

// pointer checks of a whole backward pass (fa_bwd, fa_bwd_strided)
fa_status bwd_ptrs(const FaProblem &p, const void *Q, const void *K, const void *V, const void *O, const void *dO,
                   const float *L, const void *dQ, const void *dK, const void *dV) {
    fa_status s = FA_OK;
    if ((long long)p.BH * p.Nq > 0 && (s = check_ptrs({Q, K, V, O, dO, L, dQ})) != FA_OK) return s;
    if ((long long)p.BH * p.Nk > 0 && (s = check_ptrs({dK, dV})) != FA_OK) return s;
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
        case FA_ERR_BOUNDS: return "debug build: a kernel bounds check failed";
    }
    return "unknown status";
}

void fa_set_wait_limit(uint32_t spins) { g_wait_limit.store(spins, std::memory_order_relaxed); }

void fa_debug_force_stall(int on) { g_force_stall.store(on ? 1u : 0u, std::memory_order_relaxed); }

const char *fa_path_name(int Nq, int Nk, int d, int is_causal, fa_dtype dtype) {
    FaProblem p{};
    if (check_common(1, 1, Nq, Nk, d, is_causal, dtype, 1.f, false, &p) != FA_OK) return nullptr;
    p.scale = 1.f / sqrtf((float)d);   // the default scale
    return tc_fwd_supported(p) ? "tc" : "simt";
}

int fa_set_fp32_mode(int mode) {
    if (mode < FA_FP32_AUTO || mode > FA_FP32_SPLIT) return -1;
    const int prev = tc_get_fp32_mode();
    tc_set_fp32_mode(mode);
    return prev;
}

int fa_set_dq_strategy(int strategy) {
    if (strategy < FA_DQ_AUTO || strategy > FA_DQ_REDUCTION) return -1;
    const int prev = static_cast<int>(tc_get_dq_setting());
    tc_set_dq_strategy(static_cast<DqStrategy>(strategy));
    return prev;
}

int fa_bwd_dq_strategy(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype) {
    FaProblem p{};
    if (check_common(B, H, Nq, Nk, d, is_causal, dtype, 1.f, false, &p) != FA_OK) return -1;
    return tc_bwd_dq_by_reduction(p) ? FA_DQ_REDUCTION : FA_DQ_SEPARATE_PASS;
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H, int Nq, int Nk,
                 int d, float scale, int is_causal, fa_dtype dtype, fa_stream_t stream) {
    return fa_fwd_strided(Q, nullptr, K, nullptr, V, nullptr, O, nullptr, L, B, H, Nq, Nk, d, scale, is_causal, dtype,
                          stream);
}

fa_status fa_fwd_strided(const void *Q, const fa_strides *sQ, const void *K, const fa_strides *sK, const void *V,
                         const fa_strides *sV, void *O, const fa_strides *sO, float *L, int B, int H, int Nq, int Nk,
                         int d, float scale, int is_causal, fa_dtype dtype, fa_stream_t stream) {
    FaProblem p{};
    fa_status s = check_common(B, H, Nq, Nk, d, is_causal, dtype, scale, true, &p);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0) return FA_OK;
    if ((s = take_strides(sQ, B, H, Nq, d, dtype, false, &p.sQ)) != FA_OK ||
        (s = take_strides(sK, B, H, Nk, d, dtype, false, &p.sK)) != FA_OK ||
        (s = take_strides(sV, B, H, Nk, d, dtype, false, &p.sV)) != FA_OK ||
        (s = take_strides(sO, B, H, Nq, d, dtype, true, &p.sO)) != FA_OK)
        return s;
    if ((s = check_ptrs({Q, K, V, O, L})) != FA_OK) return s;
    return run_fwd(p, Q, K, V, O, L, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype) {
    FaProblem p{};
    if (check_common(B, H, Nq, Nk, d, is_causal, dtype, 1.f, false, &p) != FA_OK) return 0;
    return workspace_layout(p).total;   // (the layout does not depend on the scale)
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
    return run_preprocess(p, w, O, dO, L, workspace, stream, false);
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
    if ((s = check_ptrs({dK, dV})) != FA_OK) return s;
    if (p.Nq > 0 && (s = check_ptrs({Q, K, V, dO, L, dQ})) != FA_OK) return s;
    return run_dkdv(p, w, Q, K, V, dO, L, dK, dV, workspace, stream);
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
    return run_dq(p, w, Q, K, V, dO, L, dQ, workspace, stream);
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
    return run_grads(p, w, Q, K, V, dO, L, dQ, dK, dV, workspace, stream);
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *L,
                 void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                 fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    return fa_bwd_strided(Q, nullptr, K, nullptr, V, nullptr, O, nullptr, dO, nullptr, L, dQ, nullptr, dK, nullptr,
                          dV, nullptr, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_strided(const void *Q, const fa_strides *sQ, const void *K, const fa_strides *sK, const void *V,
                         const fa_strides *sV, const void *O, const fa_strides *sO, const void *dO,
                         const fa_strides *sdO, const float *L, void *dQ, const fa_strides *sdQ, void *dK,
                         const fa_strides *sdK, void *dV, const fa_strides *sdV, int B, int H, int Nq, int Nk, int d,
                         float scale, int is_causal, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                         fa_stream_t stream) {
    // validate everything up front so that a bad argument launches nothing at all
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                           workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0 && (long long)p.BH * p.Nk == 0) return FA_OK;
    if ((s = take_strides(sQ, B, H, Nq, d, dtype, false, &p.sQ)) != FA_OK ||
        (s = take_strides(sK, B, H, Nk, d, dtype, false, &p.sK)) != FA_OK ||
        (s = take_strides(sV, B, H, Nk, d, dtype, false, &p.sV)) != FA_OK ||
        (s = take_strides(sO, B, H, Nq, d, dtype, false, &p.sO)) != FA_OK ||
        (s = take_strides(sdO, B, H, Nq, d, dtype, false, &p.sdO)) != FA_OK ||
        (s = take_strides(sdQ, B, H, Nq, d, dtype, true, &p.sdQ)) != FA_OK ||
        (s = take_strides(sdK, B, H, Nk, d, dtype, true, &p.sdK)) != FA_OK ||
        (s = take_strides(sdV, B, H, Nk, d, dtype, true, &p.sdV)) != FA_OK)
        return s;
    if ((s = bwd_ptrs(p, Q, K, V, O, dO, L, dQ, dK, dV)) != FA_OK) return s;
    if ((s = run_preprocess(p, w, O, dO, L, workspace, stream)) != FA_OK) return s;
    return run_grads(p, w, Q, K, V, dO, L, dQ, dK, dV, workspace, stream);
}

fa_status fa_fwd_bwd(const void *Q, const void *K, const void *V, const void *dO, void *O, float *L, void *dQ,
                     void *dK, void *dV, int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                     fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    // both passes' arguments first, so that a bad one launches nothing at all
    FaProblem p{};
    Workspace w{};
    fa_status s = bwd_args(Q, K, V, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, is_causal, dtype, workspace,
                           workspace_bytes, &p, &w, false);
    if (s != FA_OK) return s;
    if ((long long)p.BH * p.Nq == 0 && (long long)p.BH * p.Nk == 0) return FA_OK;
    if ((s = bwd_ptrs(p, Q, K, V, O, dO, L, dQ, dK, dV)) != FA_OK) return s;
    if (w.x3) {
        // fp32 on the tensor cores: Q, K, V split once into the workspace serve both passes
        if ((s = device_ok()) != FA_OK) return s;
        const cudaStream_t st = as_stream(stream);
        char *ws = static_cast<char *>(workspace);
        float *Dv = reinterpret_cast<float *>(ws + w.d_off), *Lv = reinterpret_cast<float *>(ws + w.l_off);
        cudaError_t e = split_qkv(p, Q, K, V, ws + w.q2_off, ws + w.k2_off, ws + w.v2_off, st);
        if (e == cudaSuccess) e = tc_fwd_x3(p, ws + w.q2_off, ws + w.k2_off, ws + w.v2_off, O, L, st);
        if (e == cudaSuccess) e = tc_bwd_preprocess_x3(p, O, dO, L, Dv, Lv, ws + w.do2_off, st);
        if (e == cudaSuccess)
            e = tc_bwd_grads_x3(p, ws + w.q2_off, ws + w.k2_off, ws + w.v2_off, ws + w.do2_off, Lv, Dv, dQ, dK, dV,
                                true, true, st);
        return map_cuda(e);
    }
    bool prep_done = false;
    if (w.tc && (long long)p.BH * p.Nq > 0) {
        // tensor-core path: the forward's epilogue also forms D = rowsum(dO * O) from
        // the unrounded O and stages the backward's row constants (no preprocessing kernel)
        if ((s = device_ok()) != FA_OK) return s;
        char *ws = static_cast<char *>(workspace);
        FwdPrep prep{};
        prep.dO = dO;
        prep.sdo = p.sdO;
        prep.Dp = reinterpret_cast<float *>(ws + w.d_off);
        prep.Lp = reinterpret_cast<float *>(ws + w.l_off);
        prep.dQa = w.red ? reinterpret_cast<float *>(ws + w.dqa_off) : nullptr;
        if ((s = map_cuda(tc_fwd(p, Q, K, V, O, L, as_stream(stream), &prep, &prep_done))) != FA_OK) return s;
    } else if ((s = run_fwd(p, Q, K, V, O, L, stream)) != FA_OK) {
        return s;
    }
    if (!prep_done && (s = run_preprocess(p, w, O, dO, L, workspace, stream)) != FA_OK) return s;
    return run_grads(p, w, Q, K, V, dO, L, dQ, dK, dV, workspace, stream);
}

fa_status fa_get_device_status(fa_stream_t stream) {
    if (device_ok() != FA_OK) return FA_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return FA_ERR_LAUNCH;
    unsigned a = 0, b = 0;
    if (tc_fwd_read_status(&a, st) != cudaSuccess || tc_bwd_read_status(&b, st) != cudaSuccess) return FA_ERR_LAUNCH;
    if ((a | b) & 0x100u) return FA_ERR_BOUNDS;   // a failed check also ends the kernel's waits
    return (a | b) ? FA_ERR_TIMEOUT : FA_OK;
}

int fa_debug_build(void) {
#ifdef FA_DEBUG
    return 1;
#else
    return 0;
#endif
}

fa_status fa_debug_tile_rows(unsigned long long *out, int n, fa_stream_t stream) {
    if (!out || n < 0) return FA_ERR_BAD_ARG;
    if (device_ok() != FA_OK) return FA_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long v[3] = {0, 0, 0};
    if (tc_fwd_read_rows(&v[0], st) != cudaSuccess || tc_bwd_read_rows(&v[1], st) != cudaSuccess) return FA_ERR_LAUNCH;
    for (int i = 0; i < n && i < 3; ++i) out[i] = v[i];
    return FA_OK;
}

fa_status fa_debug_reset_tile_rows(fa_stream_t stream) {
    if (device_ok() != FA_OK) return FA_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = tc_fwd_reset_rows(st);
    if (e == cudaSuccess) e = tc_bwd_reset_rows(st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return map_cuda(e);
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
