// Internal interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa.h"

// Element strides of a (B, H, N, d) tensor s: element (b, h, n, c) is at index
// b*s.b + h*s.h + n*s.n + c (the head dimension is contiguous).
struct FaStrides {
    long long b, h, n;
};

// index of the first element of row n of batch*head bh = b*H + h
__host__ __device__ __forceinline__ long long fa_row_offset(const FaStrides &s, int H, int bh, int n) {
    const int b = bh / H;
    return (long long)b * s.b + (long long)(bh - b * H) * s.h + (long long)n * s.n;
}

struct FaProblem {
    int B, H;        // batch, heads
    int BH;          // batch * heads
    int Nq, Nk;      // query / key sequence lengths
    int d;           // head dimension
    float scale;     // softmax scale (usually 1/sqrt(d))
    int causal;      // top-left causal mask
    fa_dtype dtype;  // element type of Q, K, V, O, dO, dQ, dK, dV
    uint32_t wait_limit;  // cap on device-side polling loops
    uint32_t force_stall; // fault injection: the forward's MMA issuer waits on a barrier nobody arrives on
    // strides of every (B, H, N, d) tensor (contiguous unless a *_strided entry point set them)
    FaStrides sQ, sK, sV, sO, sdO, sdQ, sdK, sdV;
};

// ---- fp32 CUDA-core kernels (fa_simt.cu): every dtype and head dim.
cudaError_t simt_fwd(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                     cudaStream_t st);
cudaError_t simt_bwd_preprocess(const FaProblem &p, const void *O, const void *dO, float *Dvec,
                                cudaStream_t st);
cudaError_t simt_bwd_dkdv(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                          const float *L, const float *Dvec, void *dK, void *dV, cudaStream_t st);
cudaError_t simt_bwd_dq(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                        const float *L, const float *Dvec, void *dQ, cudaStream_t st);
// writes zeros to the N rows of every batch*head of the (B, H, N, d) view X with strides s
cudaError_t simt_zero_rows(const FaProblem &p, void *X, const FaStrides &s, int N, cudaStream_t st);

// (B, H, N, d) bf16 tensor with strides s -> 4-D TMA map over (d, N, H, B), boxes of
// 64 columns x box_rows rows, 128-byte swizzle; a load of batch*head bh uses
// coordinates (column, row, bh % H, bh / H)
struct CUtensorMap_st;
bool tc_make_map_4d(CUtensorMap_st *m, const void *ptr, int B, int H, int N, int d, const FaStrides &s,
                    int box_rows);
// (B*H, N, d) contiguous bf16 tensor -> 3-D TMA map over (d, N, B*H), same boxes
bool tc_make_map_3d(CUtensorMap_st *m, const void *ptr, int BH, int N, int d, int box_rows);
// (BH, rows, cols) contiguous fp32 accumulator -> 3-D TMA map over (cols, rows, BH), boxes of
// 32 columns x 128 rows, 128-byte swizzle (the target of the dQ reductions)
bool tc_make_map_acc(CUtensorMap_st *m, const void *ptr, int BH, int rows, int cols);
// true when s is the contiguous layout of a (B, H, N, d) tensor (dimensions of extent 1 aside)
bool tc_plain_layout(const FaProblem &p, const FaStrides &s, int N);
// the 4-D map (view4) or the 3-D map of one tensor of the problem
bool tc_make_map(CUtensorMap_st *m, const void *ptr, const FaProblem &p, const FaStrides &s, int N, int box_rows,
                 bool view4);

// host-side launch helpers (fa_tc_fwd.cu): the dynamic shared-memory attribute set
// once per kernel and device, and the multiprocessor count cached per device
cudaError_t tc_set_smem_once(const void *kernel, int bytes);
int tc_sm_count();

// ---- tcgen05 tensor-core kernels (fa_tc_fwd.cu, fa_tc_bwd.cu): bf16, d in {16, 32, 64, 128}
// (16 and 32 run the d = 64 kernels with zero-filled columns), and fp32 with d <= 64 (X3 below).
bool tc_fwd_supported(const FaProblem &p);
bool tc_bwd_supported(const FaProblem &p);
// The backward's preprocessing done by the forward's epilogue when dO is known
// up front (the fused forward + backward call): D = rowsum(dO * O) from the
// unrounded fp32 O, and -D, -L*log2(e) written to the tensor-core backward's
// workspace rows (padding rows 0 and -inf), the dQ accumulator rows cleared.
struct FwdPrep {
    const void *dO;   // NULL: no preprocessing
    FaStrides sdo;
    float *Dp, *Lp;   // per batch*head, padded_rows(Nq) rows
    float *dQa;       // NULL unless dQ is formed by reduction
};
// ---- fp32 inputs (X3): each operand is first split into a bf16 pair (hi = bf16(x),
// lo = bf16(x - hi)) held as a contiguous (B*H, N, 2W) bf16 copy, hi in columns
// [0, W) and lo in [W, 2W), W = 64 for d <= 64 (the d = 128 kernels) and 128 for
// d = 128 (256-column kernels: one K / V slot in the forward, 32-row sub-tiles in
// the backward); every contraction takes three products (hi hi + hi lo + lo hi).
bool tc_x3(const FaProblem &p);            // this problem runs X3 (mode, shape and scale)
bool tc_x3_possible(const FaProblem &p);   // X3 for some scale (mode and shape): workspace sizing
void tc_disable_x3(bool off);   // for the calling thread's calls (off: fp32 on the CUDA cores)
void tc_set_fp32_mode(int mode);          // FA_FP32_AUTO / _EXACT / _SPLIT
int tc_get_fp32_mode();
size_t tc_x3_row_bytes(const FaProblem &p);   // bytes of one split row: 256 or 512
// count (1..4) tensors X[i] with strides s[i] and N[i] rows per batch*head -> X2[i]
cudaError_t tc_split_x3(const FaProblem &p, int count, const void *const *X, const FaStrides *s, const int *N,
                        void *const *X2, cudaStream_t st);
// forward on split copies; O (fp32) is written through p.sO
cudaError_t tc_fwd_x3(const FaProblem &p, const void *Q2, const void *K2, const void *V2, void *O, float *L,
                      cudaStream_t st);
// backward on split copies: -D, -L*log2(e) rows as tc_bwd_preprocess (from fp32 O and
// dO through p.sO, p.sdO) plus dO's split copy; then the gradient items (dQ by the
// separate pass), dQ, dK, dV written in fp32 through their strides
cudaError_t tc_bwd_preprocess_x3(const FaProblem &p, const void *O, const void *dO, const float *L, float *Dp,
                                 float *Lp, void *dO2, cudaStream_t st);
cudaError_t tc_bwd_grads_x3(const FaProblem &p, const void *Q2, const void *K2, const void *V2, const void *dO2,
                            const float *Lp, const float *Dp, void *dQ, void *dK, void *dV, bool do_kv, bool do_q,
                            cudaStream_t st);
// Forward.  With prep (dO not NULL) the forward's epilogue also does the
// backward's preprocessing (*prep_done tells whether it did).
cudaError_t tc_fwd(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                   cudaStream_t st, const FwdPrep *prep = nullptr, bool *prep_done = nullptr);
// backward workspace on this path: per batch*head, padded_rows(Nq) fp32 D then the same
// of L*log2(e); when dQ is formed by reduction, then an fp32 dQ accumulator of
// padded_rows(Nq) x max(d, 64) per batch*head
size_t tc_bwd_ld_rows(const FaProblem &p);
// dQ strategy: a separate pass over query tiles (recomputing S and dP), or fp32
// reduction by the dK/dV items (no recomputation) followed by a conversion kernel
enum class DqStrategy { kAuto = 0, kSeparatePass = 1, kReduction = 2 };
void tc_set_dq_strategy(DqStrategy s);
DqStrategy tc_get_dq_strategy();
// the strategy for the calling thread's calls until reset with kAuto (overrides the setting)
void tc_override_dq_strategy(DqStrategy s);
DqStrategy tc_get_dq_setting();   // the process-wide setting alone
bool tc_bwd_dq_by_reduction(const FaProblem &p);
size_t tc_bwd_dqa_floats(const FaProblem &p);   // 0 unless tc_bwd_dq_by_reduction(p)
// D, L staged (and the dQ accumulator, when dQa is not NULL, cleared)
cudaError_t tc_bwd_preprocess(const FaProblem &p, const void *O, const void *dO, const float *L, float *Dp,
                              float *Lp, float *dQa, cudaStream_t st);
cudaError_t tc_bwd_dkdv(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                        const float *Lp, const float *Dp, void *dK, void *dV, cudaStream_t st);
cudaError_t tc_bwd_dq(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                      const float *Lp, const float *Dp, void *dQ, cudaStream_t st);
// dK, dV and dQ: one launch of both kinds of work item (dQa NULL), or the dK/dV
// items adding dQ into dQa (cleared by the preprocess) plus the conversion kernel
cudaError_t tc_bwd_grads(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                         const float *Lp, const float *Dp, float *dQa, void *dQ, void *dK, void *dV,
                         cudaStream_t st);

// device-side status words of the tensor-core translation units
cudaError_t tc_fwd_read_status(unsigned *out, cudaStream_t st);
cudaError_t tc_bwd_read_status(unsigned *out, cudaStream_t st);
cudaError_t tc_fwd_reset_status(cudaStream_t st);
cudaError_t tc_bwd_reset_status(cudaStream_t st);
// debug build: tile rows loaded (forward: key rows; backward: query rows of the
// dK/dV items, key rows of the dQ items), read (synchronising) and reset
cudaError_t tc_fwd_read_rows(unsigned long long *out, cudaStream_t st);
cudaError_t tc_fwd_reset_rows(cudaStream_t st);
cudaError_t tc_bwd_read_rows(unsigned long long *out, cudaStream_t st);
cudaError_t tc_bwd_reset_rows(cudaStream_t st);
