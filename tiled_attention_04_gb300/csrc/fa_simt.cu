// fp32 CUDA-core FlashAttention-2 kernels: the exact-precision path for fp32
// inputs, and the path for shapes the tensor-core kernels do not take.
//
// Method (CS336 A2 field guide "Systems and Parallelism", §1.2-1.3):
//   forward, problem flash_forward: one program per (query tile, batch*head),
//   a single loop over key tiles with a running max m and running sum l;
//   the accumulator is rescaled by exp(m_prev - m_new) and divided by l once
//   at the end; L = m + ln(l) is written per row.  Causal: key tiles that lie
//   wholly above the diagonal are never visited (§1.3.3's early exit), the
//   rest compare query and key indices.
//   backward, problem flash_backward: P = exp(S - L) recomputed, D from a
//   separate preprocess, and the five matrix expressions split into a dK/dV
//   pass (one program per key tile, looping over query tiles) and a dQ pass
//   (one program per query tile, looping over key tiles), so no atomics are
//   needed (§1.3.3, "split the backward pass into two passes").
//
// Everything is computed in fp32 on CUDA cores (no TF32), so fp32 inputs keep
// fp32 accuracy.  Tiles are 64 x 64, 256 threads arranged 16 x 16; a thread
// owns a 4 x 4 block of the score tile (rows ty*4.., columns tx + 16*j) and
// a 4 x d/16 block of the output.  Exponentials are taken base 2 on scores
// pre-multiplied by scale*log2(e).
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "fa_internal.h"

namespace {

constexpr int SB = 64;    // tile edge (queries and keys)
constexpr int NT = 256;   // threads per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Heads per batch and the element strides of every (B, H, N, d) tensor.
struct Views {
    int H;
    FaStrides q, k, v, o, dO, dq, dk, dv;
};

Views views_of(const FaProblem &p) { return Views{p.H, p.sQ, p.sK, p.sV, p.sO, p.sdO, p.sdQ, p.sdK, p.sdV}; }

// rows [row0, row0+SB) of an (N, D) matrix with row stride rs into smem [SB][D+1] fp32, zero past N
template <typename T, int D>
__device__ __forceinline__ void load_tile(float *s, const T *g, long long rs, int row0, int N) {
    for (int idx = threadIdx.x; idx < SB * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        const int gr = row0 + r;
        s[r * (D + 1) + c] = gr < N ? to_f(g[(long long)gr * rs + c]) : 0.f;
    }
}

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
constexpr size_t fwd_smem() { return (size_t)(3 * SB * (D + 1) + SB * (SB + 1)) * sizeof(float); }
template <int D>
constexpr size_t bwd_smem() { return (size_t)(4 * SB * (D + 1) + SB * (SB + 1) + 2 * SB) * sizeof(float); }

// ------------------------------------------------------------------ forward
template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(NT) simt_fwd_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                      const T *__restrict__ V, T *__restrict__ O,
                                                      float *__restrict__ L, int Nq, int Nk, float scale_log2,
                                                      Views vw) {
    extern __shared__ float sm[];
    float *Qs = sm, *Ks = Qs + SB * (D + 1), *Vs = Ks + SB * (D + 1), *Ps = Vs + SB * (D + 1);
    constexpr int OC = D / 16;
    const int bh = blockIdx.y, q0 = blockIdx.x * SB;
    const T *Qg = Q + fa_row_offset(vw.q, vw.H, bh, 0);
    const T *Kg = K + fa_row_offset(vw.k, vw.H, bh, 0);
    const T *Vg = V + fa_row_offset(vw.v, vw.H, bh, 0);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    float o[4][OC], m[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < OC; ++c) o[i][c] = 0.f;
    }
    load_tile<T, D>(Qs, Qg, vw.q.n, q0, Nq);
    const int kend = CAUSAL ? min(Nk, q0 + SB) : Nk;   // keys beyond the tile's last query are never visible
    for (int k0 = 0; k0 < kend; k0 += SB) {
        __syncthreads();
        load_tile<T, D>(Ks, Kg, vw.k.n, k0, Nk);
        load_tile<T, D>(Vs, Vg, vw.v.n, k0, Nk);
        __syncthreads();
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
            float qv[4], kv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] = Qs[(ty * 4 + i) * (D + 1) + k];
#pragma unroll
            for (int j = 0; j < 4; ++j) kv[j] = Ks[(tx + 16 * j) * (D + 1) + k];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
        }
        const bool diag = CAUSAL && (k0 + SB - 1 > q0);   // only these tiles need index compares
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int qi = q0 + ty * 4 + i;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kj = k0 + tx + 16 * j;
                float v = s[i][j] * scale_log2;
                if (kj >= Nk || (diag && kj > qi)) v = -INFINITY;
                s[i][j] = v;
                mx = fmaxf(mx, v);
            }
            mx = half_warp_max(mx);
            const float mnew = fmaxf(m[i], mx);     // finite: key 0 is visible to every row
            const float alpha = exp2f(m[i] - mnew);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = exp2f(s[i][j] - mnew);
                s[i][j] = pj;
                rs += pj;
            }
            rs = half_warp_sum(rs);
            l[i] = l[i] * alpha + rs;
            m[i] = mnew;
#pragma unroll
            for (int c = 0; c < OC; ++c) o[i][c] *= alpha;
#pragma unroll
            for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * (SB + 1) + tx + 16 * j] = s[i][j];
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < SB; ++k) {
            float pv[4], vv[OC];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = Ps[(ty * 4 + i) * (SB + 1) + k];
#pragma unroll
            for (int c = 0; c < OC; ++c) vv[c] = Vs[k * (D + 1) + tx + 16 * c];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < OC; ++c) o[i][c] = fmaf(pv[i], vv[c], o[i][c]);
        }
    }
    T *Og = O + fa_row_offset(vw.o, vw.H, bh, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int qi = q0 + ty * 4 + i;
        if (qi < Nq) {
            const float inv = 1.f / l[i];
#pragma unroll
            for (int c = 0; c < OC; ++c) Og[(long long)qi * vw.o.n + tx + 16 * c] = from_f<T>(o[i][c] * inv);
            if (tx == 0) L[(size_t)bh * Nq + qi] = m[i] * kLn2 + logf(l[i]);
        }
    }
}

// ------------------------------------------------------------------ D = rowsum(dO * O)
template <typename T>
__global__ void __launch_bounds__(NT) simt_preprocess_kernel(const T *__restrict__ O, const T *__restrict__ dO,
                                                             float *__restrict__ Dvec, long long rows, int D,
                                                             int Nq, Views vw) {
    const long long row = (long long)blockIdx.x * (NT / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int bh = (int)(row / Nq), q = (int)(row % Nq);
    const T *o = O + fa_row_offset(vw.o, vw.H, bh, q), *g = dO + fa_row_offset(vw.dO, vw.H, bh, q);
    float acc = 0.f;
    for (int c = lane; c < D; c += 32) acc = fmaf(to_f(o[c]), to_f(g[c]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) Dvec[row] = acc;
}

// ------------------------------------------------------------------ dK, dV
template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(NT) simt_dkdv_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                       const T *__restrict__ V, const T *__restrict__ dO,
                                                       const float *__restrict__ L, const float *__restrict__ Dvec,
                                                       T *__restrict__ dK, T *__restrict__ dV, int Nq, int Nk,
                                                       float scale, float scale_log2, Views vw) {
    extern __shared__ float sm[];
    float *Ks = sm, *Vs = Ks + SB * (D + 1), *Qs = Vs + SB * (D + 1), *dOs = Qs + SB * (D + 1);
    float *Ps = dOs + SB * (D + 1), *Ls = Ps + SB * (SB + 1), *Ds = Ls + SB;
    constexpr int OC = D / 16;
    const int bh = blockIdx.y, k0 = blockIdx.x * SB;
    const T *Qg = Q + fa_row_offset(vw.q, vw.H, bh, 0), *dOg = dO + fa_row_offset(vw.dO, vw.H, bh, 0);
    const T *Kg = K + fa_row_offset(vw.k, vw.H, bh, 0), *Vg = V + fa_row_offset(vw.v, vw.H, bh, 0);
    const float *Lg = L + (size_t)bh * Nq, *Dg = Dvec + (size_t)bh * Nq;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    float dk[4][OC], dv[4][OC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < OC; ++c) dk[i][c] = dv[i][c] = 0.f;
    load_tile<T, D>(Ks, Kg, vw.k.n, k0, Nk);
    load_tile<T, D>(Vs, Vg, vw.v.n, k0, Nk);
    const int qstart = CAUSAL ? k0 : 0;   // queries before this key tile never see it
    for (int q0 = qstart; q0 < Nq; q0 += SB) {
        __syncthreads();
        load_tile<T, D>(Qs, Qg, vw.q.n, q0, Nq);
        load_tile<T, D>(dOs, dOg, vw.dO.n, q0, Nq);
        if (tid < SB) {
            const int qi = q0 + tid;
            Ls[tid] = qi < Nq ? Lg[qi] * kLog2e : INFINITY;   // padding rows get P = 0
            Ds[tid] = qi < Nq ? Dg[qi] : 0.f;
        }
        __syncthreads();
        float p[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) p[i][j] = dp[i][j] = 0.f;
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            float kv[4], vv[4], qv[4], gv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                kv[i] = Ks[(ty * 4 + i) * (D + 1) + k];
                vv[i] = Vs[(ty * 4 + i) * (D + 1) + k];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                qv[j] = Qs[(tx + 16 * j) * (D + 1) + k];
                gv[j] = dOs[(tx + 16 * j) * (D + 1) + k];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    p[i][j] = fmaf(kv[i], qv[j], p[i][j]);
                    dp[i][j] = fmaf(vv[i], gv[j], dp[i][j]);
                }
        }
        const bool diag = CAUSAL && (k0 + SB - 1 > q0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kj = k0 + ty * 4 + i, qi = q0 + tx + 16 * j;
                const float e = exp2f(p[i][j] * scale_log2 - Ls[tx + 16 * j]);
                p[i][j] = (diag && kj > qi) ? 0.f : e;
                Ps[(ty * 4 + i) * (SB + 1) + tx + 16 * j] = p[i][j];
            }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < SB; ++c) {       // dV += P^T dO
            float pv[4], gv[OC];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = Ps[(ty * 4 + i) * (SB + 1) + c];
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) gv[cc] = dOs[c * (D + 1) + tx + 16 * cc];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int cc = 0; cc < OC; ++cc) dv[i][cc] = fmaf(pv[i], gv[cc], dv[i][cc]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                Ps[(ty * 4 + i) * (SB + 1) + tx + 16 * j] = p[i][j] * (dp[i][j] - Ds[tx + 16 * j]);
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < SB; ++c) {       // dK += dS^T Q
            float sv[4], qv[OC];
#pragma unroll
            for (int i = 0; i < 4; ++i) sv[i] = Ps[(ty * 4 + i) * (SB + 1) + c];
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) qv[cc] = Qs[c * (D + 1) + tx + 16 * cc];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int cc = 0; cc < OC; ++cc) dk[i][cc] = fmaf(sv[i], qv[cc], dk[i][cc]);
        }
    }
    T *dKg = dK + fa_row_offset(vw.dk, vw.H, bh, 0), *dVg = dV + fa_row_offset(vw.dv, vw.H, bh, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int kj = k0 + ty * 4 + i;
        if (kj < Nk) {
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) {
                dKg[(long long)kj * vw.dk.n + tx + 16 * cc] = from_f<T>(dk[i][cc] * scale);
                dVg[(long long)kj * vw.dv.n + tx + 16 * cc] = from_f<T>(dv[i][cc]);
            }
        }
    }
}

// ------------------------------------------------------------------ dQ
template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(NT) simt_dq_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                     const T *__restrict__ V, const T *__restrict__ dO,
                                                     const float *__restrict__ L, const float *__restrict__ Dvec,
                                                     T *__restrict__ dQ, int Nq, int Nk, float scale,
                                                     float scale_log2, Views vw) {
    extern __shared__ float sm[];
    float *Qs = sm, *dOs = Qs + SB * (D + 1), *Ks = dOs + SB * (D + 1), *Vs = Ks + SB * (D + 1);
    float *Ps = Vs + SB * (D + 1);
    constexpr int OC = D / 16;
    const int bh = blockIdx.y, q0 = blockIdx.x * SB;
    const T *Qg = Q + fa_row_offset(vw.q, vw.H, bh, 0), *dOg = dO + fa_row_offset(vw.dO, vw.H, bh, 0);
    const T *Kg = K + fa_row_offset(vw.k, vw.H, bh, 0), *Vg = V + fa_row_offset(vw.v, vw.H, bh, 0);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    float dq[4][OC], lrow[4], drow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int qi = q0 + ty * 4 + i;
        lrow[i] = qi < Nq ? L[(size_t)bh * Nq + qi] * kLog2e : 0.f;
        drow[i] = qi < Nq ? Dvec[(size_t)bh * Nq + qi] : 0.f;
#pragma unroll
        for (int c = 0; c < OC; ++c) dq[i][c] = 0.f;
    }
    load_tile<T, D>(Qs, Qg, vw.q.n, q0, Nq);
    load_tile<T, D>(dOs, dOg, vw.dO.n, q0, Nq);
    const int kend = CAUSAL ? min(Nk, q0 + SB) : Nk;
    for (int k0 = 0; k0 < kend; k0 += SB) {
        __syncthreads();
        load_tile<T, D>(Ks, Kg, vw.k.n, k0, Nk);
        load_tile<T, D>(Vs, Vg, vw.v.n, k0, Nk);
        __syncthreads();
        float s[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = dp[i][j] = 0.f;
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            float qv[4], gv[4], kv[4], vv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qv[i] = Qs[(ty * 4 + i) * (D + 1) + k];
                gv[i] = dOs[(ty * 4 + i) * (D + 1) + k];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kv[j] = Ks[(tx + 16 * j) * (D + 1) + k];
                vv[j] = Vs[(tx + 16 * j) * (D + 1) + k];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
                    dp[i][j] = fmaf(gv[i], vv[j], dp[i][j]);
                }
        }
        const bool diag = CAUSAL && (k0 + SB - 1 > q0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int qi = q0 + ty * 4 + i, kj = k0 + tx + 16 * j;
                const bool masked = kj >= Nk || (diag && kj > qi);
                const float pij = masked ? 0.f : exp2f(s[i][j] * scale_log2 - lrow[i]);
                Ps[(ty * 4 + i) * (SB + 1) + tx + 16 * j] = pij * (dp[i][j] - drow[i]);
            }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < SB; ++c) {       // dQ += dS K
            float sv[4], kv[OC];
#pragma unroll
            for (int i = 0; i < 4; ++i) sv[i] = Ps[(ty * 4 + i) * (SB + 1) + c];
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) kv[cc] = Ks[c * (D + 1) + tx + 16 * cc];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int cc = 0; cc < OC; ++cc) dq[i][cc] = fmaf(sv[i], kv[cc], dq[i][cc]);
        }
    }
    T *dQg = dQ + fa_row_offset(vw.dq, vw.H, bh, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int qi = q0 + ty * 4 + i;
        if (qi < Nq) {
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) dQg[(long long)qi * vw.dq.n + tx + 16 * cc] = from_f<T>(dq[i][cc] * scale);
        }
    }
}

// ------------------------------------------------------------------ zero rows of a strided view
template <typename T>
__global__ void __launch_bounds__(NT) simt_zero_kernel(T *__restrict__ X, FaStrides s, int H, int N, int D,
                                                       long long total) {
    for (long long i = (long long)blockIdx.x * NT + threadIdx.x; i < total; i += (long long)gridDim.x * NT) {
        const long long row = i / D;
        X[fa_row_offset(s, H, (int)(row / N), (int)(row % N)) + i % D] = from_f<T>(0.f);
    }
}

// ------------------------------------------------------------------ dispatch helpers
template <typename F>
cudaError_t launch(F kernel, dim3 grid, size_t smem, cudaStream_t st, auto... args) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, NT, smem, st>>>(args...);
    return cudaGetLastError();
}

template <typename T, int D, bool C>
cudaError_t fwd_t(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                  cudaStream_t st) {
    dim3 grid((p.Nq + SB - 1) / SB, p.BH);
    return launch(simt_fwd_kernel<T, D, C>, grid, fwd_smem<D>(), st, (const T *)Q, (const T *)K, (const T *)V,
                  (T *)O, L, p.Nq, p.Nk, p.scale * kLog2e, views_of(p));
}
template <typename T, int D, bool C>
cudaError_t dkdv_t(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                   const float *L, const float *Dv, void *dK, void *dV, cudaStream_t st) {
    dim3 grid((p.Nk + SB - 1) / SB, p.BH);
    return launch(simt_dkdv_kernel<T, D, C>, grid, bwd_smem<D>(), st, (const T *)Q, (const T *)K, (const T *)V,
                  (const T *)dO, L, Dv, (T *)dK, (T *)dV, p.Nq, p.Nk, p.scale, p.scale * kLog2e, views_of(p));
}
template <typename T, int D, bool C>
cudaError_t dq_t(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO, const float *L,
                 const float *Dv, void *dQ, cudaStream_t st) {
    dim3 grid((p.Nq + SB - 1) / SB, p.BH);
    return launch(simt_dq_kernel<T, D, C>, grid, bwd_smem<D>(), st, (const T *)Q, (const T *)K, (const T *)V,
                  (const T *)dO, L, Dv, (T *)dQ, p.Nq, p.Nk, p.scale, p.scale * kLog2e, views_of(p));
}

// expands FN<T, D, C>(args) over dtype x head dim x causal
#define FA_SIMT_DISPATCH(FN, ...)                                                                    \
    do {                                                                                             \
        const bool c_ = p.causal != 0;                                                               \
        if (p.dtype == FA_DTYPE_F32) {                                                               \
            switch (p.d) {                                                                           \
                case 16: return c_ ? FN<float, 16, true>(__VA_ARGS__) : FN<float, 16, false>(__VA_ARGS__);   \
                case 32: return c_ ? FN<float, 32, true>(__VA_ARGS__) : FN<float, 32, false>(__VA_ARGS__);   \
                case 64: return c_ ? FN<float, 64, true>(__VA_ARGS__) : FN<float, 64, false>(__VA_ARGS__);   \
                case 128: return c_ ? FN<float, 128, true>(__VA_ARGS__) : FN<float, 128, false>(__VA_ARGS__); \
            }                                                                                        \
        } else {                                                                                     \
            using B_ = __nv_bfloat16;                                                                \
            switch (p.d) {                                                                           \
                case 16: return c_ ? FN<B_, 16, true>(__VA_ARGS__) : FN<B_, 16, false>(__VA_ARGS__);         \
                case 32: return c_ ? FN<B_, 32, true>(__VA_ARGS__) : FN<B_, 32, false>(__VA_ARGS__);         \
                case 64: return c_ ? FN<B_, 64, true>(__VA_ARGS__) : FN<B_, 64, false>(__VA_ARGS__);         \
                case 128: return c_ ? FN<B_, 128, true>(__VA_ARGS__) : FN<B_, 128, false>(__VA_ARGS__);      \
            }                                                                                        \
        }                                                                                            \
        return cudaErrorInvalidValue;                                                                \
    } while (0)

}  // namespace

cudaError_t simt_fwd(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                     cudaStream_t st) {
    FA_SIMT_DISPATCH(fwd_t, p, Q, K, V, O, L, st);
}

cudaError_t simt_bwd_preprocess(const FaProblem &p, const void *O, const void *dO, float *Dvec, cudaStream_t st) {
    const long long rows = (long long)p.BH * p.Nq;
    if (rows == 0) return cudaSuccess;
    dim3 grid((unsigned)((rows + NT / 32 - 1) / (NT / 32)));
    if (p.dtype == FA_DTYPE_F32)
        simt_preprocess_kernel<float><<<grid, NT, 0, st>>>((const float *)O, (const float *)dO, Dvec, rows, p.d,
                                                           p.Nq, views_of(p));
    else
        simt_preprocess_kernel<__nv_bfloat16><<<grid, NT, 0, st>>>((const __nv_bfloat16 *)O,
                                                                  (const __nv_bfloat16 *)dO, Dvec, rows, p.d,
                                                                  p.Nq, views_of(p));
    return cudaGetLastError();
}

cudaError_t simt_zero_rows(const FaProblem &p, void *X, const FaStrides &s, int N, cudaStream_t st) {
    const long long total = (long long)p.BH * N * p.d;
    if (total == 0) return cudaSuccess;
    const unsigned grid = (unsigned)std::min<long long>((total + NT - 1) / NT, 4096);
    if (p.dtype == FA_DTYPE_F32)
        simt_zero_kernel<float><<<grid, NT, 0, st>>>((float *)X, s, p.H, N, p.d, total);
    else
        simt_zero_kernel<__nv_bfloat16><<<grid, NT, 0, st>>>((__nv_bfloat16 *)X, s, p.H, N, p.d, total);
    return cudaGetLastError();
}

cudaError_t simt_bwd_dkdv(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                          const float *L, const float *Dvec, void *dK, void *dV, cudaStream_t st) {
    FA_SIMT_DISPATCH(dkdv_t, p, Q, K, V, dO, L, Dvec, dK, dV, st);
}

cudaError_t simt_bwd_dq(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                        const float *L, const float *Dvec, void *dQ, cudaStream_t st) {
    FA_SIMT_DISPATCH(dq_t, p, Q, K, V, dO, L, Dvec, dQ, st);
}
