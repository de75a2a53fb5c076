// FlashAttention-2 backward on sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Method (CS336 A2 field guide "Systems and Parallelism", problem
// flash_backward and §1.3.3): P = exp(S - L) is rebuilt from Q, K and the
// saved logsumexp L; D = rowsum(dO * O) comes from a preprocess pass;
// dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = scale dS K,
// dK = scale dS^T Q.  The work is split into two passes so that no program
// ever adds into another's output (§1.3.3, "split the backward pass into two
// passes, one for dQ and one for dK and dV"):
//
//   preprocess   -D and -L*log2(e), padded per batch*head to a multiple of
//                128 rows (padding rows get -L = -inf, so their P is exactly
//                zero), in the caller's workspace;
//   dK/dV items  one per 128-key tile, looping over query sub-tiles:
//                S^T = K Q^T and dP^T = V dO^T recomputed in TMEM, P^T and
//                dS^T (bf16) written back into TMEM, then dV += P^T dO and
//                dK += dS^T Q with A read from TMEM;
//   dQ items     one per 128-query tile, looping over key sub-tiles:
//                S = Q K^T and dP = dO V^T recomputed, dS into TMEM,
//                dQ += dS K.
// Both kinds of item run in one launch (fa_bwd_tc_kernel), interleaved
// longest first; an item whose loop would dominate the run is split over a
// two-CTA cluster and the two partial accumulators are added through
// distributed shared memory.
//
// Warp roles as in the forward: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 4-7 and 8-11 two element-wise warpgroups.  Sub-tiles:
//   d = 64   128 wide (MMA N = 128 for S and dP, which run at full rate);
//            both warpgroups work on every sub-tile, each on 64 of its
//            columns, and P^T / dS^T have TMEM columns of their own so the
//            next sub-tile's S and dP are computed under the element-wise work;
//   d = 128  64 wide, the warpgroups taking alternate sub-tiles with their
//            own double-buffered S / dP columns (TMEM has no room for
//            separate P^T / dS^T next to dK and dV at this head dimension).
// The accumulators (dK and dV, or dQ) are shared: every MMA is issued by one
// thread, in order, so the two warpgroups' contributions simply add up.
// Causal: sub-tiles wholly on the masked side of the diagonal are skipped.
// Layouts as in the forward (template argument VIEW4): contiguous tensors load
// through 3-D maps and store gradient rows at (bh*N + row)*d; strided views,
// and head dims 16 and 32 on the d = 64 items, load through 4-D (d, N, H, B)
// maps and store through the gradients' own strides, skipping the zero
// columns past d.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "fa_internal.h"
#include "tc_common.cuh"

__device__ unsigned g_fa_bwd_status;
// debug build: query rows the dK/dV items loaded, key rows the dQ items loaded
__device__ unsigned long long g_fa_bwd_rows[2];

namespace {

constexpr int NTHREADS = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;

// rows of the L/D workspace per batch*head: a multiple of 128
__host__ __device__ inline int padded_rows(int n) { return (n + 127) / 128 * 128; }

// ------------------------------------------------------------------ preprocess
// d/8 threads per query row (each reads 16 bytes of O and of dO, so a row is
// one contiguous, coalesced segment), rows reduced with shuffles.  Writes the
// negated row constants the passes add: Dn = -rowsum(dO * O), Ln = -L*log2(e);
// padding rows: Dn = 0, Ln = -inf (so their P = 2^(-inf) = 0).  A block takes
// 256/(d/8) consecutive rows of one batch*head (the padded row count is a
// multiple of 128, so no block straddles two), which leaves one 32-bit
// division per thread to find them.  When dQ is formed by reduction (dQa not
// NULL), the row's fp32 accumulator (max(D, 64) columns) is cleared here too.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ O,
                                                         const __nv_bfloat16 *__restrict__ dO,
                                                         const float *__restrict__ L, float *__restrict__ Dp,
                                                         float *__restrict__ Lp, float *__restrict__ dQa, int Nq,
                                                         int H, FaStrides so, FaStrides sdo) {
    constexpr int TPR = D / 8;          // threads per row
    constexpr int RPB = 256 / TPR;      // rows per block
    static_assert(128 % RPB == 0, "a block stays within one batch*head");
    tc::pdl_launch_dependents();
    tc::pdl_wait();   // O (from the forward) and dO are complete
    const int nqp = padded_rows(Nq);
    const int bpb = nqp / RPB;                                  // blocks per batch*head
    const int bh = (int)blockIdx.x / bpb;
    const int q = ((int)blockIdx.x - bh * bpb) * RPB + (int)threadIdx.x / TPR;
    const int sub = threadIdx.x % TPR;
    const long long gr = (long long)bh * nqp + q;
    // every load goes out before anything waits on one: the row's L with O and dO,
    // so the kernel pays one memory latency, not two
    const float lrow = (sub == 0 && q < Nq) ? __ldg(L + (long long)bh * Nq + q) : 0.f;
    uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
    if (q < Nq) {
        a = __ldg(reinterpret_cast<const uint4 *>(O + fa_row_offset(so, H, bh, q) + sub * 8));
        b = __ldg(reinterpret_cast<const uint4 *>(dO + fa_row_offset(sdo, H, bh, q) + sub * 8));
    }
    if (dQa) {
        constexpr int DK = D < 64 ? 64 : D;   // accumulator columns (head dims below 64 ride the d = 64 items)
        float4 *row = reinterpret_cast<float4 *>(dQa + gr * DK);
#pragma unroll
        for (int i = sub; i < DK / 4; i += TPR) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.f;
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(pa[i]), fb = __bfloat1622float2(pb[i]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (sub == 0) {
        if (q < Nq) {
            Dp[gr] = -acc;
            Lp[gr] = -lrow * kLog2e;
        } else {
            Dp[gr] = 0.f;
            Lp[gr] = -INFINITY;
        }
    }
}

// fp32 inputs (X3): the same row constants from fp32 O and dO, and dO split into
// its bf16 pair row [hi | lo] of 2W columns (W = 64 for d <= 64, 128 for d = 128;
// zeros past d) for the gradient launch.  W/4 threads per row, four columns each.
template <int W>
__global__ void __launch_bounds__(256) fa_bwd_pre_x3_kernel(const float *__restrict__ O, const float *__restrict__ dO,
                                                            const float *__restrict__ L, float *__restrict__ Dp,
                                                            float *__restrict__ Lp, __nv_bfloat16 *__restrict__ dO2,
                                                            int Nq, int H, int d, FaStrides so, FaStrides sdo) {
    constexpr int TPR = W / 4, RPB = 256 / TPR;   // threads per row, rows per block (divides 128)
    tc::pdl_launch_dependents();
    tc::pdl_wait();   // O (from the forward) and dO are complete
    const int nqp = padded_rows(Nq);
    const long long gr = (long long)blockIdx.x * RPB + threadIdx.x / TPR;   // padded row
    const int bh = (int)(gr / nqp), q = (int)(gr - (long long)bh * nqp);
    const int cg = threadIdx.x % TPR;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (q < Nq && 4 * cg < d) {
        a = __ldg(reinterpret_cast<const float4 *>(O + fa_row_offset(so, H, bh, q) + 4 * cg));
        b = __ldg(reinterpret_cast<const float4 *>(dO + fa_row_offset(sdo, H, bh, q) + 4 * cg));
    }
    const float lrow = (cg == 0 && q < Nq) ? __ldg(L + (long long)bh * Nq + q) : 0.f;
    float acc = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (q < Nq) {
        const uint32_t h0 = tc::pack_bf16(b.x, b.y), h1 = tc::pack_bf16(b.z, b.w);
        uint2 *dst = reinterpret_cast<uint2 *>(dO2 + ((long long)bh * Nq + q) * (2 * W));
        dst[cg] = make_uint2(h0, h1);
        dst[TPR + cg] = make_uint2(tc::pack_bf16_residual(b.x, b.y, h0), tc::pack_bf16_residual(b.z, b.w, h1));
    }
    if (cg == 0) {
        Dp[gr] = q < Nq ? -acc : 0.f;
        Lp[gr] = q < Nq ? -lrow * kLog2e : -INFINITY;
    }
}

// ------------------------------------------------------------------ dQ from its fp32 accumulator
// dQ = scale * dQa, rounded to bf16: 8 columns per thread (two 16-byte loads,
// one 16-byte store), grid-stride over the BH * Nq rows' d / 8 column groups.
template <int DK, bool VIEW4>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float *__restrict__ dQa,
                                                                __nv_bfloat16 *__restrict__ dQ, int Nq, int H,
                                                                int dv, float scale, FaStrides sdq,
                                                                long long groups) {
    tc::pdl_launch_dependents();
    tc::pdl_wait();   // every reduction into dQa has completed
    const int gpr = dv / 8;                      // column groups per row
    const int nqp = padded_rows(Nq);
    for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
         g += (long long)gridDim.x * blockDim.x) {
        const long long row = g / gpr;           // bh * Nq + q
        const int c = (int)(g - row * gpr) * 8;
        const int bh = (int)(row / Nq);
        const int q = (int)(row - (long long)bh * Nq);
        const float4 *src = reinterpret_cast<const float4 *>(dQa + ((long long)bh * nqp + q) * DK + c);
        const float4 a = src[0], b = src[1];
        uint4 o;
        o.x = tc::pack_bf16(a.x * scale, a.y * scale);
        o.y = tc::pack_bf16(a.z * scale, a.w * scale);
        o.z = tc::pack_bf16(b.x * scale, b.y * scale);
        o.w = tc::pack_bf16(b.z * scale, b.w * scale);
        __nv_bfloat16 *dst;
        if constexpr (VIEW4) dst = dQ + fa_row_offset(sdq, H, bh, q) + c;
        else dst = dQ + row * dv + c;
        *reinterpret_cast<uint4 *>(dst) = o;
    }
}

// ------------------------------------------------------------------ shared layout helpers
// A "tile" here is R rows x d bf16 held as d/64 chunks of [R rows x 128 B], 128-byte swizzled.
template <int R, int D>
struct TileShape {
    static constexpr uint32_t CHUNK = R * 128u;
    static constexpr uint32_t BYTES = (D / 64) * CHUNK;
};

// K-major descriptor for k-step kk (16 elements of d) of a tile with rows `R`
template <int R>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return tc::sdesc_sw128(tile + (kk >> 2) * (R * 128u) + (kk & 3) * 32u, 16, 1024);
}
// MN-major descriptor: the tile's rows are the MMA's K dimension; k-step kk covers rows 16kk..16kk+15
template <int R>
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return tc::sdesc_sw128(tile + kk * 16u * 128u, R * 128u, 1024);
}

// ================================================================== wide sub-tiles (d = 64)
// ------------------------------------------------------------------ dK / dV (wide)
// One CTA per 128-key tile (MMA M = 128 keys), looping over 128-query
// sub-tiles (MMA N = 128 for S^T and dP^T, which run at full rate; K = 128 for
// dV and dK).  Both element-wise warpgroups work on every sub-tile, warpgroup t
// on query columns [64t, 64t + 64).
template <int D, bool RED = false>
struct DkdvWideCfg {
    static constexpr int BK = 128;                 // keys per CTA (MMA M)
    static constexpr int BQ = 128;                 // queries per sub-tile
    // d = 64 leaves TMEM for P^T and dS^T of their own, so S^T and dP^T of the
    // next sub-tile are computed while the element-wise warps work on this one;
    // d = 128 writes P^T and dS^T over S^T and dP^T.
    static constexpr bool SEP = D == 64;
    static constexpr int STAGES = D == 128 ? 2 : 3;
    using KT = TileShape<BK, D>;
    using QT = TileShape<BQ, D>;
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + KT::BYTES;
    static constexpr uint32_t Q_OFF = V_OFF + KT::BYTES;                 // stages of Q sub-tiles
    static constexpr uint32_t DO_OFF = Q_OFF + STAGES * QT::BYTES;       // stages of dO sub-tiles
    static constexpr uint32_t LD_OFF = DO_OFF + STAGES * QT::BYTES;      // stages of 128 -L*log2e + 128 -D floats
    // RED (dQ added into an fp32 accumulator in global memory): dS^T of the current
    // sub-tile in shared memory (bf16, [128 keys x 128 B] per 64 queries, swizzled),
    // read by two MMAs -- as dS^T (K-major A of dK) and as dS (MN-major A of dQ) --
    // and the dQ partial of a sub-tile staged as fp32 [128 rows x 32 columns] boxes
    // for the TMA reduction.  Measured alternatives at batch 8, N = 4096 (gradient
    // launch 54.9 us as built): a second staging buffer, which costs a stage of the
    // Q / dO ring, 60.9 us; the two idle warps issuing red.global.add.v4.f32 from
    // the staged rows instead of the TMA reduction, 58.2 us.
    static constexpr uint32_t DS_OFF = LD_OFF + STAGES * 1024;
    static constexpr uint32_t DQS_OFF = DS_OFF + (RED ? 2 * 128 * 128 : 0);
    static constexpr uint32_t DQS_BOX = 128 * 128;                       // bytes of one staged box
    static constexpr uint32_t BAR_OFF = DQS_OFF + (RED ? (D / 32) * DQS_BOX : 0);
    // kv_full, q_full[S], q_empty[S], sd_full, sd_free, p_full, drain (+ dq_staged,
    // dq_free, and ep_staged[2]: a warpgroup's dV or dK rows are staged for their TMA store)
    static constexpr int NBAR = 1 + 2 * STAGES + 4 + (RED ? 4 : 0);
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t PEER_BAR_OFF = MISC_OFF + 16;
    static constexpr uint32_t SMEM_BYTES = (PEER_BAR_OFF + 16 + 1024 > 120u * 1024u ? PEER_BAR_OFF + 16 + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(DS_OFF % 1024 == 0 && DQS_OFF % 1024 == 0, "swizzled tiles sit on 1024-byte boundaries");
    // split items: rank 1's partial dV (rows 0..127) and dK (rows 128..255), fp32, over the tile rings
    static constexpr uint32_t PART_STRIDE = (D + 4) * 4;
    static constexpr uint32_t PART_OFF = 0;
    static_assert(PART_OFF + 256 * PART_STRIDE <= DS_OFF, "partial fits the rings");
    // TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D);
    // P^T and dS^T (bf16, 64 columns each) at [384,448) and [448,512), or over S^T / dP^T.
    // RED: dS^T lives in shared memory and the sub-tile's dQ partial (fp32) takes [448,512).
    static constexpr uint32_t ST_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D;
    static constexpr uint32_t PT_COL = SEP ? 384 : 0, DS_COL = SEP ? 448 : 128;
    static constexpr uint32_t DQ_COL = 448;
    static_assert(!RED || (D == 64 && SEP), "the dQ reduction form exists for the d = 64 wide items");
};

// one dK/dV work item: key tile kt of batch*head bh (a half of its queries when SPLIT = 2).
// RED: the item also forms each sub-tile's dQ partial, dS K, and adds it into the
// fp32 accumulator behind tmdQa (a TMA reduction issued by warp 2), so that no
// separate dQ pass recomputes S and dP.
template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool RED>
__device__ __forceinline__ void dkdv_item_wide(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                          const CUtensorMap &tmdO, const CUtensorMap *tmdQa,
                                          const CUtensorMap *tmdK, const CUtensorMap *tmdV,
                                          const float *__restrict__ Lp,
                                          const float *__restrict__ Dp, __nv_bfloat16 *__restrict__ dK,
                                          __nv_bfloat16 *__restrict__ dV, int Nq, int Nk, int kt, int bh, int H,
                                          int dv, const FaStrides &sdk, const FaStrides &sdv, float scale,
                                          float scale_log2, uint32_t wait_limit) {
    using C = DkdvWideCfg<D, RED>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t rank = SPLIT > 1 ? tc::cluster_rank() : 0u;
    const int k0 = kt * C::BK;
    const int nqp = padded_rows(Nq);
    const int i_end = (Nq + C::BQ - 1) / C::BQ;
    const int i_first = CAUSAL ? kt : 0;                      // first query sub-tile that sees a key of this tile
    const int n_all = i_end > i_first ? i_end - i_first : 0;
    // this CTA's query sub-tiles: all of them, or one half of a split item
    const int n_half = SPLIT > 1 ? (n_all + 1) / 2 : n_all;
    const int i_begin = i_first + (rank == 0 ? 0 : n_half);
    const int n = rank == 0 ? n_half : n_all - n_half;        // sub-tiles to visit

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t kv_full = bar(0);
    auto q_full = [&](int s) { return bar(1 + s); };
    auto q_empty = [&](int s) { return bar(1 + C::STAGES + s); };   // sub-tile's dV/dK MMAs done
    const uint32_t sd_full = bar(1 + 2 * C::STAGES);
    const uint32_t sd_free = bar(2 + 2 * C::STAGES);
    const uint32_t p_full = bar(3 + 2 * C::STAGES);
    const uint32_t drain = bar(4 + 2 * C::STAGES);
    const uint32_t dq_staged = bar(5 + 2 * C::STAGES);   // RED: the element-wise threads staged a dQ partial
    const uint32_t dq_free = bar(6 + 2 * C::STAGES);     // RED: the reduction has read the staged partial
    // RED, unsplit: a warpgroup's dV (t = 0) or dK (t = 1) rows are staged for their TMA store
    auto ep_staged = [&](int t) { return bar(7 + 2 * C::STAGES + t); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(kv_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(q_full(s), 1);
            tc::mbar_init(q_empty(s), 1);
        }
        tc::mbar_init(sd_full, 1);
        tc::mbar_init(sd_free, 256);
        tc::mbar_init(p_full, 256);
        tc::mbar_init(drain, 1);
        if constexpr (RED) {
            tc::mbar_init(dq_staged, 256);
            tc::mbar_init(dq_free, 1);
            tc::mbar_init(ep_staged(0), 128);
            tc::mbar_init(ep_staged(1), 128);
        }
        if (SPLIT > 1) {
            tc::mbar_init(base + C::PEER_BAR_OFF, 256);       // peer_free: the peer's 256 element-wise threads
            tc::mbar_init(base + C::PEER_BAR_OFF + 8, 128);   // peer_ready: the peer's 128 senders
        }
        *abort_flag = 0u;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (SPLIT > 1) tc::cluster_sync_all();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const tc::Waiter W{abort_flag, &g_fa_bwd_status, wait_limit, 2u};

    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            tc::tma_prefetch_desc(&tmQ);
            tc::tma_prefetch_desc(&tmdO);
            const bool kv_ok = tc::in_bounds(k0 < Nk, &g_fa_bwd_status, abort_flag);
            if (kv_ok) {
                tc::mbar_arrive_expect_tx(kv_full, 2 * C::KT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::K_OFF + c * C::KT::CHUNK, &tmK, kv_full, c * 64, k0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::V_OFF + c * C::KT::CHUNK, &tmV, kv_full, c * 64, k0, bh, H);
                }
            }
            int issued = 0;
            for (int it = 0; kv_ok && it < n; ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1;
                if (!W.wait(q_empty(s), ph ^ 1u)) break;
                const int q0 = (i_begin + it) * C::BQ;
                // debug build: a query sub-tile past the queries, or wholly on the
                // masked side of the diagonal, is never loaded
                if (!tc::in_bounds(q0 < Nq && (!CAUSAL || q0 + C::BQ - 1 >= k0), &g_fa_bwd_status, abort_flag)) break;
                tc::mbar_arrive_expect_tx(q_full(s), 2 * C::QT::BYTES + 1024);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + s * C::QT::BYTES + c * C::QT::CHUNK, &tmQ, q_full(s), c * 64,
                                    q0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::DO_OFF + s * C::QT::BYTES + c * C::QT::CHUNK, &tmdO, q_full(s),
                                    c * 64, q0, bh, H);
                }
                const size_t off = (size_t)bh * nqp + q0;
                tc::bulk_load(base + C::LD_OFF + s * 1024, Lp + off, 512, q_full(s));
                tc::bulk_load(base + C::LD_OFF + s * 1024 + 512, Dp + off, 512, q_full(s));
                issued = it + 1;
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_bwd_rows[0], (unsigned long long)issued * C::BQ);
            if (*abort_flag) {
                for (int it = issued - 1; it >= 0 && it >= issued - C::STAGES; --it) {
                    const int s = it % C::STAGES;
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full(s), (it / C::STAGES) & 1); ++i) {
                    }
                }
                if (kv_ok)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(kv_full, 0); ++i) {
                    }
            }
        }
    } else if (RED && warp == 2) {
        // ------------------------------------------------------------ dQ reduction (RED)
        // each sub-tile's staged dQ partial is added into the fp32 accumulator in
        // global memory (rows q0.. of this batch*head) by one TMA reduction per box
        if (lane == 0 && n > 0) {
            for (int it = 0; it < n; ++it) {
                if (!W.wait(dq_staged, it & 1)) break;
                const int q0 = (i_begin + it) * C::BQ;
                if (!tc::in_bounds(q0 + C::BQ <= nqp, &g_fa_bwd_status, abort_flag)) break;
#pragma unroll
                for (int x = 0; x < D / 32; ++x)
                    tc::tma_reduce_add_3d(tmdQa, base + C::DQS_OFF + x * C::DQS_BOX, 32 * x, q0, bh);
                tc::bulk_commit_group();
                tc::bulk_wait_read_all();   // the staging boxes may be rewritten
                tc::mbar_arrive(dq_free);
            }
            tc::bulk_wait_all();            // the additions have landed before the CTA exits
        }
    } else if (RED && SPLIT == 1 && warp == 3) {
        // ------------------------------------------------------------ dV / dK stores (RED, unsplit)
        // the rows, staged by the element-wise warpgroups in their halves of the dS^T
        // tile (128-byte swizzled), go out as two TMA stores (rows past Nk are not written)
        if constexpr (RED && SPLIT == 1) {
            if (lane == 0) {
                for (int t = 0; t < 2; ++t) {
                    if (!W.wait(ep_staged(t), 0)) break;
                    tc::tma_store_rows<VIEW4>(t == 0 ? tmdV : tmdK, base + C::DS_OFF + t * (128 * 128), 0, k0, bh, H);
                }
                tc::bulk_commit_group();
                tc::bulk_wait_all();   // the stores have read the tiles (and landed) before the CTA exits
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // whole warp in the loop (uniform descriptors), one elected lane issues
        const bool leader = tc::elect_one();
        if (n > 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16(128, C::BQ, false, false);
            constexpr uint32_t idesc_g = tc::idesc_bf16(128, D, false, true);
            const uint64_t kd = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);     // A of S^T, K-major
            const uint64_t vd = tc::sdesc_sw128(base + C::V_OFF, 16, 1024);     // A of dP^T
            const uint64_t qk = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);     // B of S^T, K-major, stage 0
            const uint64_t gk = tc::sdesc_sw128(base + C::DO_OFF, 16, 1024);    // B of dP^T
            const uint64_t qm = tc::sdesc_sw128(base + C::Q_OFF, C::QT::CHUNK, 1024);    // B of dK, MN-major
            const uint64_t gm = tc::sdesc_sw128(base + C::DO_OFF, C::QT::CHUNK, 1024);   // B of dV, MN-major
            // RED: dQ = dS K with A = dS (queries x keys, MN-major: the dS^T rows are keys)
            // and B = K (keys x d, MN-major), both from shared memory
            constexpr uint32_t idesc_q = tc::idesc_bf16(128, D, true, true);
            const uint64_t dsk = tc::sdesc_sw128(base + C::DS_OFF, 16, 1024);              // A of dK, K-major
            const uint64_t dsm = tc::sdesc_sw128(base + C::DS_OFF, 128 * 128, 1024);       // A of dQ, MN-major
            const uint64_t km = tc::sdesc_sw128(base + C::K_OFF, C::KT::CHUNK, 1024);      // B of dQ, MN-major
            bool ok = __all_sync(0xffffffffu, W.wait(kv_full, 0));
            // S^T = K Q^T and dP^T = V dO^T for sub-tile `it`; after the first, S^T / dP^T
            // must also have been read for sub-tile it-1 (both waits polled together)
            auto sdp = [&](int it) -> bool {
                const int s = it % C::STAGES;
                const bool ready = it > 0 ? W.wait2(sd_free, (it - 1) & 1, q_full(s), (it / C::STAGES) & 1)
                                          : W.wait(q_full(s), (it / C::STAGES) & 1);
                if (!__all_sync(0xffffffffu, ready)) return false;
                if (leader) {
                    const uint32_t st = (s * C::QT::BYTES) >> 4;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {   // two independent chains, interleaved
                        const uint32_t oa = ((kk >> 2) * C::KT::CHUNK + (kk & 3) * 32) >> 4;
                        const uint32_t ob = ((kk >> 2) * C::QT::CHUNK + (kk & 3) * 32) >> 4;
                        tc::mma_ss(tmem + C::ST_COL, kd + oa, qk + st + ob, idesc_s, kk > 0 ? 1u : 0u);
                        tc::mma_ss(tmem + C::DP_COL, vd + oa, gk + st + ob, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(sd_full);
                }
                __syncwarp();
                return true;
            };
            auto grads = [&](int it) -> bool {   // dV += P^T dO, dK += dS^T Q for sub-tile `it`
                const int s = it % C::STAGES;
                if (!__all_sync(0xffffffffu, W.wait(p_full, it & 1))) return false;
                tc::fence_after_sync();
                if (leader) {
                    const uint32_t st = (s * C::QT::BYTES) >> 4;
#pragma unroll
                    for (int kk = 0; kk < C::BQ / 16; ++kk) {
                        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                        tc::mma_ts(tmem + C::DV_COL, tmem + C::PT_COL + kk * 8, gm + st + kk * 128, idesc_g, acc);
                        if constexpr (RED)
                            tc::mma_ss(tmem + C::DK_COL, dsk + (((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4),
                                       qm + st + kk * 128, idesc_g, acc);
                        else
                            tc::mma_ts(tmem + C::DK_COL, tmem + C::DS_COL + kk * 8, qm + st + kk * 128, idesc_g, acc);
                    }
                    if constexpr (RED) {
#pragma unroll
                        for (int kk = 0; kk < C::BK / 16; ++kk)   // 16 keys per step
                            tc::mma_ss(tmem + C::DQ_COL, dsm + kk * 128, km + kk * 128, idesc_q, kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(q_empty(s));   // sub-tile done: its stage is free
                }
                __syncwarp();
                return true;
            };
            if (ok) ok = sdp(0);
            for (int it = 0; ok && it < n; ++it) {
                if constexpr (C::SEP) {
                    // the next scores once this sub-tile's have been read, then this sub-tile's gradients
                    if (it + 1 < n && !(ok = sdp(it + 1))) break;
                    ok = grads(it);
                } else {
                    // P^T and dS^T live over S^T and dP^T: the next scores follow the gradients
                    if (!(ok = grads(it))) break;
                    if (it + 1 < n) ok = sdp(it + 1);
                }
            }
            if (!ok && leader) {
                tc::mma_commit(drain);
                for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
                }
            }
            __syncwarp();
        }
    }
    } else {
        tc::regs_inc<224>();
        // ------------------------------------------------------------ element-wise warpgroups
        const int t = (warp - 4) >> 2;                       // query columns [64t, 64t + 64)
        const int r = ((warp & 3) << 5) + lane;              // key row within the tile = TMEM lane
        const int key = k0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::ST_COL + 64 * t;
        const uint32_t tD = tmem + lane_base + C::DP_COL + 64 * t;
        const uint32_t tPT = tmem + lane_base + C::PT_COL + 32 * t;
        const uint32_t tDS = tmem + lane_base + C::DS_COL + 32 * t;
        const uint32_t tDQ = tmem + lane_base + C::DQ_COL + 32 * t;   // RED: query row r, columns [32t, 32t+32)
        // RED: stage sub-tile j's dQ partial (row r, columns [32t, 32t+32)) once the
        // reduction has read sub-tile j-1's, then hand it to the reducing warp
        auto stage_dq = [&](int j, const uint32_t (&v)[32]) -> bool {
            if (j > 0 && !__all_sync(0xffffffffu, W.wait(dq_free, (j - 1) & 1))) return false;
            uint8_t *row = sb + C::DQS_OFF + t * C::DQS_BOX + r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4 *>(row + ((u ^ (r & 7)) << 4)) =
                    make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(dq_staged);
            return true;
        };
        for (int it = 0; it < n; ++it) {
            const int s = it % C::STAGES;
            const int qc = (i_begin + it) * C::BQ + 64 * t;      // this warpgroup's first query column
            // S^T, dP^T of this sub-tile, and its L and D in shared memory
            bool ok = W.wait2(sd_full, it & 1, q_full(s), (it / C::STAGES) & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            uint32_t sv[2][32], dv[2][32];
            tmem_ld_x32(tS, sv[0]);
            tmem_ld_x32(tS + 32, sv[1]);
            tmem_ld_x32(tD, dv[0]);
            tmem_ld_x32(tD + 32, dv[1]);
            tc::tmem_ld_wait();
            reg_fence_x32(sv[0]);
            reg_fence_x32(sv[1]);
            reg_fence_x32(dv[0]);
            reg_fence_x32(dv[1]);
            tc::fence_before_sync();
            tc::mbar_arrive(sd_free);                                   // this half of S^T, dP^T has been read
            if constexpr (!C::SEP) {
                // P^T / dS^T land over S^T / dP^T: wait until the other warpgroup has read its half too
                ok = W.wait(sd_free, it & 1);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            const float *lds = reinterpret_cast<const float *>(sb + C::LD_OFF + s * 1024) + 64 * t;   // -L*log2e
            // causal: query columns c < key - qc cannot see this key.  Only the
            // diagonal sub-tile has such columns; there S^T is set to -inf first
            // (P = 2^-inf = 0 and dS = 0), so the main loop carries no mask test.
            const int first_visible = key - qc;
            if (CAUSAL && __any_sync(0xffffffffu, first_visible > 0)) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c < first_visible) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            // P^T and dS^T in two halves of 16 columns each: the first half is stored
            // while the second is computed
            uint32_t pp[32], dsp[32];
            auto half = [&](int hh) {
#pragma unroll
                for (int i = 8 * hh; i < 8 * hh + 8; ++i) {
                    const float4 nl = *reinterpret_cast<const float4 *>(lds + 4 * i);
                    const float4 nd = *reinterpret_cast<const float4 *>(lds + 128 + 4 * i);   // -D
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 4 * i + 2 * h;
                        const float l0 = h ? nl.z : nl.x, l1 = h ? nl.w : nl.y;
                        const float d0 = h ? nd.z : nd.x, d1 = h ? nd.w : nd.y;
                        float x0, x1, g0, g1;
                        tc::fma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]),
                                 scale_log2, scale_log2, l0, l1);
                        const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
                        tc::add2(g0, g1, __uint_as_float(dv[c >> 5][c & 31]), __uint_as_float(dv[c >> 5][(c & 31) + 1]),
                                 d0, d1);
                        tc::mul2(g0, g1, g0, g1, p0, p1);
                        pp[2 * i + h] = tc::pack_bf16(p0, p1);
                        dsp[2 * i + h] = tc::pack_bf16(g0, g1);
                    }
                }
            };
            auto store_half = [&](int hh) {
                const uint32_t(&ph)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pp[16 * hh]);
                const uint32_t(&dh)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&dsp[16 * hh]);
                tmem_st_x16(tPT + 16 * hh, ph);
                if constexpr (RED) {
                    uint8_t *row = sb + C::DS_OFF + t * (128 * 128) + r * 128;
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu)
                        *reinterpret_cast<uint4 *>(row + (((4 * hh + uu) ^ (r & 7)) << 4)) =
                            make_uint4(dh[4 * uu], dh[4 * uu + 1], dh[4 * uu + 2], dh[4 * uu + 3]);
                } else {
                    tmem_st_x16(tDS + 16 * hh, dh);
                }
            };
            half(0);
            if (C::SEP && it > 0) {
                // P^T and dS^T are still read by the previous sub-tile's gradient MMAs until they complete
                ok = W.wait(q_empty((it - 1) % C::STAGES), ((it - 1) / C::STAGES) & 1);
                if (!__all_sync(0xffffffffu, ok)) break;
                tc::fence_after_sync();
            }
            uint32_t dq[32];
            if (RED && it > 0) tmem_ld_x32(tDQ, dq);   // sub-tile it-1's dQ, before this sub-tile's MMA rewrites it
            store_half(0);
            half(1);
            store_half(1);
            tc::tmem_st_wait();
            if constexpr (RED) {
                if (it > 0) {
                    tc::tmem_ld_wait();
                    reg_fence_x32(dq);
                }
                tc::fence_proxy_async_smem();   // dS^T is read by the tensor core
            }
            tc::fence_before_sync();
            tc::mbar_arrive(p_full);
            if (RED && it > 0 && !stage_dq(it - 1, dq)) break;
        }
        // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (rows = keys);
        // a split item's rank 1 leaves its partial sums for rank 0 to add
        tc::named_bar_sync(1, 256);
        bool fine = !*abort_flag;
        // the last sub-tile's stage release means every MMA has completed (they run in order)
        if (fine && n > 0) fine = W.wait(q_empty((n - 1) % C::STAGES), ((n - 1) / C::STAGES) & 1);
        fine = __all_sync(0xffffffffu, fine);
        if (fine && n > 0) tc::fence_after_sync();
        if constexpr (RED) {
            if (fine && n > 0) {   // the last sub-tile's dQ partial
                uint32_t dq[32];
                tmem_ld_x32(tDQ, dq);
                tc::tmem_ld_wait();
                reg_fence_x32(dq);
                fine = stage_dq(n - 1, dq);
            }
        }
        __nv_bfloat16 *dst;
        if constexpr (VIEW4)
            dst = t == 0 ? dV + fa_row_offset(sdv, tc::opaque(H), bh, key) : dK + fa_row_offset(sdk, tc::opaque(H), bh, key);
        else
            dst = (t == 0 ? dV : dK) + ((size_t)bh * Nk + key) * D;
        const float mul = t == 0 ? 1.f : scale;
        const uint32_t tA = tmem + lane_base + (t == 0 ? C::DV_COL : C::DK_COL);
        // Split items: each rank finalises one tensor (rank 0 dV, rank 1 dK) and sends
        // its partial of the other into the peer's shared memory with remote stores
        // (streamed, no round trip per access), once the peer's own MMAs are done
        // and its stages are free; the peer adds it to its own accumulator.
        const bool mine = SPLIT == 1 || t == (int)rank;
        const uint32_t peer_free = base + C::PEER_BAR_OFF, peer_ready = peer_free + 8;
        const uint32_t part = base + C::PART_OFF + r * C::PART_STRIDE;   // partial row received here
        if constexpr (SPLIT > 1) tc::mbar_arrive_remote(tc::map_to_rank(peer_free, rank ^ 1u));
        bool merge = false;
        if (SPLIT > 1 && !mine) {
            const bool dst_ok = tc::wait_peer(peer_free, &g_fa_bwd_status, 2u);
            const uint32_t rdst = tc::map_to_rank(part, rank ^ 1u);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (dst_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        tc::st_cluster_v4(rdst + 128 * c + 16 * i, a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
                }
            }
            tc::mbar_arrive_remote(tc::map_to_rank(peer_ready, rank ^ 1u));   // release: the stores above
        } else {
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 2u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (merge) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 q = reinterpret_cast<const float4 *>(pr + 32 * c)[i];
                        a[4 * i + 0] = __float_as_uint(__uint_as_float(a[4 * i + 0]) + q.x);
                        a[4 * i + 1] = __float_as_uint(__uint_as_float(a[4 * i + 1]) + q.y);
                        a[4 * i + 2] = __float_as_uint(__uint_as_float(a[4 * i + 2]) + q.z);
                        a[4 * i + 3] = __float_as_uint(__uint_as_float(a[4 * i + 3]) + q.w);
                    }
                }
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = tc::pack_bf16(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
                if constexpr (RED && SPLIT == 1) {
                    // into this warpgroup's half of the dS^T tile (free: every MMA is done),
                    // for warp 3's TMA store
                    if (fine) {
                        uint8_t *srow = sb + C::DS_OFF + t * (128 * 128) + r * 128;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            *reinterpret_cast<uint4 *>(srow + (((4 * c + i) ^ (r & 7)) << 4)) =
                                make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    }
                } else if (fine && (SPLIT == 1 || merge) && key < Nk) {
                    uint4 *o = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (!VIEW4 || 32 * c + 8 * i < dv)   // columns past a head dim below 64 are padding
                            o[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
            }
            if constexpr (RED && SPLIT == 1) {
                if (fine) {
                    tc::fence_proxy_async_smem();
                    tc::mbar_arrive(ep_staged(t));
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ dQ (wide)
// One CTA per 128-query tile (MMA M = 128 queries), looping over 128-key
// sub-tiles (MMA N = 128 for S and dP; K = 128 for dQ += dS K).  Warpgroup t
// handles key columns [64t, 64t + 64).  dS has TMEM columns of its own, so the
// next sub-tile's S and dP are computed while the element-wise warps work.
template <int D>
struct DqWideCfg {
    static constexpr int BQ = 128;                 // queries per CTA (MMA M)
    static constexpr int BK = 128;                 // keys per sub-tile
    static constexpr int STAGES = D == 128 ? 2 : 3;
    using QT = TileShape<BQ, D>;
    using KT = TileShape<BK, D>;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t DO_OFF = Q_OFF + QT::BYTES;
    static constexpr uint32_t K_OFF = DO_OFF + QT::BYTES;                // stages of K sub-tiles
    static constexpr uint32_t V_OFF = K_OFF + STAGES * KT::BYTES;        // stages of V sub-tiles
    static constexpr uint32_t BAR_OFF = V_OFF + STAGES * KT::BYTES;
    // q_full, kv_full[S], kv_empty[S], sd_full, sd_free, p_full, drain
    static constexpr int NBAR = 1 + 2 * STAGES + 4;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t PEER_BAR_OFF = MISC_OFF + 16;
    static constexpr uint32_t SMEM_BYTES = (PEER_BAR_OFF + 16 + 1024 > 120u * 1024u ? PEER_BAR_OFF + 16 + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // split items: rank 1's partial dQ (fp32) over the K/V rings
    static constexpr uint32_t PART_STRIDE = (D + 4) * 4;
    static constexpr uint32_t PART_OFF = K_OFF;
    static_assert(PART_OFF + 128 * PART_STRIDE <= BAR_OFF, "partial fits the rings");
    // TMEM: S [0,128), dP [128,256), dQ [256, 256+D), dS (bf16, 64 columns) [384, 448)
    static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256, DS_COL = 384;
};

// one dQ work item: query tile qt of batch*head bh (a half of its keys when SPLIT = 2)
template <int D, bool CAUSAL, int SPLIT, bool VIEW4>
__device__ __forceinline__ void dq_item_wide(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                        const CUtensorMap &tmdO, const float *__restrict__ Lp,
                                        const float *__restrict__ Dp, __nv_bfloat16 *__restrict__ dQ, int Nq, int Nk,
                                        int qt, int bh, int H, int dv, const FaStrides &sdq, float scale,
                                        float scale_log2,
                                        uint32_t wait_limit) {
    using C = DqWideCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t rank = SPLIT > 1 ? tc::cluster_rank() : 0u;
    const int q0 = qt * C::BQ;
    const int kend = CAUSAL ? min(Nk, q0 + C::BQ) : Nk;
    const int n_all = (kend + C::BK - 1) / C::BK;
    // this CTA's key sub-tiles [jb, jb + n): all of them, or one half of a split item
    const int n_half = SPLIT > 1 ? (n_all + 1) / 2 : n_all;
    const int jb = rank == 0 ? 0 : n_half;
    const int n = rank == 0 ? n_half : n_all - n_half;
    const int nqp = padded_rows(Nq);

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t q_full = bar(0);
    auto kv_full = [&](int s) { return bar(1 + s); };
    auto kv_empty = [&](int s) { return bar(1 + C::STAGES + s); };   // sub-tile's dQ MMAs done
    const uint32_t sd_full = bar(1 + 2 * C::STAGES);
    const uint32_t sd_free = bar(2 + 2 * C::STAGES);
    const uint32_t p_full = bar(3 + 2 * C::STAGES);
    const uint32_t drain = bar(4 + 2 * C::STAGES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(kv_full(s), 1);
            tc::mbar_init(kv_empty(s), 1);
        }
        tc::mbar_init(sd_full, 1);
        tc::mbar_init(sd_free, 256);
        tc::mbar_init(p_full, 256);
        tc::mbar_init(drain, 1);
        if (SPLIT > 1) {
            tc::mbar_init(base + C::PEER_BAR_OFF, 256);       // peer_free: the peer's 256 element-wise threads
            tc::mbar_init(base + C::PEER_BAR_OFF + 8, 128);   // peer_ready: the peer's 128 senders
        }
        *abort_flag = 0u;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (SPLIT > 1) tc::cluster_sync_all();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const tc::Waiter W{abort_flag, &g_fa_bwd_status, wait_limit, 4u};

    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmK);
            tc::tma_prefetch_desc(&tmV);
            const bool q_ok = tc::in_bounds(q0 < Nq, &g_fa_bwd_status, abort_flag);
            if (q_ok) {
                tc::mbar_arrive_expect_tx(q_full, 2 * C::QT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + c * C::QT::CHUNK, &tmQ, q_full, c * 64, q0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::DO_OFF + c * C::QT::CHUNK, &tmdO, q_full, c * 64, q0, bh, H);
                }
            }
            int issued = 0;
            for (int j = 0; q_ok && j < n; ++j) {
                const int s = j % C::STAGES;
                if (!W.wait(kv_empty(s), ((j / C::STAGES) & 1) ^ 1u)) break;
                // debug build: a key sub-tile past the keys, or wholly above the diagonal, is never loaded
                const int kj = (jb + j) * C::BK;
                if (!tc::in_bounds(kj < Nk && (!CAUSAL || kj <= q0 + C::BQ - 1), &g_fa_bwd_status, abort_flag)) break;
                tc::mbar_arrive_expect_tx(kv_full(s), 2 * C::KT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::K_OFF + s * C::KT::BYTES + c * C::KT::CHUNK, &tmK, kv_full(s), c * 64,
                                    (jb + j) * C::BK, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::V_OFF + s * C::KT::BYTES + c * C::KT::CHUNK, &tmV, kv_full(s), c * 64,
                                    (jb + j) * C::BK, bh, H);
                }
                issued = j + 1;
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_bwd_rows[1], (unsigned long long)issued * C::BK);
            if (*abort_flag) {
                for (int j = issued - 1; j >= 0 && j >= issued - C::STAGES; --j) {
                    const int s = j % C::STAGES;
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(kv_full(s), (j / C::STAGES) & 1); ++i) {
                    }
                }
                if (q_ok)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full, 0); ++i) {
                    }
            }
        }
    } else if (warp == 1) {
        // whole warp in the loop (uniform descriptors), one elected lane issues
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc_s = tc::idesc_bf16(128, C::BK, false, false);
        constexpr uint32_t idesc_g = tc::idesc_bf16(128, D, false, true);
        const uint64_t qd = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);      // A of S, K-major
        const uint64_t gd = tc::sdesc_sw128(base + C::DO_OFF, 16, 1024);     // A of dP
        const uint64_t kk_ = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);    // B of S, K-major, stage 0
        const uint64_t vk = tc::sdesc_sw128(base + C::V_OFF, 16, 1024);     // B of dP
        const uint64_t km = tc::sdesc_sw128(base + C::K_OFF, C::KT::CHUNK, 1024);   // B of dQ, MN-major
        bool ok = __all_sync(0xffffffffu, W.wait(q_full, 0));
        // S = Q K_j^T and dP = dO V_j^T; after the first, S / dP must also have been read
        // for sub-tile j-1 (both waits polled together)
        auto sdp = [&](int j) -> bool {
            const int s = j % C::STAGES;
            const bool ready = j > 0 ? W.wait2(sd_free, (j - 1) & 1, kv_full(s), (j / C::STAGES) & 1)
                                     : W.wait(kv_full(s), (j / C::STAGES) & 1);
            if (!__all_sync(0xffffffffu, ready)) return false;
            if (leader) {
                const uint32_t st = (s * C::KT::BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {   // two independent chains, interleaved
                    const uint32_t oa = ((kk >> 2) * C::QT::CHUNK + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * C::KT::CHUNK + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + C::S_COL, qd + oa, kk_ + st + ob, idesc_s, kk > 0 ? 1u : 0u);
                    tc::mma_ss(tmem + C::DP_COL, gd + oa, vk + st + ob, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(sd_full);
            }
            __syncwarp();
            return true;
        };
        auto grads = [&](int j) -> bool {   // dQ += dS K_j
            const int s = j % C::STAGES;
            if (!__all_sync(0xffffffffu, W.wait(p_full, j & 1))) return false;
            tc::fence_after_sync();
            if (leader) {
                const uint32_t st = (s * C::KT::BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    tc::mma_ts(tmem + C::DQ_COL, tmem + C::DS_COL + kk * 8, km + st + kk * 128, idesc_g,
                               (j > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(kv_empty(s));   // sub-tile done: its stage is free
            }
            __syncwarp();
            return true;
        };
        if (ok && n > 0) ok = sdp(0);
        for (int j = 0; ok && j < n; ++j) {
            if (j + 1 < n && !(ok = sdp(j + 1))) break;
            ok = grads(j);
        }
        if (!ok && leader) {
            tc::mma_commit(drain);
            for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
            }
        }
        __syncwarp();
    }
    } else {
        tc::regs_inc<224>();
        const int t = (warp - 4) >> 2;                       // key columns [64t, 64t + 64)
        const int r = ((warp & 3) << 5) + lane;
        const int row = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::S_COL + 64 * t;
        const uint32_t tD = tmem + lane_base + C::DP_COL + 64 * t;
        const uint32_t tDS = tmem + lane_base + C::DS_COL + 32 * t;
        const float nlrow = Lp[(size_t)bh * nqp + row];     // -L*log2e (-inf on padding rows)
        const float ndrow = Dp[(size_t)bh * nqp + row];     // -D
        for (int j = 0; j < n; ++j) {
            const int kc = (jb + j) * C::BK + 64 * t;        // this warpgroup's first key column
            bool ok = W.wait(sd_full, j & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            uint32_t sv[2][32], dv[2][32];
            tmem_ld_x32(tS, sv[0]);
            tmem_ld_x32(tS + 32, sv[1]);
            tmem_ld_x32(tD, dv[0]);
            tmem_ld_x32(tD + 32, dv[1]);
            tc::tmem_ld_wait();
            reg_fence_x32(sv[0]);
            reg_fence_x32(sv[1]);
            reg_fence_x32(dv[0]);
            reg_fence_x32(dv[1]);
            tc::fence_before_sync();
            tc::mbar_arrive(sd_free);                         // S and dP may be overwritten
            // key columns past the diagonal (causal) or past Nk: S set to -inf first
            // (P = 0, dS = 0), so the main loop carries no mask test
            const int lim = min(Nk - 1, CAUSAL ? row : Nk - 1) - kc;   // last visible key column
            if (__any_sync(0xffffffffu, lim < 63)) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c > lim) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            uint32_t dsp[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 2 * i;
                float x0, x1, g0, g1;
                tc::fma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]),
                         scale_log2, scale_log2, nlrow, nlrow);
                const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
                tc::add2(g0, g1, __uint_as_float(dv[c >> 5][c & 31]), __uint_as_float(dv[c >> 5][(c & 31) + 1]),
                         ndrow, ndrow);
                tc::mul2(g0, g1, g0, g1, p0, p1);
                dsp[i] = tc::pack_bf16(g0, g1);
            }
            if (j > 0) {
                // dS is still read by the previous sub-tile's dQ MMAs until they complete
                ok = W.wait(kv_empty((j - 1) % C::STAGES), ((j - 1) / C::STAGES) & 1);
                if (!__all_sync(0xffffffffu, ok)) break;
                tc::fence_after_sync();
            }
            tmem_st_x32(tDS, dsp);
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(p_full);
        }
        tc::named_bar_sync(1, 256);
        bool fine = !*abort_flag;
        // the last sub-tile's stage release means every MMA has completed (they run in order)
        if (fine && n > 0) fine = W.wait(kv_empty((n - 1) % C::STAGES), ((n - 1) / C::STAGES) & 1);
        fine = __all_sync(0xffffffffu, fine);
        if (fine && n > 0) tc::fence_after_sync();
        __nv_bfloat16 *dst;
        if constexpr (VIEW4) dst = dQ + fa_row_offset(sdq, tc::opaque(H), bh, row);
        else dst = dQ + ((size_t)bh * Nq + row) * D;
        const uint32_t tA = tmem + lane_base + C::DQ_COL;
        // Split items: rank r finalises the columns of warpgroup r and sends its partial
        // of the other half into the peer's shared memory with remote stores, once the
        // peer's own MMAs are done and its stages are free.
        const bool mine = SPLIT == 1 || t == (int)rank;
        const uint32_t peer_free = base + C::PEER_BAR_OFF, peer_ready = peer_free + 8;
        const uint32_t part = base + C::PART_OFF + r * C::PART_STRIDE;   // half row received here
        if constexpr (SPLIT > 1) tc::mbar_arrive_remote(tc::map_to_rank(peer_free, rank ^ 1u));
        if (SPLIT > 1 && !mine) {
            const bool dst_ok = tc::wait_peer(peer_free, &g_fa_bwd_status, 4u);
            const uint32_t rdst = tc::map_to_rank(part, rank ^ 1u);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int col = t * (D / 2) + 32 * c;
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + col, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (dst_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        tc::st_cluster_v4(rdst + 128 * c + 16 * i, a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
                }
            }
            tc::mbar_arrive_remote(tc::map_to_rank(peer_ready, rank ^ 1u));   // release: the stores above
        } else {
            bool merge = false;
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 4u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int col = t * (D / 2) + 32 * c;
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + col, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (merge) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 q = reinterpret_cast<const float4 *>(pr + 32 * c)[i];
                        a[4 * i + 0] = __float_as_uint(__uint_as_float(a[4 * i + 0]) + q.x);
                        a[4 * i + 1] = __float_as_uint(__uint_as_float(a[4 * i + 1]) + q.y);
                        a[4 * i + 2] = __float_as_uint(__uint_as_float(a[4 * i + 2]) + q.z);
                        a[4 * i + 3] = __float_as_uint(__uint_as_float(a[4 * i + 3]) + q.w);
                    }
                }
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = tc::pack_bf16(__uint_as_float(a[2 * i]) * scale, __uint_as_float(a[2 * i + 1]) * scale);
                if (fine && (SPLIT == 1 || merge) && row < Nq) {
                    uint4 *o = reinterpret_cast<uint4 *>(dst + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (!VIEW4 || col + 8 * i < dv)   // columns past a head dim below 64 are padding
                            o[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ================================================================== narrow sub-tiles (d = 128)
// dK / dV and dQ with 64-wide sub-tiles, each warpgroup taking whole
// alternate sub-tiles with its own S/dP TMEM buffers (double-buffered), which
// measures faster than the 128-wide form at d = 128, where TMEM has no room to
// keep P^T / dS^T apart from S^T / dP^T.
// ------------------------------------------------------------------ dK / dV (narrow)
template <int D>
struct DkdvNarrowCfg {
    static constexpr int BK = 128;                 // keys per CTA (MMA M)
    // queries per sub-tile (MMA N of S^T, K of dV/dK); 32 for the 256-column split rows
    static constexpr int BQ = D == 256 ? 32 : 64;
    // deep ring: a stage is refilled only after its sub-tile's dV/dK MMAs finish, and
    // an L2-resident TMA reload takes ~2000 cycles, several sub-tiles' worth of MMA time
    // (D = 256, the split pairs of fp32 head dim 128: 32-row sub-tiles, two stages next to
    // the 64 KB K and V tiles)
    static constexpr int STAGES = D == 256 ? 2 : D == 128 ? 4 : 8;
    // dV / dK accumulator columns: d, but 128 for the 256-column split rows
    static constexpr int OW = D == 256 ? 128 : D;
    using KT = TileShape<BK, D>;
    using QT = TileShape<BQ, D>;
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + KT::BYTES;
    static constexpr uint32_t Q_OFF = V_OFF + KT::BYTES;                 // stages of Q sub-tiles
    static constexpr uint32_t DO_OFF = Q_OFF + STAGES * QT::BYTES;       // stages of dO sub-tiles
    static constexpr uint32_t LD_OFF = DO_OFF + STAGES * QT::BYTES;      // stages of BQ Lp + BQ D floats (512 B)
    static constexpr uint32_t BAR_OFF = LD_OFF + STAGES * 512;
    // kv_full, q_full[S], q_empty[S], sd_full[2], p_full[2], mma_done[2], drain
    static constexpr int NBAR = 1 + 2 * STAGES + 6 + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t PEER_BAR_OFF = MISC_OFF + 16;
    static constexpr uint32_t SMEM_BYTES = (PEER_BAR_OFF + 16 + 1024 > 120u * 1024u ? PEER_BAR_OFF + 16 + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // split items: rank 1's partial dV (rows 0..127) and dK (rows 128..255), fp32, over the tile rings
    static constexpr uint32_t PART_STRIDE = (OW + 4) * 4;
    static constexpr uint32_t PART_OFF = 0;
    static_assert(PART_OFF + 256 * PART_STRIDE <= BAR_OFF, "partial fits the rings");
    // TMEM: S^T_t [128t, 128t+64), dP^T_t [128t+64, 128t+128), dV [256, 256+OW), dK [256+OW, 256+2OW)
    static constexpr uint32_t DV_COL = 256, DK_COL = 256 + OW;
    static_assert(DK_COL + OW <= TMEM_COLS, "dV and dK after the score buffers");
};

// one dK/dV work item: key tile kt of batch*head bh (a half of it when SPLIT = 2).
// X3 (fp32 inputs, head dim up to 64, operands as bf16 pairs [hi | lo] in the
// d = 128 layout): S^T and dP^T take the chunk pairs (hi, hi), (hi, lo), (lo, hi);
// P^T and dS^T are split too (lo in the second 32 columns of their TMEM
// buffers), dV = Phi^T [dOhi | dOlo] + Plo^T dOhi and dK likewise; output column
// c is accumulator column c plus 64 + c, written in fp32.
template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool X3 = false>
__device__ __forceinline__ void dkdv_item_narrow(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                          const CUtensorMap &tmdO, const float *__restrict__ Lp,
                                          const float *__restrict__ Dp, void *__restrict__ dKv,
                                          void *__restrict__ dVv, int Nq, int Nk, int kt, int bh, int H,
                                          int dv, const FaStrides &sdk, const FaStrides &sdv, float scale,
                                          float scale_log2, uint32_t wait_limit) {
    static_assert(!X3 || ((D == 128 || D == 256) && !VIEW4), "split fp32 operands: 128- or 256-column copies");
    static_assert(X3 || D <= 128, "the 256-column layout holds split pairs only");
    using C = DkdvNarrowCfg<D>;
    constexpr bool FOLD = X3 && D == 128;   // outputs folded from [hi | lo] accumulator columns
    __nv_bfloat16 *dK = static_cast<__nv_bfloat16 *>(dKv), *dV = static_cast<__nv_bfloat16 *>(dVv);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t rank = SPLIT > 1 ? tc::cluster_rank() : 0u;
    const int k0 = kt * C::BK;
    const int nqp = padded_rows(Nq);
    const int i_end = (Nq + C::BQ - 1) / C::BQ;
    const int i_first = CAUSAL ? k0 / C::BQ : 0;              // first query sub-tile that sees a key of this tile
    const int n_all = i_end > i_first ? i_end - i_first : 0;
    // this CTA's query sub-tiles: all of them, or one half of a split item
    const int n_half = SPLIT > 1 ? (n_all + 1) / 2 : n_all;
    const int i_begin = i_first + (rank == 0 ? 0 : n_half);
    const int n = rank == 0 ? n_half : n_all - n_half;        // sub-tiles to visit

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t kv_full = bar(0);
    auto q_full = [&](int s) { return bar(1 + s); };
    auto q_empty = [&](int s) { return bar(1 + C::STAGES + s); };
    auto sd_full = [&](int t) { return bar(1 + 2 * C::STAGES + t); };
    auto p_full = [&](int t) { return bar(3 + 2 * C::STAGES + t); };
    auto mma_done = [&](int t) { return bar(5 + 2 * C::STAGES + t); };
    const uint32_t drain = bar(7 + 2 * C::STAGES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(kv_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(q_full(s), 1);
            tc::mbar_init(q_empty(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(sd_full(t), 1);
            tc::mbar_init(p_full(t), 128);
            tc::mbar_init(mma_done(t), 1);
        }
        tc::mbar_init(drain, 1);
        if (SPLIT > 1) {
            tc::mbar_init(base + C::PEER_BAR_OFF, 256);       // peer_free: the peer's 256 element-wise threads
            tc::mbar_init(base + C::PEER_BAR_OFF + 8, 128);   // peer_ready: the peer's 128 senders
        }
        *abort_flag = 0u;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (SPLIT > 1) tc::cluster_sync_all();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const tc::Waiter W{abort_flag, &g_fa_bwd_status, wait_limit, 2u};

    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            tc::tma_prefetch_desc(&tmQ);
            tc::tma_prefetch_desc(&tmdO);
            const bool kv_ok = tc::in_bounds(k0 < Nk, &g_fa_bwd_status, abort_flag);
            if (kv_ok) {
                tc::mbar_arrive_expect_tx(kv_full, 2 * C::KT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::K_OFF + c * C::KT::CHUNK, &tmK, kv_full, c * 64, k0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::V_OFF + c * C::KT::CHUNK, &tmV, kv_full, c * 64, k0, bh, H);
                }
            }
            int issued = 0;
            for (int it = 0; kv_ok && it < n; ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1;
                if (!W.wait(q_empty(s), ph ^ 1u)) break;
                const int q0 = (i_begin + it) * C::BQ;
                // debug build: a query sub-tile past the queries, or wholly on the
                // masked side of the diagonal, is never loaded
                if (!tc::in_bounds(q0 < Nq && (!CAUSAL || q0 + C::BQ - 1 >= k0), &g_fa_bwd_status, abort_flag)) break;
                tc::mbar_arrive_expect_tx(q_full(s), 2 * C::QT::BYTES + 2 * C::BQ * 4);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + s * C::QT::BYTES + c * C::QT::CHUNK, &tmQ, q_full(s), c * 64,
                                    q0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::DO_OFF + s * C::QT::BYTES + c * C::QT::CHUNK, &tmdO, q_full(s),
                                    c * 64, q0, bh, H);
                }
                const size_t off = (size_t)bh * nqp + q0;
                tc::bulk_load(base + C::LD_OFF + s * 512, Lp + off, C::BQ * 4, q_full(s));
                tc::bulk_load(base + C::LD_OFF + s * 512 + 256, Dp + off, C::BQ * 4, q_full(s));
                issued = it + 1;
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_bwd_rows[0], (unsigned long long)issued * C::BQ);
            if (*abort_flag) {
                for (int it = issued - 1; it >= 0 && it >= issued - C::STAGES; --it) {
                    const int s = it % C::STAGES;
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full(s), (it / C::STAGES) & 1); ++i) {
                    }
                }
                if (kv_ok)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(kv_full, 0); ++i) {
                    }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // whole warp in the loop (uniform descriptors), one elected lane issues
        const bool leader = tc::elect_one();
        if (n > 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16(128, C::BQ, false, false);
            constexpr uint32_t idesc_g = tc::idesc_bf16(128, C::OW, false, true);
            constexpr uint32_t idesc_g_hi = tc::idesc_bf16(128, 64, false, true);   // X3, D = 128: lo times hi
            const uint64_t kd = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);     // A of S^T, K-major
            const uint64_t vd = tc::sdesc_sw128(base + C::V_OFF, 16, 1024);     // A of dP^T
            const uint64_t qk = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);     // B of S^T, K-major, stage 0
            const uint64_t ok_ = tc::sdesc_sw128(base + C::DO_OFF, 16, 1024);   // B of dP^T
            const uint64_t qm = tc::sdesc_sw128(base + C::Q_OFF, C::QT::CHUNK, 1024);    // B of dK, MN-major
            const uint64_t om = tc::sdesc_sw128(base + C::DO_OFF, C::QT::CHUNK, 1024);   // B of dV, MN-major
            bool ok = __all_sync(0xffffffffu, W.wait(kv_full, 0));
            auto grads = [&](int it) -> bool {   // dV += P^T dO, dK += dS^T Q for sub-tile `it`
                const int s = it % C::STAGES, t = it & 1, k = it >> 1;
                if (!__all_sync(0xffffffffu, W.wait(p_full(t), k & 1))) return false;
                tc::fence_after_sync();
                if (leader) {
                    const uint32_t st = (s * C::QT::BYTES) >> 4;
#pragma unroll
                    for (int kk = 0; kk < C::BQ / 16; ++kk) {   // two independent chains, interleaved
                        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                        tc::mma_ts(tmem + C::DV_COL, tmem + 128 * t + kk * 8, om + st + kk * 128, idesc_g, acc);
                        tc::mma_ts(tmem + C::DK_COL, tmem + 128 * t + 64 + kk * 8, qm + st + kk * 128, idesc_g, acc);
                    }
                    if constexpr (FOLD) {   // Plo^T dOhi and dSlo^T Qhi into the first 64 columns
#pragma unroll
                        for (int kk = 0; kk < C::BQ / 16; ++kk) {
                            tc::mma_ts(tmem + C::DV_COL, tmem + 128 * t + C::BQ / 2 + kk * 8, om + st + kk * 128,
                                       idesc_g_hi, 1u);
                            tc::mma_ts(tmem + C::DK_COL, tmem + 128 * t + 64 + C::BQ / 2 + kk * 8, qm + st + kk * 128,
                                       idesc_g_hi, 1u);
                        }
                    } else if constexpr (X3) {
                        // D = 256: Phi^T dOlo, dShi^T Qlo (chunks 2, 3), then Plo^T dOhi, dSlo^T Qhi, all
                        // into the same dV / dK columns
                        const uint32_t lo = (2 * C::QT::CHUNK) >> 4;
#pragma unroll
                        for (int kk = 0; kk < C::BQ / 16; ++kk) {
                            tc::mma_ts(tmem + C::DV_COL, tmem + 128 * t + kk * 8, om + st + lo + kk * 128, idesc_g, 1u);
                            tc::mma_ts(tmem + C::DK_COL, tmem + 128 * t + 64 + kk * 8, qm + st + lo + kk * 128, idesc_g, 1u);
                        }
#pragma unroll
                        for (int kk = 0; kk < C::BQ / 16; ++kk) {
                            tc::mma_ts(tmem + C::DV_COL, tmem + 128 * t + C::BQ / 2 + kk * 8, om + st + kk * 128,
                                       idesc_g, 1u);
                            tc::mma_ts(tmem + C::DK_COL, tmem + 128 * t + 64 + C::BQ / 2 + kk * 8, qm + st + kk * 128,
                                       idesc_g, 1u);
                        }
                    }
                    tc::mma_commit(q_empty(s));   // sub-tile `it` done: its stage is free
                }
                __syncwarp();
                return true;
            };
            for (int it = 0; ok && it < n; ++it) {
                const int s = it % C::STAGES, t = it & 1;
                if (!(ok = __all_sync(0xffffffffu, W.wait(q_full(s), (it / C::STAGES) & 1)))) break;
                if (leader) {
                    const uint32_t st = (s * C::QT::BYTES) >> 4;
                    // S^T = K Q^T and dP^T = V dO^T, interleaved, four k-steps per chunk pair:
                    // (c, c) for each chunk, or X3: (hi, hi), (hi, lo), (lo, hi) for each of the
                    // HC hi chunks (the lo chunks follow them)
                    constexpr int HC = X3 ? D / 128 : 1;
                    constexpr int PAIRS = X3 ? 3 * HC : D / 64;
                    auto pair = [&](int pr) {
                        int ca = pr, cb = pr;
                        if constexpr (X3) {
                            const int grp = pr / HC, c = pr % HC;
                            ca = grp == 2 ? HC + c : c;
                            cb = grp == 1 ? HC + c : c;
                        }
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint32_t oa = (ca * C::KT::CHUNK + k4 * 32) >> 4;
                            const uint32_t ob = (cb * C::QT::CHUNK + k4 * 32) >> 4;
                            const uint32_t acc = (pr > 0 || k4 > 0) ? 1u : 0u;
                            tc::mma_ss(tmem + 128 * t, kd + oa, qk + st + ob, idesc_s, acc);
                            tc::mma_ss(tmem + 128 * t + 64, vd + oa, ok_ + st + ob, idesc_s, acc);
                        }
                    };
                    if constexpr (PAIRS <= 3) {
#pragma unroll
                        for (int pr = 0; pr < PAIRS; ++pr) pair(pr);
                    } else {
#pragma unroll 1
                        for (int pr = 0; pr < PAIRS; ++pr) pair(pr);
                    }
                    tc::mma_commit(sd_full(t));
                }
                __syncwarp();
                if (it >= 1) ok = grads(it - 1);
            }
            if (ok) ok = grads(n - 1);
            if (!ok && leader) {
                tc::mma_commit(drain);
                for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
                }
            }
            __syncwarp();
        }
    }
    } else {
        tc::regs_inc<224>();
        // ------------------------------------------------------------ element-wise warpgroups
        const int t = (warp - 4) >> 2;
        const int r = ((warp & 3) << 5) + lane;              // key row within the tile = TMEM lane
        const int key = k0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + 128 * t;
        const uint32_t tP = tS + 64;
        const int nt = (n - t + 1) >> 1;
        for (int k = 0; k < nt; ++k) {
            const int it = 2 * k + t;
            const int s = it % C::STAGES;
            const int q0 = (i_begin + it) * C::BQ;
            bool ok = W.wait(sd_full(t), k & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            ok = W.wait(q_full(s), (it / C::STAGES) & 1);      // L and D of this sub-tile are in smem
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            constexpr int NC = C::BQ / 32;   // 32-column TMEM loads per buffer
            uint32_t sv[NC][32], dv[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                tmem_ld_x32(tS + 32 * c, sv[c]);
                tmem_ld_x32(tP + 32 * c, dv[c]);
            }
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                reg_fence_x32(sv[c]);
                reg_fence_x32(dv[c]);
            }
            const float *lds = reinterpret_cast<const float *>(sb + C::LD_OFF + s * 512);   // -L*log2e, -D
            // causal: query columns c < key - q0 cannot see this key; where a sub-tile
            // has such columns, S^T is set to -inf first (P = 0, dS = 0)
            const int first_visible = key - q0;
            if (CAUSAL && __any_sync(0xffffffffu, first_visible > 0)) {
#pragma unroll
                for (int c = 0; c < C::BQ; ++c)
                    if (c < first_visible) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            uint32_t pp[C::BQ / 2], dsp[C::BQ / 2];
            uint32_t ppl[X3 ? C::BQ / 2 : 1], dspl[X3 ? C::BQ / 2 : 1];   // X3: the bf16 residuals
#pragma unroll
            for (int i = 0; i < C::BQ / 4; ++i) {
                const float4 nl = *reinterpret_cast<const float4 *>(lds + 4 * i);
                const float4 nd = *reinterpret_cast<const float4 *>(lds + 64 + 4 * i);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = 4 * i + 2 * h;
                    const float l0 = h ? nl.z : nl.x, l1 = h ? nl.w : nl.y;
                    const float d0 = h ? nd.z : nd.x, d1 = h ? nd.w : nd.y;
                    float x0, x1, g0, g1;
                    tc::fma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]),
                             scale_log2, scale_log2, l0, l1);
                    const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
                    tc::add2(g0, g1, __uint_as_float(dv[c >> 5][c & 31]), __uint_as_float(dv[c >> 5][(c & 31) + 1]),
                             d0, d1);
                    tc::mul2(g0, g1, g0, g1, p0, p1);
                    pp[2 * i + h] = tc::pack_bf16(p0, p1);
                    dsp[2 * i + h] = tc::pack_bf16(g0, g1);
                    if constexpr (X3) {
                        ppl[2 * i + h] = tc::pack_bf16_residual(p0, p1, pp[2 * i + h]);
                        dspl[2 * i + h] = tc::pack_bf16_residual(g0, g1, dsp[2 * i + h]);
                    }
                }
            }
            if constexpr (C::BQ == 64) {
                tmem_st_x32(tS, pp);
                tmem_st_x32(tP, dsp);
                if constexpr (X3) {   // over S^T / dP^T columns 32..63, already read
                    tmem_st_x32(tS + 32, ppl);
                    tmem_st_x32(tP + 32, dspl);
                }
            } else {   // 32-query sub-tiles: 16 packed columns each, lo over columns 16..31
                tmem_st_x16(tS, pp);
                tmem_st_x16(tP, dsp);
                if constexpr (X3) {
                    tmem_st_x16(tS + 16, ppl);
                    tmem_st_x16(tP + 16, dspl);
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(p_full(t));
        }
        // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (rows = keys);
        // a split item's rank 1 leaves its partial sums for rank 0 to add
        tc::named_bar_sync(1, 256);
        bool fine = !*abort_flag;
        // the last sub-tile's stage release means every MMA has completed (they run in order)
        if (fine && n > 0) fine = W.wait(q_empty((n - 1) % C::STAGES), ((n - 1) / C::STAGES) & 1);
        fine = __all_sync(0xffffffffu, fine);
        if (fine && n > 0) tc::fence_after_sync();
        __nv_bfloat16 *dst;
        if constexpr (VIEW4)
            dst = t == 0 ? dV + fa_row_offset(sdv, tc::opaque(H), bh, key) : dK + fa_row_offset(sdk, tc::opaque(H), bh, key);
        else
            dst = (t == 0 ? dV : dK) + ((size_t)bh * Nk + key) * D;
        const float mul = t == 0 ? 1.f : scale;
        const uint32_t tA = tmem + lane_base + (t == 0 ? C::DV_COL : C::DK_COL);
        // Split items: each rank finalises one tensor (rank 0 dV, rank 1 dK) and sends
        // its partial of the other into the peer's shared memory with remote stores
        // (streamed, no round trip per access), once the peer's own MMAs are done
        // and its stages are free; the peer adds it to its own accumulator.
        const bool mine = SPLIT == 1 || t == (int)rank;
        const uint32_t peer_free = base + C::PEER_BAR_OFF, peer_ready = peer_free + 8;
        const uint32_t part = base + C::PART_OFF + r * C::PART_STRIDE;   // partial row received here
        if constexpr (SPLIT > 1) tc::mbar_arrive_remote(tc::map_to_rank(peer_free, rank ^ 1u));
        bool merge = false;
        if (SPLIT > 1 && !mine) {
            const bool dst_ok = tc::wait_peer(peer_free, &g_fa_bwd_status, 2u);
            const uint32_t rdst = tc::map_to_rank(part, rank ^ 1u);
#pragma unroll
            for (int c = 0; c < C::OW / 32; ++c) {
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (dst_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        tc::st_cluster_v4(rdst + 128 * c + 16 * i, a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
                }
            }
            tc::mbar_arrive_remote(tc::map_to_rank(peer_ready, rank ^ 1u));   // release: the stores above
        } else if constexpr (X3 && !FOLD) {
            // D = 256: the accumulator columns are the output columns, written in fp32
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 2u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
            float *drow = static_cast<float *>(t == 0 ? dVv : dKv) +
                          fa_row_offset(t == 0 ? sdv : sdk, tc::opaque(H), bh, key);
#pragma unroll
            for (int c = 0; c < C::OW / 32; ++c) {
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(a[i]);
                    if (merge) x += pr[32 * c + i];
                    o[i] = x * mul;
                }
                if (fine && (SPLIT == 1 || merge) && key < Nk) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (32 * c + 4 * i < dv)
                            reinterpret_cast<float4 *>(drow + 32 * c)[i] =
                                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
        } else if constexpr (X3) {
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 2u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
            float *drow = static_cast<float *>(t == 0 ? dVv : dKv) +
                          fa_row_offset(t == 0 ? sdv : sdk, tc::opaque(H), bh, key);
            // accumulator chunk c (hi products) plus chunk c + 2 (hi x lo products): output columns 32c..32c+31
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t a[32], b[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tmem_ld_x32(tA + 32 * (c + 2), b);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                    reg_fence_x32(b);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = b[i] = 0u;
                }
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(a[i]) + __uint_as_float(b[i]);
                    if (merge) x += pr[32 * c + i] + pr[32 * (c + 2) + i];
                    o[i] = x * mul;
                }
                if (fine && (SPLIT == 1 || merge) && key < Nk) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (32 * c + 4 * i < dv)   // columns past the head dim are padding
                            reinterpret_cast<float4 *>(drow + 32 * c)[i] =
                                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
        } else {
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 2u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + 32 * c, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (merge) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 q = reinterpret_cast<const float4 *>(pr + 32 * c)[i];
                        a[4 * i + 0] = __float_as_uint(__uint_as_float(a[4 * i + 0]) + q.x);
                        a[4 * i + 1] = __float_as_uint(__uint_as_float(a[4 * i + 1]) + q.y);
                        a[4 * i + 2] = __float_as_uint(__uint_as_float(a[4 * i + 2]) + q.z);
                        a[4 * i + 3] = __float_as_uint(__uint_as_float(a[4 * i + 3]) + q.w);
                    }
                }
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = tc::pack_bf16(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
                if (fine && (SPLIT == 1 || merge) && key < Nk) {
                    uint4 *o = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (!VIEW4 || 32 * c + 8 * i < dv)   // columns past a head dim below 64 are padding
                            o[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ dQ (narrow)
template <int D>
struct DqNarrowCfg {
    static constexpr int BQ = 128;                 // queries per CTA (MMA M)
    static constexpr int BK = D == 256 ? 32 : 64;  // keys per sub-tile (32 for the 256-column split rows)
    static constexpr int STAGES = D == 256 ? 2 : D == 128 ? 4 : 8;    // see DkdvNarrowCfg
    static constexpr int OW = D == 256 ? 128 : D;                     // dQ accumulator columns
    using QT = TileShape<BQ, D>;
    using KT = TileShape<BK, D>;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t DO_OFF = Q_OFF + QT::BYTES;
    static constexpr uint32_t K_OFF = DO_OFF + QT::BYTES;                // stages of K sub-tiles
    static constexpr uint32_t V_OFF = K_OFF + STAGES * KT::BYTES;        // stages of V sub-tiles
    static constexpr uint32_t BAR_OFF = V_OFF + STAGES * KT::BYTES;
    // q_full, kv_full[S], kv_empty[S], sd_full[2], p_full[2], mma_done[2], drain
    static constexpr int NBAR = 1 + 2 * STAGES + 6 + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t PEER_BAR_OFF = MISC_OFF + 16;
    static constexpr uint32_t SMEM_BYTES = (PEER_BAR_OFF + 16 + 1024 > 120u * 1024u ? PEER_BAR_OFF + 16 + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // split items: rank 1's partial dQ (fp32) over the K/V rings
    // (the 256-column layout, never split, would need the Q and dO tiles' room as well)
    static constexpr uint32_t PART_STRIDE = (OW + 4) * 4;
    static constexpr uint32_t PART_OFF = D == 256 ? 0 : K_OFF;
    static_assert(PART_OFF + 128 * PART_STRIDE <= BAR_OFF, "partial fits the rings");
    // TMEM: S_t [128t, 128t+BK), dP_t [128t+64, 128t+64+BK), dQ [256, 256+OW)
    static constexpr uint32_t DQ_COL = 256;
};

// one dQ work item: query tile qt of batch*head bh (a half of its keys when SPLIT = 2).
// X3 as in dkdv_item_narrow: S and dP from three chunk pairs, dS split in TMEM
// (lo in the second 32 columns of its buffer), dQ = dShi [Khi | Klo] + dSlo Khi,
// output column c = accumulator column c plus 64 + c, written in fp32.
template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool X3 = false>
__device__ __forceinline__ void dq_item_narrow(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                        const CUtensorMap &tmdO, const float *__restrict__ Lp,
                                        const float *__restrict__ Dp, void *__restrict__ dQv, int Nq, int Nk,
                                        int qt, int bh, int H, int dv, const FaStrides &sdq, float scale,
                                        float scale_log2,
                                        uint32_t wait_limit) {
    static_assert(!X3 || ((D == 128 || D == 256) && !VIEW4), "split fp32 operands: 128- or 256-column copies");
    static_assert(X3 || D <= 128, "the 256-column layout holds split pairs only");
    using C = DqNarrowCfg<D>;
    constexpr bool FOLD = X3 && D == 128;   // outputs folded from [hi | lo] accumulator columns
    __nv_bfloat16 *dQ = static_cast<__nv_bfloat16 *>(dQv);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t rank = SPLIT > 1 ? tc::cluster_rank() : 0u;
    const int q0 = qt * C::BQ;
    const int kend = CAUSAL ? min(Nk, q0 + C::BQ) : Nk;
    const int n_all = (kend + C::BK - 1) / C::BK;
    // this CTA's key sub-tiles [jb, jb + n): all of them, or one half of a split item
    const int n_half = SPLIT > 1 ? (n_all + 1) / 2 : n_all;
    const int jb = rank == 0 ? 0 : n_half;
    const int n = rank == 0 ? n_half : n_all - n_half;
    const int nqp = padded_rows(Nq);

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t q_full = bar(0);
    auto kv_full = [&](int s) { return bar(1 + s); };
    auto kv_empty = [&](int s) { return bar(1 + C::STAGES + s); };
    auto sd_full = [&](int t) { return bar(1 + 2 * C::STAGES + t); };
    auto p_full = [&](int t) { return bar(3 + 2 * C::STAGES + t); };
    auto mma_done = [&](int t) { return bar(5 + 2 * C::STAGES + t); };
    const uint32_t drain = bar(7 + 2 * C::STAGES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(kv_full(s), 1);
            tc::mbar_init(kv_empty(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(sd_full(t), 1);
            tc::mbar_init(p_full(t), 128);
            tc::mbar_init(mma_done(t), 1);
        }
        tc::mbar_init(drain, 1);
        if (SPLIT > 1) {
            tc::mbar_init(base + C::PEER_BAR_OFF, 256);       // peer_free: the peer's 256 element-wise threads
            tc::mbar_init(base + C::PEER_BAR_OFF + 8, 128);   // peer_ready: the peer's 128 senders
        }
        *abort_flag = 0u;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (SPLIT > 1) tc::cluster_sync_all();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const tc::Waiter W{abort_flag, &g_fa_bwd_status, wait_limit, 4u};

    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmK);
            tc::tma_prefetch_desc(&tmV);
            const bool q_ok = tc::in_bounds(q0 < Nq, &g_fa_bwd_status, abort_flag);
            if (q_ok) {
                tc::mbar_arrive_expect_tx(q_full, 2 * C::QT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + c * C::QT::CHUNK, &tmQ, q_full, c * 64, q0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::DO_OFF + c * C::QT::CHUNK, &tmdO, q_full, c * 64, q0, bh, H);
                }
            }
            int issued = 0;
            for (int j = 0; q_ok && j < n; ++j) {
                const int s = j % C::STAGES;
                if (!W.wait(kv_empty(s), ((j / C::STAGES) & 1) ^ 1u)) break;
                // debug build: a key sub-tile past the keys, or wholly above the diagonal, is never loaded
                const int kj = (jb + j) * C::BK;
                if (!tc::in_bounds(kj < Nk && (!CAUSAL || kj <= q0 + C::BQ - 1), &g_fa_bwd_status, abort_flag)) break;
                tc::mbar_arrive_expect_tx(kv_full(s), 2 * C::KT::BYTES);
                for (int c = 0; c < D / 64; ++c) {
                    tc::tma_load_rows<VIEW4>(base + C::K_OFF + s * C::KT::BYTES + c * C::KT::CHUNK, &tmK, kv_full(s), c * 64,
                                    (jb + j) * C::BK, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::V_OFF + s * C::KT::BYTES + c * C::KT::CHUNK, &tmV, kv_full(s), c * 64,
                                    (jb + j) * C::BK, bh, H);
                }
                issued = j + 1;
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_bwd_rows[1], (unsigned long long)issued * C::BK);
            if (*abort_flag) {
                for (int j = issued - 1; j >= 0 && j >= issued - C::STAGES; --j) {
                    const int s = j % C::STAGES;
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(kv_full(s), (j / C::STAGES) & 1); ++i) {
                    }
                }
                if (q_ok)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full, 0); ++i) {
                    }
            }
        }
    } else if (warp == 1) {
        // whole warp in the loop (uniform descriptors), one elected lane issues
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc_s = tc::idesc_bf16(128, C::BK, false, false);
        constexpr uint32_t idesc_g = tc::idesc_bf16(128, C::OW, false, true);
        constexpr uint32_t idesc_g_hi = tc::idesc_bf16(128, 64, false, true);   // X3, D = 128: dSlo Khi
        const uint64_t qd = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);      // A of S, K-major
        const uint64_t od = tc::sdesc_sw128(base + C::DO_OFF, 16, 1024);     // A of dP
        const uint64_t kk_ = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);    // B of S, K-major, stage 0
        const uint64_t vk = tc::sdesc_sw128(base + C::V_OFF, 16, 1024);     // B of dP
        const uint64_t km = tc::sdesc_sw128(base + C::K_OFF, C::KT::CHUNK, 1024);   // B of dQ, MN-major
        bool ok = __all_sync(0xffffffffu, W.wait(q_full, 0));
        auto grads = [&](int j) -> bool {   // dQ += dS K_j
            const int s = j % C::STAGES, t = j & 1, k = j >> 1;
            if (!__all_sync(0xffffffffu, W.wait(p_full(t), k & 1))) return false;
            tc::fence_after_sync();
            if (leader) {
                const uint32_t st = (s * C::KT::BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    tc::mma_ts(tmem + C::DQ_COL, tmem + 128 * t + 64 + kk * 8, km + st + kk * 128, idesc_g,
                               (j > 0 || kk > 0) ? 1u : 0u);
                if constexpr (FOLD) {
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc::mma_ts(tmem + C::DQ_COL, tmem + 128 * t + 64 + C::BK / 2 + kk * 8, km + st + kk * 128,
                                   idesc_g_hi, 1u);
                } else if constexpr (X3) {
                    // D = 256: dShi Klo (chunks 2, 3), then dSlo Khi, into the same dQ columns
                    const uint32_t lo = (2 * C::KT::CHUNK) >> 4;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc::mma_ts(tmem + C::DQ_COL, tmem + 128 * t + 64 + kk * 8, km + st + lo + kk * 128, idesc_g, 1u);
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        tc::mma_ts(tmem + C::DQ_COL, tmem + 128 * t + 64 + C::BK / 2 + kk * 8, km + st + kk * 128,
                                   idesc_g, 1u);
                }
                tc::mma_commit(kv_empty(s));   // sub-tile j done: its stage is free
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; ok && j < n; ++j) {
            const int s = j % C::STAGES, t = j & 1;
            if (!(ok = __all_sync(0xffffffffu, W.wait(kv_full(s), (j / C::STAGES) & 1)))) break;
            if (leader) {
                const uint32_t st = (s * C::KT::BYTES) >> 4;
                // S = Q K^T and dP = dO V^T, interleaved, four k-steps per chunk pair: (c, c)
                // for each chunk, or X3: (hi, hi), (hi, lo), (lo, hi) for each of the HC hi
                // chunks (the lo chunks follow them)
                constexpr int HC = X3 ? D / 128 : 1;
                constexpr int PAIRS = X3 ? 3 * HC : D / 64;
                auto pair = [&](int pr) {
                    int ca = pr, cb = pr;
                    if constexpr (X3) {
                        const int grp = pr / HC, c = pr % HC;
                        ca = grp == 2 ? HC + c : c;
                        cb = grp == 1 ? HC + c : c;
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const uint32_t oa = (ca * C::QT::CHUNK + k4 * 32) >> 4;
                        const uint32_t ob = (cb * C::KT::CHUNK + k4 * 32) >> 4;
                        const uint32_t acc = (pr > 0 || k4 > 0) ? 1u : 0u;
                        tc::mma_ss(tmem + 128 * t, qd + oa, kk_ + st + ob, idesc_s, acc);
                        tc::mma_ss(tmem + 128 * t + 64, od + oa, vk + st + ob, idesc_s, acc);
                    }
                };
                if constexpr (PAIRS <= 3) {
#pragma unroll
                    for (int pr = 0; pr < PAIRS; ++pr) pair(pr);
                } else {
#pragma unroll 1
                    for (int pr = 0; pr < PAIRS; ++pr) pair(pr);
                }
                tc::mma_commit(sd_full(t));
            }
            __syncwarp();
            if (j >= 1) ok = grads(j - 1);
        }
        if (ok && n > 0) ok = grads(n - 1);
        if (!ok && leader) {
            tc::mma_commit(drain);
            for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
            }
        }
        __syncwarp();
    }
    } else {
        tc::regs_inc<224>();
        const int t = (warp - 4) >> 2;
        const int r = ((warp & 3) << 5) + lane;
        const int row = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + 128 * t;
        const uint32_t tP = tS + 64;
        const float nlrow = Lp[(size_t)bh * nqp + row];     // -L*log2e (-inf on padding rows)
        const float ndrow = Dp[(size_t)bh * nqp + row];     // -D
        const int nt = (n - t + 1) >> 1;
        for (int k = 0; k < nt; ++k) {
            const int j = 2 * k + t;
            const int kb0 = (jb + j) * C::BK;
            bool ok = W.wait(sd_full(t), k & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            constexpr int NC = C::BK / 32;   // 32-column TMEM loads per buffer
            uint32_t sv[NC][32], dv[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                tmem_ld_x32(tS + 32 * c, sv[c]);
                tmem_ld_x32(tP + 32 * c, dv[c]);
            }
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                reg_fence_x32(sv[c]);
                reg_fence_x32(dv[c]);
            }
            // key columns past the diagonal (causal) or past Nk: S set to -inf first (P = 0, dS = 0)
            const int lim = min(Nk - 1, CAUSAL ? row : Nk - 1) - kb0;   // last visible key column
            if (__any_sync(0xffffffffu, lim < C::BK - 1)) {
#pragma unroll
                for (int c = 0; c < C::BK; ++c)
                    if (c > lim) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            uint32_t dsp[C::BK / 2];
            uint32_t dspl[X3 ? C::BK / 2 : 1];   // X3: the bf16 residuals
#pragma unroll
            for (int i = 0; i < C::BK / 2; ++i) {
                const int c = 2 * i;
                float x0, x1, g0, g1;
                tc::fma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]),
                         scale_log2, scale_log2, nlrow, nlrow);
                const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
                tc::add2(g0, g1, __uint_as_float(dv[c >> 5][c & 31]), __uint_as_float(dv[c >> 5][(c & 31) + 1]),
                         ndrow, ndrow);
                tc::mul2(g0, g1, g0, g1, p0, p1);
                dsp[i] = tc::pack_bf16(g0, g1);
                if constexpr (X3) dspl[i] = tc::pack_bf16_residual(g0, g1, dsp[i]);
            }
            if constexpr (C::BK == 64) {
                tmem_st_x32(tP, dsp);
                if constexpr (X3) tmem_st_x32(tP + 32, dspl);   // over dP columns 32..63, already read
            } else {   // 32-key sub-tiles: 16 packed columns, lo over columns 16..31
                tmem_st_x16(tP, dsp);
                if constexpr (X3) tmem_st_x16(tP + 16, dspl);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(p_full(t));
        }
        tc::named_bar_sync(1, 256);
        bool fine = !*abort_flag;
        // the last sub-tile's stage release means every MMA has completed (they run in order)
        if (fine && n > 0) fine = W.wait(kv_empty((n - 1) % C::STAGES), ((n - 1) / C::STAGES) & 1);
        fine = __all_sync(0xffffffffu, fine);
        if (fine && n > 0) tc::fence_after_sync();
        __nv_bfloat16 *dst;
        if constexpr (VIEW4) dst = dQ + fa_row_offset(sdq, tc::opaque(H), bh, row);
        else dst = dQ + ((size_t)bh * Nq + row) * D;
        const uint32_t tA = tmem + lane_base + C::DQ_COL;
        // Split items: rank r finalises the columns of warpgroup r and sends its partial
        // of the other half into the peer's shared memory with remote stores, once the
        // peer's own MMAs are done and its stages are free.
        const bool mine = SPLIT == 1 || t == (int)rank;
        const uint32_t peer_free = base + C::PEER_BAR_OFF, peer_ready = peer_free + 8;
        const uint32_t part = base + C::PART_OFF + r * C::PART_STRIDE;   // half row received here
        if constexpr (SPLIT > 1) tc::mbar_arrive_remote(tc::map_to_rank(peer_free, rank ^ 1u));
        if (SPLIT > 1 && !mine) {
            const bool dst_ok = tc::wait_peer(peer_free, &g_fa_bwd_status, 4u);
            const uint32_t rdst = tc::map_to_rank(part, rank ^ 1u);
#pragma unroll
            for (int c = 0; c < C::OW / 64; ++c) {
                const int col = FOLD ? t * 32 + 64 * c : t * (C::OW / 2) + 32 * c;
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + col, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (dst_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        tc::st_cluster_v4(rdst + 128 * c + 16 * i, a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
                }
            }
            tc::mbar_arrive_remote(tc::map_to_rank(peer_ready, rank ^ 1u));   // release: the stores above
        } else if constexpr (X3 && !FOLD) {
            // D = 256: this warpgroup's output columns [64t, 64t + 64) are its accumulator columns
            bool merge = false;
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 4u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
            float *drow = static_cast<float *>(dQv) + fa_row_offset(sdq, tc::opaque(H), bh, row);
#pragma unroll
            for (int c = 0; c < C::OW / 64; ++c) {
                const int col = t * (C::OW / 2) + 32 * c;
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + col, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(a[i]);
                    if (merge) x += pr[32 * c + i];
                    o[i] = x * scale;
                }
                if (fine && (SPLIT == 1 || merge) && row < Nq) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (col + 4 * i < dv)
                            reinterpret_cast<float4 *>(drow + col)[i] =
                                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
        } else if constexpr (X3) {
            // this warpgroup's output columns [32t, 32t + 32): accumulator columns 32t + i and 64 + 32t + i
            bool merge = false;
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 4u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
            uint32_t a[32], b[32];
            if (fine && n > 0) {
                tmem_ld_x32(tA + 32 * t, a);
                tmem_ld_x32(tA + 64 + 32 * t, b);
                tc::tmem_ld_wait();
                reg_fence_x32(a);
                reg_fence_x32(b);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) a[i] = b[i] = 0u;
            }
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float x = __uint_as_float(a[i]) + __uint_as_float(b[i]);
                if (merge) x += pr[i] + pr[32 + i];
                o[i] = x * scale;
            }
            if (fine && (SPLIT == 1 || merge) && row < Nq) {
                float *drow = static_cast<float *>(dQv) + fa_row_offset(sdq, tc::opaque(H), bh, row) + 32 * t;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (32 * t + 4 * i < dv)   // columns past the head dim are padding
                        reinterpret_cast<float4 *>(drow)[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
        } else {
            bool merge = false;
            if constexpr (SPLIT > 1) merge = tc::wait_peer(peer_ready, &g_fa_bwd_status, 4u);
            const float *pr = reinterpret_cast<const float *>(sb + (part - base));
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int col = t * (D / 2) + 32 * c;
                uint32_t a[32];
                if (fine && n > 0) {
                    tmem_ld_x32(tA + col, a);
                    tc::tmem_ld_wait();
                    reg_fence_x32(a);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
                if (merge) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 q = reinterpret_cast<const float4 *>(pr + 32 * c)[i];
                        a[4 * i + 0] = __float_as_uint(__uint_as_float(a[4 * i + 0]) + q.x);
                        a[4 * i + 1] = __float_as_uint(__uint_as_float(a[4 * i + 1]) + q.y);
                        a[4 * i + 2] = __float_as_uint(__uint_as_float(a[4 * i + 2]) + q.z);
                        a[4 * i + 3] = __float_as_uint(__uint_as_float(a[4 * i + 3]) + q.w);
                    }
                }
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = tc::pack_bf16(__uint_as_float(a[2 * i]) * scale, __uint_as_float(a[2 * i + 1]) * scale);
                if (fine && (SPLIT == 1 || merge) && row < Nq) {
                    uint4 *o = reinterpret_cast<uint4 *>(dst + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (!VIEW4 || col + 8 * i < dv)   // columns past a head dim below 64 are padding
                            o[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ================================================================== persistent dK/dV items (d = 64, dQ by reduction)
// One CTA per SM walks a snake-ordered list of dK/dV items (longest first), with
// the work of the 128-wide d = 64 items and dQ formed by reduction.  Unlike the
// one-item-per-CTA launch, nothing is set up per item: TMEM is allocated once,
// the barriers are initialised once and their phases run on across items (the
// query sub-tiles are numbered over all of the CTA's items), and the register
// split is set once.  Between items the next item's K/V tile loads once the
// previous item's MMAs are done, and its first S^T / dP^T MMAs start while the
// element-wise warps still store the previous item's dK and dV.
struct DkdvPersistCfg : DkdvWideCfg<64, true> {
    using Base = DkdvWideCfg<64, true>;
    // the base barriers, then kv_empty (an item's MMAs are done: K/V may be
    // reloaded), acc_free (the epilogue has read dV / dK from TMEM) and ds_free[2]
    // (the TMA store of a warpgroup's dV or dK rows has read them out of the dS^T tile)
    static constexpr int NBAR = Base::NBAR + 4;
    static constexpr uint32_t MISC_OFF = Base::BAR_OFF + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = (MISC_OFF + 16 + 1024 > 120u * 1024u ? MISC_OFF + 16 + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <bool CAUSAL, bool VIEW4>
__global__ void __launch_bounds__(NTHREADS, 1)
    fa_bwd_red_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                                 const __grid_constant__ CUtensorMap dqa, const __grid_constant__ CUtensorMap tmdK,
                                 const __grid_constant__ CUtensorMap tmdV, const float *__restrict__ Lp,
                                 const float *__restrict__ Dp, __nv_bfloat16 *__restrict__ dK,
                                 __nv_bfloat16 *__restrict__ dV, int Nq, int Nk, int BH, int k_tiles, float scale,
                                 float scale_log2, uint32_t wait_limit, int H, int dv, FaStrides sdk, FaStrides sdv) {
    constexpr int D = 64;
    using C = DkdvPersistCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    tc::pdl_launch_dependents();

    const int nqp = padded_rows(Nq);
    const int i_end = (Nq + C::BQ - 1) / C::BQ;
    const int num_items = k_tiles * BH;
    const int G = (int)gridDim.x, cb = (int)blockIdx.x;
    // item r of this CTA (snake order over the longest-first list): key tile kt of
    // batch*head bh, with query sub-tiles [first, first + n)
    auto item_of = [&](int r, int &kt, int &bh, int &first, int &n) -> bool {
        const int u = r * G + ((r & 1) ? G - 1 - cb : cb);
        if (u >= num_items) return false;
        const int rr = u / BH;
        kt = CAUSAL ? rr : k_tiles - 1 - rr;   // causal: the first key tiles see the most queries
        bh = u % BH;
        first = CAUSAL ? kt : 0;
        n = i_end > first ? i_end - first : 0;
        return true;
    };

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t kv_full = bar(0);
    auto q_full = [&](int s) { return bar(1 + s); };
    auto q_empty = [&](int s) { return bar(1 + C::STAGES + s); };
    const uint32_t sd_full = bar(1 + 2 * C::STAGES);
    const uint32_t sd_free = bar(2 + 2 * C::STAGES);
    const uint32_t p_full = bar(3 + 2 * C::STAGES);
    const uint32_t drain = bar(4 + 2 * C::STAGES);
    const uint32_t dq_staged = bar(5 + 2 * C::STAGES);
    const uint32_t dq_free = bar(6 + 2 * C::STAGES);
    auto ep_staged = [&](int t) { return bar(7 + 2 * C::STAGES + t); };   // a warpgroup's dV / dK rows staged
    const uint32_t kv_empty = bar(9 + 2 * C::STAGES);
    const uint32_t acc_free = bar(10 + 2 * C::STAGES);
    auto ds_free = [&](int t) { return bar(11 + 2 * C::STAGES + t); };    // ... and read out by their TMA store
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(kv_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(q_full(s), 1);
            tc::mbar_init(q_empty(s), 1);
        }
        tc::mbar_init(sd_full, 1);
        tc::mbar_init(sd_free, 256);
        tc::mbar_init(p_full, 256);
        tc::mbar_init(drain, 1);
        tc::mbar_init(dq_staged, 256);
        tc::mbar_init(dq_free, 1);
        tc::mbar_init(kv_empty, 1);
        tc::mbar_init(acc_free, 256);
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(ep_staged(t), 128);
            tc::mbar_init(ds_free(t), 1);
        }
        *abort_flag = 0u;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    tc::pdl_wait();   // D and L staged by the preprocessing (or the forward) are complete
    const tc::Waiter W{abort_flag, &g_fa_bwd_status, wait_limit, 2u};

    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmQ);
            tc::tma_prefetch_desc(&tmdO);
            int g = 0, issued = 0, kt, bh, first, n;
            int kv_r = -1;   // the last item whose K/V load was issued
            for (int r = 0; item_of(r, kt, bh, first, n); ++r) {
                // the K/V buffer is refilled once the previous item's MMAs have completed
                if (r > 0 && !W.wait(kv_empty, (r - 1) & 1)) break;
                const int k0 = kt * C::BK;
                if (!tc::in_bounds(k0 < Nk && bh < BH, &g_fa_bwd_status, abort_flag)) break;
                if (n > 0) {
                    tc::mbar_arrive_expect_tx(kv_full, 2 * C::KT::BYTES);
                    tc::tma_load_rows<VIEW4>(base + C::K_OFF, &tmK, kv_full, 0, k0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::V_OFF, &tmV, kv_full, 0, k0, bh, H);
                    kv_r = r;
                } else {
                    tc::mbar_arrive(kv_full);   // an item with no queries still moves the phase on
                }
                bool ok = true;
                for (int it = 0; it < n; ++it, ++g) {
                    const int s = g % C::STAGES;
                    if (!(ok = W.wait(q_empty(s), ((g / C::STAGES) & 1) ^ 1u))) break;
                    const int q0 = (first + it) * C::BQ;
                    if (!(ok = tc::in_bounds(q0 < Nq && (!CAUSAL || q0 + C::BQ - 1 >= k0), &g_fa_bwd_status,
                                             abort_flag)))
                        break;
                    tc::mbar_arrive_expect_tx(q_full(s), 2 * C::QT::BYTES + 1024);
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + s * C::QT::BYTES, &tmQ, q_full(s), 0, q0, bh, H);
                    tc::tma_load_rows<VIEW4>(base + C::DO_OFF + s * C::QT::BYTES, &tmdO, q_full(s), 0, q0, bh, H);
                    const size_t off = (size_t)bh * nqp + q0;
                    tc::bulk_load(base + C::LD_OFF + s * 1024, Lp + off, 512, q_full(s));
                    tc::bulk_load(base + C::LD_OFF + s * 1024 + 512, Dp + off, 512, q_full(s));
                    issued = g + 1;
                }
                if (!ok) break;
                if constexpr (tc::kDebug) atomicAdd(&g_fa_bwd_rows[0], (unsigned long long)n * C::BQ);
            }
            if (*abort_flag) {
                for (int gg = issued - 1; gg >= 0 && gg >= issued - C::STAGES; --gg)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full(gg % C::STAGES), (gg / C::STAGES) & 1);
                         ++i) {
                    }
                // the last K/V load lands before the CTA may exit
                if (kv_r >= 0)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(kv_full, kv_r & 1); ++i) {
                    }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ dQ reduction
        if (lane == 0) {
            int g = 0, kt, bh, first, n;
            bool ok = true;
            for (int r = 0; ok && item_of(r, kt, bh, first, n); ++r) {
                for (int it = 0; it < n; ++it, ++g) {
                    if (!(ok = W.wait(dq_staged, g & 1))) break;
                    const int q0 = (first + it) * C::BQ;
                    if (!(ok = tc::in_bounds(q0 + C::BQ <= nqp, &g_fa_bwd_status, abort_flag))) break;
#pragma unroll
                    for (int x = 0; x < D / 32; ++x)
                        tc::tma_reduce_add_3d(&dqa, base + C::DQS_OFF + x * C::DQS_BOX, 32 * x, q0, bh);
                    tc::bulk_commit_group();
                    tc::bulk_wait_read_all();
                    tc::mbar_arrive(dq_free);
                }
            }
            tc::bulk_wait_all();
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ dV / dK stores
        // each item's rows, staged by the element-wise warpgroups in their halves of
        // the dS^T tile (128-byte swizzled), go out as two TMA stores (rows past Nk
        // are not written); the halves are handed back once the stores have read them
        if (lane == 0) {
            int kt, bh, first, n;
            for (int r = 0; item_of(r, kt, bh, first, n); ++r) {
                bool ok = true;
                for (int t = 0; ok && t < 2; ++t) {
                    if (!(ok = W.wait(ep_staged(t), r & 1))) break;
                    tc::tma_store_rows<VIEW4>(t == 0 ? &tmdV : &tmdK, base + C::DS_OFF + t * (128 * 128), 0,
                                              kt * C::BK, bh, H);
                }
                tc::bulk_commit_group();
                tc::bulk_wait_read_all();
                if (!ok) break;
                tc::mbar_arrive(ds_free(0));
                tc::mbar_arrive(ds_free(1));
            }
            tc::bulk_wait_all();   // the stores have landed before the CTA exits
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc_s = tc::idesc_bf16(128, C::BQ, false, false);
        constexpr uint32_t idesc_g = tc::idesc_bf16(128, D, false, true);
        constexpr uint32_t idesc_q = tc::idesc_bf16(128, D, true, true);
        const uint64_t kd = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);
        const uint64_t vd = tc::sdesc_sw128(base + C::V_OFF, 16, 1024);
        const uint64_t qk = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);
        const uint64_t gk = tc::sdesc_sw128(base + C::DO_OFF, 16, 1024);
        const uint64_t qm = tc::sdesc_sw128(base + C::Q_OFF, C::QT::CHUNK, 1024);
        const uint64_t gm = tc::sdesc_sw128(base + C::DO_OFF, C::QT::CHUNK, 1024);
        const uint64_t dsk = tc::sdesc_sw128(base + C::DS_OFF, 16, 1024);
        const uint64_t dsm = tc::sdesc_sw128(base + C::DS_OFF, 128 * 128, 1024);
        const uint64_t km = tc::sdesc_sw128(base + C::K_OFF, C::KT::CHUNK, 1024);
        // S^T = K Q^T and dP^T = V dO^T of global sub-tile gg (its S^T / dP^T columns
        // must have been read for sub-tile gg-1 first)
        auto sdp = [&](int gg) -> bool {
            const int s = gg % C::STAGES;
            const bool ready = gg > 0 ? W.wait2(sd_free, (gg - 1) & 1, q_full(s), (gg / C::STAGES) & 1)
                                      : W.wait(q_full(s), (gg / C::STAGES) & 1);
            if (!__all_sync(0xffffffffu, ready)) return false;
            if (leader) {
                const uint32_t st = (s * C::QT::BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + C::ST_COL, kd + oa, qk + st + oa, idesc_s, kk > 0 ? 1u : 0u);
                    tc::mma_ss(tmem + C::DP_COL, vd + oa, gk + st + oa, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(sd_full);
            }
            __syncwarp();
            return true;
        };
        // dV += P^T dO, dK += dS^T Q (fresh at an item's first sub-tile), dQ partial = dS K
        auto grads = [&](int gg, bool fresh) -> bool {
            const int s = gg % C::STAGES;
            if (!__all_sync(0xffffffffu, W.wait(p_full, gg & 1))) return false;
            tc::fence_after_sync();
            if (leader) {
                const uint32_t st = (s * C::QT::BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < C::BQ / 16; ++kk) {
                    const uint32_t acc = (!fresh || kk > 0) ? 1u : 0u;
                    tc::mma_ts(tmem + C::DV_COL, tmem + C::PT_COL + kk * 8, gm + st + kk * 128, idesc_g, acc);
                    tc::mma_ss(tmem + C::DK_COL, dsk + (((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4), qm + st + kk * 128,
                               idesc_g, acc);
                }
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    tc::mma_ss(tmem + C::DQ_COL, dsm + kk * 128, km + kk * 128, idesc_q, kk > 0 ? 1u : 0u);
                tc::mma_commit(q_empty(s));
            }
            __syncwarp();
            return true;
        };
        int g = 0, kt, bh, first, n;
        bool ok = true;
        for (int r = 0; ok && item_of(r, kt, bh, first, n); ++r) {
            if (!(ok = __all_sync(0xffffffffu, W.wait(kv_full, r & 1)))) break;
            if (n > 0) {
                if (!(ok = sdp(g))) break;
                for (int it = 0; ok && it < n; ++it) {
                    if (it + 1 < n && !(ok = sdp(g + it + 1))) break;
                    // dV / dK of the previous item must have been read before the first
                    // gradient MMAs of this one overwrite them
                    if (it == 0 && r > 0 && !(ok = __all_sync(0xffffffffu, W.wait(acc_free, (r - 1) & 1)))) break;
                    ok = grads(g + it, it == 0);
                }
            }
            if (ok && leader) tc::mma_commit(kv_empty);   // this item's MMAs are done with K and V
            __syncwarp();
            g += n;
        }
        if (!ok && leader) {
            tc::mma_commit(drain);
            for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
            }
        }
        __syncwarp();
    }
    } else {
        tc::regs_inc<224>();
        // ------------------------------------------------------------ element-wise warpgroups
        const int t = (warp - 4) >> 2;                       // query columns [64t, 64t + 64)
        const int rrow = ((warp & 3) << 5) + lane;           // key row within the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::ST_COL + 64 * t;
        const uint32_t tD = tmem + lane_base + C::DP_COL + 64 * t;
        const uint32_t tPT = tmem + lane_base + C::PT_COL + 32 * t;
        const uint32_t tDQ = tmem + lane_base + C::DQ_COL + 32 * t;
        auto stage_dq = [&](int gg, const uint32_t (&v)[32]) -> bool {
            if (gg > 0 && !__all_sync(0xffffffffu, W.wait(dq_free, (gg - 1) & 1))) return false;
            uint8_t *row = sb + C::DQS_OFF + t * C::DQS_BOX + rrow * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4 *>(row + ((u ^ (rrow & 7)) << 4)) =
                    make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(dq_staged);
            return true;
        };
        int g = 0, kt, bh, first, n;
        bool alive = true;
        for (int r = 0; item_of(r, kt, bh, first, n); ++r) {
            const int k0 = kt * C::BK, key = k0 + rrow;
            for (int it = 0; alive && it < n; ++it) {
                const int gg = g + it, s = gg % C::STAGES;
                const int qc = (first + it) * C::BQ + 64 * t;
                bool ok = W.wait2(sd_full, gg & 1, q_full(s), (gg / C::STAGES) & 1);
                if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
                tc::fence_after_sync();
                uint32_t sv[2][32], dv_[2][32];
                tmem_ld_x32(tS, sv[0]);
                tmem_ld_x32(tS + 32, sv[1]);
                tmem_ld_x32(tD, dv_[0]);
                tmem_ld_x32(tD + 32, dv_[1]);
                tc::tmem_ld_wait();
                reg_fence_x32(sv[0]);
                reg_fence_x32(sv[1]);
                reg_fence_x32(dv_[0]);
                reg_fence_x32(dv_[1]);
                tc::fence_before_sync();
                tc::mbar_arrive(sd_free);
                const float *lds = reinterpret_cast<const float *>(sb + C::LD_OFF + s * 1024) + 64 * t;
                const int first_visible = key - qc;
                if (CAUSAL && __any_sync(0xffffffffu, first_visible > 0)) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c < first_visible) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
                // P^T and dS^T in two halves of 16 columns each: the first half is stored
                // while the second is computed
                uint32_t pp[32], dsp[32];
                auto half = [&](int hh) {
#pragma unroll
                    for (int i = 8 * hh; i < 8 * hh + 8; ++i) {
                        const float4 nl = *reinterpret_cast<const float4 *>(lds + 4 * i);
                        const float4 nd = *reinterpret_cast<const float4 *>(lds + 128 + 4 * i);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int c = 4 * i + 2 * h;
                            const float l0 = h ? nl.z : nl.x, l1 = h ? nl.w : nl.y;
                            const float d0 = h ? nd.z : nd.x, d1 = h ? nd.w : nd.y;
                            float x0, x1, g0, g1;
                            tc::fma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]),
                                     __uint_as_float(sv[c >> 5][(c & 31) + 1]), scale_log2, scale_log2, l0, l1);
                            const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
                            tc::add2(g0, g1, __uint_as_float(dv_[c >> 5][c & 31]),
                                     __uint_as_float(dv_[c >> 5][(c & 31) + 1]), d0, d1);
                            tc::mul2(g0, g1, g0, g1, p0, p1);
                            pp[2 * i + h] = tc::pack_bf16(p0, p1);
                            dsp[2 * i + h] = tc::pack_bf16(g0, g1);
                        }
                    }
                };
                auto store_half = [&](int hh) {
                    const uint32_t(&ph)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pp[16 * hh]);
                    tmem_st_x16(tPT + 16 * hh, ph);
                    uint8_t *row = sb + C::DS_OFF + t * (128 * 128) + rrow * 128;
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu)
                        *reinterpret_cast<uint4 *>(row + (((4 * hh + uu) ^ (rrow & 7)) << 4)) =
                            make_uint4(dsp[16 * hh + 4 * uu], dsp[16 * hh + 4 * uu + 1], dsp[16 * hh + 4 * uu + 2],
                                       dsp[16 * hh + 4 * uu + 3]);
                };
                half(0);
                uint32_t dq[32];
                if (it > 0) {
                    // the previous sub-tile's MMAs read P^T and dS and wrote its dQ partial
                    ok = W.wait(q_empty((gg - 1) % C::STAGES), ((gg - 1) / C::STAGES) & 1);
                    if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
                    tc::fence_after_sync();
                    tmem_ld_x32(tDQ, dq);
                } else if (r > 0) {
                    // the previous item's dV / dK rows left this warpgroup's dS^T half
                    if (!__all_sync(0xffffffffu, W.wait(ds_free(t), (r - 1) & 1))) { alive = false; break; }
                }
                store_half(0);
                half(1);
                store_half(1);
                tc::tmem_st_wait();
                if (it > 0) {
                    tc::tmem_ld_wait();
                    reg_fence_x32(dq);
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                tc::mbar_arrive(p_full);
                if (it > 0 && !stage_dq(gg - 1, dq)) { alive = false; break; }
            }
            // ---- item epilogue: the last dQ partial, then dV (warpgroup 0) / dK (1)
            bool fine = alive && !*abort_flag;
            if (fine && n > 0) fine = W.wait(q_empty((g + n - 1) % C::STAGES), ((g + n - 1) / C::STAGES) & 1);
            fine = __all_sync(0xffffffffu, fine);
            if (fine && n > 0) {
                tc::fence_after_sync();
                uint32_t dq[32];
                tmem_ld_x32(tDQ, dq);
                tc::tmem_ld_wait();
                reg_fence_x32(dq);
                fine = stage_dq(g + n - 1, dq);
            }
            const float mul = t == 0 ? 1.f : scale;
            const uint32_t tA = tmem + lane_base + (t == 0 ? C::DV_COL : C::DK_COL);
            uint32_t a[2][32];
            if (fine && n > 0) {
                tmem_ld_x32(tA, a[0]);
                tmem_ld_x32(tA + 32, a[1]);
                tc::tmem_ld_wait();
                reg_fence_x32(a[0]);
                reg_fence_x32(a[1]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) a[0][i] = a[1][i] = 0u;
            }
            tc::fence_before_sync();
            tc::mbar_arrive(acc_free);   // dV / dK may be overwritten by the next item
            // the row, in bf16, into this warpgroup's half of the dS^T tile (free: the
            // item's MMAs are done, and an item without sub-tiles waits for the previous
            // item's store here), then warp 3 stores the tile
            bool stage = fine || n == 0;
            if (n == 0 && r > 0 && !__all_sync(0xffffffffu, W.wait(ds_free(t), (r - 1) & 1))) stage = false;
            if (!stage) alive = false;
            if (stage) {
                uint8_t *srow = sb + C::DS_OFF + t * (128 * 128) + rrow * 128;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[i] = tc::pack_bf16(__uint_as_float(a[c][2 * i]) * mul,
                                                  __uint_as_float(a[c][2 * i + 1]) * mul);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4 *>(srow + (((4 * c + i) ^ (rrow & 7)) << 4)) =
                            make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(ep_staged(t));
            }
            g += n;
            if (!fine && n > 0) alive = false;
            if (!alive) break;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Both gradient passes in one launch.  The two lists of work items (dK/dV per
// key tile, dQ per query tile; each longest first) are interleaved so that the
// long items of both start first and the short ones of both fill the end --
// one kernel tail instead of two, and the passes balance each other's load.
// RED: dK/dV items only, each adding its dQ partials into the fp32 accumulator
// behind dqa (no dQ items; a short kernel converts the accumulator afterwards).
template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool RED, bool X3 = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    fa_bwd_tc_kernel(const __grid_constant__ CUtensorMap qA, const __grid_constant__ CUtensorMap kA,
                     const __grid_constant__ CUtensorMap vA, const __grid_constant__ CUtensorMap dOA,
                     const __grid_constant__ CUtensorMap qB, const __grid_constant__ CUtensorMap kB,
                     const __grid_constant__ CUtensorMap vB, const __grid_constant__ CUtensorMap dOB,
                     const __grid_constant__ CUtensorMap dqa, const __grid_constant__ CUtensorMap tmdK,
                     const __grid_constant__ CUtensorMap tmdV, const float *__restrict__ Lp, const float *__restrict__ Dp,
                     void *__restrict__ dQ, void *__restrict__ dK, void *__restrict__ dV, int Nq, int Nk, int BH,
                     int k_tiles, int q_tiles, int n_kv_items, int n_q_items, float scale, float scale_log2,
                     uint32_t wait_limit, int H, int dv, FaStrides sdq, FaStrides sdk, FaStrides sdv) {
    tc::pdl_launch_dependents();
    tc::pdl_wait();   // D and L staged by the preprocessing kernel are complete
    const int item = blockIdx.x / SPLIT;
    const int both = min(n_kv_items, n_q_items);
    int role, idx;
    if (item < 2 * both) {
        role = item & 1;
        idx = item >> 1;
    } else {
        role = n_kv_items > n_q_items ? 0 : 1;
        idx = item - both;
    }
    const int bh = idx % BH;
    if (role == 0) {
        const int r = idx / BH;
        const int kt = CAUSAL ? r : k_tiles - 1 - r;    // causal: the first key tiles see the most queries
        if constexpr (D == 64)
            dkdv_item_wide<D, CAUSAL, SPLIT, VIEW4, RED>(qA, kA, vA, dOA, &dqa, &tmdK, &tmdV, Lp, Dp,
                                                         static_cast<__nv_bfloat16 *>(dK),
                                                         static_cast<__nv_bfloat16 *>(dV), Nq, Nk, kt, bh, H, dv,
                                                         sdk, sdv, scale, scale_log2, wait_limit);
        else
            dkdv_item_narrow<D, CAUSAL, SPLIT, VIEW4, X3>(qA, kA, vA, dOA, Lp, Dp, dK, dV, Nq, Nk, kt, bh, H, dv, sdk,
                                                          sdv, scale, scale_log2, wait_limit);
    } else if constexpr (!RED) {
        const int qt = q_tiles - 1 - idx / BH;           // causal: the last query tiles see the most keys
        if constexpr (D == 64)
            dq_item_wide<D, CAUSAL, SPLIT, VIEW4>(qB, kB, vB, dOB, Lp, Dp, static_cast<__nv_bfloat16 *>(dQ), Nq, Nk,
                                                  qt, bh, H, dv, sdq, scale, scale_log2, wait_limit);
        else
            dq_item_narrow<D, CAUSAL, SPLIT, VIEW4, X3>(qB, kB, vB, dOB, Lp, Dp, dQ, Nq, Nk, qt, bh, H, dv, sdq, scale,
                                                        scale_log2, wait_limit);
    }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes) {
    return tc_set_smem_once(reinterpret_cast<const void *>(k), (int)bytes);
}

struct Maps {
    CUtensorMap q, k, v, dO;
};

template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern kern, uint32_t smem, long long grid, int split, cudaStream_t st, Args... args) {
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split > 1 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int sm_count() { return tc_sm_count(); }

// Split an item over a two-CTA cluster when the longest item's loop is more than
// 1.5x the average loop length per SM (it, not the total work, would set the time).
bool worth_splitting(long long n_max, long long total) { return n_max >= 2 && 2 * n_max * sm_count() > 3 * total; }

bool dkdv_split(const FaProblem &p) {
    const long long ktiles = (p.Nk + 127) / 128, i_end = (p.Nq + 127) / 128;
    long long total = 0, n_max = 0;
    for (long long kt = 0; kt < ktiles; ++kt) {
        const long long first = p.causal ? kt : 0;
        const long long n = i_end > first ? i_end - first : 0;
        total += n;
        n_max = std::max(n_max, n);
    }
    return worth_splitting(n_max, total * p.BH);
}

bool dq_split(const FaProblem &p) {
    const long long qtiles = (p.Nq + 127) / 128;
    long long total = 0, n_max = 0;
    for (long long qt = 0; qt < qtiles; ++qt) {
        const long long kend = p.causal ? std::min<long long>(p.Nk, (qt + 1) * 128) : p.Nk;
        const long long n = (kend + 127) / 128;
        total += n;
        n_max = std::max(n_max, n);
    }
    return worth_splitting(n_max, total * p.BH);
}

struct Maps2 {
    Maps a, b;        // tensor maps of the dK/dV pass (a) and of the dQ pass (b)
    CUtensorMap dqa;  // the fp32 dQ accumulator (dQ by reduction), else unused
    CUtensorMap dk, dv;   // dK and dV (dQ by reduction: their rows leave through TMA stores), else unused
    bool view4;       // 4-D maps over strided views (else 3-D maps over contiguous tensors)
};

template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool RED, bool X3 = false>
cudaError_t launch_bwd(const FaProblem &p, const Maps2 &m, const float *Lp, const float *Dp, void *dQ, void *dK,
                       void *dV, bool do_kv, bool do_q, cudaStream_t st) {
    static_assert(!RED || D == 64, "the dQ reduction form exists for the d = 64 items");
    static_assert(!X3 || ((D == 128 || D == 256) && !RED && !VIEW4),
                  "split fp32 operands: 128- or 256-column items, dQ by the separate pass");
    static_assert(!X3 || D == 128 || SPLIT == 1, "256-column split rows run one item per CTA");
    using KvC = std::conditional_t<D == 64, DkdvWideCfg<D, RED>, DkdvNarrowCfg<D>>;
    using QC = std::conditional_t<D == 64, DqWideCfg<D>, DqNarrowCfg<D>>;
    constexpr uint32_t smem = KvC::SMEM_BYTES > QC::SMEM_BYTES ? KvC::SMEM_BYTES : QC::SMEM_BYTES;
    const int kt = (p.Nk + 127) / 128, qt = (p.Nq + 127) / 128;
    const long long na = do_kv ? (long long)kt * p.BH : 0, nb = (do_q && !RED) ? (long long)qt * p.BH : 0;
    return launch_cluster(fa_bwd_tc_kernel<D, CAUSAL, SPLIT, VIEW4, RED, X3>, smem, (na + nb) * SPLIT, SPLIT, st, m.a.q,
                          m.a.k, m.a.v, m.a.dO, m.b.q, m.b.k, m.b.v, m.b.dO, m.dqa, m.dk, m.dv, Lp, Dp, dQ, dK, dV, p.Nq, p.Nk,
                          p.BH, kt, qt, (int)na, (int)nb, p.scale,
                          p.scale * kLog2e, p.wait_limit, p.H, p.d, p.sdQ, p.sdK, p.sdV);
}

template <int D, bool CAUSAL, bool RED>
cudaError_t launch_bwd_any(const FaProblem &p, const Maps2 &m, const float *Lp, const float *Dp, void *dQ, void *dK,
                           void *dV, bool do_kv, bool do_q, cudaStream_t st) {
    const bool split = (do_kv && dkdv_split(p)) || (do_q && !RED && dq_split(p));
    if (m.view4)
        return split ? launch_bwd<D, CAUSAL, 2, true, RED>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                     : launch_bwd<D, CAUSAL, 1, true, RED>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
    return split ? launch_bwd<D, CAUSAL, 2, false, RED>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                 : launch_bwd<D, CAUSAL, 1, false, RED>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
}

// the persistent dK/dV items of dQ by reduction (d = 64): one CTA per SM
template <bool CAUSAL, bool VIEW4>
cudaError_t launch_red_persistent(const FaProblem &p, const Maps2 &m, const float *Lp, const float *Dp, void *dK,
                                  void *dV, cudaStream_t st) {
    using C = DkdvPersistCfg;
    const int kt = (p.Nk + 127) / 128;
    const long long items = (long long)kt * p.BH;
    const long long grid = std::min<long long>(items, sm_count());
    cudaError_t e = set_smem(fa_bwd_red_persistent_kernel<CAUSAL, VIEW4>, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fa_bwd_red_persistent_kernel<CAUSAL, VIEW4>, m.a.q, m.a.k, m.a.v, m.a.dO, m.dqa, m.dk,
                           m.dv, Lp,
                           Dp, static_cast<__nv_bfloat16 *>(dK), static_cast<__nv_bfloat16 *>(dV), p.Nq, p.Nk, p.BH,
                           kt, p.scale, p.scale * kLog2e, p.wait_limit, p.H, p.d, p.sdK, p.sdV);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Persistent dK/dV items where there are many short ones: at least two items per
// SM and no item whose loop alone would set the run time.  Measured (gradient
// launch, persistent / one item per CTA): 4 x 25 x 1024 causal 68.6 / 80.0 us,
// non-causal 99.3 / 108.3 us; batch 8 x N 4096 causal and N 65536 causal (long
// items, not chosen) equal within 0.3 %.
bool red_persistent(const FaProblem &p) {
    const long long ktiles = (p.Nk + 127) / 128, i_end = (p.Nq + 127) / 128;
    return ktiles * p.BH >= 2LL * sm_count() && i_end <= 16 && !dkdv_split(p);
}

bool make_maps(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO, int q_rows,
               int k_rows, bool view4, Maps *m) {
    return tc_make_map(&m->q, Q, p, p.sQ, p.Nq, q_rows, view4) && tc_make_map(&m->dO, dO, p, p.sdO, p.Nq, q_rows, view4) &&
           tc_make_map(&m->k, K, p, p.sK, p.Nk, k_rows, view4) && tc_make_map(&m->v, V, p, p.sV, p.Nk, k_rows, view4);
}

}  // namespace

bool tc_bwd_supported(const FaProblem &p) { return tc_fwd_supported(p); }

size_t tc_bwd_ld_rows(const FaProblem &p) { return (size_t)p.BH * padded_rows(p.Nq); }

namespace {
std::atomic<int> g_dq_strategy{0};
thread_local int t_dq_override = 0;   // DqStrategy for this thread's calls; 0: the library setting
}

void tc_set_dq_strategy(DqStrategy s) { g_dq_strategy.store(static_cast<int>(s)); }
DqStrategy tc_get_dq_strategy() {
    return static_cast<DqStrategy>(t_dq_override ? t_dq_override : g_dq_strategy.load());
}
void tc_override_dq_strategy(DqStrategy s) { t_dq_override = static_cast<int>(s); }
DqStrategy tc_get_dq_setting() { return static_cast<DqStrategy>(g_dq_strategy.load()); }

// dQ by fp32 reduction inside the dK/dV items exists for head dims up to 64 (the
// 128-wide items).  Measured on GB300 (gradient launch, reduction / separate pass):
// batch 8 x N 4096 causal 54.9 / 58.6 us, N 65536 causal 1204 / 1279 us, the
// 4 x 25 x 1024 layer causal 75.6 / 78.2 us (68.6 with the reduction's persistent
// items) but non-causal 103.8 / 101.0 us one item per CTA -- the reductions (32 KB
// per key tile and query tile) cost more where every key tile meets every query
// tile -- and 99.3 / 107.5 us with persistent items.  So: the reduction for causal
// shapes and wherever its items run persistent, the separate pass otherwise.  A
// forced strategy overrides the choice.
bool tc_bwd_dq_by_reduction(const FaProblem &p) {
    // (split fp32 operands run the d = 128 items, which form dQ by the separate pass)
    if (!tc_bwd_supported(p) || p.d > 64 || p.dtype != FA_DTYPE_BF16) return false;
    switch (tc_get_dq_strategy()) {
        case DqStrategy::kSeparatePass: return false;
        case DqStrategy::kReduction: return true;
        default: return p.causal != 0 || red_persistent(p);
    }
}

size_t tc_bwd_dqa_floats(const FaProblem &p) {
    return tc_bwd_dq_by_reduction(p) ? (size_t)p.BH * padded_rows(p.Nq) * (p.d < 64 ? 64 : p.d) : 0;
}

cudaError_t tc_bwd_preprocess(const FaProblem &p, const void *O, const void *dO, const float *L, float *Dp,
                              float *Lp, float *dQa, cudaStream_t st) {
    const long long rows = (long long)p.BH * padded_rows(p.Nq);
    if (rows == 0) return cudaSuccess;
    const auto *o = static_cast<const __nv_bfloat16 *>(O);
    const auto *g = static_cast<const __nv_bfloat16 *>(dO);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows / (256 / (p.d / 8))));   // rows is a multiple of 128
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (p.d) {
        case 128: e = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<128>, o, g, L, Dp, Lp, dQa, p.Nq, p.H, p.sO, p.sdO); break;
        case 64: e = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<64>, o, g, L, Dp, Lp, dQa, p.Nq, p.H, p.sO, p.sdO); break;
        case 32: e = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<32>, o, g, L, Dp, Lp, dQa, p.Nq, p.H, p.sO, p.sdO); break;
        default: e = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<16>, o, g, L, Dp, Lp, dQa, p.Nq, p.H, p.sO, p.sdO); break;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

namespace {

template <int DK>
cudaError_t launch_dq_convert(const FaProblem &p, const float *dQa, void *dQ, bool view4, cudaStream_t st) {
    const long long groups = (long long)p.BH * p.Nq * (p.d / 8);
    if (groups == 0) return cudaSuccess;
    const long long blocks = std::min<long long>((groups + 255) / 256, (long long)sm_count() * 8);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto *q = static_cast<__nv_bfloat16 *>(dQ);
    const cudaError_t e =
        view4 ? cudaLaunchKernelEx(&cfg, fa_bwd_dq_convert_kernel<DK, true>, dQa, q, p.Nq, p.H, p.d, p.scale, p.sdQ, groups)
              : cudaLaunchKernelEx(&cfg, fa_bwd_dq_convert_kernel<DK, false>, dQa, q, p.Nq, p.H, p.d, p.scale, p.sdQ,
                                   groups);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// the whole backward's gradient launches; dQa != NULL selects dQ by reduction
cudaError_t grads_impl(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                       const float *Lp, const float *Dp, float *dQa, void *dQ, void *dK, void *dV, bool do_kv,
                       bool do_q, cudaStream_t st) {
    // Contiguous tensors keep 3-D (d, N, B*H) maps and plain row addressing; any
    // strided view, or a head dim below 64 (run on the d = 64 kernels with the
    // columns past d read as zero and never stored), switches the whole launch to
    // 4-D maps and strided rows.
    Maps2 m;
    m.view4 = p.d < 64 || !tc_plain_layout(p, p.sQ, p.Nq) || !tc_plain_layout(p, p.sK, p.Nk) ||
              !tc_plain_layout(p, p.sV, p.Nk) || !tc_plain_layout(p, p.sdO, p.Nq) ||
              !tc_plain_layout(p, p.sdQ, p.Nq) || !tc_plain_layout(p, p.sdK, p.Nk) ||
              !tc_plain_layout(p, p.sdV, p.Nk);
    // box heights: wide sub-tiles (d <= 64) load 128-row tiles everywhere; narrow ones
    // (d = 128) load 64-row sub-tiles of the looped-over operand
    if (p.d <= 64) {
        if (!make_maps(p, Q, K, V, dO, 128, 128, m.view4, &m.a)) return cudaErrorInvalidValue;
        m.b = m.a;
    } else if (!make_maps(p, Q, K, V, dO, 64, 128, m.view4, &m.a) ||
               !make_maps(p, Q, K, V, dO, 128, 64, m.view4, &m.b)) {
        return cudaErrorInvalidValue;
    }
    const bool red = dQa != nullptr && do_kv && do_q;
    if (red) {
        if (p.d > 64) return cudaErrorInvalidValue;
        if (!tc_make_map_acc(reinterpret_cast<CUtensorMap_st *>(&m.dqa), dQa, p.BH, padded_rows(p.Nq), 64))
            return cudaErrorInvalidValue;
        if (!tc_make_map(&m.dk, dK, p, p.sdK, p.Nk, 128, m.view4) || !tc_make_map(&m.dv, dV, p, p.sdV, p.Nk, 128, m.view4))
            return cudaErrorInvalidValue;
        cudaError_t e;
        if (red_persistent(p))
            e = m.view4 ? (p.causal ? launch_red_persistent<true, true>(p, m, Lp, Dp, dK, dV, st)
                                    : launch_red_persistent<false, true>(p, m, Lp, Dp, dK, dV, st))
                        : (p.causal ? launch_red_persistent<true, false>(p, m, Lp, Dp, dK, dV, st)
                                    : launch_red_persistent<false, false>(p, m, Lp, Dp, dK, dV, st));
        else
            e = p.causal ? launch_bwd_any<64, true, true>(p, m, Lp, Dp, dQ, dK, dV, true, true, st)
                         : launch_bwd_any<64, false, true>(p, m, Lp, Dp, dQ, dK, dV, true, true, st);
        if (e != cudaSuccess) return e;
        return launch_dq_convert<64>(p, dQa, dQ, !tc_plain_layout(p, p.sdQ, p.Nq), st);
    }
    m.dqa = m.a.q;   // unused by the two-pass launch
    m.dk = m.dv = m.a.q;
    if (p.d == 128) return p.causal ? launch_bwd_any<128, true, false>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                                    : launch_bwd_any<128, false, false>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
    return p.causal ? launch_bwd_any<64, true, false>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                    : launch_bwd_any<64, false, false>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
}

}  // namespace

cudaError_t tc_bwd_grads(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                         const float *Lp, const float *Dp, float *dQa, void *dQ, void *dK, void *dV,
                         cudaStream_t st) {
    return grads_impl(p, Q, K, V, dO, Lp, Dp, dQa, dQ, dK, dV, true, true, st);
}

cudaError_t tc_bwd_dkdv(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                        const float *Lp, const float *Dp, void *dK, void *dV, cudaStream_t st) {
    return grads_impl(p, Q, K, V, dO, Lp, Dp, nullptr, nullptr, dK, dV, true, false, st);
}

cudaError_t tc_bwd_dq(const FaProblem &p, const void *Q, const void *K, const void *V, const void *dO,
                      const float *Lp, const float *Dp, void *dQ, cudaStream_t st) {
    return grads_impl(p, Q, K, V, dO, Lp, Dp, nullptr, dQ, nullptr, nullptr, false, true, st);
}

// ------------------------------------------------------------------ fp32 inputs (X3)
cudaError_t tc_bwd_preprocess_x3(const FaProblem &p, const void *O, const void *dO, const float *L, float *Dp,
                                 float *Lp, void *dO2, cudaStream_t st) {
    const long long rows = (long long)p.BH * padded_rows(p.Nq);
    if (rows == 0) return cudaSuccess;
    if (!tc_x3_possible(p)) return cudaErrorInvalidValue;
    const int rpb = p.d <= 64 ? 16 : 8;   // rows per block: 256 / (W / 4)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows / rpb));   // rows is a multiple of 128
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto *o = static_cast<const float *>(O), *g = static_cast<const float *>(dO);
    auto *g2 = static_cast<__nv_bfloat16 *>(dO2);
    cudaError_t e = p.d <= 64
                        ? cudaLaunchKernelEx(&cfg, fa_bwd_pre_x3_kernel<64>, o, g, L, Dp, Lp, g2, p.Nq, p.H, p.d, p.sO, p.sdO)
                        : cudaLaunchKernelEx(&cfg, fa_bwd_pre_x3_kernel<128>, o, g, L, Dp, Lp, g2, p.Nq, p.H, p.d, p.sO,
                                             p.sdO);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_bwd_grads_x3(const FaProblem &p, const void *Q2, const void *K2, const void *V2, const void *dO2,
                            const float *Lp, const float *Dp, void *dQ, void *dK, void *dV, bool do_kv, bool do_q,
                            cudaStream_t st) {
    if (!tc_x3(p)) return cudaErrorInvalidValue;
    // the d = 128 items over the contiguous (B*H, N, 128) copies: 64-row sub-tiles of
    // the looped-over operand, 128-row tiles of the item's own
    // columns of a split row, and rows of a looped-over sub-tile (the 256-column items
    // take 32-row sub-tiles, so that two stages fit next to the 64 KB K / V or Q / dO tiles)
    const int width = p.d <= 64 ? 128 : 256, sub = p.d <= 64 ? 64 : 32;
    auto map = [&](CUtensorMap *m, const void *ptr, int N, int rows) {
        return tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(m), ptr, p.BH, N, width, rows);
    };
    Maps2 m;
    m.view4 = false;
    if (!map(&m.a.q, Q2, p.Nq, sub) || !map(&m.a.dO, dO2, p.Nq, sub) || !map(&m.a.k, K2, p.Nk, 128) ||
        !map(&m.a.v, V2, p.Nk, 128) || !map(&m.b.q, Q2, p.Nq, 128) || !map(&m.b.dO, dO2, p.Nq, 128) ||
        !map(&m.b.k, K2, p.Nk, sub) || !map(&m.b.v, V2, p.Nk, sub))
        return cudaErrorInvalidValue;
    m.dqa = m.a.q;   // unused
    m.dk = m.dv = m.a.q;
    if (p.d == 128)   // 256-column rows: one item per CTA
        return p.causal ? launch_bwd<256, true, 1, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                        : launch_bwd<256, false, 1, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
    const bool split = (do_kv && dkdv_split(p)) || (do_q && dq_split(p));
    if (p.causal)
        return split ? launch_bwd<128, true, 2, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                     : launch_bwd<128, true, 1, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
    return split ? launch_bwd<128, false, 2, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st)
                 : launch_bwd<128, false, 1, false, false, true>(p, m, Lp, Dp, dQ, dK, dV, do_kv, do_q, st);
}

cudaError_t tc_bwd_read_status(unsigned *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_bwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

cudaError_t tc_bwd_read_rows(unsigned long long *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_bwd_rows, 2 * sizeof(unsigned long long), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

cudaError_t tc_bwd_reset_rows(cudaStream_t st) {
    static const unsigned long long zero[2] = {0, 0};
    return cudaMemcpyToSymbolAsync(g_fa_bwd_rows, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
}

cudaError_t tc_bwd_reset_status(cudaStream_t st) {
    static const unsigned zero = 0;
    return cudaMemcpyToSymbolAsync(g_fa_bwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
}
