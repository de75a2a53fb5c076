// FlashAttention-2 forward on sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Method (CS336 A2 field guide "Systems and Parallelism", §1.2-1.3, problem
// flash_forward; FlashAttention-2): for one tile of 128 query rows, walk the
// key tiles with a running row max m and running row sum l, rescale the output
// accumulator when m moves, divide by l once at the end and write
// L = m + ln(l).  S and P never leave the SM.  Causal: key tiles wholly above
// the diagonal are never loaded (§1.3.3's early exit); only tiles that cross
// the diagonal (or the ragged end of the keys) pay for index compares.
//
// GB300 mapping (one CTA = one 128-row query tile of one batch*head):
//   warp 0      TMA producer: Q once, then K_j and V_j into a ring of smem
//               stages (128-byte swizzle), each stage guarded by mbarriers.
//   warp 1      MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T into
//               TMEM (tcgen05.mma, bf16 in, fp32 accumulate), then
//               O_t += P_j V_j with P read straight from TMEM.
//   warps 4-7   softmax warpgroup 0: key tiles j = 0, 2, 4, ...
//   warps 8-11  softmax warpgroup 1: key tiles j = 1, 3, 5, ...
// Each softmax thread owns one query row (TMEM lane = row), so row max and
// row sum need no shuffles.  The two warpgroups keep separate (m, l, O) over
// interleaved halves of the key range -- while one computes exponentials the
// tensor core works on the other's tile -- and merge the two partial results
// exactly at the end (O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1), a_t = 2^(m_t - M)).
// The running max is only moved when it grows by more than 8 (in log2 units),
// so O is rescaled in TMEM rarely; P stays below 2^8 and the final division
// by l makes the result exact regardless of the max used.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256, 256+d), O1 [256+d,
// 256+2d).  P (packed bf16, 64 columns) aliases the first half of its S for
// d = 128; for d = 64 it has its own columns [384 + 64t, 448 + 64t), and the
// MMA warp issues S_{j+2} as soon as the softmax has read S_j (one barrier
// per tile), so the tensor core computes the next scores under the softmax.
//
// Split work items (SPLIT = 2): when there are too few query tiles to fill the
// GPU, or the longest causal row would dominate the run, a cluster of two CTAs
// shares one query tile: rank 0 takes the first half of the key tiles, rank 1
// the rest.  Each rank then finalises half of the columns: it stores its
// unnormalised partial of the other half, with the row's (m, l), into the
// peer's shared memory with remote stores (once the peer's MMAs are done),
// and merges the half it keeps exactly like the two warpgroups' halves.  The
// hand-over uses mbarriers arrived on from the other CTA, waited on with a
// bound.
//
// Many short units (at least two per SM, at most 12 key tiles on average):
// fa_fwd_tc_persistent_kernel runs one CTA per SM over a snake-ordered list of
// units, numbering tiles across units so that every ring slot, barrier phase
// and TMEM buffer carries over; the next unit's Q and first K/V tiles load and
// its first S MMAs run while the softmax warps finish the previous unit.
//
// Every kernel here is launched with programmatic stream serialisation: it
// lets the next kernel be scheduled as soon as all of its CTAs have started,
// and waits (griddepcontrol.wait) for the previous one before touching global
// memory, so launch latency overlaps the previous kernel's tail.
//
// Layouts (template argument VIEW4): contiguous (B*H, N, d) tensors load
// through 3-D tensor maps (d, N, B*H) and store O rows at (bh*Nq + row)*d.
// Strided (B, H, N, d) views -- the method's block pointers keep one stride per
// dimension, and here batch and heads keep theirs -- load through 4-D maps
// (d, N, H, B) at coordinates (col, row, bh % H, bh / H) and store through O's
// own strides.  Head dims 16 and 32 run the d = 64 kernels in this form: the
// 64-column boxes read zeros past d, so Q K^T is unchanged and the zero output
// columns past d are never stored.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "fa_internal.h"
#include "tc_common.cuh"

__device__ unsigned g_fa_fwd_status;
__device__ unsigned long long g_fa_fwd_rows;   // debug build: key rows the forward loaded

namespace {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 128;          // keys per tile
constexpr int NTHREADS = 384;    // 12 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct FwdCfg {
    // separate K and V rings: a K slot frees when its S MMAs finish, a V slot
    // when its PV MMAs finish; K runs one tile ahead of V.  Deep enough to
    // cover an L2-resident TMA reload (~2000 cycles).
    // (D = 256: fp32 head dim 128 as split bf16 pairs; one 64 KB tile per ring)
    static constexpr int KST = D == 256 ? 1 : D == 128 ? 3 : 6;
    static constexpr int VST = D == 256 ? 1 : D == 128 ? 2 : 4;
    // one "PV_j complete" barrier per tile in a ring of R > KST, VST: it frees K_j's
    // and V_j's slots (in-order completion covers S_j) and tells the softmax that
    // P_j / O may be touched again -- one commit instead of three
    static constexpr int R = D == 64 ? 8 : 4;
    static constexpr int CHUNKS = D / 64;                      // 128-byte swizzle chunks per row
    // O accumulator columns per warpgroup: d, except for the 256-column split rows of
    // a head dim of 128, whose three products all add into the 128 output columns
    static constexpr int OW = D == 256 ? 128 : D;
    static constexpr uint32_t CHUNK_BYTES = 128u * 128u;       // 128 rows x 128 bytes
    static constexpr uint32_t TILE_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = Q_OFF + TILE_BYTES;
    static constexpr uint32_t V_OFF = K_OFF + KST * TILE_BYTES;
    static constexpr uint32_t BAR_OFF = V_OFF + VST * TILE_BYTES;
    static constexpr int NBAR = 1 + KST + VST + R + 17;
    // per-row (m, l) of both warpgroups, double-buffered by work unit: 2 x (256 + 256) floats
    static constexpr uint32_t STAT_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t MISC_OFF = STAT_OFF + 2 * 512 * 4;
    static constexpr uint32_t PEER_BAR_OFF = MISC_OFF + 16;                  // peer_free, peer_ready, peer_d
    // persistent kernel: per softmax thread, the element offset of its output row in the current unit
    static constexpr uint32_t OROW_OFF = PEER_BAR_OFF + 32;
    // fused backward preprocessing: the two halves of each row's rowsum(dO * O)
    // (double-buffered by work unit in the persistent kernel; the split form's
    // rank 1 stores its half into rank 0's copy)
    static constexpr uint32_t DSUM_OFF = OROW_OFF + 256 * 8;
    // fused backward preprocessing, d = 64: the tile's dO rows (128 bytes each, the
    // 16-byte chunks of row r swizzled by r mod 8 so that the epilogue's row-per-thread
    // reads hit eight different bank groups), fetched by TMA from an otherwise idle
    // warp during the main loop; two buffers, alternating by unit in the persistent
    // kernel (the 128-byte swizzle wants 1024-byte aligned destinations; the barrier
    // block above leaves the offsets after it only 8-byte aligned, hence the rounding)
    static constexpr uint32_t DOS_OFF = (DSUM_OFF + 2 * 256 * 4 + 1023) / 1024 * 1024;
    static constexpr uint32_t DOS_BYTES = 128 * 64 * 2;
    static_assert(DOS_OFF % 1024 == 0 && DOS_BYTES % 1024 == 0, "swizzled TMA destinations on 1024-byte boundaries");
    static constexpr uint32_t USED = DOS_OFF + (D == 64 ? 2 * DOS_BYTES : 0);
    // split items: rank 1's partial O (fp32, rows padded by 4 floats) and its m, l, in the K ring
    static constexpr uint32_t PART_STRIDE = (OW + 4) * 4;
    static constexpr uint32_t PART_OFF = K_OFF;
    static constexpr uint32_t PART_ML_OFF = PART_OFF + 128 * PART_STRIDE;
    static_assert(PART_ML_OFF + 2 * 128 * 4 <= V_OFF + VST * TILE_BYTES, "partial fits the K and V rings");
    // at least ~116 KB so that one CTA (which owns all 512 TMEM columns) runs per SM
    static constexpr uint32_t SMEM_BYTES = (USED + 1024 > 120u * 1024u ? USED + 1024 : 120u * 1024u);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static constexpr uint32_t S_COL0 = 0, O_COL0 = 256;
    static_assert(O_COL0 + 2 * OW <= TMEM_COLS, "two O accumulators after the two S buffers");
    // d = 64 leaves 128 TMEM columns free: P gets its own columns there, so the
    // next S of a warpgroup can be issued as soon as the current S has been read
    static constexpr bool SEP_P = D == 64;
    static constexpr uint32_t P_COL0 = SEP_P ? 384 : 0;   // P_t at P_COL0 + (SEP_P ? 64 : 128) * t
    static constexpr uint32_t P_STRIDE = SEP_P ? 64 : 128;
};

// ------------------------------------------------------------------ fused backward preprocessing
// One 16-byte chunk (8 columns) of a dO row staged by a 128-byte-swizzled TMA
// load: chunk j of tile row r sits at chunk position j ^ (r mod 8) of the row.
__device__ __forceinline__ uint4 swizzled_chunk(const uint8_t *srow, int r, int j) {
    return *reinterpret_cast<const uint4 *>(srow + ((j ^ (r & 7)) << 4));
}

// Half of rowsum(dO * O) for one query row: this thread's D/2 output columns of
// the unrounded fp32 O (vals * inv) against the same columns of dO, read from
// global memory or (srow not NULL) from tile row r staged in shared memory.
template <int D, bool VIEW4>
__device__ __forceinline__ float prep_half_rowsum(const FwdPrep &prep, const float *vals, float inv, int bh, int row,
                                                  int Nq, int H, int dv, int t, const uint8_t *srow = nullptr,
                                                  int r = 0) {
    const __nv_bfloat16 *g;
    if constexpr (VIEW4) g = static_cast<const __nv_bfloat16 *>(prep.dO) + fa_row_offset(prep.sdo, H, bh, row) + t * (D / 2);
    else g = static_cast<const __nv_bfloat16 *>(prep.dO) + ((size_t)bh * Nq + row) * D + t * (D / 2);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        if (!VIEW4 || t * (D / 2) + 8 * c < dv) {   // columns past a head dim below 64 are padding
            const uint4 x = srow ? swizzled_chunk(srow, r, t * (D / 16) + c) : __ldg(reinterpret_cast<const uint4 *>(g) + c);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(h[k]);
                acc = fmaf(vals[8 * c + 2 * k] * inv, f.x, acc);
                acc = fmaf(vals[8 * c + 2 * k + 1] * inv, f.y, acc);
            }
        }
    }
    return acc;
}

// The backward's per-row constants from the forward's epilogue: -D (half0 +
// half1) and -L*log2(e), L exactly as stored (padding rows: 0 and -inf, so
// their P is exactly zero); and this warpgroup's half of the row's dQ
// accumulator cleared (d <= 64 kernels, when dQ is formed by reduction).
template <int D>
__device__ __forceinline__ void prep_row_finish(const FwdPrep &prep, float half0, float half1, bool write_consts,
                                                float Mrow, float lrow, int bh, int row, int Nq, int t,
                                                bool clear_acc = true) {
    const size_t gr = (size_t)bh * ((Nq + 127) / 128 * 128) + row;
    if (write_consts) {
        if (row < Nq) {
            const float L = Mrow * kLn2 + logf(lrow);
            prep.Dp[gr] = -(half0 + half1);
            prep.Lp[gr] = -L * kLog2e;
        } else {
            prep.Dp[gr] = 0.f;
            prep.Lp[gr] = -INFINITY;
        }
    }
    if constexpr (D == 64) {
        if (prep.dQa && clear_acc) {
            float4 *z = reinterpret_cast<float4 *>(prep.dQa + gr * 64 + t * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// ------------------------------------------------------------------ fp32 operands as bf16 pairs
// X (B, H, N, d) fp32, through its strides -> X2, B*H*N contiguous rows of 2W
// bf16 (W = 64 for d <= 64, 128 for d = 128): hi = bf16(x) in columns [0, W),
// lo = bf16(x - hi) in [W, 2W), zeros past d.  x - hi is exact in fp32, so
// hi + lo meets x to within 2^-16 relative.  W/4 threads per row, four
// columns each.
struct SplitJob {
    const float *X;
    __nv_bfloat16 *X2;
    FaStrides s;
    int N;
};
struct SplitJobs {
    SplitJob j[4];   // blockIdx.y selects the tensor
};
template <int W>
__global__ void __launch_bounds__(256) fa_split_x3_kernel(const __grid_constant__ SplitJobs jobs, int BH, int H,
                                                          int d) {
    constexpr int TPR = W / 4;   // threads per row
    tc::pdl_launch_dependents();
    tc::pdl_wait();   // the tensors may come from the previous kernel
    const SplitJob &J = jobs.j[blockIdx.y];
    const long long g = (long long)blockIdx.x * 256 + threadIdx.x;
    const long long row = g / TPR;
    const int cg = (int)(g % TPR);
    if (row >= (long long)BH * J.N) return;
    const int bh = (int)(row / J.N), n = (int)(row - (long long)bh * J.N);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (4 * cg < d) x = __ldg(reinterpret_cast<const float4 *>(J.X + fa_row_offset(J.s, H, bh, n) + 4 * cg));
    const uint32_t h0 = tc::pack_bf16(x.x, x.y), h1 = tc::pack_bf16(x.z, x.w);
    uint2 *dst = reinterpret_cast<uint2 *>(J.X2 + row * (2 * W));
    dst[cg] = make_uint2(h0, h1);
    dst[TPR + cg] = make_uint2(tc::pack_bf16_residual(x.x, x.y, h0), tc::pack_bf16_residual(x.z, x.w, h1));
}

// X3 (fp32 inputs, head dim up to 64): Q, K and V arrive as bf16 pairs, each
// 128-column row holding hi = bf16(x) in columns [0, 64) and lo = bf16(x - hi) in
// [64, 128), and the kernel runs the d = 128 layout with three products per
// contraction: Q K^T = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T (12 k-steps instead of
// 8), and P V = Phi [Vhi | Vlo] + Plo Vhi, with P split the same way in TMEM (hi
// over the first 64 columns of its S, lo over the other 64).  Output column c
// is then accumulator column c plus column 64 + c, and O is written in fp32.
// The product lo * lo and the rounding of lo leave a relative error near 2^-16
// per product, against 2^-8 for one bf16 product.
template <int D, bool CAUSAL, int SPLIT, bool VIEW4, bool X3 = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     void *__restrict__ Ov,
                     float *__restrict__ Lout, int Nq, int Nk, int BH, int num_q_tiles, float scale_log2,
                     uint32_t wait_limit, uint32_t force_stall, int H, int dv, FaStrides so, FwdPrep prep) {
    static_assert(!X3 || ((D == 128 || D == 256) && !VIEW4), "split fp32 operands: 128- or 256-column copies");
    static_assert(X3 || D <= 128, "the 256-column layout holds split pairs only");
    static_assert(!X3 || D == 128 || SPLIT == 1, "256-column split rows run one unit per CTA");
    using C = FwdCfg<D>;
    // X3 at D = 128 (head dims up to 64): output column c is accumulator column c plus
    // 64 + c (hi and lo products of V); at D = 256 all products add into the same columns
    constexpr bool FOLD = X3 && D == 128;
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(Ov);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    tc::pdl_launch_dependents();

    // longest work first: high query tiles (more key tiles under causal) start first
    const int item = blockIdx.x / SPLIT;
    const uint32_t rank = SPLIT > 1 ? tc::cluster_rank() : 0u;
    const int qt = num_q_tiles - 1 - item / BH;
    const int bh = item % BH;
    const int q0 = qt * BM;
    const int kend = CAUSAL ? min(Nk, q0 + BM) : Nk;
    const int n_all = (kend + BN - 1) / BN;
    // this CTA's key tiles [jb, jb + n): all of them, or one half of a split item
    const int n_first = SPLIT > 1 ? (n_all + 1) / 2 : n_all;
    const int jb = rank == 0 ? 0 : n_first;
    const int n = rank == 0 ? n_first : n_all - n_first;

    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t q_full = bar(0);
    constexpr int RB = 1 + C::KST + C::VST + C::R;          // first non-ring barrier
    auto k_full = [&](int s) { return bar(1 + s); };
    auto v_full = [&](int s) { return bar(1 + C::KST + s); };
    auto pv_done_bar = [&](int j) { return bar(1 + C::KST + C::VST + j % C::R); };
    auto s_full = [&](int t) { return bar(RB + t); };
    auto p_full = [&](int t) { return bar(RB + 2 + t); };
    const uint32_t drain = bar(RB + 4);
    const uint32_t never = bar(RB + 5);   // fault injection: nothing ever arrives here
    auto s_free = [&](int t) { return bar(RB + 6 + t); };   // softmax has read S_t (separate-P layout)
    const uint32_t do_full = bar(RB + 8);   // fused preprocessing (d = 64): the tile's dO rows have landed
    float *m_sm = reinterpret_cast<float *>(sb + C::STAT_OFF);
    float *l_sm = m_sm + 256;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < C::KST; ++s) tc::mbar_init(k_full(s), 1);
        for (int s = 0; s < C::VST; ++s) tc::mbar_init(v_full(s), 1);
        for (int s = 0; s < C::R; ++s) tc::mbar_init(pv_done_bar(s), 1);
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(s_full(t), 1);
            tc::mbar_init(p_full(t), 128);
            tc::mbar_init(s_free(t), 128);
        }
        tc::mbar_init(drain, 1);
        tc::mbar_init(never, 1);
        tc::mbar_init(do_full, 1);
        if (SPLIT > 1) {
            tc::mbar_init(base + C::PEER_BAR_OFF, 256);       // peer_free: the peer's 256 softmax threads
            tc::mbar_init(base + C::PEER_BAR_OFF + 8, 128);   // peer_ready: the peer's 128 senders
            tc::mbar_init(base + C::PEER_BAR_OFF + 16, 128);  // peer_d: rank 1's half rowsums (fused preprocessing)
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
    if (SPLIT > 1) tc::cluster_sync_all();   // the peer's barriers are initialised before anyone arrives
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    tc::pdl_wait();   // the previous kernel's writes (Q, K, V; readers of O and L) are done
    const tc::Waiter W{abort_flag, &g_fa_fwd_status, wait_limit, 1u};
    // registers: warps 0-3 (producer, MMA issuer, two idle) give theirs to the softmax warpgroups

    // registers: warpgroup 0 (producer, MMA issuer, two idle warps) hands its share
    // to the two softmax warpgroups; each warpgroup changes its budget in one place
    if (warp < 4) {
    tc::regs_dec<(SPLIT > 1 ? 72 : 56)>();   // split items keep cluster state: 72 avoids a spill
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmQ);
            tc::tma_prefetch_desc(&tmK);
            tc::tma_prefetch_desc(&tmV);
            const bool q_ok = tc::in_bounds(q0 < Nq && bh < BH, &g_fa_fwd_status, abort_flag);
            if (q_ok) {
                tc::mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
                for (int c = 0; c < C::CHUNKS; ++c)
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + c * C::CHUNK_BYTES, &tmQ, q_full, c * 64, q0, bh, H);
            }
            int k_issued = 0, v_issued = 0;
            // The slot of tile j last held tile j - st.  A V slot is free once PV of that
            // tile has completed.  A K slot is read only by S of that tile; with P over S
            // the MMA warp issues S_{x+1} before PV_x (and S_0, S_1 before PV_0), so the
            // K slot is free once PV_{j-st-1} has completed.  (With P in its own columns
            // the K ring is deep enough to keep waiting for PV_{j-st}.)
            auto load = [&](const CUtensorMap *m, uint32_t ring, int st, int j, uint32_t full, int lag) {
                // debug build: a key tile past the keys, or wholly above the diagonal, is never loaded
                const int key0 = (jb + j) * BN;
                if (!tc::in_bounds(key0 < Nk && (!CAUSAL || key0 <= q0 + BM - 1), &g_fa_fwd_status, abort_flag))
                    return false;
                if (st == 1 && lag == 1) {
                    // one K slot (256-column rows): it last held tile j - 1, whose S MMAs are
                    // issued before PV_{j-2} completes, so wait for S_{j-1} itself
                    if (j >= 1 && !W.wait(s_full((j - 1) & 1), ((j - 1) >> 1) & 1)) return false;
                } else {
                    const int g = j - st - lag < 0 ? 0 : j - st - lag;
                    if (j >= st && !W.wait(pv_done_bar(g), (g / C::R) & 1)) return false;
                }
                tc::mbar_arrive_expect_tx(full, C::TILE_BYTES);
                for (int c = 0; c < C::CHUNKS; ++c)
                    tc::tma_load_rows<VIEW4>(ring + (j % st) * C::TILE_BYTES + c * C::CHUNK_BYTES, m, full, c * 64,
                                    (jb + j) * BN, bh, H);
                return true;
            };
            // order K_0, K_1, V_0, K_2, V_1, ...: the MMA warp uses K_{j+1} before V_j
            for (int j = 0; q_ok && j <= n; ++j) {
                if (j < n) {
                    if (!load(&tmK, base + C::K_OFF, C::KST, j, k_full(j % C::KST), C::SEP_P ? 0 : 1)) break;
                    k_issued = j + 1;
                }
                if (j >= 1) {
                    const int v = j - 1;
                    if (!load(&tmV, base + C::V_OFF, C::VST, v, v_full(v % C::VST), 0)) break;
                    v_issued = v + 1;
                }
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_fwd_rows, (unsigned long long)k_issued * BN);
            if (*abort_flag) {
                // let the copies already in flight land before the CTA exits
                for (int j = k_issued - 1; j >= 0 && j >= k_issued - C::KST; --j)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(k_full(j % C::KST), (j / C::KST) & 1); ++i) {
                    }
                for (int j = v_issued - 1; j >= 0 && j >= v_issued - C::VST; --j)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(v_full(j % C::VST), (j / C::VST) & 1); ++i) {
                    }
                if (q_ok)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full, 0); ++i) {
                    }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ fused preprocessing
        // While the tile runs: fetch its dO rows into shared memory for the epilogue's
        // rowsum (d = 64: one swizzled TMA tile; rows past Nq and columns past a head
        // dim below 64 read as zeros) and clear its rows of the dQ accumulator (rank 0
        // of a split item), off the epilogue's path.
        if (prep.dO && q0 < Nq) {
            if (D == 64 && lane == 0) {
                tc::mbar_arrive_expect_tx(do_full, C::DOS_BYTES);
                tc::tma_load_rows<VIEW4>(base + C::DOS_OFF, &tmdO, do_full, 0, q0, bh, H);
            }
            if (D == 64 && prep.dQa && rank == 0) {
                float4 *z = reinterpret_cast<float4 *>(prep.dQa + ((size_t)bh * ((Nq + 127) / 128 * 128) + q0) * 64);
                for (int i = lane; i < BM * 64 / 4; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (D == 64 && lane == 0)   // the copy lands before the CTA may exit
                for (uint32_t i = 0; i < (1u << 22) && !tc::mbar_try_wait(do_full, 0); ++i) {
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop so that descriptors stay warp-uniform and
        // cheap to form; one elected lane issues the tcgen05 instructions.
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc_s = tc::idesc_bf16(BM, BN, false, false);
        constexpr uint32_t idesc_o = tc::idesc_bf16(BM, C::OW, false, true);
        constexpr uint32_t idesc_o_hi = tc::idesc_bf16(BM, 64, false, true);   // X3, D = 128: Plo Vhi
        const uint64_t qd = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);
        const uint64_t kd = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);
        const uint64_t vd = tc::sdesc_sw128(base + C::V_OFF, C::CHUNK_BYTES, 1024);
        bool ok = __all_sync(0xffffffffu, W.wait(q_full, 0));
        if (force_stall) ok = __all_sync(0xffffffffu, W.wait(never, 0));
        auto pv = [&](int j) -> bool {
            const int s = j % C::VST, t = j & 1, k = j >> 1;
            if (!__all_sync(0xffffffffu, W.wait2(p_full(t), k & 1, v_full(s), (j / C::VST) & 1))) return false;
            tc::fence_after_sync();
            if (leader) {
                const uint64_t vs = vd + ((s * C::TILE_BYTES) >> 4);
                const uint32_t tP = tmem + C::P_COL0 + t * C::P_STRIDE;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)   // 16 keys = 16 rows of V = 2048 bytes per k-step
                    tc::mma_ts(tmem + C::O_COL0 + t * C::OW, tP + kk * 8, vs + kk * 128, idesc_o,
                               (k > 0 || kk > 0) ? 1u : 0u);
                if constexpr (X3 && D == 128) {
                    // Plo (TMEM columns 64..127 of P_t) times Vhi (the first 64 columns) into O's first 64
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc::mma_ts(tmem + C::O_COL0 + t * C::OW, tP + 64 + kk * 8, vs + kk * 128, idesc_o_hi, 1u);
                } else if constexpr (X3) {
                    // D = 256: Phi times Vlo (chunks 2, 3), then Plo times Vhi (chunks 0, 1), into the same O
                    const uint64_t vlo = vs + ((2 * C::CHUNK_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc::mma_ts(tmem + C::O_COL0 + t * C::OW, tP + kk * 8, vlo + kk * 128, idesc_o, 1u);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc::mma_ts(tmem + C::O_COL0 + t * C::OW, tP + 64 + kk * 8, vs + kk * 128, idesc_o, 1u);
                }
                tc::mma_commit(pv_done_bar(j));
            }
            __syncwarp();
            return true;
        };
        // S_j = Q K_j^T into S_{j&1}; with P in its own columns S_{j&1} must first have
        // been read by the softmax (tile j - 2): both waits are polled together
        auto issue_s = [&](int j) -> bool {
            const int s = j % C::KST, t = j & 1;
            const bool ok_k = (C::SEP_P && j >= 2)
                                  ? W.wait2(s_free(t), ((j - 2) >> 1) & 1, k_full(s), (j / C::KST) & 1)
                                  : W.wait(k_full(s), (j / C::KST) & 1);
            if (!__all_sync(0xffffffffu, ok_k)) return false;
            if (leader) {
                const uint64_t ks = kd + ((s * C::TILE_BYTES) >> 4);
                if constexpr (X3) {
                    // chunk pairs (Q, K): (hi, hi), (hi, lo), (lo, hi) for each of the HC hi chunks
                    // (the lo chunks follow them), four k-steps each
                    constexpr int HC = D / 128;
                    auto pair = [&](int pr) {
                        const int grp = pr / HC, c = pr % HC;
                        const uint32_t bq = (grp == 2 ? HC + c : c) * C::CHUNK_BYTES;
                        const uint32_t bk = (grp == 1 ? HC + c : c) * C::CHUNK_BYTES;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            tc::mma_ss(tmem + C::S_COL0 + t * 128, qd + ((bq + k4 * 32) >> 4),
                                       ks + ((bk + k4 * 32) >> 4), idesc_s, (pr > 0 || k4 > 0) ? 1u : 0u);
                    };
                    if constexpr (HC == 1) {
#pragma unroll
                        for (int pr = 0; pr < 3; ++pr) pair(pr);
                    } else {
                        // (kept rolled: unrolled, the 24 descriptors spill the issuer's 56 registers)
#pragma unroll 1
                        for (int pr = 0; pr < 3 * HC; ++pr) pair(pr);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4;
                        tc::mma_ss(tmem + C::S_COL0 + t * 128, qd + off, ks + off, idesc_s, kk > 0 ? 1u : 0u);
                    }
                }
                tc::mma_commit(s_full(t));
            }
            __syncwarp();
            return true;
        };
        if constexpr (C::SEP_P) {
            // S_0, S_1, then per tile: S_{j+2} once S_j has been read, then PV_j once P_j is ready
            for (int j = 0; ok && j < n && j < 2; ++j) ok = issue_s(j);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 2 < n && !(ok = issue_s(j + 2))) break;
                ok = pv(j);
            }
        } else {
            // P aliases S: S_{j+2} can only follow PV_j
            for (int j = 0; ok && j < n; ++j) {
                if (!(ok = issue_s(j))) break;
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok && n > 0) ok = pv(n - 1);
        }
        if (!ok && leader) {
            // wait (bounded) for the MMAs already issued before TMEM is released
            tc::mma_commit(drain);
            for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
            }
        }
        __syncwarp();
    }
    } else {
        tc::regs_inc<(SPLIT > 1 ? 216 : 224)>();
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 4) >> 2;
        const int r = ((warp & 3) << 5) + lane;            // row within the tile = TMEM lane
        const int row = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::S_COL0 + t * 128;
        const uint32_t tP = tmem + lane_base + C::P_COL0 + t * C::P_STRIDE;
        const uint32_t tO = tmem + lane_base + C::O_COL0 + t * C::OW;
        const int nt = (n - t + 1) >> 1;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int k = 0; k < nt; ++k) {
            const int k0 = (jb + 2 * k + t) * BN;
            ok = W.wait(s_full(t), k & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_x32(tS + 32 * c, sr[c]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence_x32(sr[c]);
            if constexpr (C::SEP_P) {
                tc::fence_before_sync();
                tc::mbar_arrive(s_free(t));   // S_t may now be overwritten by S_{j+2}
            }
            float s[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
            const bool need_mask = (CAUSAL && k0 + BN - 1 > q0) || (k0 + BN > Nk);
            if (need_mask) {
                const int lim = min(Nk - 1, CAUSAL ? row : Nk - 1) - k0;   // last visible column
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i > lim) s[i] = -INFINITY;
            }
            // row max as four independent chains (short dependency paths)
            float mq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) mq[q] = tc::fmax3(s[q], s[4 + q], s[8 + q]);
#pragma unroll
            for (int i = 12; i < 124; i += 8)
#pragma unroll
                for (int q = 0; q < 4; ++q) mq[q] = tc::fmax3(mq[q], s[i + q], s[i + 4 + q]);
#pragma unroll
            for (int q = 0; q < 4; ++q) mq[q] = fmaxf(mq[q], s[124 + q]);
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            const float m_cand = fmaxf(m, mx * scale_log2);
            const bool rescale = m_cand > m + kRescaleThreshold;
            float alpha = 1.f;
            if (rescale) {
                alpha = tc::ex2(m - m_cand);
                m = m_cand;
            }
            l *= alpha;
            const float nm = -m;
            uint32_t p[64];
            float rs[4][2] = {};
            if constexpr (X3) {
                // P = hi + lo: hi over P_t's first 64 columns, lo over the other 64, stored
                // half by half (S_t has been read into registers; P aliases it)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ph[32], pl[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int ii = 32 * h + i;
                        float x0, x1;
                        tc::fma2(x0, x1, s[2 * ii], s[2 * ii + 1], scale_log2, scale_log2, nm, nm);
                        const float e0 = tc::ex2(x0), e1 = tc::ex2(x1);
                        tc::add2(rs[i & 3][0], rs[i & 3][1], rs[i & 3][0], rs[i & 3][1], e0, e1);
                        ph[i] = tc::pack_bf16(e0, e1);
                        pl[i] = tc::pack_bf16_residual(e0, e1, ph[i]);
                    }
                    tmem_st_x32(tP + 32 * h, ph);
                    tmem_st_x32(tP + 64 + 32 * h, pl);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float x0, x1;
                    tc::fma2(x0, x1, s[2 * i], s[2 * i + 1], scale_log2, scale_log2, nm, nm);
                    const float e0 = tc::ex2(x0), e1 = tc::ex2(x1);
                    tc::add2(rs[i & 3][0], rs[i & 3][1], rs[i & 3][0], rs[i & 3][1], e0, e1);
                    p[i] = tc::pack_bf16(e0, e1);
                }
            }
            l += ((rs[0][0] + rs[0][1]) + (rs[1][0] + rs[1][1])) + ((rs[2][0] + rs[2][1]) + (rs[3][0] + rs[3][1]));
            if (C::SEP_P && k > 0) {
                // P_t is still read by PV of this warpgroup's previous tile until that completes
                ok = W.wait(pv_done_bar(2 * k + t - 2), ((2 * k + t - 2) / C::R) & 1);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::fence_after_sync();
            }
            if constexpr (!X3) {
                tmem_st_x32(tP, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                tmem_st_x32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
            }
            if (k > 0 && __any_sync(0xffffffffu, rescale)) {
                // O_t holds the sum up to this warpgroup's previous tile: rescale it in place
                ok = W.wait(pv_done_bar(2 * k + t - 2), ((2 * k + t - 2) / C::R) & 1);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < C::OW / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + 32 * c, o);
                    tc::tmem_ld_wait();
                    reg_fence_x32(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_x32(tO + 32 * c, o);
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(p_full(t));
        }
        // ---- merge the two warpgroups' partial results (and, for split items, the peer CTA's)
        m_sm[t * 128 + r] = m;
        l_sm[t * 128 + r] = l;
        tc::named_bar_sync(1, 256);
        const int n0 = (n + 1) >> 1, n1 = n >> 1;
        bool fine = !*abort_flag;
        if (fine && n0 > 0) fine = W.wait(pv_done_bar(2 * n0 - 2), ((2 * n0 - 2) / C::R) & 1);
        if (fine && n1 > 0) fine = W.wait(pv_done_bar(2 * n1 - 1), ((2 * n1 - 1) / C::R) & 1);
        if (D == 64 && prep.dO && fine) fine = W.wait(do_full, 0);   // the dO rows are in shared memory
        fine = __all_sync(0xffffffffu, fine);
        // this CTA's partial for row r, output columns [t*VW, (t+1)*VW), relative to max Mc
        // (unnormalised); X3: output column c sums accumulator columns c and 64 + c
        constexpr int VW = FOLD ? 32 : C::OW / 2;
        float v[VW];
        float Mc = -INFINITY, lc = 0.f;
#pragma unroll
        for (int i = 0; i < VW; ++i) v[i] = 0.f;
        if (fine && n0 > 0) {
            tc::fence_after_sync();
            const float m0 = m_sm[r], l0 = l_sm[r];
            const float m1 = m_sm[128 + r], l1 = l_sm[128 + r];
            Mc = fmaxf(m0, m1);
            const float a0 = exp2f(m0 - Mc);
            const float a1 = n1 > 0 ? exp2f(m1 - Mc) : 0.f;
            lc = l0 * a0 + l1 * a1;
            const uint32_t tO0 = tmem + lane_base + C::O_COL0, tO1 = tO0 + C::OW;
#pragma unroll
            for (int c = 0; c < (FOLD ? 2 : C::OW / 64); ++c) {
                const int col = FOLD ? t * VW + 64 * c : t * (C::OW / 2) + 32 * c;
                uint32_t o0[32], o1[32] = {};
                tmem_ld_x32(tO0 + col, o0);
                if (n1 > 0) tmem_ld_x32(tO1 + col, o1);
                tc::tmem_ld_wait();
                reg_fence_x32(o0);
                reg_fence_x32(o1);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(o0[i]) * a0;
                    if (n1 > 0) x = fmaf(__uint_as_float(o1[i]), a1, x);
                    if (FOLD) v[i] += x;
                    else v[32 * c + i] = x;
                }
            }
        }
        // stores this thread's half row of O (and L); returns the half's part of
        // rowsum(dO * O) from the unrounded O when the preprocessing is fused
        auto store_row = [&](const float *vals, float Mrow, float lrow) -> float {
            const float inv = 1.f / lrow;
            if constexpr (X3) {
                // fp32 output row through O's strides; columns past the head dim are padding
                float *orow = static_cast<float *>(Ov) + fa_row_offset(so, tc::opaque(H), bh, row) + t * VW;
                if (row < Nq) {
#pragma unroll
                    for (int c = 0; c < VW / 4; ++c)
                        if (t * VW + 4 * c < dv)
                            reinterpret_cast<float4 *>(orow)[c] =
                                make_float4(vals[4 * c] * inv, vals[4 * c + 1] * inv, vals[4 * c + 2] * inv,
                                            vals[4 * c + 3] * inv);
                    if (t == 0) Lout[(size_t)bh * Nq + row] = Mrow * kLn2 + logf(lrow);
                }
                return 0.f;
            }
            __nv_bfloat16 *orow;
            if constexpr (VIEW4) orow = O + fa_row_offset(so, tc::opaque(H), bh, row) + t * (D / 2);
            else orow = O + ((size_t)bh * Nq + row) * D + t * (D / 2);
            float part = 0.f;
            if (row < Nq) {
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint4 q;
                    q.x = tc::pack_bf16(vals[8 * c + 0] * inv, vals[8 * c + 1] * inv);
                    q.y = tc::pack_bf16(vals[8 * c + 2] * inv, vals[8 * c + 3] * inv);
                    q.z = tc::pack_bf16(vals[8 * c + 4] * inv, vals[8 * c + 5] * inv);
                    q.w = tc::pack_bf16(vals[8 * c + 6] * inv, vals[8 * c + 7] * inv);
                    if (!VIEW4 || t * (D / 2) + 8 * c < dv)   // columns past a head dim below 64 are padding
                        reinterpret_cast<uint4 *>(orow)[c] = q;
                }
                if (t == 0) Lout[(size_t)bh * Nq + row] = Mrow * kLn2 + logf(lrow);
                if (prep.dO) {
                    const uint8_t *srow = nullptr;
                    if constexpr (D == 64) srow = sb + C::DOS_OFF + r * 128;
                    part = prep_half_rowsum<D, VIEW4>(prep, vals, inv, bh, row, Nq, H, dv, t, srow, r);
                }
            }
            return part;
        };
        // hand-over waits: bounded, but not cut short by this CTA's own abort flag, so
        // that neither CTA exits while the other may still touch its shared memory
        auto wait_peer = [&](uint32_t b) -> bool {
            uint64_t deadline = 0;
            for (uint32_t i = 0;; ++i) {
                if (tc::mbar_try_wait_cluster(b, 0)) return true;
                if ((i & 255u) == 0) {
                    const uint64_t now = tc::globaltimer();
                    if (deadline == 0) deadline = now + 2000000000ull;
                    else if (now > deadline) break;
                }
            }
            atomicOr(&g_fa_fwd_status, 1u);
            return false;
        };
        if constexpr (SPLIT == 1) {
            const float part = fine ? store_row(v, Mc, lc) : 0.f;
            if (!X3 && prep.dO) {   // the same for every thread: all 256 reach the barrier
                float *dsum = reinterpret_cast<float *>(sb + C::DSUM_OFF);
                dsum[t * 128 + r] = part;
                tc::named_bar_sync(1, 256);
                if (fine)
                    prep_row_finish<D>(prep, part, t == 0 ? dsum[128 + r] : 0.f, t == 0, Mc, lc, bh, row, Nq, t, false);
            }
        } else {
            // rank r finalises the columns of warpgroup r; the other warpgroup sends its
            // half row and the row's (m, l) into the peer's shared memory with remote
            // stores, once the peer's MMAs are done (its K ring holds the partials)
            const uint32_t peer_free = base + C::PEER_BAR_OFF, peer_ready = peer_free + 8;
            tc::mbar_arrive_remote(tc::map_to_rank(peer_free, rank ^ 1u));
            if (t != (int)rank) {
                const bool dst_ok = wait_peer(peer_free);
                if (dst_ok) {
                    const uint32_t prow = tc::map_to_rank(base + C::PART_OFF + r * C::PART_STRIDE, rank ^ 1u);
                    const uint32_t pml = tc::map_to_rank(base + C::PART_ML_OFF, rank ^ 1u);
                    const bool ok_part = fine && n > 0;
#pragma unroll
                    for (int c = 0; c < VW / 4; ++c)
                        tc::st_cluster_v4(prow + 16 * c, __float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                          __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
                    tc::st_cluster_f32(pml + r * 4, ok_part ? Mc : -INFINITY);
                    tc::st_cluster_f32(pml + (128 + r) * 4, ok_part ? lc : 0.f);
                }
                tc::mbar_arrive_remote(tc::map_to_rank(peer_ready, rank ^ 1u));   // release: the stores above
            } else {
                const bool got = wait_peer(peer_ready);
                const bool both = __all_sync(0xffffffffu, fine && got);
                float part = 0.f, M = Mc, lrow = lc;
                if (both) {
                    const float *prow = reinterpret_cast<const float *>(sb + C::PART_OFF + r * C::PART_STRIDE);
                    const float *ml = reinterpret_cast<const float *>(sb + C::PART_ML_OFF);
                    const float M1 = ml[r], l1 = ml[128 + r];
                    M = fmaxf(Mc, M1);
                    const float b0 = Mc > -INFINITY ? exp2f(Mc - M) : 0.f;
                    const float b1 = l1 > 0.f ? exp2f(M1 - M) : 0.f;
#pragma unroll
                    for (int c = 0; c < VW / 4; ++c) {
                        const float4 pv = reinterpret_cast<const float4 *>(prow)[c];
                        v[4 * c + 0] = fmaf(pv.x, b1, v[4 * c + 0] * b0);
                        v[4 * c + 1] = fmaf(pv.y, b1, v[4 * c + 1] * b0);
                        v[4 * c + 2] = fmaf(pv.z, b1, v[4 * c + 2] * b0);
                        v[4 * c + 3] = fmaf(pv.w, b1, v[4 * c + 3] * b0);
                    }
                    lrow = lc * b0 + l1 * b1;
                    part = store_row(v, M, lrow);
                }
                if (prep.dO) {
                    // The row's other half was finalised by the other rank: rank 1 hands
                    // its half rowsum to rank 0 (always, so that rank 0 never waits in
                    // vain nor exits before the store lands), and rank 0 writes the
                    // row's constants.
                    const uint32_t peer_d = base + C::PEER_BAR_OFF + 16;
                    if (rank == 1) {
                        tc::st_cluster_f32(tc::map_to_rank(base + C::DSUM_OFF + 4u * r, 0u), part);
                        tc::mbar_arrive_remote(tc::map_to_rank(peer_d, 0u));   // release: the store above
                        if (both) prep_row_finish<D>(prep, part, 0.f, false, M, lrow, bh, row, Nq, t, false);
                    } else {
                        const bool got_d = wait_peer(peer_d);
                        if (both) {
                            const float other = got_d ? reinterpret_cast<const float *>(sb + C::DSUM_OFF)[r] : 0.f;
                            prep_row_finish<D>(prep, part, other, got_d, M, lrow, bh, row, Nq, t, false);
                        }
                    }
                }
            }
        }
    }
    // ------------------------------------------------------------ teardown
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Persistent form for many short query tiles: one CTA per SM walks a list of
// work units (one 128-row query tile of one batch*head each).  Same roles,
// TMEM layout and per-tile pipeline as fa_fwd_tc_kernel; what it adds is the
// hand-over between units -- the next unit's Q and first K/V tiles load, and
// its first S MMAs run, under the previous unit's last tiles and epilogue.
template <int D, bool CAUSAL, bool VIEW4>
__global__ void __launch_bounds__(NTHREADS, 1)
    fa_fwd_tc_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     void *__restrict__ Ov,
                     float *__restrict__ Lout, int Nq, int Nk, int BH, int num_q_tiles, float scale_log2,
                     uint32_t wait_limit, uint32_t force_stall, int H, int dv, FaStrides so, FwdPrep prep) {
    using C = FwdCfg<D>;
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(Ov);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    tc::pdl_launch_dependents();

    // Work units are numbered longest first (high query tiles see the most keys
    // under causal masking) and dealt to the CTAs in snake order: round r gives
    // CTA b unit r*G + b when r is even and r*G + G-1-b when r is odd, which
    // evens out the causal lengths.
    const int num_units = num_q_tiles * BH;
    const int G = (int)gridDim.x, cb = (int)blockIdx.x;
    struct Unit {
        int bh, q0, jb, n;   // batch*head, first query row, first key tile (0), key tiles
    };
    auto unit_of = [&](int r, Unit &w) -> bool {
        const int u = r * G + ((r & 1) ? G - 1 - cb : cb);
        if (u >= num_units) return false;
        const int qt = num_q_tiles - 1 - u / BH;
        w.bh = u % BH;
        w.q0 = qt * BM;
        const int kend = CAUSAL ? min(Nk, w.q0 + BM) : Nk;
        w.jb = 0;
        w.n = (kend + BN - 1) / BN;
        return true;
    };

    // Tiles are numbered globally over this CTA's units (g); the two S / P / O
    // buffers and softmax warpgroups alternate with g, and every ring index and
    // barrier phase below follows from g, so one unit runs into the next: its
    // Q and first K/V tiles load, and its first S MMAs run, under the previous
    // unit's last tiles and epilogue.
    auto bar = [&](int i) { return base + C::BAR_OFF + 8u * i; };
    const uint32_t q_full = bar(0);
    constexpr int RB = 1 + C::KST + C::VST + C::R;          // first non-ring barrier
    auto k_full = [&](int s) { return bar(1 + s); };
    auto v_full = [&](int s) { return bar(1 + C::KST + s); };
    auto pv_done_bar = [&](int g) { return bar(1 + C::KST + C::VST + (int)((uint32_t)g % C::R)); };
    auto pv_done_par = [&](int g) { return ((uint32_t)g / C::R) & 1u; };
    auto s_full = [&](int t) { return bar(RB + t); };
    auto p_full = [&](int t) { return bar(RB + 2 + t); };
    const uint32_t drain = bar(RB + 4);
    const uint32_t never = bar(RB + 5);   // fault injection: nothing ever arrives here
    auto s_free = [&](int t) { return bar(RB + 6 + t); };   // softmax has read S_t (separate-P layout)
    const uint32_t q_empty = bar(RB + 8);     // S MMAs of the unit done: the Q buffer may be refilled
    const uint32_t o_free = bar(RB + 9);      // epilogue has read O_0, O_1: the next unit may overwrite them
    // the warpgroup not holding unit u's last tile has published its (m, l); one barrier
    // per unit parity, so that it can publish unit u + 1's before the merge of u waits
    auto merge_bar = [&](int u) { return bar(u & 1 ? RB + 16 : RB + 10); };
    // fused preprocessing, d = 64: a unit's dO rows have landed in buffer b (do_full) /
    // have been read by the epilogue (do_free); buffers alternate by unit
    auto do_full = [&](int b) { return bar(RB + 12 + b); };
    auto do_free = [&](int b) { return bar(RB + 14 + b); };
    float *stat_sm = reinterpret_cast<float *>(sb + C::STAT_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::MISC_OFF);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < C::KST; ++s) tc::mbar_init(k_full(s), 1);
        for (int s = 0; s < C::VST; ++s) tc::mbar_init(v_full(s), 1);
        for (int s = 0; s < C::R; ++s) tc::mbar_init(pv_done_bar(s), 1);
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(s_full(t), 1);
            tc::mbar_init(p_full(t), 128);
            tc::mbar_init(s_free(t), 128);
        }
        tc::mbar_init(drain, 1);
        tc::mbar_init(never, 1);
        tc::mbar_init(q_empty, 1);
        tc::mbar_init(o_free, 128);
        tc::mbar_init(merge_bar(0), 128);
        tc::mbar_init(merge_bar(1), 128);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(do_full(b), 1);
            tc::mbar_init(do_free(b), 128);
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
    tc::pdl_wait();   // the previous kernel's writes (Q, K, V; readers of O and L) are done
    const tc::Waiter W{abort_flag, &g_fa_fwd_status, wait_limit, 1u};

    // registers: warpgroup 0 (producer, MMA issuer, two idle warps) hands its share
    // to the two softmax warpgroups; each warpgroup changes its budget in one place
    if (warp < 4) {
    tc::regs_dec<56>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmQ);
            tc::tma_prefetch_desc(&tmK);
            tc::tma_prefetch_desc(&tmV);
            int g0 = 0, k_issued = 0, v_issued = 0, q_issued = 0;
            bool ok = true;
            Unit w;
            for (int u = 0; ok && unit_of(u, w); ++u) {
                // the Q buffer is refilled once the previous unit's S MMAs have completed
                if (u > 0 && !(ok = W.wait(q_empty, (u - 1) & 1))) break;
                if (!(ok = tc::in_bounds(w.q0 < Nq && w.bh < BH, &g_fa_fwd_status, abort_flag))) break;
                tc::mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
                for (int c = 0; c < C::CHUNKS; ++c)
                    tc::tma_load_rows<VIEW4>(base + C::Q_OFF + c * C::CHUNK_BYTES, &tmQ, q_full, c * 64, w.q0, w.bh, H);
                q_issued = u + 1;
                auto load = [&](const CUtensorMap *m, uint32_t ring, uint32_t st, int g, int key0, uint32_t full) {
                    // debug build: a key tile past the keys, or wholly above the diagonal, is never loaded
                    if (!tc::in_bounds(key0 < Nk && (!CAUSAL || key0 <= w.q0 + BM - 1), &g_fa_fwd_status, abort_flag))
                        return false;
                    // the slot last held tile g - st: wait until PV of that tile has completed
                    if (g >= (int)st && !W.wait(pv_done_bar(g - (int)st), pv_done_par(g - (int)st))) return false;
                    tc::mbar_arrive_expect_tx(full, C::TILE_BYTES);
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tc::tma_load_rows<VIEW4>(ring + ((uint32_t)g % st) * C::TILE_BYTES + c * C::CHUNK_BYTES, m, full,
                                        c * 64, key0, w.bh, H);
                    return true;
                };
                // order K_0, K_1, V_0, K_2, V_1, ...: the MMA warp uses K_{j+1} before V_j
                for (int j = 0; j <= w.n; ++j) {
                    if (j < w.n) {
                        const int g = g0 + j;
                        if (!(ok = load(&tmK, base + C::K_OFF, C::KST, g, (w.jb + j) * BN, k_full((uint32_t)g % C::KST))))
                            break;
                        k_issued = g + 1;
                    }
                    if (j >= 1) {
                        const int g = g0 + j - 1;
                        if (!(ok = load(&tmV, base + C::V_OFF, C::VST, g, (w.jb + j - 1) * BN,
                                        v_full((uint32_t)g % C::VST))))
                            break;
                        v_issued = g + 1;
                    }
                }
                g0 += w.n;
            }
            if constexpr (tc::kDebug) atomicAdd(&g_fa_fwd_rows, (unsigned long long)k_issued * BN);
            if (*abort_flag) {
                // let the copies already in flight land before the CTA exits
                for (int g = k_issued - 1; g >= 0 && g >= k_issued - C::KST; --g)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(k_full(g % C::KST), (g / C::KST) & 1); ++i) {
                    }
                for (int g = v_issued - 1; g >= 0 && g >= v_issued - C::VST; --g)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(v_full(g % C::VST), (g / C::VST) & 1); ++i) {
                    }
                if (q_issued > 0)
                    for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(q_full, (q_issued - 1) & 1); ++i) {
                    }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ fused preprocessing
        // d = 64: each unit's dO rows into the unit's buffer (one bulk copy of the
        // contiguous rows), and the unit's rows of the dQ accumulator cleared, ahead of
        // the epilogue that reads them
        if (D == 64 && prep.dO) {
            Unit w;
            int issued = 0;
            bool ok = true;
            for (int u = 0; ok && unit_of(u, w); ++u) {
                const int b = u & 1;
                if (lane == 0) {
                    // the buffer last held unit u - 2's rows: wait until its epilogue read them
                    if (u >= 2) ok = W.wait(do_free(b), ((u - 2) >> 1) & 1);
                    if (ok) {
                        tc::mbar_arrive_expect_tx(do_full(b), C::DOS_BYTES);
                        tc::tma_load_rows<VIEW4>(base + C::DOS_OFF + b * C::DOS_BYTES, &tmdO, do_full(b), 0, w.q0, w.bh,
                                                 H);
                        issued = u + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok && prep.dQa) {
                    float4 *z = reinterpret_cast<float4 *>(prep.dQa + ((size_t)w.bh * ((Nq + 127) / 128 * 128) + w.q0) * 64);
                    for (int i = lane; i < BM * 64 / 4; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            // the copies land before the CTA may exit
            if (lane == 0)
                for (int u = issued - 1; u >= 0 && u >= issued - 2; --u)
                    for (uint32_t i = 0; i < (1u << 22) && !tc::mbar_try_wait(do_full(u & 1), (u >> 1) & 1); ++i) {
                    }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop so that descriptors stay warp-uniform and
        // cheap to form; one elected lane issues the tcgen05 instructions.
        const bool leader = tc::elect_one();
        constexpr uint32_t idesc_s = tc::idesc_bf16(BM, BN, false, false);
        constexpr uint32_t idesc_o = tc::idesc_bf16(BM, D, false, true);
        const uint64_t qd = tc::sdesc_sw128(base + C::Q_OFF, 16, 1024);
        const uint64_t kd = tc::sdesc_sw128(base + C::K_OFF, 16, 1024);
        const uint64_t vd = tc::sdesc_sw128(base + C::V_OFF, C::CHUNK_BYTES, 1024);
        bool ok = true;
        if (force_stall) ok = __all_sync(0xffffffffu, W.wait(never, 0));
        auto wait_all = [&](uint32_t b, uint32_t par) { return __all_sync(0xffffffffu, W.wait(b, par)); };
        // ring positions advance by one per S (K ring) and per PV (V ring); g_s and
        // g_pv are the global indices of the next S and the next PV
        int k_slot = 0, v_slot = 0, g_s = 0, g_pv = 0;
        uint32_t k_par = 0, v_par = 0;
        // S runs LAG tiles ahead of PV: with P in its own columns S_{j+2} can be
        // computed while the softmax works on S_j; with P over S, S_{j+1} only
        constexpr int LAG = C::SEP_P ? 2 : 1;
        Unit w;
        for (int u = 0; ok && unit_of(u, w); ++u) {
            const int n = w.n;
            if (!(ok = wait_all(q_full, u & 1))) break;
            for (int i = 0; ok && i < n + LAG; ++i) {
                if (i < n) {
                    // S_g = Q K_g^T into S_{g&1}; with separate P, S_{g&1} is free once S_{g-2} has been read
                    const int t = g_s & 1;
                    const bool ready = (C::SEP_P && g_s >= 2)
                                           ? W.wait2(s_free(t), ((g_s - 2) >> 1) & 1, k_full(k_slot), k_par)
                                           : W.wait(k_full(k_slot), k_par);
                    if (!(ok = __all_sync(0xffffffffu, ready))) break;
                    tc::fence_after_sync();
                    if (leader) {
                        const uint64_t ks = kd + ((k_slot * C::TILE_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4;
                            tc::mma_ss(tmem + C::S_COL0 + t * 128, qd + off, ks + off, idesc_s, kk > 0 ? 1u : 0u);
                        }
                        tc::mma_commit(s_full(t));
                        if (i == n - 1) tc::mma_commit(q_empty);   // last S of the unit: Q may be refilled
                    }
                    __syncwarp();
                    ++g_s;
                    if (++k_slot == C::KST) { k_slot = 0; k_par ^= 1u; }
                }
                if (i >= LAG) {
                    // O_t (+)= P_g V_g; the first PV of a unit overwrites O, so the
                    // previous unit's epilogue must have read it
                    const int j = i - LAG, t = g_pv & 1;
                    if (j == 0 && u > 0 && !(ok = wait_all(o_free, (u - 1) & 1))) break;
                    if (!(ok = __all_sync(0xffffffffu, W.wait2(p_full(t), (g_pv >> 1) & 1, v_full(v_slot), v_par))))
                        break;
                    tc::fence_after_sync();
                    if (leader) {
                        const uint64_t vs = vd + ((v_slot * C::TILE_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)   // 16 keys = 16 rows of V = 2048 bytes per k-step
                            tc::mma_ts(tmem + C::O_COL0 + t * D, tmem + C::P_COL0 + t * C::P_STRIDE + kk * 8,
                                       vs + kk * 128, idesc_o, (j >= 2 || kk > 0) ? 1u : 0u);
                        tc::mma_commit(pv_done_bar(g_pv));
                    }
                    __syncwarp();
                    ++g_pv;
                    if (++v_slot == C::VST) { v_slot = 0; v_par ^= 1u; }
                }
            }
            if (ok && n == 0) {
                if (leader) tc::mma_commit(q_empty);   // nothing reads Q: release it at once
                __syncwarp();
            }
        }
        if (!ok && leader) {
            // wait (bounded) for the MMAs already issued before TMEM is released
            tc::mma_commit(drain);
            for (uint32_t i = 0; i < (1u << 20) && !tc::mbar_try_wait(drain, 0); ++i) {
            }
        }
        __syncwarp();
    }
    } else {
        tc::regs_inc<224>();
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 4) >> 2;
        const int r = ((warp & 3) << 5) + lane;            // row within the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_base + C::S_COL0 + t * 128;
        const uint32_t tP = tmem + lane_base + C::P_COL0 + t * C::P_STRIDE;
        const uint32_t tO = tmem + lane_base + C::O_COL0 + t * D;
        bool ok = true;
        int g0 = 0;
        Unit w;
        for (int u = 0; ok && unit_of(u, w); ++u) {
            const int n = w.n, bh = w.bh, row = w.q0 + r;
            // a strided output row's offset, taken now and parked in shared memory:
            // computed at the epilogue it would compete for registers with the row
            volatile long long *orow_sm = reinterpret_cast<volatile long long *>(sb + C::OROW_OFF) + (threadIdx.x - 128);
            if constexpr (VIEW4) *orow_sm = fa_row_offset(so, H, bh, row);
            // this warpgroup's tiles of the unit: local j = jt, jt + 2, ... (global g = g0 + j has parity t)
            const int j_0 = (0 - g0) & 1, j_1 = (1 - g0) & 1;
            const int jt = t == 0 ? j_0 : j_1;
            const int nt = n > jt ? (n - jt + 1) >> 1 : 0;
            float m = -INFINITY, l = 0.f;
            for (int k = 0; k < nt; ++k) {
                const int j = jt + 2 * k, g = g0 + j;
                const int k0 = (w.jb + j) * BN;
                ok = W.wait(s_full(t), (g >> 1) & 1);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc::fence_after_sync();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_x32(tS + 32 * c, sr[c]);
                tc::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence_x32(sr[c]);
                if constexpr (C::SEP_P) {
                    tc::fence_before_sync();
                    tc::mbar_arrive(s_free(t));   // S_t may now be overwritten by S_{g+2}
                }
                float s[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
                const bool need_mask = (CAUSAL && k0 + BN - 1 > w.q0) || (k0 + BN > Nk);
                if (need_mask) {
                    const int lim = min(Nk - 1, CAUSAL ? row : Nk - 1) - k0;   // last visible column
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i > lim) s[i] = -INFINITY;
                }
                // row max as four independent chains (short dependency paths)
                float mq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) mq[q] = tc::fmax3(s[q], s[4 + q], s[8 + q]);
#pragma unroll
                for (int i = 12; i < 124; i += 8)
#pragma unroll
                    for (int q = 0; q < 4; ++q) mq[q] = tc::fmax3(mq[q], s[i + q], s[i + 4 + q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) mq[q] = fmaxf(mq[q], s[124 + q]);
                const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                const float m_cand = fmaxf(m, mx * scale_log2);
                const bool rescale = m_cand > m + kRescaleThreshold;
                float alpha = 1.f;
                if (rescale) {
                    alpha = tc::ex2(m - m_cand);
                    m = m_cand;
                }
                l *= alpha;
                const float nm = -m;
                uint32_t p[64];
                float rs[4][2] = {};
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float x0, x1;
                    tc::fma2(x0, x1, s[2 * i], s[2 * i + 1], scale_log2, scale_log2, nm, nm);
                    const float e0 = tc::ex2(x0), e1 = tc::ex2(x1);
                    tc::add2(rs[i & 3][0], rs[i & 3][1], rs[i & 3][0], rs[i & 3][1], e0, e1);
                    p[i] = tc::pack_bf16(e0, e1);
                }
                l += ((rs[0][0] + rs[0][1]) + (rs[1][0] + rs[1][1])) + ((rs[2][0] + rs[2][1]) + (rs[3][0] + rs[3][1]));
                if (C::SEP_P && g >= 2) {
                    // P_t is still read by the PV of this warpgroup's previous tile until that completes
                    ok = W.wait(pv_done_bar(g - 2), pv_done_par(g - 2));
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc::fence_after_sync();
                }
                tmem_st_x32(tP, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                tmem_st_x32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                if (k > 0 && __any_sync(0xffffffffu, rescale)) {
                    // O_t holds the sum up to this warpgroup's previous tile: rescale it in place
                    ok = W.wait(pv_done_bar(g - 2), pv_done_par(g - 2));
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + 32 * c, o);
                        tc::tmem_ld_wait();
                        reg_fence_x32(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st_x32(tO + 32 * c, o);
                    }
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();
                tc::mbar_arrive(p_full(t));
            }
            // ---- merge.  The warpgroup holding the unit's last tile merges both partial
            // results and writes the rows; the other publishes its (m, l) and goes on to
            // the next unit at once, so the epilogue overlaps its tiles.
            const int t_last = n > 0 ? (g0 + n - 1) & 1 : 0;
            float *m_sm = stat_sm + (u & 1) * 512;
            float *l_sm = m_sm + 256;
            bool fine = ok;
            if (t != t_last) {
                m_sm[t * 128 + r] = m;
                l_sm[t * 128 + r] = l;
                tc::mbar_arrive(merge_bar(u));   // release: the stores above
            } else {
                const int to = t ^ 1;
                const bool has_o = n > (to == 0 ? j_0 : j_1);   // the other warpgroup had tiles
                fine = W.wait(merge_bar(u), (u >> 1) & 1) && fine;
                if (fine && n > 0) fine = W.wait(pv_done_bar(g0 + n - 1), pv_done_par(g0 + n - 1));
                fine = __all_sync(0xffffffffu, fine);
                float mo = -INFINITY, lo = 0.f;
                if (fine && has_o) {
                    mo = m_sm[to * 128 + r];
                    lo = l_sm[to * 128 + r];
                }
                const float Mc = fmaxf(m, mo);
                const float am = exp2f(m - Mc), ao = has_o ? exp2f(mo - Mc) : 0.f;
                const float lc = l * am + lo * ao;
                const float inv = 1.f / lc;
                const uint32_t tOm = tmem + lane_base + C::O_COL0 + t * D;
                const uint32_t tOo = tmem + lane_base + C::O_COL0 + to * D;
                __nv_bfloat16 *orow;
                if constexpr (VIEW4) orow = O + *orow_sm;
                else orow = O + ((size_t)bh * Nq + row) * D;
                if (D == 64 && prep.dO && fine)
                    fine = __all_sync(0xffffffffu, W.wait(do_full(u & 1), (u >> 1) & 1));
                const uint8_t *srow = nullptr;   // d = 64: the row of dO in shared memory (swizzled)
                if constexpr (D == 64) srow = sb + C::DOS_OFF + (u & 1) * C::DOS_BYTES + r * 128;
                if (fine) tc::fence_after_sync();
                // 32 columns at a time: both accumulators, the merged and normalised row, its
                // store, and (fused preprocessing) its part of rowsum(dO * O)
                float part = 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t om[32] = {}, oo[32] = {};
                    if (fine) {
                        tmem_ld_x32(tOm + 32 * c, om);
                        if (has_o) tmem_ld_x32(tOo + 32 * c, oo);
                        tc::tmem_ld_wait();
                    }
                    reg_fence_x32(om);
                    reg_fence_x32(oo);
                    float x[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        x[i] = fmaf(__uint_as_float(oo[i]), ao, __uint_as_float(om[i]) * am) * inv;
                    if (fine && row < Nq) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 q;
                            q.x = tc::pack_bf16(x[8 * q4 + 0], x[8 * q4 + 1]);
                            q.y = tc::pack_bf16(x[8 * q4 + 2], x[8 * q4 + 3]);
                            q.z = tc::pack_bf16(x[8 * q4 + 4], x[8 * q4 + 5]);
                            q.w = tc::pack_bf16(x[8 * q4 + 6], x[8 * q4 + 7]);
                            if (!VIEW4 || 32 * c + 8 * q4 < dv)   // columns past a head dim below 64 are padding
                                reinterpret_cast<uint4 *>(orow + 32 * c)[q4] = q;
                        }
                        if (prep.dO) {
                            const __nv_bfloat16 *g = nullptr;
                            if (!srow) {
                                if constexpr (VIEW4)
                                    g = static_cast<const __nv_bfloat16 *>(prep.dO) +
                                        fa_row_offset(prep.sdo, H, bh, row) + 32 * c;
                                else
                                    g = static_cast<const __nv_bfloat16 *>(prep.dO) + ((size_t)bh * Nq + row) * D + 32 * c;
                            }
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                if (!VIEW4 || 32 * c + 8 * q4 < dv) {
                                    const uint4 y = srow ? swizzled_chunk(srow, r, 4 * c + q4)
                                                         : __ldg(reinterpret_cast<const uint4 *>(g) + q4);
                                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 f = __bfloat1622float2(h[e]);
                                        part = fmaf(x[8 * q4 + 2 * e], f.x, part);
                                        part = fmaf(x[8 * q4 + 2 * e + 1], f.y, part);
                                    }
                                }
                            }
                        }
                    }
                }
                // O_0 and O_1 have been read: the next unit's first PV may overwrite them
                tc::fence_before_sync();
                tc::mbar_arrive(o_free);
                if (D == 64 && prep.dO) {
                    // this unit's dO rows have been read: the buffer may take unit u + 2's
                    tc::fence_proxy_async_smem();
                    tc::mbar_arrive(do_free(u & 1));
                }
                if (fine && row < Nq) Lout[(size_t)bh * Nq + row] = Mc * kLn2 + logf(lc);
                if (fine && prep.dO)   // d = 64: warp 2 cleared the accumulator rows
                    prep_row_finish<D>(prep, part, 0.f, true, Mc, lc, bh, row, Nq, 0, D != 64);
            }
            g0 += n;
            if (!fine) ok = false;
        }
    }
    // ------------------------------------------------------------ teardown
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// (B*H, N, d) contiguous bf16 tensor -> 3-D map with 64 x rows x 1 boxes, 128-byte
// swizzle.  Rows past N in a batch*head read as zero.
bool tc_make_map_3d(CUtensorMap_st *m, const void *ptr, int BH, int N, int d, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_plain_layout(const FaProblem &p, const FaStrides &s, int N) {
    const long long n = p.d, h = (long long)N * p.d, b = (long long)p.H * N * p.d;
    return (N <= 1 || s.n == n) && (p.H <= 1 || s.h == h) && (p.B <= 1 || s.b == b);
}

// Encoded maps are kept in a small table keyed by everything they encode (pointer,
// sizes, strides, box, rank): a step's launches reuse the same few tensors, and a
// hit costs a short scan instead of a descriptor encode.  A map holds only the
// address and geometry, so an entry never goes stale.
namespace {
struct MapKey {
    const void *ptr;
    long long b, h, n, sb, sh, sn;
    int d, box_rows, view4;
    bool operator==(const MapKey &o) const {
        return ptr == o.ptr && b == o.b && h == o.h && n == o.n && sb == o.sb && sh == o.sh && sn == o.sn &&
               d == o.d && box_rows == o.box_rows && view4 == o.view4;
    }
};
constexpr int kMapCache = 32;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_used = 0, g_map_next = 0;
}  // namespace

bool tc_make_map(CUtensorMap_st *m, const void *ptr, const FaProblem &p, const FaStrides &s, int N, int box_rows,
                 bool view4) {
    const MapKey key{ptr, p.B, p.H, N, s.b, s.h, s.n, p.d, box_rows, view4 ? 1 : 0};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (int i = 0; i < g_map_used; ++i)
            if (g_map_key[i] == key) {
                *reinterpret_cast<CUtensorMap *>(m) = g_map_val[i];
                return true;
            }
    }
    const bool ok = view4 ? tc_make_map_4d(m, ptr, p.B, p.H, N, p.d, s, box_rows)
                          : tc_make_map_3d(m, ptr, p.BH, N, p.d, box_rows);
    if (ok) {
        std::lock_guard<std::mutex> lock(g_map_mu);
        const int i = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
        g_map_key[i] = key;
        g_map_val[i] = *reinterpret_cast<CUtensorMap *>(m);
    }
    return ok;
}

// (BH, rows, cols) contiguous fp32 accumulator -> 3-D map with 32 x 128 x 1 boxes
// (one 128-byte swizzled row of 32 floats per row), for TMA reductions into it
bool tc_make_map_acc(CUtensorMap_st *m, const void *ptr, int BH, int rows, int cols) {
    const MapKey key{ptr, BH, 0, rows, 0, 0, 0, cols, 128, 2};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (int i = 0; i < g_map_used; ++i)
            if (g_map_key[i] == key) {
                *reinterpret_cast<CUtensorMap *>(m) = g_map_val[i];
                return true;
            }
    }
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)rows * cols * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const bool ok = enc(reinterpret_cast<CUtensorMap *>(m), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (ok) {
        std::lock_guard<std::mutex> lock(g_map_mu);
        const int i = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
        g_map_key[i] = key;
        g_map_val[i] = *reinterpret_cast<CUtensorMap *>(m);
    }
    return ok;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and device
cudaError_t tc_set_smem_once(const void *kernel, int bytes) {
    static std::mutex mu;
    static const void *fn[128];
    static unsigned long long mask[128];
    static int used = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    while (i < used && fn[i] != kernel) ++i;
    if (i < used && bit && (mask[i] & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) {
        if (i == used && used < 128) fn[used++] = kernel;
        if (i < used) mask[i] |= bit;
    }
    return e;
}

// multiprocessor count of the current device, looked up once per device
int tc_sm_count() {
    static std::atomic<int> sms[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64) {
        const int v = sms[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 148;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

// (B, H, N, d) bf16 view -> 4-D map over (d, N, H, B) with 64 x rows x 1 x 1 boxes,
// 128-byte swizzle.  Rows past N in a batch*head read as zero.  The strides are
// the view's own (positive multiples of 16 bytes below 2^40 bytes), in any order.
bool tc_make_map_4d(CUtensorMap_st *m, const void *ptr, int B, int H, int N, int d, const FaStrides &s,
                    int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)s.n * 2, (cuuint64_t)s.h * 2, (cuuint64_t)s.b * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 with d in {16, 32, 64, 128}.  Head dims 16 and 32 run the d = 64 kernels:
// their TMA boxes are 64 columns wide and the columns past d read as zero, which
// adds nothing to Q K^T and leaves zero output columns that are never stored.
// fp32 with d in {16, 32, 64} may run the same kernels on split bf16 pairs (X3):
// always (FA_FP32_SPLIT), never (FA_FP32_EXACT), or (FA_FP32_AUTO) when
// |scale| * sqrt(d) <= 1, where unit-variance inputs give unit-variance scores and
// the split products' relative error (about 3 * 2^-16 of sum |x y|) stays well
// inside fp32's tolerance; larger scales take the CUDA-core kernels.  A thread may
// turn X3 off for its own calls (the no-allocation entry point does, where the
// split copies do not fit its scratch).
static std::atomic<int> g_fp32_mode{FA_FP32_AUTO};
static thread_local bool t_x3_off = false;
void tc_disable_x3(bool off) { t_x3_off = off; }
void tc_set_fp32_mode(int mode) { g_fp32_mode.store(mode); }
int tc_get_fp32_mode() { return g_fp32_mode.load(); }

static bool tiles_fit(const FaProblem &p) { return p.Nq >= 128 && p.Nk >= 128 && p.BH >= 1; }

bool tc_x3_possible(const FaProblem &p) {
    return p.dtype == FA_DTYPE_F32 && (p.d == 16 || p.d == 32 || p.d == 64 || p.d == 128) && tiles_fit(p) &&
           !t_x3_off && g_fp32_mode.load() != FA_FP32_EXACT;
}

size_t tc_x3_row_bytes(const FaProblem &p) { return p.d <= 64 ? 256 : 512; }

bool tc_x3(const FaProblem &p) {
    return tc_x3_possible(p) &&
           (g_fp32_mode.load() == FA_FP32_SPLIT || fabsf(p.scale) * sqrtf((float)p.d) <= 1.0001f);
}

bool tc_fwd_supported(const FaProblem &p) {
    if (p.dtype == FA_DTYPE_F32) return tc_x3(p);
    return p.dtype == FA_DTYPE_BF16 && (p.d == 16 || p.d == 32 || p.d == 64 || p.d == 128) && tiles_fit(p);
}

static int sm_count() { return tc_sm_count(); }

template <int D, bool CAUSAL, int SPLIT, bool PERSIST, bool VIEW4, bool X3 = false>
static cudaError_t launch_fwd(const FaProblem &p, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                              const CUtensorMap &mdo, void *O, float *L, const FwdPrep &prep, cudaStream_t st) {
    static_assert(!(PERSIST && SPLIT > 1), "persistent units are not split");
    static_assert(!(PERSIST && X3), "split fp32 operands run one unit per CTA (or cluster)");
    using C = FwdCfg<D>;
    void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, void *, float *, int, int,
                 int, int, float, uint32_t, uint32_t, int, int, FaStrides, FwdPrep);
    if constexpr (PERSIST) kern = fa_fwd_tc_persistent_kernel<D, CAUSAL, VIEW4>;
    else kern = fa_fwd_tc_kernel<D, CAUSAL, SPLIT, VIEW4, X3>;
    cudaError_t e = tc_set_smem_once(reinterpret_cast<const void *>(kern), (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int qtiles = (p.Nq + BM - 1) / BM;
    // persistent: one CTA per SM walking its share of the work units; otherwise
    // one CTA (or cluster) per unit, handed out by the hardware as SMs free up
    const long long units = (long long)qtiles * p.BH;
    const long long grid = PERSIST ? std::min<long long>(units, sm_count()) : units * SPLIT;
    const float scale_log2 = p.scale * 1.4426950408889634f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = SPLIT;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = SPLIT > 1 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mdo, O, L, p.Nq, p.Nk, p.BH, qtiles,
                           scale_log2, p.wait_limit, p.force_stall, p.H, p.d, p.sO, prep);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

enum class FwdMode { kStream, kSplit, kPersist };

// Work units are split over a cluster of two CTAs when the longest one (a whole
// row of key tiles) is more than 1.5x the average number of key tiles per SM:
// then it, not the total work, would set the run time.  Many short units (at
// least two per SM, at most 12 key tiles on average) run on persistent CTAs,
// which overlap one unit's epilogue with the next unit's loads and first MMAs;
// otherwise the hardware hands out one unit per CTA, which balances uneven
// causal lengths by itself.
static FwdMode fwd_mode(const FaProblem &p) {
    const int sms = sm_count();
    const long long qtiles = (p.Nq + BM - 1) / BM;
    long long total = 0, n_max = 0;
    for (long long qt = 0; qt < qtiles; ++qt) {
        const long long kend = p.causal ? std::min<long long>(p.Nk, (qt + 1) * BM) : p.Nk;
        const long long n = (kend + BN - 1) / BN;
        total += n;
        n_max = std::max(n_max, n);
    }
    total *= p.BH;
    const long long units = qtiles * p.BH;
    if (n_max >= 4 && 2 * n_max * sms > 3 * total) return FwdMode::kSplit;
    if (units >= 2LL * sms && total <= 12 * units) return FwdMode::kPersist;
    return FwdMode::kStream;
}

template <int D, bool CAUSAL, bool VIEW4>
static cudaError_t launch_fwd_mode(const FaProblem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                   const CUtensorMap &mv, const CUtensorMap &mdo, void *O, float *L, const FwdPrep &prep,
                                   cudaStream_t st) {
    switch (fwd_mode(p)) {
        case FwdMode::kSplit: return launch_fwd<D, CAUSAL, 2, false, VIEW4>(p, mq, mk, mv, mdo, O, L, prep, st);
        case FwdMode::kPersist: return launch_fwd<D, CAUSAL, 1, true, VIEW4>(p, mq, mk, mv, mdo, O, L, prep, st);
        default: return launch_fwd<D, CAUSAL, 1, false, VIEW4>(p, mq, mk, mv, mdo, O, L, prep, st);
    }
}

template <int D, bool CAUSAL>
static cudaError_t launch_fwd_any(const FaProblem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                  const CUtensorMap &mv, const CUtensorMap &mdo, void *O, float *L, bool view4,
                                  const FwdPrep &prep, cudaStream_t st) {
    return view4 ? launch_fwd_mode<D, CAUSAL, true>(p, mq, mk, mv, mdo, O, L, prep, st)
                 : launch_fwd_mode<D, CAUSAL, false>(p, mq, mk, mv, mdo, O, L, prep, st);
}

cudaError_t tc_fwd(const FaProblem &p, const void *Q, const void *K, const void *V, void *O, float *L,
                   cudaStream_t st, const FwdPrep *prep, bool *prep_done) {
    // contiguous tensors keep 3-D (d, N, B*H) maps and plain row addressing; any
    // strided view, or a head dim below 64 (whose rows are narrower than the
    // kernel's), switches the whole launch to 4-D maps and strided rows
    const bool view4 = p.d < 64 || !tc_plain_layout(p, p.sQ, p.Nq) || !tc_plain_layout(p, p.sK, p.Nk) ||
                       !tc_plain_layout(p, p.sV, p.Nk) || !tc_plain_layout(p, p.sO, p.Nq) ||
                       (prep && prep->dO && !tc_plain_layout(p, prep->sdo, p.Nq));
    CUtensorMap mq, mk, mv;
    if (!tc_make_map(&mq, Q, p, p.sQ, p.Nq, BM, view4) || !tc_make_map(&mk, K, p, p.sK, p.Nk, BN, view4) ||
        !tc_make_map(&mv, V, p, p.sV, p.Nk, BN, view4))
        return cudaErrorInvalidValue;
    FwdPrep none{};
    const FwdPrep &pr = (prep && prep->dO) ? *prep : none;
    // d <= 64 kernels stage the tile's dO rows in shared memory through their own map
    CUtensorMap mdo = mq;
    if (pr.dO && p.d <= 64 && !tc_make_map(&mdo, pr.dO, p, pr.sdo, p.Nq, BM, view4)) return cudaErrorInvalidValue;
    if (prep_done) *prep_done = pr.dO != nullptr;   // every kernel form does it
    if (p.d == 128) return p.causal ? launch_fwd_any<128, true>(p, mq, mk, mv, mdo, O, L, view4, pr, st)
                                    : launch_fwd_any<128, false>(p, mq, mk, mv, mdo, O, L, view4, pr, st);
    return p.causal ? launch_fwd_any<64, true>(p, mq, mk, mv, mdo, O, L, view4, pr, st)
                    : launch_fwd_any<64, false>(p, mq, mk, mv, mdo, O, L, view4, pr, st);
}

// ------------------------------------------------------------------ fp32 inputs (X3)
cudaError_t tc_split_x3(const FaProblem &p, int count, const void *const *X, const FaStrides *s, const int *N,
                        void *const *X2, cudaStream_t st) {
    if (count < 1 || count > 4) return cudaErrorInvalidValue;
    SplitJobs jobs{};
    long long rows_max = 0;
    for (int i = 0; i < count; ++i) {
        jobs.j[i] = SplitJob{static_cast<const float *>(X[i]), static_cast<__nv_bfloat16 *>(X2[i]), s[i], N[i]};
        rows_max = std::max(rows_max, (long long)p.BH * N[i]);
    }
    if (rows_max == 0) return cudaSuccess;
    const int tpr = p.d <= 64 ? 16 : 32;   // threads per row: W / 4
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows_max * tpr + 255) / 256), (unsigned)count);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = p.d <= 64 ? cudaLaunchKernelEx(&cfg, fa_split_x3_kernel<64>, jobs, p.BH, p.H, p.d)
                              : cudaLaunchKernelEx(&cfg, fa_split_x3_kernel<128>, jobs, p.BH, p.H, p.d);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_fwd_x3(const FaProblem &p, const void *Q2, const void *K2, const void *V2, void *O, float *L,
                      cudaStream_t st) {
    if (!tc_x3(p)) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&mq), Q2, p.BH, p.Nq, 128, BM) ||
        !tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&mk), K2, p.BH, p.Nk, 128, BN) ||
        !tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&mv), V2, p.BH, p.Nk, 128, BN))
        return cudaErrorInvalidValue;
    const FwdPrep none{};
    if (p.d == 128) {   // 256-column rows: one unit per CTA
        CUtensorMap wq, wk, wv;
        if (!tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&wq), Q2, p.BH, p.Nq, 256, BM) ||
            !tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&wk), K2, p.BH, p.Nk, 256, BN) ||
            !tc_make_map_3d(reinterpret_cast<CUtensorMap_st *>(&wv), V2, p.BH, p.Nk, 256, BN))
            return cudaErrorInvalidValue;
        return p.causal ? launch_fwd<256, true, 1, false, false, true>(p, wq, wk, wv, wq, O, L, none, st)
                        : launch_fwd<256, false, 1, false, false, true>(p, wq, wk, wv, wq, O, L, none, st);
    }
    // the split form where it pays; otherwise one unit per CTA (no persistent form)
    const bool split = fwd_mode(p) == FwdMode::kSplit;
    if (p.causal)
        return split ? launch_fwd<128, true, 2, false, false, true>(p, mq, mk, mv, mq, O, L, none, st)
                     : launch_fwd<128, true, 1, false, false, true>(p, mq, mk, mv, mq, O, L, none, st);
    return split ? launch_fwd<128, false, 2, false, false, true>(p, mq, mk, mv, mq, O, L, none, st)
                 : launch_fwd<128, false, 1, false, false, true>(p, mq, mk, mv, mq, O, L, none, st);
}

cudaError_t tc_fwd_read_status(unsigned *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_fwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

cudaError_t tc_fwd_read_rows(unsigned long long *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa_fwd_rows, sizeof(unsigned long long), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

cudaError_t tc_fwd_reset_rows(cudaStream_t st) {
    static const unsigned long long zero = 0;
    return cudaMemcpyToSymbolAsync(g_fa_fwd_rows, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
}

cudaError_t tc_fwd_reset_status(cudaStream_t st) {
    static const unsigned zero = 0;
    return cudaMemcpyToSymbolAsync(g_fa_fwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
}
