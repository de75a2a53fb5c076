/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 library, libfa.so.
 *
 * What it computes (CS336 A2 field guide "Systems and Parallelism", §1.2-1.3;
 * FlashAttention-2, Dao 2023):
 *
 *   forward  (problem flash_forward (a)-(c)):
 *     S = scale * Q K^T; causal: keys with index > query index are masked
 *     (contribute exactly zero, the same as adding -1e6 then exponentiating);
 *     P = softmax over each row of S; O = P V; L = m + ln(l) per row, the
 *     natural-log logsumexp of the row that the backward pass reuses.
 *     S and P are never written to memory: the kernels walk key tiles with an
 *     online (running max m, running sum l) softmax.
 *
 *   backward (problem flash_backward):
 *     P = exp(S - L) recomputed from Q, K and L; D = rowsum(dO * O);
 *     dV = P^T dO; dP = dO V^T; dS = P * (dP - D);
 *     dQ = scale * dS K; dK = scale * dS^T Q.
 *
 * Layout.  Q, O, dO, dQ: (B, H, Nq, d) row-major contiguous, i.e. (B*H, Nq, d)
 * with batch and heads flattened in front (problem flash_forward (b)).
 * K, V, dK, dV: (B, H, Nk, d).  L: (B*H, Nq) fp32.  All tensors but L and the
 * workspace share one element type (fa_dtype); O, dQ, dK, dV are written in
 * that type; accumulation is always fp32.  fa_fwd_strided / fa_bwd_strided
 * (below) take any of these tensors as a strided (B, H, N, d) view instead.
 *
 * Causal alignment: top-left.  Key j is visible to query i iff j <= i
 * (absolute indices), so every query row sees key 0 and no row is empty.
 *
 * Ownership.  The caller owns every buffer (device memory), including the
 * backward workspace.  The library allocates no device memory per call, with
 * one exception: fa_fwd / fa_fwd_strided with fp32 inputs on the tensor-core
 * path (fa_set_fp32_mode below) take the split bf16 copies of Q, K and V
 * (256 bytes per row each, 512 at head dim 128) from a stream-ordered memory
 * pool the library owns, one per device; the pool keeps its memory between
 * calls, so only the first call, or the first larger one, allocates.  Calls are asynchronous and
 * ordered on the caller's stream; nothing synchronises inside a call.
 *
 * Errors.  Every entry point returns fa_status and never throws.  Arguments
 * are checked before anything is launched; on a bad argument nothing runs and
 * no output is touched.  A launch failure maps to FA_ERR_LAUNCH.  The kernels
 * bound every wait; a wait that runs out sets a device-side status word that
 * fa_get_device_status() reports as FA_ERR_TIMEOUT.
 *
 * Supported: d in {16, 32, 64, 128}; dtype fp32 or bf16 (fp32 on the tensor
 * cores as split bf16 pairs, see fa_set_fp32_mode); Nq >= 0, Nk >= 1
 * (Nk >= 0 when Nq == 0); B*H*max(Nq,Nk) < 2^31; every pointer 16-byte
 * aligned; scale finite.  B*H*Nq == 0 (and B*H*Nk == 0) is a valid empty call.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL_PTR = 1,             /* a required pointer is NULL                      */
    FA_ERR_BAD_SHAPE = 2,            /* negative / overflowing sizes, Nk == 0 with Nq>0 */
    FA_ERR_UNSUPPORTED_HEAD_DIM = 3, /* d not in {16,32,64,128}                         */
    FA_ERR_UNSUPPORTED_DTYPE = 4,    /* dtype not an fa_dtype value                     */
    FA_ERR_MISALIGNED = 5,           /* a pointer not 16-byte aligned                   */
    FA_ERR_WORKSPACE = 6,            /* workspace NULL or smaller than required         */
    FA_ERR_LAUNCH = 7,               /* CUDA launch or descriptor error                 */
    FA_ERR_TIMEOUT = 8,              /* a device-side bounded wait ran out              */
    FA_ERR_NO_DEVICE = 9,            /* no usable CUDA device                           */
    FA_ERR_BAD_ARG = 10,             /* other invalid argument (is_causal, scale)       */
    FA_ERR_BOUNDS = 11               /* debug build: an in-kernel bounds check failed   */
} fa_status;

typedef enum {
    FA_DTYPE_F32 = 0,
    FA_DTYPE_BF16 = 1
} fa_dtype;

/*
 * Forward pass (flash_forward).  Reads Q, K, V; writes O (input dtype) and
 * L (fp32, natural-log logsumexp per query row).
 */
FA_API fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *L,
                 int B, int H, int Nq, int Nk, int d, float scale, int is_causal,
                 fa_dtype dtype, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for this shape (fp32 D per query row;
 * on the tensor-core path fp32 D and L per query row, rows padded to a
 * multiple of 128, plus, for fp32 inputs on that path, the split bf16 copies of
 * Q, dO, K and V at 256 bytes per row each, 512 at head dim 128).  Returns 0
 * for unsupported arguments.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype);

/*
 * Backward pass (flash_backward).  Reads Q, K, V, O, dO (input dtype) and L
 * (fp32, from fa_fwd on the same inputs); writes dQ, dK, dV (input dtype).
 * Runs fa_bwd_preprocess, then fa_bwd_grads, on `stream`.
 * `workspace` must hold fa_bwd_workspace_size(...) bytes, 16-byte aligned;
 * its contents need not be initialised and are scratch afterwards.
 */
FA_API fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *L, void *dQ, void *dK, void *dV,
                 int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                 void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * The phases of fa_bwd, exported so each kernel can be launched and timed on
 * its own.  On one stream, with the same arguments and workspace, run
 * fa_bwd_preprocess first, then either fa_bwd_grads or both fa_bwd_dkdv and
 * fa_bwd_dq (any order):
 *   fa_bwd_preprocess: D = rowsum(dO * O) into the workspace (the tensor-core
 *                      path also stages L there, scaled by log2(e) and padded);
 *   fa_bwd_dkdv:       dK, dV (one program per key tile, looping over query tiles);
 *   fa_bwd_dq:         dQ (one program per query tile, looping over key tiles);
 *   fa_bwd_grads:      dK, dV and dQ; on the tensor-core path one launch whose
 *                      programs take either kind of work, longest first.
 */
FA_API fa_status fa_bwd_preprocess(const void *O, const void *dO, const float *L,
                            int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype,
                            void *workspace, size_t workspace_bytes, fa_stream_t stream);
FA_API fa_status fa_bwd_dkdv(const void *Q, const void *K, const void *V, const void *dO,
                      const float *L, void *dQ, void *dK, void *dV,
                      int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                      void *workspace, size_t workspace_bytes, fa_stream_t stream);
FA_API fa_status fa_bwd_dq(const void *Q, const void *K, const void *V, const void *dO,
                    const float *L, void *dQ,
                    int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                    void *workspace, size_t workspace_bytes, fa_stream_t stream);
FA_API fa_status fa_bwd_grads(const void *Q, const void *K, const void *V, const void *dO,
                       const float *L, void *dQ, void *dK, void *dV,
                       int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                       void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Forward then backward in one call: the unit the field guide's §1.3.3
 * leaderboard times (a forward plus backward at a fixed configuration, with a
 * given dO).  Writes O and L, then dQ, dK and dV.  Every argument of both
 * passes is checked before the first launch.  On the tensor-core path dO is
 * known to the forward, so its epilogue also forms D = rowsum(dO * O) from the
 * unrounded fp32 O (not from O rounded to the input dtype, as fa_bwd must) and
 * stages the backward's row constants: no preprocessing kernel runs, and the
 * kernels (forward, gradients, plus the dQ conversion when dQ is formed by
 * reduction) go out back to back, each starting while its predecessor drains.
 * O, L and dV are bit for bit those of fa_fwd followed by fa_bwd; dQ and dK
 * differ from them only through that more accurate D.  The CUDA-core path runs
 * fa_fwd then fa_bwd (four kernels).  Contiguous layout; `workspace` as for fa_bwd.
 */
FA_API fa_status fa_fwd_bwd(const void *Q, const void *K, const void *V, const void *dO,
                            void *O, float *L, void *dQ, void *dK, void *dV,
                            int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                            void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd without a caller-supplied workspace.  (No counterpart in the method's
 * description: this exists for callers, not for the algorithm.)
 *
 * For callers that cannot allocate device memory -- code that only receives
 * raw pointers from a host framework and has no allocator of its own, or code
 * that must not call cudaMalloc/cudaFree because those calls can synchronise
 * the device and stall unrelated work.  The scratch lives in a fixed array of
 * FA_NOALLOC_SCRATCH_BYTES of device global memory inside the library, present
 * on every GPU that loads the library until the process exits.  The caller
 * still owns and passes every input and output.  Same arguments, layout and
 * results as fa_bwd.
 *
 *  - Where fa_bwd would form dQ by reduction (FA_DQ_REDUCTION: an fp32 dQ
 *    accumulator of 256 bytes per query row in the workspace) and that does
 *    not fit, this call forms dQ by the separate pass, whose workspace is 8
 *    bytes per query row; shapes needing more than FA_NOALLOC_SCRATCH_BYTES
 *    even so return FA_ERR_WORKSPACE and launch nothing.  8 MiB covers about
 *    one million query rows (B*H*Nq).
 *  - Every call shares the one array: calls whose GPU work overlaps (other
 *    streams, other host threads) race on it.  Serialise them.
 *  - The array's previous contents never matter: each call writes every
 *    scratch word before reading it.
 *  - The first call on each device looks up the array's address with that
 *    device current; make it before any stream capture starts.  The address
 *    is kept for the life of the process: after cudaDeviceReset the array is
 *    loaded again elsewhere, so do not call this entry point after a reset.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
FA_API fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                const float *L, void *dQ, void *dK, void *dV,
                                int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                                fa_stream_t stream);
/* FA_NOALLOC_SCRATCH_BYTES as compiled into the library. */
FA_API size_t fa_noalloc_scratch_bytes(void);

/*
 * Strided (B, H, N, d) views.  The field guide's "Systems and Parallelism"
 * §1.3 builds every tile load from a base pointer, a shape and per-dimension
 * strides, with batch and heads flattened into one batch stride.  Here batch
 * and heads keep a stride each, so a view such as the (B, N, H, d) output of a
 * projection, transposed to (B, H, N, d), is read and written in place with no
 * reshape copy.
 *
 * Element (b, h, n, c) of a tensor with strides s sits at element index
 * b*s.b + h*s.h + n*s.n + c from its base pointer: the head dimension d is
 * contiguous; the other three strides are in elements, not bytes.  A NULL
 * fa_strides pointer means the contiguous layout of the plain entry points,
 * {H*N*d, N*d, d}.
 *
 * Rules (checked before anything is launched):
 *  - for every dimension of extent > 1 (B, H, or N of that tensor) the stride
 *    is positive, a multiple of 16 bytes (8 elements for bf16, 4 for fp32) and
 *    below 2^40 bytes -- else FA_ERR_BAD_SHAPE (not positive or too large) or
 *    FA_ERR_MISALIGNED (not a multiple of 16 bytes); the stride of a
 *    dimension of extent 1 is ignored;
 *  - input views (Q, K, V, O read by the backward, dO) may overlap each other
 *    and themselves (for example two rows sharing elements);
 *  - output views (O written by the forward, dQ, dK, dV) must not overlap
 *    themselves: sorted by stride, each of the four dimensions' strides must be
 *    at least the previous one times its extent -- else FA_ERR_BAD_SHAPE.  An
 *    output must not overlap any input or another output (not checked);
 *  - L stays a contiguous (B*H, Nq) fp32 array, and the workspace is the one
 *    fa_bwd_workspace_size gives.
 * Results are the same, bit for bit, as those of the plain entry points on
 * contiguous copies of the same values.
 */
typedef struct {
    int64_t b, h, n;
} fa_strides;

/* fa_fwd over strided views: reads Q, K, V through sQ, sK, sV; writes O through sO. */
FA_API fa_status fa_fwd_strided(const void *Q, const fa_strides *sQ, const void *K, const fa_strides *sK,
                                const void *V, const fa_strides *sV, void *O, const fa_strides *sO, float *L,
                                int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                                fa_stream_t stream);

/* fa_bwd over strided views: reads Q, K, V, O, dO through their strides; writes
 * dQ, dK, dV through sdQ, sdK, sdV. */
FA_API fa_status fa_bwd_strided(const void *Q, const fa_strides *sQ, const void *K, const fa_strides *sK,
                                const void *V, const fa_strides *sV, const void *O, const fa_strides *sO,
                                const void *dO, const fa_strides *sdO, const float *L,
                                void *dQ, const fa_strides *sdQ, void *dK, const fa_strides *sdK,
                                void *dV, const fa_strides *sdV,
                                int B, int H, int Nq, int Nk, int d, float scale, int is_causal, fa_dtype dtype,
                                void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Name of the kernel family fa_fwd / fa_bwd would use for these arguments and
 * the default scale 1/sqrt(d): "tc" (tcgen05 tensor-core kernels) or "simt"
 * (fp32 CUDA-core kernels), or NULL for unsupported arguments.  Host-only;
 * launches nothing.
 */
FA_API const char *fa_path_name(int Nq, int Nk, int d, int is_causal, fa_dtype dtype);

/*
 * fp32 inputs.  The CUDA-core kernels compute in fp32 throughout.  With Nq and
 * Nk >= 128, fp32 inputs of every head dim can instead run on the tensor
 * cores: every operand x is split into two bf16 numbers, hi = bf16(x) and
 * lo = bf16(x - hi), and every product of the method (S = Q K^T, O = P V, and
 * the backward's five) takes three bf16 products with fp32 accumulation,
 * hi*hi + hi*lo + lo*hi.  With u = 2^-8 (bf16's unit roundoff) each such sum
 * of products x_i y_i carries an error of at most about 3 u^2 sum |x_i y_i|
 * (3 * 2^-16 relative, against about 2^-7 for a product of two bf16-rounded
 * operands and 2^-24 for fp32);
 * through the softmax the scores' absolute error becomes P's relative error,
 * so the outputs' error grows with the size of the scores.
 *   FA_FP32_AUTO   the split path when |scale| * sqrt(d) <= 1 (unit-variance
 *                  inputs then give unit-variance scores, and the outputs meet
 *                  an elementwise 1e-4 tolerance with room to spare), the
 *                  CUDA-core kernels otherwise;
 *   FA_FP32_EXACT  always the CUDA-core kernels;
 *   FA_FP32_SPLIT  the split path wherever the shape allows.
 * The split path forms dQ by the separate pass.  fa_bwd_workspace_size covers
 * the split copies whenever some scale may take them.  Returns the previous
 * mode, or -1 for an unknown value (which changes nothing); do not change it
 * while calls are queued on a stream.
 */
#define FA_FP32_AUTO 0
#define FA_FP32_EXACT 1
#define FA_FP32_SPLIT 2
FA_API int fa_set_fp32_mode(int mode);

/*
 * How the backward forms dQ = scale * dS K (problem flash_backward; the field
 * guide's §1.3.3 names both options: a separate pass, or adding partial sums
 * into one buffer):
 *   FA_DQ_SEPARATE_PASS  one program per query tile loops over the key tiles,
 *                        recomputing S and dP (seven N x N x d products for the
 *                        five of the method; bit-reproducible);
 *   FA_DQ_REDUCTION      each key tile's program also forms dS K for every query
 *                        tile it visits and adds it into an fp32 dQ accumulator
 *                        in the workspace (TMA reductions in L2), then a short
 *                        kernel writes dQ = scale * accumulator in the input
 *                        dtype (five products; dQ's fp32 sums are added in a
 *                        run-dependent order, so dQ can differ between runs in
 *                        the last bit of its fp32 sum, about one bf16 rounding
 *                        step at most; dK, dV, O and L stay bit-reproducible);
 *   FA_DQ_AUTO           per shape, the faster form as measured on GB300: the
 *                        reduction for head dims up to 64 on the tensor-core path
 *                        when causal, or when there are many short key tiles
 *                        (their items then run on persistent CTAs); the separate
 *                        pass otherwise.
 * The CUDA-core (fp32) path always uses the separate pass.
 */
#define FA_DQ_AUTO 0
#define FA_DQ_SEPARATE_PASS 1
#define FA_DQ_REDUCTION 2
/* Sets the process-wide dQ strategy and returns the previous one (-1 for an
 * unknown value, which changes nothing).  The workspace size depends on it:
 * query fa_bwd_workspace_size after setting it, and do not change it while a
 * backward pass is queued on a stream. */
FA_API int fa_set_dq_strategy(int strategy);
/* The strategy fa_bwd would use for these arguments (FA_DQ_SEPARATE_PASS or
 * FA_DQ_REDUCTION), or -1 for unsupported arguments.  Host-only. */
FA_API int fa_bwd_dq_strategy(int B, int H, int Nq, int Nk, int d, int is_causal, fa_dtype dtype);

/*
 * Synchronises `stream`, then returns FA_ERR_TIMEOUT if any kernel since the
 * last fa_reset_device_status() gave up a bounded wait, else the stream's
 * CUDA status mapped to FA_OK / FA_ERR_LAUNCH.
 */
FA_API fa_status fa_get_device_status(fa_stream_t stream);
FA_API fa_status fa_reset_device_status(fa_stream_t stream);

/*
 * Fault injection on the host side: caps every device-side wait loop at
 * `spins` polls (0 restores the default, about a second of polling).  With a
 * tiny cap the tensor-core kernels give up early, record FA_ERR_TIMEOUT and
 * return without hanging; their outputs are then undefined.
 */
FA_API void fa_set_wait_limit(uint32_t spins);

/*
 * Fault injection on the host side: while `on` is nonzero, the tensor-core
 * forward kernel's MMA issuer first waits on a barrier that nothing ever
 * arrives on.  The bounded wait gives up (after the fa_set_wait_limit cap,
 * else about two seconds), the kernel records FA_ERR_TIMEOUT for
 * fa_get_device_status, releases its resources and returns; O and L are then
 * undefined.  For testing the failure path without faulting the GPU.
 */
FA_API void fa_debug_force_stall(int on);

/*
 * Debug build.  libfa_debug.so is the same library compiled with FA_DEBUG: its
 * kernels check, before each tile load and each store of a row, that the index
 * lies inside its tensor and (causal) on or below the diagonal; a failed check
 * records a bit that fa_get_device_status reports as FA_ERR_BOUNDS, skips the
 * access and ends the kernel's waits (never a trap).  It also counts the tile
 * rows that the kernels load.  The release library (libfa.so) carries neither.
 */
FA_API int fa_debug_build(void);   /* 1 in libfa_debug.so, 0 in libfa.so */
/*
 * Rows of tiles loaded since the last reset (debug build; zeros otherwise):
 *   out[0]  key rows the forward loaded (K; V follows tile for tile),
 *   out[1]  query rows the backward's dK/dV work items loaded (Q; dO alike),
 *   out[2]  key rows the backward's dQ work items loaded (K; V alike).
 * A tile counts with its full height (128 rows; 64 for the d = 128 backward's
 * sub-tiles), ragged ends included.  Synchronises `stream`; n entries (at most 3).
 */
FA_API fa_status fa_debug_tile_rows(unsigned long long *out, int n, fa_stream_t stream);
FA_API fa_status fa_debug_reset_tile_rows(fa_stream_t stream);

FA_API const char *fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif
#endif /* FA_H */
