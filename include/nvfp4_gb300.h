/*
 * nvfp4_gb300.h -- C ABI of the GB300 (sm_103a) NVFP4 linear-projection library.
 *
 * What it computes follows "Full-Stack FP4: Stable LLM Pretraining with
 * Quantized Projections, Optimizers, and Attention" (gist.science explainer):
 *   - section 1 (Problem statement): NVFP4 tensor-core arithmetic on Blackwell
 *     for the linear projections of LLM pretraining;
 *   - section 2.1 (LoRA-SVD linear projections), "Mechanism": the weight is
 *     W = W_res + beta * L2 L1 with the rank-r subspace L2 L1 kept in BF16 and
 *     the residual W_res in NVFP4;
 *   - section 3 (Key contributions): "standard NVFP4" quantization; section 2.2
 *     names stochastic rounding (SR), used here for gradients.
 * The pages do not define the NVFP4 encoding; this library reads it as:
 *   E2M1 element codes (grid +-{0,0.5,1,1.5,2,3,4,6}), one unsigned E4M3 scale
 *   per 16 contiguous elements, one FP32 tensor scale S_t = amax / 2688;
 *   s_b = E4M3_rn_satfinite(amax_b / (6 S_t)); d = s_b S_t; y = x * (1/d);
 *   code = E2M1_rn_satfinite(y) (RTN) or stochastic rounding of y driven by
 *   16 bits of Philox4x32-10 per element (SR).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory.  fp4_tensor and the other structs passed by
 *     pointer live in HOST memory and are read during the call only.
 *   - Every call is asynchronous on the caller's stream (cudaStream_t passed as
 *     void*; NULL = legacy default stream) and returns an fp4_status at once.
 *     Its work is ordered after everything queued earlier on that stream
 *     (kernels, copies, memsets, event waits): only the kernels inside one call
 *     overlap one another (programmatic dependent launch).
 *     Argument errors are detected on the host before anything is launched.
 *   - Device-side timeouts (a bounded wait that expired) are recorded in a
 *     device status word; fp4_check_status() synchronises the stream and reads
 *     (and clears) it.
 *   - fp4_last_error() returns a thread-local message for the last failure.
 *   - BF16 tensors are row-major with a leading dimension (in elements);
 *     base pointers and row pitches must be 16-byte aligned.
 *   - Inputs must be finite (no Inf/NaN).
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size      */
    FP4_ERR_MISALIGNED = 2,        /* pointer or pitch not 16-byte aligned       */
    FP4_ERR_UNSUPPORTED_SHAPE = 3, /* shape outside what a kernel supports      */
    FP4_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed          */
    FP4_ERR_TIMEOUT = 5,           /* a device-side bounded wait expired         */
    FP4_ERR_WORKSPACE = 6          /* workspace pointer/size too small           */
} fp4_status;

typedef enum { FP4_ROUND_RTN = 0, FP4_ROUND_SR = 1 } fp4_round_mode;
typedef enum { FP4_OUT_BF16 = 0, FP4_OUT_F32 = 1 } fp4_out_dtype;

/* An NVFP4 tensor of logical shape rows x cols, blocks of 16 along cols.
 *   codes:  rows * cols / 2 bytes, row-major; element 2i of a row sits in the
 *           low nibble of byte i, element 2i+1 in the high nibble; a code is
 *           sign << 3 | magnitude index (0..7 over the E2M1 grid).
 *   scales: fp4_scale_bytes(rows, cols) bytes of UE4M3 block scales in the
 *           layout the block-scaled tensor-core MMA reads: the [rows][cols/16]
 *           scale matrix is cut into 128-row x 4-column atoms of 512 bytes,
 *           atoms ordered by 128-row block then by column group; inside an atom
 *           scale (r, k) is at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + k % 4.
 *           Padding bytes (rows or column groups beyond the tensor) are zero.
 *   scale:  2 floats: scale[0] = S_t (FP32 decode tensor scale), scale[1] = amax.
 * All three pointers are device pointers, 16-byte aligned. */
typedef struct {
    void* codes;
    void* scales;
    float* scale;
    int64_t rows;
    int64_t cols;
} fp4_tensor;

/* Bytes of the MMA-layout scale buffer for a rows x cols NVFP4 tensor. */
int64_t fp4_scale_bytes(int64_t rows, int64_t cols);

/* Tensor amax: *amax_out (device) = max |x| over x[rows][cols] (BF16, pitch ld).
 * The value is written, not accumulated.  rows >= 1, cols % 8 == 0. */
fp4_status fp4_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                    float* amax_out, void* stream);

/* Quantize x[rows][cols] (BF16, pitch ld) row-wise: out is rows x cols with
 * blocks of 16 along cols.  round_mode RTN, or SR with Philox key = seed and
 * counter stream id `sr_stream`; the SR draw of element (r, c) uses element
 * index e = r * cols + c.  amax_opt: device pointer to a precomputed amax of
 * x (or NULL: the call computes it into out->scale[1]).  Requires
 * cols % 16 == 0; out->rows/cols must equal rows/cols.
 * Passage: section 3 "standard NVFP4"; section 2.2 (SR). */
fp4_status fp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                        int round_mode, uint64_t seed, uint32_t sr_stream,
                        const float* amax_opt, fp4_tensor* out, void* stream);

/* Quantize x[rows][cols] column-wise (blocks of 16 along rows) and emit the
 * transposed tensor: out is cols x rows, out row c holding source column c.
 * SR element index is the SOURCE index e = r * cols + c.  Requires rows % 16
 * == 0 and cols % 16 == 0; out->rows == cols, out->cols == rows.
 * This is the K-major operand form of x^T needed by dX = dY W and dW = dY^T X
 * (section 2.1, the backward pass of the projection). */
fp4_status fp4_quantize_transposed(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                   int round_mode, uint64_t seed, uint32_t sr_stream,
                                   const float* amax_opt, fp4_tensor* out, void* stream);

/* Both orientations from one read of x: out_row as fp4_quantize (SR stream
 * sr_stream_row), out_col as fp4_quantize_transposed (SR stream sr_stream_col).
 * Either output may be NULL. */
fp4_status fp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld,
                             int round_mode, uint64_t seed, uint32_t sr_stream_row,
                             uint32_t sr_stream_col, const float* amax_opt,
                             fp4_tensor* out_row, fp4_tensor* out_col, void* stream);

/* Block-scaled NVFP4 GEMM with the fused BF16 low-rank branch.  In exact
 * arithmetic it is
 *   C[m][n] = S_tA * S_tB * sum_k A[m][k] B[n][k]  +  beta * sum_j P[m][j] Q[n][j];
 * what it computes is that sum with the branch folded into the residual's
 * FP32 accumulator, so the output is rounded once:
 *   alpha = fl32(S_tA * S_tB)   (alpha = 1 when that product is 0)
 *   P~[m][j] = bf16(fl32(P[m][j] * fl32(beta / alpha)))
 *   C[m][n] = round_c(fl32(alpha * acc)),  acc = sum_k A B + sum_j P~ Q  (FP32)
 * with A, B their dequantized E2M1 x E4M3 values (exact products), round_c the
 * RN-even conversion to C's type.  P~ adds one BF16 rounding to the branch
 * beyond the BF16 P and Q themselves (relative 2^-9 at most per element of P).
 * A: M x K NVFP4, B: N x K NVFP4 (both blocks along K), P: M x r BF16 (pitch r),
 * Q: N x r BF16 (pitch r); r in {0, 16, 32, 48, 64} (r = 0: P, Q ignored).
 * C: M x N, BF16 or FP32 (c_dtype), pitch ldc elements.
 * Requires M % 128 == 0, N % 128 == 0, K % 64 == 0, and S_tA * S_tB not
 * below the FP32 normal range unless one of them is 0.
 * Passage: section 2.1 "Mechanism" (residual in NVFP4, subspace in BF16,
 * added into the same output). */
fp4_status fp4_gemm_blockscaled(const fp4_tensor* A, const fp4_tensor* B,
                                const void* P, const void* Q, int r, float beta,
                                void* C, int c_dtype, int64_t ldc, void* stream);

/* Bytes of device workspace with which a GEMM may split its last partial wave
 * of tiles along K (one 256 x 256 FP32 partial per pair of SMs of the current
 * device: 19 MiB on a 152-SM GPU). */
size_t fp4_gemm_split_workspace(void);

/* Bytes of workspace for fp4_gemm_blockscaled_ws with A of M rows and rank r:
 * fp4_gemm_split_workspace(), plus M * r BF16 values for P~ when r > 0. */
size_t fp4_gemm_blockscaled_workspace(int64_t M, int r);

/* fp4_gemm_blockscaled with a workspace.  With r > 0 the call first writes
 * P~ (the fold above) into the workspace by a launch of its own, so that the
 * GEMM loads P~ like any operand tile instead of rewriting P in shared memory
 * (the same values, so the same result).  And it may split its tail: when M and
 * N are multiples of 256, K is at least 48 * 256 and the 256 x 256 tiles fill
 * W >= 1 whole waves over the SM pairs plus R < pairs more, each of the last
 * R tiles is cut into S = pairs / R consecutive K ranges, computed by S pairs
 * in parallel; a second launch adds the S FP32 partial accumulators in K order
 * (the branch is in the last range) and rounds once, as for a whole tile.  So
 * the result equals fp4_gemm_blockscaled's up to the FP32 summation order
 * inside those tiles, and it is the same from run to run.
 * ws: NULL (exactly fp4_gemm_blockscaled) or at least
 * fp4_gemm_blockscaled_workspace(M, r) bytes, 256-byte aligned (else
 * FP4_ERR_WORKSPACE); its content is scratch.  Calls that share one ws must be
 * ordered. */
fp4_status fp4_gemm_blockscaled_ws(const fp4_tensor* A, const fp4_tensor* B,
                                   const void* P, const void* Q, int r, float beta,
                                   void* C, int c_dtype, int64_t ldc,
                                   void* ws, size_t ws_bytes, void* stream);

/* Low-rank branch factor: P[m][j] = bf16( sum_k X[m][k] L[j][k] ), FP32
 * accumulation.  X: M x K BF16 (pitch ldx), L: r x K BF16 (pitch K), P: M x r
 * BF16 (pitch r).  Requires M % 128 == 0, K % 16 == 0, r in {16,32,48,64}.
 * Forward: P = X L1^T; backward: P' = dY L2 (pass L = L2^T).
 * amax_out (optional, device, 4-byte aligned; NULL to skip): also receives
 * max |X| over the whole tensor, the same value fp4_amax returns, taken from
 * this call's own read of X; the call zeroes it first.  The linear calls use
 * it so that X (or dY) is read once for the factor and the tensor scale. */
fp4_status fp4_branch_factor(const void* X, int64_t M, int64_t K, int64_t ldx,
                             const void* L, int r, void* P, float* amax_out, void* stream);

/* Workspace bytes needed by fp4_linear_fwd / fp4_linear_bwd. */
size_t fp4_linear_fwd_workspace(int64_t M, int64_t N, int64_t K, int r);
size_t fp4_linear_bwd_workspace(int64_t M, int64_t N, int64_t K, int r);

/* Linear projection forward (section 2.1):
 *   Y = X W^T = S_tX S_tW Xq Wq^T + beta * bf16(X L1^T) L2^T      (M x N, BF16)
 * (the GEMM of fp4_gemm_blockscaled with P = bf16(X L1^T), Q = L2: the same
 * branch fold and single rounding of Y)
 * X: M x K BF16 (pitch ldx); Wq: N x K NVFP4 (RTN-quantized W_res, prepared by
 * the caller, reused across micro-batches); L1: r x K, L2: N x r BF16.
 * X is quantized RTN in both orientations from one read; the column form
 * (K x M) is written to xqT_saved (caller-owned) for the dW product of the
 * backward pass.  The quantization of X also writes the GEMM's P~ (the fold of
 * fp4_gemm_blockscaled) over P in the workspace, so the GEMM loads it as it is.
 * ws/ws_bytes: device workspace of at least
 * fp4_linear_fwd_workspace(M, N, K, r) bytes, 256-byte aligned; with
 * fp4_gemm_split_workspace() bytes more, the GEMM may split its tail as
 * fp4_gemm_blockscaled_ws does. */
fp4_status fp4_linear_fwd(const void* X, int64_t M, int64_t K, int64_t ldx,
                          const fp4_tensor* Wq, const void* L1, const void* L2, int r,
                          float beta, void* Y, int64_t ldy, fp4_tensor* xqT_saved,
                          void* ws, size_t ws_bytes, void* stream);

/* fp4_linear_fwd without a caller workspace; the call allocates nothing.
 * Same arguments, result and launches as fp4_linear_fwd minus ws/ws_bytes
 * (given a workspace with the split-tail room): the workspace lives in a
 * 32 MiB file-scope device buffer of this library, followed by 20 MiB for the
 * GEMM's split tail (a static __device__ array, created when the module
 * loads; on a GPU with more than 160 SMs the tail is not split).  The pages have
 * no counterpart to this call: it is an interface variant, not part of the
 * method.
 * For callers that cannot allocate device memory: plain C host code linked
 * only against this library, which has no device allocator of its own, and
 * callers that must not call cudaMalloc/cudaFree in the middle of a step
 * (cudaFree synchronises the device; with the rest of HBM reserved by a
 * caching allocator, cudaMalloc fails for lack of memory).
 * Limit: fp4_linear_fwd_workspace(M, N, K, r) <= 32 MiB (about M * K <= 50e6
 * at r = 64, e.g. M = 16384, K = 3072); larger shapes return
 * FP4_ERR_WORKSPACE, with the sizes in fp4_last_error(), before anything is
 * launched.
 * Nothing in the scratch has to start at zero: each call zeroes what it
 * reduces into (the amax slot) before use and overwrites the rest.
 * The first call on each device looks the buffer's address up
 * (cudaGetSymbolAddress, which can load the module) and caches it for the
 * life of the process.  cudaDeviceReset unloads the module and leaves the
 * cached address stale: do not use this call after resetting a device it has
 * run on.
 * All calls on one device share the one buffer: calls whose executions can
 * overlap (unordered streams, several host threads) race on it and give wrong
 * results.  Order them (one stream, or events). */
fp4_status fp4_linear_fwd_noalloc(const void* X, int64_t M, int64_t K, int64_t ldx,
                                  const fp4_tensor* Wq, const void* L1, const void* L2, int r,
                                  float beta, void* Y, int64_t ldy, fp4_tensor* xqT_saved,
                                  void* stream);

/* Linear projection backward (section 2.1, backward pass; the subspace
 * constraint on the factor update is not part of this call):
 *   dX = S_tdY S_tW dYq WqT^T + beta * bf16(dY L2) L1     (M x K, BF16)
 *   dW = S_tdY' S_tX dYqT XqT^T                          (N x K, BF16 or FP32)
 * dY: M x N BF16 (pitch lddy), quantized with SR (seed; Philox stream 0 for
 * the row form used by dX, stream 1 for the column form used by dW).
 * WqT: K x N NVFP4 (W_res quantized column-wise, RTN); xqT_saved: K x M from
 * fp4_linear_fwd.  The quantization of dY also folds P' = bf16(dY L2) for the
 * dX GEMM (as the forward does).  ws: at least fp4_linear_bwd_workspace(M, N,
 * K, r) bytes;
 * with fp4_gemm_split_workspace() bytes more, the dX and dW GEMMs may split
 * their tails as fp4_gemm_blockscaled_ws does. */
fp4_status fp4_linear_bwd(const void* dY, int64_t M, int64_t N, int64_t lddy,
                          const fp4_tensor* WqT, const fp4_tensor* xqT_saved,
                          const void* L1, const void* L2, int r, float beta, uint64_t seed,
                          void* dX, int64_t lddx, void* dW, int dw_dtype, int64_t lddw,
                          void* ws, size_t ws_bytes, void* stream);

/* Gradients of the LoRA-SVD branch factors (section 2.1: W = W_res + beta L2 L1,
 * the subspace in BF16, the backward pass restricted to the subspace), straight
 * through the BF16 branch factors P = bf16(X L1^T) (forward) and
 * P' = bf16(dY L2) (backward):
 *   dL2 = beta * dY^T P   (N x r):  A = dY (T x N), B = P,  transpose_c = 0
 *   dL1 = beta * P'^T X   (r x K):  A = X (T x K),  B = P', transpose_c = 1
 * i.e. C = beta * A^T B with the sum over the T tokens, FP32 accumulation.
 * A: T x M BF16, row pitch lda elements (16-byte aligned base and pitch);
 * B: T x r BF16, pitch r; C: FP32, M x r at C[m * ldc + j] (transpose_c = 0) or
 * r x M at C[j * ldc + m] (transpose_c = 1).  M % 128 == 0, r in {16,32,48,64},
 * any T >= 1.  ws: at least fp4_lora_factor_grad_workspace(T, M, r) bytes,
 * 256-byte aligned (FP32 partial sums of the token splits; the size depends on
 * the device's SM count).  Deterministic: the partials are added in a fixed
 * order.  The Cholesky-QR constraint the pages name is not specified there and
 * is not applied. */
size_t fp4_lora_factor_grad_workspace(int64_t T, int64_t M, int r);
fp4_status fp4_lora_factor_grad(const void* A, int64_t T, int64_t M, int64_t lda,
                                const void* B, int r, float beta, float* C, int64_t ldc,
                                int transpose_c, void* ws, size_t ws_bytes, void* stream);

/* Realignment of the LoRA-SVD subspace by a randomized SVD (section 2.1,
 * Realignment: the subspace is reset periodically with a randomized SVD; the
 * pages give no parameters).  The randomized subspace iteration and direct SVD
 * of Halko, Martinsson and Tropp (SIAM Review 2011, Algorithms 4.4 and 5.1) on
 * W = W_res + beta L2 L1:
 *   Y = W Omega;  q times Y = W orth(W^T orth(Y));  Q = orth(Y);  B = Q^T W;
 *   B = Ub Sigma V^T;  L2_out = bf16(Q Ub_r Sigma_r / beta);  L1_out = bf16(V_r^T);
 *   W_res_out = bf16(W - beta L2_out L1_out),
 * each L1_out row's largest-magnitude entry made positive (L2_out's column
 * follows).  FP32 arithmetic: the products with W and W^T on the tensor cores
 * as three TF32 products each (high and low parts of both operands; within a
 * small multiple of FP32 rounding), the others in this library's own tiled
 * FP32 GEMM (outputs with few tiles split over K, the slices added in a fixed
 * order: deterministic), Cholesky-QR twice for orth(), a one-CTA Jacobi
 * eigensolver for B B^T.  Allocates nothing.
 * W_res: N x K BF16, row pitch ldw (W_res_out the same); L1: r x K (pitch K);
 * L2: N x r (pitch r); Omega: K x s BF16 test matrix (pitch s), Gaussian,
 * supplied by the caller.  Outputs may be the inputs.  r in {16,32,48,64},
 * s a multiple of 16 in [r, 128], N, K >= s, N, K < 2^31, 0 <= q <= 8, beta > 0.
 * W must have numerical rank >= s.  info (device int): 0, or nonzero when a
 * Cholesky factorisation failed (then no output is written).
 * ws: fp4_lora_realign_workspace(N, K, r, s) bytes (about 8 N K + 8 MB),
 * 256-byte aligned. */
size_t fp4_lora_realign_workspace(int64_t N, int64_t K, int r, int s);
fp4_status fp4_lora_realign(const void* W_res, int64_t N, int64_t K, int64_t ldw,
                            const void* L1, const void* L2, int r, float beta,
                            const void* Omega, int s, int q, void* W_res_out, void* L1_out,
                            void* L2_out, int* info, void* ws, size_t ws_bytes, void* stream);

/* Cholesky-QR step of the LoRA-SVD branch (section 2.1: the backward pass is
 * restricted to the subspace under a Cholesky-QR constraint; no formula on the
 * pages).  Reading: the rows of L1 are re-orthonormalised through the Cholesky
 * factor of their Gram matrix and L2 takes the factor, so beta L2 L1 is kept:
 *   L1 L1^T = L L^T,   L1_out = bf16(L^-1 L1),   L2_out = bf16(L2 L).
 * FP32 arithmetic (Gram partials over 128-column chunks added in a fixed order).
 * L1: r x K BF16, row pitch ld1 elements; L2: N x r BF16, pitch r; the outputs
 * have the same layouts and may be the inputs (in-place update).  All 16-byte
 * aligned.  r in {16, 32, 48, 64}.  info (device int): 0 on success, else j >= 1
 * when the leading minor of order j of L1 L1^T is not positive definite, and
 * then the outputs are not written.  ws: fp4_lora_cholqr_workspace(K, r) bytes,
 * 256-byte aligned. */
size_t fp4_lora_cholqr_workspace(int64_t K, int r);
fp4_status fp4_lora_cholqr(const void* L1, int64_t K, int64_t ld1, const void* L2, int64_t N,
                           int r, void* L1_out, void* L2_out, int* info, void* ws,
                           size_t ws_bytes, void* stream);

/* Q-Root orthogonalisation: Newton-Schulz iterations with every matrix product
 * in NVFP4 (section 2.3, NVFP4 Root optimizer: direct NVFP4 execution, shape-
 * dependent coefficients a, b, c, p99 outlier clipping; the pages print neither
 * the coefficients nor the clipping rule).  With normalize = 1,
 *   X_0 = bf16(G / max(||G||_F, 1e-7))          (the norm in FP64)
 * else X_0 = G; then `steps` times:
 *   if clip: X <- sign(X) min(|X|, v), v = the ceil(0.99 m n)-th smallest |x|
 *   A  = bf16(Q(X) Q(X)^T)                       (m x m; Q = NVFP4 RTN, blocks along n)
 *   B  = bf16(fl32(b A) + fl32(c bf16(Q(A) Q(A)^T)))   (c = 0: B = bf16(fl32(b A)),
 *                                                 the A^2 product is not formed)
 *   X  <- bf16(fl32(a X) + bf16(Q(B) Q_T(X)))     (Q_T: blocks along m)
 * G: m x n BF16, row pitch ldg; X: m x n BF16 output, row pitch ldx (X may be G);
 * both 16-byte aligned with 16-byte pitches.  m % 128 == 0, n % 128 == 0,
 * m * n < 2^32; m <= n is the efficient orientation (the caller transposes a tall
 * matrix).  0 <= steps <= 1000.  ws: at least fp4_newton_schulz_workspace(m, n, c)
 * bytes, 256-byte aligned.  Deterministic (the norm's partial sums and the
 * histograms reduce in a fixed order or in integers). */
size_t fp4_newton_schulz_workspace(int64_t m, int64_t n, float c);
fp4_status fp4_newton_schulz(const void* G, int64_t m, int64_t n, int64_t ldg, int normalize,
                             int steps, float a, float b, float c, int clip, void* X,
                             int64_t ldx, void* ws, size_t ws_bytes, void* stream);

/* Q-AdamW second-moment codec (section 2.2, Quantized-state AdamW: v_t is
 * stored in NVFP4 after a square root, a tile mean kept in BF16 and a Hadamard
 * transform of the residual; it is rebuilt by inverting the transform and the
 * mean, then squaring).  The pages give no tile or transform size; here both
 * span one 16-element NVFP4 block along a row:
 *   u = sqrt(v)                        mean = bf16((pairwise-tree sum of u) / 16)
 *   h = WHT16(u - mean) / 4            (Walsh-Hadamard butterfly, natural order)
 *   out = NVFP4 RTN of h               (tensor scale from max |h|)
 * and decode: v' = (WHT16(deq) / 4 + mean)^2, deq = fl32(e2m1 * e4m3 * S_t).
 * Every step is one FP32 operation in that order (bit-reproducible).
 * v: rows x cols FP32, v >= 0 (a negative or NaN entry is unsupported), row
 * pitch ldv elements (16-byte aligned base and pitch), cols % 16 == 0.
 * out: rows x cols NVFP4 tensor (scales in the MMA layout, out->scale[0] = S_t,
 * [1] = max |h|).  mean: rows x cols/16 BF16, row-major, pitch cols/16.
 * Encode reads v twice (max |h|, then the codes).  Decode writes v_out
 * (rows x cols FP32, pitch ldo, 16-byte aligned) from in and mean. */
fp4_status fp4_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, int64_t ldv,
                               fp4_tensor* out, uint16_t* mean, void* stream);
fp4_status fp4_qadamw_v_decode(const fp4_tensor* in, const uint16_t* mean, float* v_out,
                               int64_t ldo, void* stream);

/* Synchronise `stream`, then read and clear the device status word.
 * Returns FP4_ERR_TIMEOUT if any kernel recorded an expired wait. */
fp4_status fp4_check_status(void* stream);

/* Thread-local text of the last error (never NULL). */
const char* fp4_last_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t fp4_launch_count(void);

/* Diagnostic: convert n floats (device) with the quantizer's own E2M1 RTN
 * routine (codes, one per byte) and E4M3 scale routine (bytes) so tests can
 * check the conversion conventions against the oracle.  n % 2 == 0. */
fp4_status fp4_debug_convert(const float* in, int64_t n, uint8_t* e2m1_out,
                             uint8_t* e4m3_out, void* stream);

/* Diagnostic: stochastically round n floats (device) to E2M1 with the
 * quantizer's own rounding routine, element i using the 16 random bits
 * rnd16[i] (device), so tests can drive exact ties and denormals that Philox
 * draws reach only by chance.  Element i rounds up in magnitude iff
 * rnd16[i] < frac * 2^16, frac its position between the two neighbouring grid
 * points (magnitude clamped to 6 first; sign kept).  One code per byte in
 * e2m1_out.  0 < n <= 2^34.  Stochastic rounding is the one "Full-Stack FP4"
 * (gist.science explainer) names in section 2.2; the 16-bit comparison is this
 * library's reading of it (see the encoding note at the top). */
fp4_status fp4_debug_sr_round(const float* in, const uint16_t* rnd16, int64_t n,
                              uint8_t* e2m1_out, void* stream);

/* Diagnostic: on != 0 makes every later SR quantization (until called with 0)
 * take its kernels' general form, which computes the Philox counter word 1
 * (the high half of the element group index) instead of assuming it zero.
 * Tensors of 2^35 or more elements take that form anyway; this lets tests
 * check it on small ones.  The results are the same either way.  Not for use
 * while other host threads launch quantizations. */
void fp4_debug_force_counter64(int on);

/* Diagnostic: dense NVFP4 tensor-core rate probe.  Launches one CTA per SM;
 * each issues 4 * iters block-scaled MMAs of shape M=128 x N=n x K=64
 * (n in {128, 256}) on operands resident in shared memory.  The caller times
 * the launch (e.g. with CUDA events on `stream`); the work is
 * num_sms * 4 * iters * 2 * 128 * n * 64 FLOP.  *num_sms_out (host, may be
 * NULL) receives the SM count used. */
fp4_status fp4_mma_peak_probe(int n, int iters, int* num_sms_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_GB300_H */
