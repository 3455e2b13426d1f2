// Internal launcher declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace nvfp4 {

// 2-D row-major tensor map over a rows x cols matrix (`inner` contiguous elements per row,
// `outer` rows, row pitch `pitch_bytes`), box box_inner x box_outer, built with the driver's
// cuTensorMapEncodeTiled (resolved at run time).  False if the driver rejects it.
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Output buffers of one quantized tensor (device pointers).
struct QOut {
  void* codes;
  void* scales;
  float* scale;
};

void count_launch();

// Programmatic dependent launch is used only from one of this library's kernels to the next: a
// kernel launched with it may start as soon as the previous kernel in the stream lets it, and its
// griddepcontrol.wait is defined to wait for prerequisite kernels, so the library does not rely on
// it to order a copy, memset or event wait queued between the two.  g_pdl_chain is true while the
// last operation this thread queued was one of the library's kernels; every C-ABI call clears it on
// entry, and so does every memset the library queues, so the first kernel after either is launched
// normally (ordered after everything before it in the stream).
inline thread_local bool g_pdl_chain = false;
inline void pdl_chain_break() { g_pdl_chain = false; }

// Launches `kernel` with programmatic stream serialization when the previous operation in the stream
// is one of this library's kernels (its CTAs may then be scheduled while that kernel drains, and
// they wait in pdl_wait() before touching its data), else with a normal launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl_chain ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  g_pdl_chain = e == cudaSuccess;
  return e;
}

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* out, int num_sms,
                        cudaStream_t s);

// clip (optional, device, both orientations with RTN only): |x| is clipped to this BF16
// magnitude pattern before quantization.
// The block-scaled GEMM's branch fold, P~ = bf16(fl32(P * fl32(beta / alpha))) in place with
// alpha = fl32(S_tA * S_tB) (1 when 0): P rows x r BF16 (pitch r); other_scale: the S_t of the
// GEMM's other operand (device).
struct BranchFold {
  void* P;
  int r;
  const float* other_scale;
  float beta;
};
// fold (optional): the quantizer also folds P for the GEMM that consumes its row form (x's rows
// are P's rows; S_tA is the quantizer's own tensor scale).
cudaError_t launch_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, bool sr, uint64_t seed,
                                 uint32_t stream_r, uint32_t stream_c, const float* amax, const QOut* row_out,
                                 const QOut* col_out, cudaStream_t s, const uint32_t* clip = nullptr,
                                 const BranchFold* fold = nullptr);
void set_force_counter64(bool on);
cudaError_t launch_debug_convert(const float* in, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t s);
cudaError_t launch_debug_sr_round(const float* in, const uint16_t* rnd, int64_t n, uint8_t* e2m1, cudaStream_t s);

// Block-scaled NVFP4 GEMM with the fused BF16 branch.  Tensor maps are built
// inside; `sm_count` sizes the persistent grid.
struct GemmArgs {
  const void* a_codes;
  const void* a_scales;
  const float* a_scale;  // device: S_tA
  const void* b_codes;
  const void* b_scales;
  const float* b_scale;  // device: S_tB
  int64_t M, N, K;
  const void* P;  // M x r bf16
  const void* Q;  // N x r bf16
  int r;
  float beta;
  void* C;
  int c_f32;
  int64_t ldc;
  // optional (nullptr: none): room for the split tail's FP32 partials, gemm_splitk_ws_bytes() bytes
  float* sk_ws = nullptr;
  size_t sk_ws_bytes = 0;
  // P already holds P~ (the branch fold done before the GEMM): the GEMM loads it as it is
  bool p_folded = false;
};
cudaError_t launch_gemm_nvf4(const GemmArgs& g, int num_sms, cudaStream_t s);
// Workspace that lets launch_gemm_nvf4 split the K range of its last partial wave of 256 x 256
// tiles over the idle CTA pairs: one 256 x 256 FP32 slot per pair.
size_t gemm_splitk_ws_bytes(int num_sms);
// The branch fold on its own: Pt = P~ for the GEMM of a_scale's and b_scale's operands.
cudaError_t launch_fold_branch(const void* P, int64_t M, int r, const float* a_scale, const float* b_scale,
                               float beta, void* Pt, cudaStream_t s);

// P = bf16(X L^T): X M x K (pitch ldx), L r x K, P M x r.
// amax_out (optional, device): also reduces max |X| into it (zeroed by the launcher).
cudaError_t launch_branch_factor(const void* X, int64_t M, int64_t K, int64_t ldx, const void* L, int r, void* P,
                                 float* amax_out, int num_sms, cudaStream_t s);

// Dense NVFP4 MMA rate probe: every SM issues 4 * iters M=128 x N=n x K=64 MMAs.
cudaError_t launch_mma_peak(int n, int iters, int num_sms, cudaStream_t s);

// Read and clear the status word of the GEMM kernels (synchronous on s).
cudaError_t gemm_status_read_clear(unsigned int* out, cudaStream_t s);

// out[c][r] = in[r][c] for a BF16 rows x cols matrix (pitches = widths).
cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, void* out, cudaStream_t s);

// LoRA factor gradients: C = beta * A^T B (A: T x M, B: T x r, row-major BF16), the token range
// split over `splits` CTAs per 128-row block with FP32 partials in `partial` (splits x M x r).
uint32_t lora_grad_splits(int64_t T, int64_t M, int num_sms);
cudaError_t launch_lora_grad(const void* A, int64_t T, int64_t M, int64_t lda, const void* B, int r, float beta,
                             float* C, int64_t ldc, int transpose_c, float* partial, uint32_t splits, cudaStream_t s);

// Newton-Schulz elementwise kernels (BF16 matrices, cols % 8 == 0, rows * cols / 8 < 2^32).
// Normalisation: X = bf16(G / max(||G||_F, 1e-7)); `partial` holds ns_sumsq_blocks(num_sms)
// doubles; hist (optional, zeroed, 32768 counters) receives the |X| histogram.
constexpr int kNsHistBins = 32768;
int ns_sumsq_blocks(int num_sms);
cudaError_t launch_ns_normalize(const void* G, int64_t rows, int64_t cols, int64_t ldg, void* X, int64_t ldx,
                                double* partial, uint32_t* hist, int num_sms, cudaStream_t s);
// The k-th smallest |x| pattern from `hist` (then zeroed) into *clip_slot and, as a float, into
// *amax_out (the clipped tensor's max |x|).
cudaError_t launch_ns_select(uint32_t* hist, uint32_t k, uint32_t* clip_slot, float* amax_out, cudaStream_t s);
// out = bf16(fl32(p x') + fl32(q y)) (y optional), x' = x clipped to +-*clip_x (optional);
// amax_out (optional): max |out| (zeroed here); hist (optional, zeroed): the |out| histogram.
// out may alias x or y.
cudaError_t launch_ns_lincomb(const void* x, int64_t ldx, float p, const void* y, int64_t ldy, float q, void* out,
                              int64_t ldo, int64_t rows, int64_t cols, const uint32_t* clip_x, float* amax_out,
                              uint32_t* hist, int num_sms, cudaStream_t s);

// Cholesky-QR of the LoRA factors: L1 (r x K, pitch ld1) <- L^-1 L1 and L2 (N x r) <- L2 L with
// L1 L1^T = L L^T; ws holds cholqr_parts(K) * r * r + 2 * r * r floats; *info (device) = 0 or the
// order of the first non-positive-definite leading minor (then nothing is written).
int cholqr_parts(int64_t K);
cudaError_t launch_lora_cholqr(const void* L1, int64_t K, int64_t ld1, const void* L2, int64_t N, int r,
                               void* L1_out, void* L2_out, int* info, float* ws, cudaStream_t s);

// Randomized-SVD realignment of the LoRA-SVD subspace (FP32; the products with W on the tensor
// cores as three TF32 products, the rest in the library's tiled FP32 GEMM); ws holds realign_workspace_floats(N, K, r, s) floats; *info (device) = 0, or a
// failed Cholesky (1000 * stage + pivot order), in which case no output is written.
size_t realign_workspace_floats(int64_t N, int64_t K, int r, int s);
cudaError_t launch_lora_realign(const void* W_res, int64_t N, int64_t K, int64_t ldw, const void* L1, const void* L2,
                                int r, float beta, const void* Omega, int s_cols, int q, void* W_res_out,
                                void* L1_out, void* L2_out, int* info, float* ws, int num_sms, cudaStream_t st);

// Q-AdamW second-moment codec: v (FP32 rows x cols, pitch ldv, cols % 16 == 0) to NVFP4
// codes/scales/S_t (out; out.scale[1] receives the amax) and BF16 tile means (rows x cols/16);
// and back to FP32 (pitch ldo).
cudaError_t launch_vt_encode(const float* v, int64_t rows, int64_t cols, int64_t ldv, const QOut& out,
                             uint16_t* mean, int num_sms, cudaStream_t s);
cudaError_t launch_vt_decode(const void* codes, const void* scales, const float* scale, const uint16_t* mean,
                             int64_t rows, int64_t cols, float* out, int64_t ldo, int num_sms, cudaStream_t s);

}  // namespace nvfp4
