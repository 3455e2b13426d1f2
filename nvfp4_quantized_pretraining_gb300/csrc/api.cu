// C ABI of the NVFP4 linear-projection library: argument validation, the
// composition of the linear forward/backward passes, and error reporting.
// Every entry point is declared (with its contract) in include/nvfp4_gb300.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "kernels.h"
#include "nvfp4_gb300.h"

namespace nvfp4 {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static thread_local std::string t_err = "no error";

static fp4_status fail(fp4_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static fp4_status fail(fp4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                      \
  do {                                                                                      \
    cudaError_t e_ = (expr);                                                                \
    if (e_ != cudaSuccess)                                                                  \
      return fail(FP4_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));            \
  } while (0)

static int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load();
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev].store(n);
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static int64_t scale_bytes(int64_t rows, int64_t cols) {
  const int64_t kb = cols / 16;
  return ((rows + 127) / 128) * 128 * ((kb + 3) / 4) * 4;
}
static bool scale_padded(int64_t rows, int64_t cols) { return (rows % 128) != 0 || ((cols / 16) % 4) != 0; }

static fp4_status check_tensor(const fp4_tensor* t, const char* name) {
  if (!t) return fail(FP4_ERR_INVALID_ARG, "%s is NULL", name);
  if (!t->codes || !t->scales || !t->scale) return fail(FP4_ERR_INVALID_ARG, "%s has a NULL buffer", name);
  if (!aligned16(t->codes) || !aligned16(t->scales) || (reinterpret_cast<uintptr_t>(t->scale) & 7u))
    return fail(FP4_ERR_MISALIGNED, "%s buffers must be 16-byte aligned (scale 8-byte)", name);
  if (t->rows <= 0 || t->cols <= 0 || t->cols % 16 != 0)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "%s shape %lld x %lld: cols must be a positive multiple of 16", name,
                (long long)t->rows, (long long)t->cols);
  return FP4_OK;
}

static fp4_status check_bf16_input(const void* x, int64_t rows, int64_t cols, int64_t ld, const char* name) {
  if (!x) return fail(FP4_ERR_INVALID_ARG, "%s is NULL", name);
  if (rows <= 0 || cols <= 0) return fail(FP4_ERR_INVALID_ARG, "%s has a non-positive size", name);
  if (ld < cols) return fail(FP4_ERR_INVALID_ARG, "%s: ld %lld < cols %lld", name, (long long)ld, (long long)cols);
  if (!aligned16(x) || (ld * 2) % 16 != 0)
    return fail(FP4_ERR_MISALIGNED, "%s: base and row pitch must be 16-byte aligned", name);
  if (rows * (cols / 8) >= (int64_t(1) << 32) || rows >= (int64_t(1) << 31))
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "%s: tensor too large (%lld x %lld)", name, (long long)rows,
                (long long)cols);
  return FP4_OK;
}

static QOut qout(const fp4_tensor* t) { return QOut{t->codes, t->scales, t->scale}; }

// Quantize in one or both orientations.  amax: precomputed (device) or NULL.
// clip (optional, device; both forms, RTN): |x| is clipped to that BF16 magnitude pattern first.
static fp4_status quantize_impl(const void* x, int64_t rows, int64_t cols, int64_t ld, int round_mode,
                                uint64_t seed, uint32_t sr_row, uint32_t sr_col, const float* amax_opt,
                                const fp4_tensor* out_row, const fp4_tensor* out_col, cudaStream_t s,
                                const uint32_t* clip = nullptr, const BranchFold* fold = nullptr) {
  fp4_status st = check_bf16_input(x, rows, cols, ld, "x");
  if (st) return st;
  if (round_mode != FP4_ROUND_RTN && round_mode != FP4_ROUND_SR)
    return fail(FP4_ERR_INVALID_ARG, "round_mode %d is not RTN (0) or SR (1)", round_mode);
  if (cols % 16 != 0) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "cols %lld is not a multiple of 16", (long long)cols);
  if (!out_row && !out_col) return fail(FP4_ERR_INVALID_ARG, "no output tensor");
  if (out_row) {
    if ((st = check_tensor(out_row, "out"))) return st;
    if (out_row->rows != rows || out_row->cols != cols)
      return fail(FP4_ERR_INVALID_ARG, "out is %lld x %lld, expected %lld x %lld", (long long)out_row->rows,
                  (long long)out_row->cols, (long long)rows, (long long)cols);
  }
  if (out_col) {
    if (rows % 16 != 0)
      return fail(FP4_ERR_UNSUPPORTED_SHAPE, "transposed quantization needs rows %% 16 == 0 (rows = %lld)",
                  (long long)rows);
    if ((st = check_tensor(out_col, "out_col"))) return st;
    if (out_col->rows != cols || out_col->cols != rows)
      return fail(FP4_ERR_INVALID_ARG, "transposed out is %lld x %lld, expected %lld x %lld",
                  (long long)out_col->rows, (long long)out_col->cols, (long long)cols, (long long)rows);
  }
  if ((rows + 63) / 64 > 65535)  // one 64-row tile per grid row
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rows %lld too large (at most 65535 x 64)", (long long)rows);
  if (amax_opt && (reinterpret_cast<uintptr_t>(amax_opt) & 3u))
    return fail(FP4_ERR_MISALIGNED, "amax_opt must be 4-byte aligned");
  if (out_row && scale_padded(rows, cols)) {
    CUDA_TRY(cudaMemsetAsync(out_row->scales, 0, scale_bytes(rows, cols), s));
    pdl_chain_break();
  }
  if (out_col && scale_padded(cols, rows)) {
    CUDA_TRY(cudaMemsetAsync(out_col->scales, 0, scale_bytes(cols, rows), s));
    pdl_chain_break();
  }
  const float* amax = amax_opt;
  if (!amax) {
    float* slot = out_row ? &out_row->scale[1] : &out_col->scale[1];
    CUDA_TRY(launch_amax(x, rows, cols, ld, slot, sm_count(), s));
    amax = slot;
  }
  const bool sr = round_mode == FP4_ROUND_SR;
  // one tiled kernel for every orientation request: the tile is staged once and each requested
  // form is produced from it
  QOut r{}, c{};
  if (out_row) r = qout(out_row);
  if (out_col) c = qout(out_col);
  CUDA_TRY(launch_quantize_dual(x, rows, cols, ld, sr, seed, sr_row, sr_col, amax, out_row ? &r : nullptr,
                                out_col ? &c : nullptr, s, clip, fold));
  return FP4_OK;
}

// sk_ws (optional, 256-byte aligned, sk_bytes of room): lets the GEMM split its last partial wave
// of tiles along K (gemm_splitk_ws_bytes() bytes are enough for any shape).
// p_folded: P holds P~ already (the branch fold done by the caller's launch before this one).
static fp4_status gemm_impl(const fp4_tensor* A, const fp4_tensor* B, const void* P, const void* Q, int r,
                            float beta, void* C, int c_dtype, int64_t ldc, cudaStream_t s, void* sk_ws = nullptr,
                            size_t sk_bytes = 0, bool p_folded = false) {
  fp4_status st;
  if ((st = check_tensor(A, "A")) || (st = check_tensor(B, "B"))) return st;
  const int64_t M = A->rows, N = B->rows, K = A->cols;
  if (B->cols != K) return fail(FP4_ERR_INVALID_ARG, "A is ? x %lld but B is ? x %lld", (long long)K, (long long)B->cols);
  if (M % 128 || N % 128 || K % 64)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "GEMM needs M %% 128 == 0, N %% 128 == 0, K %% 64 == 0 (M=%lld N=%lld K=%lld)",
                (long long)M, (long long)N, (long long)K);
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "GEMM dimension too large");
  if (r != 0 && r != 16 && r != 32 && r != 48 && r != 64)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {0,16,32,48,64}", r);
  if (r > 0) {
    if (!P || !Q) return fail(FP4_ERR_INVALID_ARG, "r > 0 needs P and Q");
    if (!aligned16(P) || !aligned16(Q)) return fail(FP4_ERR_MISALIGNED, "P and Q must be 16-byte aligned");
  }
  if (!C) return fail(FP4_ERR_INVALID_ARG, "C is NULL");
  if (c_dtype != FP4_OUT_BF16 && c_dtype != FP4_OUT_F32) return fail(FP4_ERR_INVALID_ARG, "bad c_dtype %d", c_dtype);
  const int esz = c_dtype == FP4_OUT_F32 ? 4 : 2;
  if (ldc < N) return fail(FP4_ERR_INVALID_ARG, "ldc %lld < N %lld", (long long)ldc, (long long)N);
  if (!aligned16(C) || (ldc * esz) % 16) return fail(FP4_ERR_MISALIGNED, "C base and row pitch must be 16-byte aligned");
  GemmArgs g;
  g.a_codes = A->codes;
  g.a_scales = A->scales;
  g.a_scale = A->scale;
  g.b_codes = B->codes;
  g.b_scales = B->scales;
  g.b_scale = B->scale;
  g.M = M;
  g.N = N;
  g.K = K;
  g.P = P;
  g.Q = Q;
  g.r = r;
  g.beta = beta;
  g.C = C;
  g.c_f32 = c_dtype == FP4_OUT_F32;
  g.ldc = ldc;
  g.sk_ws = static_cast<float*>(sk_ws);
  g.sk_ws_bytes = sk_ws ? sk_bytes : 0;
  g.p_folded = p_folded;
  CUDA_TRY(launch_gemm_nvf4(g, sm_count(), s));
  return FP4_OK;
}

static fp4_status branch_impl(const void* X, int64_t M, int64_t K, int64_t ldx, const void* L, int r, void* P,
                              cudaStream_t s, float* amax_out = nullptr) {
  fp4_status st = check_bf16_input(X, M, K, ldx, "X");
  if (st) return st;
  if (!L || !P) return fail(FP4_ERR_INVALID_ARG, "L and P must be non-NULL");
  if (!aligned16(L) || !aligned16(P)) return fail(FP4_ERR_MISALIGNED, "L and P must be 16-byte aligned");
  if (M % 128 || K % 16) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "branch factor needs M %% 128 == 0, K %% 16 == 0");
  if (r != 16 && r != 32 && r != 48 && r != 64) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {16,32,48,64}", r);
  CUDA_TRY(launch_branch_factor(X, M, K, ldx, L, r, P, amax_out, sm_count(), s));
  return FP4_OK;
}

// Carves a workspace into 256-byte-aligned regions.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += round256(bytes);
    return p;
  }
};

static fp4_tensor carve_tensor(Carver& c, int64_t rows, int64_t cols) {
  fp4_tensor t;
  t.codes = c.take(static_cast<size_t>(rows * cols / 2));
  t.scales = c.take(static_cast<size_t>(scale_bytes(rows, cols)));
  t.scale = static_cast<float*>(c.take(2 * sizeof(float)));
  t.rows = rows;
  t.cols = cols;
  return t;
}

static size_t fwd_ws(int64_t M, int64_t N, int64_t K, int r, Carver* c, fp4_tensor* xq, void** P) {
  (void)N;
  Carver local(nullptr);
  Carver& cv = c ? *c : local;
  fp4_tensor t = carve_tensor(cv, M, K);
  void* p = cv.take(static_cast<size_t>(M) * (r > 0 ? r : 0) * 2);
  if (xq) *xq = t;
  if (P) *P = p;
  return cv.off;
}

static size_t bwd_ws(int64_t M, int64_t N, int64_t K, int r, Carver* c, fp4_tensor* dyq, fp4_tensor* dyqT, void** P2,
                     void** L2T, void** L1T) {
  Carver local(nullptr);
  Carver& cv = c ? *c : local;
  fp4_tensor a = carve_tensor(cv, M, N);
  fp4_tensor b = carve_tensor(cv, N, M);
  const int rr = r > 0 ? r : 0;
  void* p = cv.take(static_cast<size_t>(M) * rr * 2);
  void* l2t = cv.take(static_cast<size_t>(rr) * N * 2);
  void* l1t = cv.take(static_cast<size_t>(K) * rr * 2);
  if (dyq) *dyq = a;
  if (dyqT) *dyqT = b;
  if (P2) *P2 = p;
  if (L2T) *L2T = l2t;
  if (L1T) *L1T = l1t;
  return cv.off;
}

// Argument checks shared by the two forward entry points.
static fp4_status check_linear_fwd(const void* X, int64_t M, int64_t K, int64_t ldx, const fp4_tensor* Wq,
                                   const void* L1, const void* L2, int r, const fp4_tensor* xqT_saved) {
  fp4_status st;
  if ((st = check_bf16_input(X, M, K, ldx, "X"))) return st;
  if ((st = check_tensor(Wq, "Wq")) || (st = check_tensor(xqT_saved, "xqT_saved"))) return st;
  if (Wq->cols != K)
    return fail(FP4_ERR_INVALID_ARG, "Wq has %lld columns, X has K = %lld", (long long)Wq->cols, (long long)K);
  const int64_t N = Wq->rows;
  if (xqT_saved->rows != K || xqT_saved->cols != M)
    return fail(FP4_ERR_INVALID_ARG, "xqT_saved must be K x M (%lld x %lld)", (long long)K, (long long)M);
  if (M % 128 || N % 128 || K % 64)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "linear needs M %% 128, N %% 128 == 0 and K %% 64 == 0");
  if (r > 0 && (!L1 || !L2)) return fail(FP4_ERR_INVALID_ARG, "r > 0 needs L1 and L2");
  return FP4_OK;
}

// Room for the GEMMs' split tail after the required part of a caller workspace of ws_bytes
// bytes, or nullptr when it does not fit.
static void* split_region(void* ws, size_t ws_bytes, size_t need) {
  return ws_bytes >= need + gemm_splitk_ws_bytes(sm_count()) ? static_cast<uint8_t*>(ws) + need : nullptr;
}

// The forward's launches on a workspace `ws` already checked to hold fwd_ws(M, N, K, r) bytes:
// the branch factor of X (its read of X also yields max |X|), the dual RTN quantization of X,
// then the block-scaled GEMM with the fused branch.  With r = 0: amax, quantize, GEMM.
// sk_ws: the GEMM's split-tail room (gemm_splitk_ws_bytes() bytes) or nullptr.
static fp4_status linear_fwd_on(void* ws, void* sk_ws, const void* X, int64_t M, int64_t K, int64_t ldx,
                                const fp4_tensor* Wq, const void* L1, const void* L2, int r, float beta, void* Y,
                                int64_t ldy, const fp4_tensor* xqT_saved, cudaStream_t s) {
  fp4_status st;
  Carver c(ws);
  fp4_tensor xq;
  void* P = nullptr;
  fwd_ws(M, Wq->rows, K, r, &c, &xq, &P);
  if (r > 0) {
    // the quantizer also folds P for the GEMM (P~ = bf16(P * beta / (S_tX S_tW)), in place)
    const BranchFold fold{P, r, Wq->scale, beta};
    if ((st = branch_impl(X, M, K, ldx, L1, r, P, s, &xq.scale[1]))) return st;
    if ((st = quantize_impl(X, M, K, ldx, FP4_ROUND_RTN, 0, 0, 0, &xq.scale[1], &xq, xqT_saved, s, nullptr, &fold)))
      return st;
  } else if ((st = quantize_impl(X, M, K, ldx, FP4_ROUND_RTN, 0, 0, 0, nullptr, &xq, xqT_saved, s))) {
    return st;
  }
  return gemm_impl(&xq, Wq, P, L2, r, beta, Y, FP4_OUT_BF16, ldy, s, sk_ws, gemm_splitk_ws_bytes(sm_count()), r > 0);
}

// Workspace of fp4_newton_schulz: the iterate's two NVFP4 forms, the m x m Gram
// matrix (B overwrites it), A's NVFP4 form and A^2 when c != 0, B's NVFP4 form,
// the m x n product B X, the magnitude histogram, the norm's partial sums and a
// clip-value slot.
struct NsBufs {
  fp4_tensor xq, xqT, aq, bq;
  void* A;
  void* A2;
  void* BX;
  uint32_t* hist;
  double* partial;
  uint32_t* clip;
};

static size_t ns_ws(int64_t m, int64_t n, float c, Carver* c_opt, NsBufs* out) {
  Carver local(nullptr);
  Carver& cv = c_opt ? *c_opt : local;
  NsBufs w{};
  w.xq = carve_tensor(cv, m, n);
  w.xqT = carve_tensor(cv, n, m);
  w.A = cv.take(static_cast<size_t>(m * m * 2));
  if (c != 0.0f) {
    w.aq = carve_tensor(cv, m, m);
    w.A2 = cv.take(static_cast<size_t>(m * m * 2));
  }
  w.bq = carve_tensor(cv, m, m);
  w.BX = cv.take(static_cast<size_t>(m * n * 2));
  w.hist = static_cast<uint32_t*>(cv.take(kNsHistBins * sizeof(uint32_t)));
  w.partial = static_cast<double*>(cv.take(static_cast<size_t>(ns_sumsq_blocks(sm_count())) * sizeof(double)));
  w.clip = static_cast<uint32_t*>(cv.take(16));
  if (out) *out = w;
  return cv.off;
}

// Scratch of fp4_linear_fwd_noalloc: one file-scope device buffer, created with
// the module, so that call needs no allocation.  32 MiB holds the forward
// workspace up to M * K ~ 50e6 elements at r = 64 (e.g. M = 16384, K = 3072).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
// followed by the GEMM's split-tail room: 256 KB per CTA pair, enough for 160 SMs
constexpr size_t kNoAllocSplitBytes = size_t(20) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes + kNoAllocSplitBytes];

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call per device and cached for the life of the process (a
// cudaDeviceReset unloads the module, after which the cached address is stale).
static fp4_status noalloc_scratch(void** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(FP4_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
  static std::atomic<void*> cache[64];
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    cache[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return FP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

int64_t fp4_scale_bytes(int64_t rows, int64_t cols) { return scale_bytes(rows, cols); }

fp4_status fp4_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax_out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st = check_bf16_input(x, rows, cols, ld, "x");
  if (st) return st;
  if (cols % 8) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "amax needs cols %% 8 == 0");
  if (!amax_out) return fail(FP4_ERR_INVALID_ARG, "amax_out is NULL");
  CUDA_TRY(launch_amax(x, rows, cols, ld, amax_out, sm_count(), static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

fp4_status fp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int round_mode, uint64_t seed,
                        uint32_t sr_stream, const float* amax_opt, fp4_tensor* out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if (!out) return fail(FP4_ERR_INVALID_ARG, "out is NULL");
  return quantize_impl(x, rows, cols, ld, round_mode, seed, sr_stream, 0, amax_opt, out, nullptr,
                       static_cast<cudaStream_t>(stream));
}

fp4_status fp4_quantize_transposed(const void* x, int64_t rows, int64_t cols, int64_t ld, int round_mode,
                                   uint64_t seed, uint32_t sr_stream, const float* amax_opt, fp4_tensor* out,
                                   void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if (!out) return fail(FP4_ERR_INVALID_ARG, "out is NULL");
  return quantize_impl(x, rows, cols, ld, round_mode, seed, 0, sr_stream, amax_opt, nullptr, out,
                       static_cast<cudaStream_t>(stream));
}

fp4_status fp4_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, int round_mode, uint64_t seed,
                             uint32_t sr_stream_row, uint32_t sr_stream_col, const float* amax_opt,
                             fp4_tensor* out_row, fp4_tensor* out_col, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  return quantize_impl(x, rows, cols, ld, round_mode, seed, sr_stream_row, sr_stream_col, amax_opt, out_row, out_col,
                       static_cast<cudaStream_t>(stream));
}

fp4_status fp4_gemm_blockscaled(const fp4_tensor* A, const fp4_tensor* B, const void* P, const void* Q, int r,
                                float beta, void* C, int c_dtype, int64_t ldc, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  return gemm_impl(A, B, P, Q, r, beta, C, c_dtype, ldc, static_cast<cudaStream_t>(stream));
}

size_t fp4_gemm_split_workspace(void) { return gemm_splitk_ws_bytes(sm_count()); }

size_t fp4_gemm_blockscaled_workspace(int64_t M, int r) {
  return gemm_splitk_ws_bytes(sm_count()) + (r > 0 && M > 0 ? round256(static_cast<size_t>(M) * r * 2) : 0);
}

fp4_status fp4_gemm_blockscaled_ws(const fp4_tensor* A, const fp4_tensor* B, const void* P, const void* Q, int r,
                                   float beta, void* C, int c_dtype, int64_t ldc, void* ws, size_t ws_bytes,
                                   void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!ws) return gemm_impl(A, B, P, Q, r, beta, C, c_dtype, ldc, s);
  fp4_status st;
  if ((st = check_tensor(A, "A")) || (st = check_tensor(B, "B"))) return st;
  if (r != 0 && r != 16 && r != 32 && r != 48 && r != 64)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {0,16,32,48,64}", r);
  if (r > 0 && (!P || !Q)) return fail(FP4_ERR_INVALID_ARG, "r > 0 needs P and Q");
  if (r > 0 && (!aligned16(P) || !aligned16(Q))) return fail(FP4_ERR_MISALIGNED, "P and Q must be 16-byte aligned");
  const size_t split = gemm_splitk_ws_bytes(sm_count());
  const size_t need = fp4_gemm_blockscaled_workspace(A->rows, r);
  if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  if (r > 0) {
    // the branch fold by its own launch, into the workspace after the split-tail room
    void* Pt = static_cast<uint8_t*>(ws) + split;
    CUDA_TRY(launch_fold_branch(P, A->rows, r, A->scale, B->scale, beta, Pt, s));
    return gemm_impl(A, B, Pt, Q, r, beta, C, c_dtype, ldc, s, ws, split, true);
  }
  return gemm_impl(A, B, P, Q, r, beta, C, c_dtype, ldc, s, ws, split);
}

fp4_status fp4_branch_factor(const void* X, int64_t M, int64_t K, int64_t ldx, const void* L, int r, void* P,
                             float* amax_out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if (amax_out && (reinterpret_cast<uintptr_t>(amax_out) & 3u))
    return fail(FP4_ERR_MISALIGNED, "amax_out must be 4-byte aligned");
  return branch_impl(X, M, K, ldx, L, r, P, static_cast<cudaStream_t>(stream), amax_out);
}

size_t fp4_linear_fwd_workspace(int64_t M, int64_t N, int64_t K, int r) {
  return fwd_ws(M, N, K, r, nullptr, nullptr, nullptr);
}

size_t fp4_linear_bwd_workspace(int64_t M, int64_t N, int64_t K, int r) {
  return bwd_ws(M, N, K, r, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
}

fp4_status fp4_linear_fwd(const void* X, int64_t M, int64_t K, int64_t ldx, const fp4_tensor* Wq, const void* L1,
                          const void* L2, int r, float beta, void* Y, int64_t ldy, fp4_tensor* xqT_saved, void* ws,
                          size_t ws_bytes, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if ((st = check_linear_fwd(X, M, K, ldx, Wq, L1, L2, r, xqT_saved))) return st;
  const size_t need = fp4_linear_fwd_workspace(M, Wq->rows, K, r);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  return linear_fwd_on(ws, split_region(ws, ws_bytes, need), X, M, K, ldx, Wq, L1, L2, r, beta, Y, ldy, xqT_saved,
                       static_cast<cudaStream_t>(stream));
}

fp4_status fp4_linear_fwd_noalloc(const void* X, int64_t M, int64_t K, int64_t ldx, const fp4_tensor* Wq,
                                  const void* L1, const void* L2, int r, float beta, void* Y, int64_t ldy,
                                  fp4_tensor* xqT_saved, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if ((st = check_linear_fwd(X, M, K, ldx, Wq, L1, L2, r, xqT_saved))) return st;
  const size_t need = fp4_linear_fwd_workspace(M, Wq->rows, K, r);
  if (need > kNoAllocScratchBytes)
    return fail(FP4_ERR_WORKSPACE,
                "fp4_linear_fwd_noalloc: M = %lld, K = %lld, r = %d needs %zu bytes of scratch but the static "
                "scratch holds %zu; use fp4_linear_fwd with a caller workspace",
                (long long)M, (long long)K, r, need, kNoAllocScratchBytes);
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws))) return st;
  void* sk = gemm_splitk_ws_bytes(sm_count()) <= kNoAllocSplitBytes ? static_cast<uint8_t*>(ws) + kNoAllocScratchBytes
                                                                     : nullptr;
  return linear_fwd_on(ws, sk, X, M, K, ldx, Wq, L1, L2, r, beta, Y, ldy, xqT_saved, static_cast<cudaStream_t>(stream));
}

fp4_status fp4_linear_bwd(const void* dY, int64_t M, int64_t N, int64_t lddy, const fp4_tensor* WqT,
                          const fp4_tensor* xqT_saved, const void* L1, const void* L2, int r, float beta,
                          uint64_t seed, void* dX, int64_t lddx, void* dW, int dw_dtype, int64_t lddw, void* ws,
                          size_t ws_bytes, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fp4_status st;
  if ((st = check_bf16_input(dY, M, N, lddy, "dY"))) return st;
  if ((st = check_tensor(WqT, "WqT")) || (st = check_tensor(xqT_saved, "xqT_saved"))) return st;
  if (WqT->cols != N) return fail(FP4_ERR_INVALID_ARG, "WqT has %lld columns, dY has N = %lld", (long long)WqT->cols, (long long)N);
  const int64_t K = WqT->rows;
  if (xqT_saved->rows != K || xqT_saved->cols != M)
    return fail(FP4_ERR_INVALID_ARG, "xqT_saved must be K x M (%lld x %lld)", (long long)K, (long long)M);
  if (M % 128 || N % 128 || K % 128)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "linear backward needs M, N, K multiples of 128");
  if (r > 0 && (!L1 || !L2)) return fail(FP4_ERR_INVALID_ARG, "r > 0 needs L1 and L2");
  if (r > 0 && (!aligned16(L1) || !aligned16(L2))) return fail(FP4_ERR_MISALIGNED, "L1 and L2 must be 16-byte aligned");
  const size_t need = fp4_linear_bwd_workspace(M, N, K, r);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  Carver c(ws);
  fp4_tensor dyq, dyqT;
  void *P2 = nullptr, *L2T = nullptr, *L1T = nullptr;
  bwd_ws(M, N, K, r, &c, &dyq, &dyqT, &P2, &L2T, &L1T);
  if (r > 0) {
    // the branch factor's read of dY also yields max |dY| for the quantizer (no separate amax pass)
    CUDA_TRY(launch_transpose_bf16(L2, N, r, L2T, s));
    if ((st = branch_impl(dY, M, N, lddy, L2T, r, P2, s, &dyq.scale[1]))) return st;
    CUDA_TRY(launch_transpose_bf16(L1, r, K, L1T, s));
    // the quantizer also folds P' for the dX GEMM (P'~ = bf16(P' * beta / (S_tdY S_tW)), in place)
    const BranchFold fold{P2, r, WqT->scale, beta};
    if ((st = quantize_impl(dY, M, N, lddy, FP4_ROUND_SR, seed, 0, 1, &dyq.scale[1], &dyq, &dyqT, s, nullptr, &fold)))
      return st;
  } else if ((st = quantize_impl(dY, M, N, lddy, FP4_ROUND_SR, seed, 0, 1, nullptr, &dyq, &dyqT, s))) {
    return st;
  }
  void* sk = split_region(ws, ws_bytes, need);  // one region serves both GEMMs (same stream, in order)
  const size_t skb = gemm_splitk_ws_bytes(sm_count());
  if ((st = gemm_impl(&dyq, WqT, P2, L1T, r, beta, dX, FP4_OUT_BF16, lddx, s, sk, skb, r > 0))) return st;
  return gemm_impl(&dyqT, xqT_saved, nullptr, nullptr, 0, 0.0f, dW, dw_dtype, lddw, s, sk, skb);
}

fp4_status fp4_check_status(void* stream) {
  unsigned int v = 0;
  CUDA_TRY(gemm_status_read_clear(&v, static_cast<cudaStream_t>(stream)));
  if (v & (1u << FP4_ERR_TIMEOUT)) return fail(FP4_ERR_TIMEOUT, "a device-side wait timed out");
  return FP4_OK;
}

const char* fp4_last_error(void) { return t_err.c_str(); }

uint64_t fp4_launch_count(void) { return g_launches.load(); }

size_t fp4_lora_factor_grad_workspace(int64_t T, int64_t M, int r) {
  if (T <= 0 || M <= 0 || r <= 0) return 0;
  return round256(static_cast<size_t>(lora_grad_splits(T, M, sm_count())) * static_cast<size_t>(M) *
                  static_cast<size_t>(r) * sizeof(float));
}

fp4_status fp4_lora_factor_grad(const void* A, int64_t T, int64_t M, int64_t lda, const void* B, int r, float beta,
                                float* C, int64_t ldc, int transpose_c, void* ws, size_t ws_bytes, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if ((st = check_bf16_input(A, T, M, lda, "A"))) return st;
  if (!B || !C) return fail(FP4_ERR_INVALID_ARG, "B and C must be non-NULL");
  if (!aligned16(B)) return fail(FP4_ERR_MISALIGNED, "B must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(C) & 3u) return fail(FP4_ERR_MISALIGNED, "C must be 4-byte aligned");
  if (M % 128) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "M %lld is not a multiple of 128", (long long)M);
  if (r != 16 && r != 32 && r != 48 && r != 64) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {16,32,48,64}", r);
  if (transpose_c != 0 && transpose_c != 1) return fail(FP4_ERR_INVALID_ARG, "transpose_c must be 0 or 1");
  if (ldc < (transpose_c ? M : r))
    return fail(FP4_ERR_INVALID_ARG, "ldc %lld too small for %s output", (long long)ldc, transpose_c ? "r x M" : "M x r");
  const size_t need = fp4_lora_factor_grad_workspace(T, M, r);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  const uint32_t splits = lora_grad_splits(T, M, sm_count());
  CUDA_TRY(launch_lora_grad(A, T, M, lda, B, r, beta, C, ldc, transpose_c, static_cast<float*>(ws), splits,
                            static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

size_t fp4_newton_schulz_workspace(int64_t m, int64_t n, float c) {
  if (m <= 0 || n <= 0) return 0;
  return ns_ws(m, n, c, nullptr, nullptr);
}

fp4_status fp4_newton_schulz(const void* G, int64_t m, int64_t n, int64_t ldg, int normalize, int steps, float a,
                             float b, float c, int clip, void* X, int64_t ldx, void* ws, size_t ws_bytes,
                             void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fp4_status st;
  if ((st = check_bf16_input(G, m, n, ldg, "G")) || (st = check_bf16_input(X, m, n, ldx, "X"))) return st;
  if (m % 128 || n % 128)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "Newton-Schulz needs m %% 128 == 0 and n %% 128 == 0 (m=%lld n=%lld)",
                (long long)m, (long long)n);
  if (m * n >= (int64_t(1) << 32))  // 32-bit histogram counts
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "Newton-Schulz matrix too large (m n >= 2^32)");
  if (steps < 0 || steps > 1000) return fail(FP4_ERR_INVALID_ARG, "steps %d not in [0, 1000]", steps);
  if ((normalize != 0 && normalize != 1) || (clip != 0 && clip != 1))
    return fail(FP4_ERR_INVALID_ARG, "normalize and clip must be 0 or 1");
  if (G != X && ldg == ldx) {
    const uint8_t* g0 = static_cast<const uint8_t*>(G);
    const uint8_t* x0 = static_cast<const uint8_t*>(X);
    const int64_t span = ((m - 1) * ldx + n) * 2;
    if (g0 < x0 + span && x0 < g0 + span) return fail(FP4_ERR_INVALID_ARG, "G and X overlap without being equal");
  }
  const size_t need = fp4_newton_schulz_workspace(m, n, c);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  Carver cv(ws);
  NsBufs w;
  ns_ws(m, n, c, &cv, &w);
  const int sms = sm_count();
  // k-th smallest magnitude: k = ceil(0.99 m n)
  const int64_t count = m * n;
  const uint32_t k = static_cast<uint32_t>((count * 99 + 99) / 100);
  uint32_t* hist = clip ? w.hist : nullptr;
  if (clip && steps > 0) {
    CUDA_TRY(cudaMemsetAsync(w.hist, 0, kNsHistBins * sizeof(uint32_t), s));
    pdl_chain_break();
  }
  uint32_t* hist0 = steps > 0 ? hist : nullptr;
  if (normalize) {
    CUDA_TRY(launch_ns_normalize(G, m, n, ldg, X, ldx, w.partial, hist0, sms, s));
  } else if (G != X || hist0) {
    CUDA_TRY(launch_ns_lincomb(G, ldg, 1.0f, nullptr, 0, 0.0f, X, ldx, m, n, nullptr, nullptr, hist0, sms, s));
  }
  // The clip is applied by the iterate's readers (the quantizer and the update), so X stays unclipped
  // in memory between the two.
  const uint32_t* clip_v = clip ? w.clip : nullptr;
  for (int it = 0; it < steps; ++it) {
    const float* amax_x = nullptr;
    if (clip) {
      CUDA_TRY(launch_ns_select(w.hist, k, w.clip, &w.xq.scale[1], s));
      amax_x = &w.xq.scale[1];  // the clipped iterate's max |x| is the clip value itself
    }
    if ((st = quantize_impl(X, m, n, ldx, FP4_ROUND_RTN, 0, 0, 0, amax_x, &w.xq, &w.xqT, s, clip_v))) return st;
    if ((st = gemm_impl(&w.xq, &w.xq, nullptr, nullptr, 0, 0.0f, w.A, FP4_OUT_BF16, m, s))) return st;
    const void* A2 = nullptr;
    if (c != 0.0f) {
      if ((st = quantize_impl(w.A, m, m, m, FP4_ROUND_RTN, 0, 0, 0, nullptr, &w.aq, nullptr, s))) return st;
      if ((st = gemm_impl(&w.aq, &w.aq, nullptr, nullptr, 0, 0.0f, w.A2, FP4_OUT_BF16, m, s))) return st;
      A2 = w.A2;
    }
    // B overwrites A in place; its max |B| goes straight to the quantizer
    CUDA_TRY(launch_ns_lincomb(w.A, m, b, A2, m, c, w.A, m, m, m, nullptr, &w.bq.scale[1], nullptr, sms, s));
    if ((st = quantize_impl(w.A, m, m, m, FP4_ROUND_RTN, 0, 0, 0, &w.bq.scale[1], &w.bq, nullptr, s))) return st;
    if ((st = gemm_impl(&w.bq, &w.xqT, nullptr, nullptr, 0, 0.0f, w.BX, FP4_OUT_BF16, n, s))) return st;
    CUDA_TRY(launch_ns_lincomb(X, ldx, a, w.BX, n, 1.0f, X, ldx, m, n, clip_v, nullptr,
                               it + 1 < steps ? hist : nullptr, sms, s));
  }
  return FP4_OK;
}

size_t fp4_lora_cholqr_workspace(int64_t K, int r) {
  if (K <= 0 || r <= 0) return 0;
  return round256((static_cast<size_t>(cholqr_parts(K)) + 2) * static_cast<size_t>(r) * r * sizeof(float));
}

fp4_status fp4_lora_cholqr(const void* L1, int64_t K, int64_t ld1, const void* L2, int64_t N, int r, void* L1_out,
                           void* L2_out, int* info, void* ws, size_t ws_bytes, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if (r != 16 && r != 32 && r != 48 && r != 64) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {16,32,48,64}", r);
  if ((st = check_bf16_input(L1, r, K, ld1, "L1")) || (st = check_bf16_input(L2, N, r, r, "L2"))) return st;
  if (!L1_out || !L2_out || !info) return fail(FP4_ERR_INVALID_ARG, "L1_out, L2_out and info must be non-NULL");
  if (!aligned16(L1_out) || !aligned16(L2_out) || (reinterpret_cast<uintptr_t>(info) & 3u))
    return fail(FP4_ERR_MISALIGNED, "L1_out and L2_out must be 16-byte aligned, info 4-byte aligned");
  const size_t need = fp4_lora_cholqr_workspace(K, r);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  CUDA_TRY(launch_lora_cholqr(L1, K, ld1, L2, N, r, L1_out, L2_out, info, static_cast<float*>(ws),
                              static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

size_t fp4_lora_realign_workspace(int64_t N, int64_t K, int r, int s) {
  if (N <= 0 || K <= 0 || r <= 0 || s <= 0) return 0;
  return round256(realign_workspace_floats(N, K, r, s) * sizeof(float));
}

fp4_status fp4_lora_realign(const void* W_res, int64_t N, int64_t K, int64_t ldw, const void* L1, const void* L2,
                            int r, float beta, const void* Omega, int s, int q, void* W_res_out, void* L1_out,
                            void* L2_out, int* info, void* ws, size_t ws_bytes, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if (r != 16 && r != 32 && r != 48 && r != 64) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "rank r=%d not in {16,32,48,64}", r);
  if (s < r || s > 128 || s % 16 != 0)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "sketch width s=%d must be a multiple of 16 in [r, 128]", s);
  if (q < 0 || q > 8) return fail(FP4_ERR_INVALID_ARG, "power iterations q=%d not in [0, 8]", q);
  if (!(beta > 0.0f)) return fail(FP4_ERR_INVALID_ARG, "beta must be positive");
  if ((st = check_bf16_input(W_res, N, K, ldw, "W_res")) || (st = check_bf16_input(L1, r, K, K, "L1")) ||
      (st = check_bf16_input(L2, N, r, r, "L2")) || (st = check_bf16_input(Omega, K, s, s, "Omega")))
    return st;
  if (N < s || K < s) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "N and K must be at least s");
  if (N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "W dimensions must be below 2^31");
  if (!W_res_out || !L1_out || !L2_out || !info) return fail(FP4_ERR_INVALID_ARG, "outputs and info must be non-NULL");
  if (!aligned16(W_res_out) || !aligned16(L1_out) || !aligned16(L2_out) || (reinterpret_cast<uintptr_t>(info) & 3u))
    return fail(FP4_ERR_MISALIGNED, "outputs must be 16-byte aligned, info 4-byte aligned");
  const size_t need = fp4_lora_realign_workspace(N, K, r, s);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FP4_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  CUDA_TRY(launch_lora_realign(W_res, N, K, ldw, L1, L2, r, beta, Omega, s, q, W_res_out, L1_out, L2_out, info,
                               static_cast<float*>(ws), sm_count(), static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

static fp4_status check_f32_matrix(const float* p, int64_t rows, int64_t cols, int64_t ld, const char* name) {
  if (!p) return fail(FP4_ERR_INVALID_ARG, "%s is NULL", name);
  if (rows <= 0 || cols <= 0 || cols % 16 != 0)
    return fail(FP4_ERR_UNSUPPORTED_SHAPE, "%s is %lld x %lld: cols must be a positive multiple of 16", name,
                (long long)rows, (long long)cols);
  if (ld < cols) return fail(FP4_ERR_INVALID_ARG, "%s: ld %lld < cols %lld", name, (long long)ld, (long long)cols);
  if (!aligned16(p) || ld % 4 != 0)
    return fail(FP4_ERR_MISALIGNED, "%s: base and row pitch must be 16-byte aligned", name);
  if (rows * (cols / 16) >= (int64_t(1) << 32)) return fail(FP4_ERR_UNSUPPORTED_SHAPE, "%s too large", name);
  return FP4_OK;
}

fp4_status fp4_qadamw_v_encode(const float* v, int64_t rows, int64_t cols, int64_t ldv, fp4_tensor* out,
                               uint16_t* mean, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fp4_status st;
  if ((st = check_f32_matrix(v, rows, cols, ldv, "v")) || (st = check_tensor(out, "out"))) return st;
  if (out->rows != rows || out->cols != cols)
    return fail(FP4_ERR_INVALID_ARG, "out is %lld x %lld, expected %lld x %lld", (long long)out->rows,
                (long long)out->cols, (long long)rows, (long long)cols);
  if (!mean || (reinterpret_cast<uintptr_t>(mean) & 1u)) return fail(FP4_ERR_INVALID_ARG, "mean must be non-NULL and 2-byte aligned");
  if (scale_padded(rows, cols)) {
    CUDA_TRY(cudaMemsetAsync(out->scales, 0, scale_bytes(rows, cols), s));
    pdl_chain_break();
  }
  CUDA_TRY(launch_vt_encode(v, rows, cols, ldv, qout(out), mean, sm_count(), s));
  return FP4_OK;
}

fp4_status fp4_qadamw_v_decode(const fp4_tensor* in, const uint16_t* mean, float* v_out, int64_t ldo, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  fp4_status st;
  if ((st = check_tensor(in, "in"))) return st;
  if ((st = check_f32_matrix(v_out, in->rows, in->cols, ldo, "v_out"))) return st;
  if (!mean || (reinterpret_cast<uintptr_t>(mean) & 1u)) return fail(FP4_ERR_INVALID_ARG, "mean must be non-NULL and 2-byte aligned");
  CUDA_TRY(launch_vt_decode(in->codes, in->scales, in->scale, mean, in->rows, in->cols, v_out, ldo, sm_count(),
                            static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

fp4_status fp4_debug_convert(const float* in, int64_t n, uint8_t* e2m1_out, uint8_t* e4m3_out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if (!in || !e2m1_out || !e4m3_out || n <= 0) return fail(FP4_ERR_INVALID_ARG, "bad debug_convert arguments");
  CUDA_TRY(launch_debug_convert(in, n, e2m1_out, e4m3_out, static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

void fp4_debug_force_counter64(int on) { set_force_counter64(on != 0); }

fp4_status fp4_debug_sr_round(const float* in, const uint16_t* rnd16, int64_t n, uint8_t* e2m1_out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if (!in || !rnd16 || !e2m1_out || n <= 0 || n > (int64_t(1) << 34))
    return fail(FP4_ERR_INVALID_ARG, "bad debug_sr_round arguments");
  CUDA_TRY(launch_debug_sr_round(in, rnd16, n, e2m1_out, static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

fp4_status fp4_mma_peak_probe(int n, int iters, int* num_sms_out, void* stream) {
  pdl_chain_break();  // the call's first kernel is ordered after all earlier stream work
  if ((n != 128 && n != 256) || iters <= 0) return fail(FP4_ERR_INVALID_ARG, "probe needs n in {128, 256}, iters > 0");
  const int sms = sm_count();
  if (num_sms_out) *num_sms_out = sms;
  CUDA_TRY(launch_mma_peak(n, iters, sms, static_cast<cudaStream_t>(stream)));
  return FP4_OK;
}

}  // extern "C"
