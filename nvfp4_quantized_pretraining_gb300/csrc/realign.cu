// Periodic realignment of the LoRA-SVD subspace by a randomized SVD ("Full-Stack
// FP4", section 2.1, Realignment: the subspace is reset with a randomized SVD so
// that the BF16 branch stays optimal).  The method is the randomized subspace
// iteration and direct SVD of Halko, Martinsson and Tropp (SIAM Review 2011,
// Algorithms 4.4 and 5.1) on W = W_res + beta L2 L1:
//   Y = W Omega;  q times: Y = W basis(W^T basis(Y));  Q = orth(Y);  B = Q^T W;
//   B B^T = Ub Lambda Ub^T (Jacobi);  L2 = Q Ub_r Sigma_r / beta;  L1 = Ub_r^T B / Sigma_r;
//   W_res = W - beta bf16(L2) bf16(L1).
// FP32 throughout.  The sketch products with W and W^T (Y = W Omega, the power
// iterations, B^T = W^T Q) run on the tensor cores as three TF32 products per
// FP32 product (rl_tf32x3_kernel, FP32-class accuracy); the other products in
// this file's own tiled FP32 GEMM (rl_sgemm_kernel); both split over K into a
// fixed-order sum when the output has few tiles.  orth() is Cholesky-QR (the factor and its
// inverse in one CTA, Y L^-T as a product): twice for the final basis,
// once between the products of the subspace iteration, which depend on the span
// only.  The first pass adds a small diagonal shift: the column space is that of
// Y whatever the triangular factor, so the shift only guards the factorisation
// of a near-rank-deficient sketch.  The small symmetric eigenproblem is a cyclic
// Jacobi iteration with round-robin pairs in one CTA.
#include <atomic>

#include "bf16_convert.cuh"
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kRlThreads = 256;
constexpr int kRlMaxS = 128;

// ---------------------------------------------------------------------------
// Conversions
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRlThreads) rl_bf16_to_f32(const uint16_t* __restrict__ in, int64_t ld,
                                                             float* __restrict__ out, int64_t ldo, int64_t rows,
                                                             int64_t cols) {
  const int64_t n = rows * cols;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / cols, c = e - r * cols;
    out[r * ldo + c] = __uint_as_float(static_cast<uint32_t>(in[r * ld + c]) << 16);
  }
}

// out = bf16(in * rs[row] * cs[col]) (rs, cs optional); nothing is written when *info != 0.
__global__ void __launch_bounds__(kRlThreads) rl_f32_to_bf16(const float* __restrict__ in, int64_t ld,
                                                             uint16_t* __restrict__ out, int64_t ldo, int64_t rows,
                                                             int64_t cols, const float* __restrict__ rs,
                                                             const float* __restrict__ cs,
                                                             const int* __restrict__ info) {
  if (*info != 0) return;
  const int64_t n = rows * cols;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / cols, c = e - r * cols;
    float v = in[r * ld + c];
    if (rs) v *= rs[r];
    if (cs) v *= cs[c];
    out[r * ldo + c] = static_cast<uint16_t>(bf16_rn_bits(v));
  }
}

// ---------------------------------------------------------------------------
// FP32 GEMM on row-major operands: C (m x n, ldc) = alpha op(A) op(B) + beta C, op(A) m x k
// (A stored m x k, or k x m when ta), op(B) k x n (B stored k x n, or n x k when tb).  A CTA
// of 256 threads computes a BM x BN tile, TM x TN outputs per thread (128 x 32, 64 x 64 or
// 32 x 128 with 4 x 4; 128 x 80 or 80 x 128 with 8 x 5 or 5 x 8 for the products whose one
// side is the sketch width 80; whichever pads the output least), over the K slice of blockIdx.z: with one slice it
// writes C; with several, each slice's sum goes to partial[z] (m x n) and rl_sgemm_reduce adds
// the slices in order, so the result is deterministic.  Tiles of op(A) and op(B), 16 deep in K,
// are staged in shared memory k-major; the loads run along whichever dimension is contiguous.
// ---------------------------------------------------------------------------
namespace rg {
constexpr int BK = 16, THREADS = 256;
}

template <bool TA, bool TB, int BM, int BN, int TM, int TN>
__global__ void __launch_bounds__(rg::THREADS) rl_sgemm_kernel(int64_t m, int64_t n, int64_t k, int64_t kslice,
                                                              float alpha, const float* __restrict__ A, int64_t lda,
                                                              const float* __restrict__ B, int64_t ldb, float beta,
                                                              float* __restrict__ C, int64_t ldc,
                                                              float* __restrict__ partial) {
  using namespace rg;
  static_assert(BM * BN == TM * TN * THREADS && BM % TM == 0 && BN % TN == 0, "TM x TN outputs per thread");
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Bs[BK][BN + 4];
  const int tid = threadIdx.x, tx = tid % (BN / TN), ty = tid / (BN / TN);
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM, n0 = static_cast<int64_t>(blockIdx.x) * BN;
  const int64_t k0 = static_cast<int64_t>(blockIdx.z) * kslice;
  const int64_t k1 = k0 + kslice < k ? k0 + kslice : k;
  float acc[TM][TN] = {};
  for (int64_t kt = k0; kt < k1; kt += BK) {
#pragma unroll
    for (int u = 0; u < BM * BK / THREADS; ++u) {
      const int e = tid + u * THREADS;
      int mi, ki;
      if (TA) { ki = e / BM; mi = e % BM; }  // A stored k x m: contiguous along m
      else { mi = e / BK; ki = e % BK; }     // A stored m x k: contiguous along k
      const int64_t gm = m0 + mi, gk = kt + ki;
      As[ki][mi] = (gm < m && gk < k1) ? (TA ? A[gk * lda + gm] : A[gm * lda + gk]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < BN * BK / THREADS; ++u) {
      const int e = tid + u * THREADS;
      int nj, kj;
      if (TB) { nj = e / BK; kj = e % BK; }  // B stored n x k: contiguous along k
      else { kj = e / BN; nj = e % BN; }     // B stored k x n: contiguous along n
      const int64_t gn = n0 + nj, gk = kt + kj;
      Bs[kj][nj] = (gn < n && gk < k1) ? (TB ? B[gn * ldb + gk] : B[gk * ldb + gn]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[TM], bv[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) av[i] = As[kk][TM * ty + i];
#pragma unroll
      for (int j = 0; j < TN; ++j) bv[j] = Bs[kk][TN * tx + j];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = partial ? partial + static_cast<int64_t>(blockIdx.z) * m * n : nullptr;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t gm = m0 + TM * ty + i;
    if (gm >= m) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int64_t gn = n0 + TN * tx + j;
      if (gn >= n) continue;
      if (out) out[gm * n + gn] = acc[i][j];
      else C[gm * ldc + gn] = beta == 0.0f ? alpha * acc[i][j] : fmaf(alpha, acc[i][j], beta * C[gm * ldc + gn]);
    }
  }
}

// C = alpha (partial[0] + partial[1] + ... + partial[splits - 1]) + beta C, slices added in order.
__global__ void __launch_bounds__(kRlThreads) rl_sgemm_reduce(int64_t m, int64_t n, int splits, float alpha,
                                                              const float* __restrict__ partial, float beta,
                                                              float* __restrict__ C, int64_t ldc) {
  const int64_t total = m * n;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.0f;
    for (int z = 0; z < splits; ++z) s += partial[z * total + e];
    const int64_t r = e / n, c = e - r * n;
    C[r * ldc + c] = beta == 0.0f ? alpha * s : fmaf(alpha, s, beta * C[r * ldc + c]);
  }
}

// Elements of split-K scratch the products of one realignment need at most (see Rl::gemm).
constexpr int64_t kRlSplitFloats = int64_t(1) << 21;

// ---------------------------------------------------------------------------
// FP32 products on the tensor cores: out (M x n, pitch n) = A B^T with A (M x Kc) and B (n x Kc)
// both row-major and contiguous along Kc, n a multiple of 16 up to 128, as three TF32 products
// (tcgen05.mma kind::tf32, FP32 accumulation in tensor memory):
//   A B^T ~ A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T,  x_hi = x with its 13 low mantissa bits
//   cleared (exactly a TF32 value), x_lo = x - x_hi (exact in FP32).
// The dropped term A_lo B_lo^T is below 2^-20 |a||b| per product, and the tensor core's
// conversion of x_lo to TF32 loses at most 2^-21 |x|, so the result is within a small multiple of
// FP32 rounding.  A's tiles arrive
// by TMA in FP32 and four warps split them in shared memory (the high part in place, the low
// part beside it); B is split once beforehand, its high and low parts stacked as the rows
// [0, n) and [n, 2n) of one 2n x Kc matrix.  blockIdx.x takes 128 rows of A, blockIdx.y the
// K stages [y * kss, (y + 1) * kss): with one slice it writes out directly, with several
// out is slice y's partial sum (M x n) and rl_sgemm_reduce adds the slices in order.
// ---------------------------------------------------------------------------
namespace rt {
constexpr int BM = 128;
constexpr int BK = 32;                    // FP32 elements of K per stage: one 128-byte row
constexpr int MAX_STAGES = 4;
constexpr int TILE_BYTES = BM * BK * 4;   // 16 KB: 128 rows of A
constexpr int NUM_THREADS = 192;          // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 split + epilogue
constexpr int SMEM_MAX = 232448;
// A stage holds A_hi, A_lo (16 KB each), then B_hi and B_lo (n rows of 128 bytes each: a
// multiple of 1024 bytes for n % 8 == 0); as many stages as fit, up to four.
__host__ __device__ constexpr uint32_t stage_bytes(uint32_t n) { return 2 * TILE_BYTES + 2 * n * BK * 4; }
__host__ __device__ constexpr uint32_t num_stages(uint32_t n) {
  return (SMEM_MAX - 1024 - 256) / stage_bytes(n) < MAX_STAGES ? (SMEM_MAX - 1024 - 256) / stage_bytes(n)
                                                                : MAX_STAGES;
}
__host__ __device__ constexpr uint32_t smem_bytes(uint32_t n) { return num_stages(n) * stage_bytes(n) + 1024 + 256; }
static_assert(num_stages(128) >= 3 && num_stages(80) == 4 && smem_bytes(96) <= SMEM_MAX, "stages");
}  // namespace rt

// Instruction descriptor, kind::tf32: TF32 x TF32 -> FP32, K-major A and B.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
  return (1u << 4)             // D format FP32
         | (2u << 7)           // A format TF32
         | (2u << 10)          // B format TF32
         | ((N >> 3) << 17) | ((M >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void rl_tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

__global__ void __launch_bounds__(rt::NUM_THREADS, 1)
    rl_tf32x3_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     uint32_t M, uint32_t n, uint32_t Kc, uint32_t kss, float* __restrict__ out) {
  using namespace rt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t STAGES = num_stages(n), STAGE_BYTES = stage_bytes(n), B_BYTES = n * BK * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* ready = full + STAGES;
  uint64_t* empty = ready + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* done_bar = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 4);  // the four split warps
      mbar_init(&empty[s], 1);  // the MMA commit
    }
    mbar_init(acc_full, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t num_k_all = (Kc + BK - 1) / BK;
  const uint32_t k_begin = blockIdx.y * kss;
  const uint32_t num_k = min(kss, num_k_all - k_begin);  // >= 1: the host makes no empty slice
  const uint32_t m0 = blockIdx.x * BM;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int armed[MAX_STAGES];
      uint32_t armed_phase[MAX_STAGES];
      for (int s = 0; s < MAX_STAGES; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
        uint8_t* st = smem + stage * STAGE_BYTES;
        // A's 128 rows (rows past M and columns past Kc arrive zero-filled), then B's high and low rows
        mbar_arrive_expect_tx(&full[stage], TILE_BYTES + 2 * B_BYTES);
        const int32_t kx = (int32_t)((k_begin + it) * BK);
        tma_load_2d(st, &tmap_a, &full[stage], kx, (int32_t)m0);
        tma_load_2d(st + 2 * TILE_BYTES, &tmap_b, &full[stage], kx, 0);
        tma_load_2d(st + 2 * TILE_BYTES + B_BYTES, &tmap_b, &full[stage], kx, (int32_t)n);
        armed[stage] = 1;
        armed_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        for (uint32_t s = 0; s < STAGES; ++s)
          if (armed[s]) mbar_wait(&full[s], armed_phase[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(BM, n);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait(&ready[stage], phase)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
#pragma unroll
        for (uint32_t kk = 0; kk < BK / 8; ++kk) {  // 8 TF32 elements (32 bytes) of K per MMA
          const uint32_t o = kk * 32;
          const uint64_t a_hi = smem_desc(sa + o, 16, 1024, kSwizzle128B);
          const uint64_t a_lo = smem_desc(sa + TILE_BYTES + o, 16, 1024, kSwizzle128B);
          const uint64_t b_hi = smem_desc(sa + 2 * TILE_BYTES + o, 16, 1024, kSwizzle128B);
          const uint64_t b_lo = smem_desc(sa + 2 * TILE_BYTES + B_BYTES + o, 16, 1024, kSwizzle128B);
          mma_tf32(tmem, a_lo, b_hi, idesc, (it | kk) != 0);
          mma_tf32(tmem, a_hi, b_lo, idesc, 1);
          mma_tf32(tmem, a_hi, b_hi, idesc, 1);
        }
        tc_commit(&empty[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (ok) tc_commit(acc_full);
      else *abort_flag = 1;
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
  } else {
    // warps 2..5: split each landed A tile (an elementwise map, so the swizzle does not matter),
    // then drain the accumulator: warp w reads TMEM lanes 32 (w % 4) .. + 31, one row per lane
    const int t = (warp - 2) * 32 + lane;
    uint32_t stage = 0, phase = 0;
    for (uint32_t it = 0; it < num_k; ++it) {
      if (*abort_flag || !mbar_wait_warp(&full[stage], phase)) {
        *abort_flag = 1;
        break;
      }
      float4* hi = reinterpret_cast<float4*>(smem + stage * STAGE_BYTES);
      float4* lo = reinterpret_cast<float4*>(smem + stage * STAGE_BYTES + TILE_BYTES);
#pragma unroll
      for (int i = 0; i < TILE_BYTES / 16 / 128; ++i) {
        const int u = t + 128 * i;
        const float4 v = hi[u];
        const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
        hi[u] = h;
        lo[u] = make_float4(__fsub_rn(v.x, h.x), __fsub_rn(v.y, h.y), __fsub_rn(v.z, h.z), __fsub_rn(v.w, h.w));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[stage]);
      if (++stage == STAGES) stage = 0, phase ^= 1;
    }
    const uint32_t quad = warp & 3;
    if (!*abort_flag && mbar_wait_warp(acc_full, 0)) {
      tc_fence_after();
      const uint32_t row = m0 + quad * 32 + lane;
      for (uint32_t j = 0; j < n / 16; ++j) {
        uint32_t v[16];
        rl_tmem_ld16(tmem + ((quad * 32) << 16) + 16 * j, v);
        if (row < M) {
          float* dst = out + (size_t)blockIdx.y * M * n + (size_t)row * n + 16 * j;
          if ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) {  // n % 16 == 0: every row starts aligned
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<float4*>(dst)[q] =
                  make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                              __uint_as_float(v[4 * q + 3]));
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) dst[q] = __uint_as_float(v[q]);
          }
        }
      }
      tc_fence_before();
    } else {
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (*abort_flag) {  // a wait expired: let copies still in flight land first
    if (threadIdx.x == 0) drain_pause();
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Transpose of an FP32 matrix (rows x cols, pitch cols) into out (cols x rows, pitch rows); with
// SPLIT, the TF32 high part goes to out's rows [0, cols) and the low part to rows [cols, 2 cols).
template <bool SPLIT>
__global__ void rl_transpose_kernel(const float* __restrict__ in, int64_t rows, int64_t cols,
                                    float* __restrict__ out) {
  __shared__ float t[32][33];
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t r = static_cast<int64_t>(blockIdx.y) * 32 + i;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[r * cols + c];
  }
  __syncthreads();
  const int64_t r2 = static_cast<int64_t>(blockIdx.y) * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t c2 = static_cast<int64_t>(blockIdx.x) * 32 + i;
    if (r2 < rows && c2 < cols) {
      const float v = t[threadIdx.x][i];
      if (SPLIT) {
        const float h = tf32_hi(v);
        out[c2 * rows + r2] = h;
        out[(cols + c2) * rows + r2] = __fsub_rn(v, h);
      } else {
        out[c2 * rows + r2] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Cholesky of an S x S Gram matrix (S <= 128, a multiple of 16) in one CTA, and
// the inverse of the factor: G + shift * mean(diag) I = L L^T (right-looking on
// the unscaled columns: with d_j the pivot, G_ik -= (G_ij / d_j) G_kj, and
// L_ij = G_ij / sqrt(d_j) at the end), then M = L^-1 with thread c computing
// column c by forward substitution: x_i = (delta_ic - sum_{k < i} L_ik x_k) / L_ii.
// The 256 threads hold G as a 16 x 16 grid of (S/16) x (S/16) register blocks
// (thread (ty, tx) has rows ty + 16a and columns tx + 16b), so each step's update
// is local: the owners of column j publish it in shared memory, one barrier, and
// every thread updates its own elements.  The substitution runs right-looking
// (once x_i is known, every later row's partial sum takes its term), which adds
// each row's terms in the same order as the left-looking form but leaves the
// multiply-adds of a step independent of each other.  The partial sums of rows
// i, i + 1, .. sit in registers r[0], r[1], .. and shift down by one each step
// (r[t] <- r[t + 1] - L_{i+1+t,i} x_i), so that every index is a compile-time
// one; step i's coefficients L_{i+1+t,i} are stored from the start of a padded
// row of shared memory (zeros past the end), read 16 bytes at a time.  Writes M
// (lower, row-major S x S); a non-positive pivot sets *info (if still 0) to
// 1000 * stage + its order.
// ---------------------------------------------------------------------------
constexpr int kRlCholThreads = 256;

template <int S>
constexpr int chol_smem_floats() {
  return S * (S + 4) + 4 * S;  // sub-diagonal coefficients (rows padded), two column buffers, pivots, diagonal
}

template <int S>
__global__ void __launch_bounds__(kRlCholThreads) rl_cholesky_kernel(const float* __restrict__ Gin, float shift,
                                                                     float* __restrict__ Mout, int* __restrict__ info,
                                                                     int stage) {
  constexpr int B = S / 16;
  constexpr int ld = S + 4;
  extern __shared__ float sh[];
  float* LS = sh;             // LS[k * ld + t] = L_{k+1+t, k} for t < S - 1 - k, 0 beyond
  float* col = sh + S * ld;   // column j of the partly factored matrix, in col[(j & 1) * S + i]
  float* piv = col + 2 * S;   // the pivots d_j
  float* diag = piv + S;      // L_kk
  __shared__ float mean_diag;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float g[B][B];
#pragma unroll
  for (int a = 0; a < B; ++a)
#pragma unroll
    for (int b = 0; b < B; ++b) g[a][b] = Gin[(ty + 16 * a) * S + tx + 16 * b];
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int i = 0; i < S; ++i) t += Gin[i * S + i];
    mean_diag = t / S;
  }
  // zero the coefficient rows (their tails past each step's last row stay zero; the barriers of the
  // factorization order this before the coefficients are written)
  for (int e = threadIdx.x; e < S * ld; e += kRlCholThreads) LS[e] = 0.0f;
  __syncthreads();
  if (tx == ty) {
    const float add = shift * mean_diag;
#pragma unroll
    for (int a = 0; a < B; ++a) g[a][a] += add;
  }
  int bad = 0;
#pragma unroll
  for (int bj = 0; bj < B; ++bj) {
    for (int jj = 0; jj < 16 && !bad; ++jj) {
      const int j = 16 * bj + jj;
      float* cj = col + (j & 1) * S;
      if (tx == jj) {  // this thread column owns column j: publish rows j.. of it
#pragma unroll
        for (int a = 0; a < B; ++a)
          if (ty + 16 * a >= j) cj[ty + 16 * a] = g[a][bj];
      }
      __syncthreads();  // column j visible; every read of column j - 2's buffer is done
      const float d = cj[j];  // every thread reads the same pivot: the test is uniform
      if (!(d > 0.0f)) {
        bad = j + 1;
        break;
      }
      if (threadIdx.x == 0) piv[j] = d;
      const float inv = 1.0f / d;
      float li[B], lk[B];
#pragma unroll
      for (int a = 0; a < B; ++a) li[a] = ty + 16 * a > j ? cj[ty + 16 * a] * inv : 0.0f;
#pragma unroll
      for (int b = 0; b < B; ++b) lk[b] = tx + 16 * b > j ? cj[tx + 16 * b] : 0.0f;
#pragma unroll
      for (int a = 0; a < B; ++a)
#pragma unroll
        for (int b = 0; b < B; ++b)
          if (tx + 16 * b > j && tx + 16 * b <= ty + 16 * a) g[a][b] = fmaf(-li[a], lk[b], g[a][b]);
    }
  }
  if (bad) {
    if (threadIdx.x == 0) atomicCAS(info, 0, 1000 * stage + bad);
    return;
  }
  __syncthreads();  // every pivot written
#pragma unroll
  for (int a = 0; a < B; ++a)
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int i = ty + 16 * a, k = tx + 16 * b;
      if (k < i) LS[k * ld + (i - k - 1)] = g[a][b] * rsqrtf(piv[k]);
      else if (k == i) diag[k] = sqrtf(piv[k]);
    }
  __syncthreads();
  if (threadIdx.x < S) {
    const int c = threadIdx.x;
    float r[S];
#pragma unroll
    for (int t = 0; t < S; ++t) r[t] = t == c ? 1.0f : 0.0f;
    for (int i = 0; i < S; ++i) {
      const float x = i < c ? 0.0f : r[0] / diag[i];
      Mout[i * S + c] = x;
      const float4* row = reinterpret_cast<const float4*>(LS + i * ld);
#pragma unroll
      for (int q = 0; q < S / 4; ++q) {
        const float4 l = row[q];
        r[4 * q] = fmaf(-l.x, x, r[4 * q + 1]);
        r[4 * q + 1] = fmaf(-l.y, x, r[4 * q + 2]);
        r[4 * q + 2] = fmaf(-l.z, x, r[4 * q + 3]);
        if (4 * q + 4 < S) r[4 * q + 3] = fmaf(-l.w, x, r[4 * q + 4]);
      }
    }
  }
}

template <int S>
static cudaError_t cholesky_launch(const float* G, float shift, float* M, int* info, int stage, cudaStream_t st) {
  const int smem = chol_smem_floats<S>() * static_cast<int>(sizeof(float));
  static const cudaError_t attr =
      cudaFuncSetAttribute(rl_cholesky_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  rl_cholesky_kernel<S><<<1, kRlCholThreads, smem, st>>>(G, shift, M, info, stage);
  count_launch();
  return cudaGetLastError();
}

static cudaError_t launch_cholesky(int s, const float* G, float shift, float* M, int* info, int stage,
                                   cudaStream_t st) {
  switch (s) {
    case 16: return cholesky_launch<16>(G, shift, M, info, stage, st);
    case 32: return cholesky_launch<32>(G, shift, M, info, stage, st);
    case 48: return cholesky_launch<48>(G, shift, M, info, stage, st);
    case 64: return cholesky_launch<64>(G, shift, M, info, stage, st);
    case 80: return cholesky_launch<80>(G, shift, M, info, stage, st);
    case 96: return cholesky_launch<96>(G, shift, M, info, stage, st);
    case 112: return cholesky_launch<112>(G, shift, M, info, stage, st);
    case 128: return cholesky_launch<128>(G, shift, M, info, stage, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------
// Symmetric eigenproblem C = V diag(lambda) V^T (s x s, s even, s <= 128) in one
// CTA: cyclic Jacobi (Golub and Van Loan, Matrix Computations, the symmetric
// Schur rotation), each round rotating s / 2 disjoint pairs chosen by the
// round-robin schedule (pair 0 is (s - 1, r), pair k is ((r + k) mod (s - 1),
// (r - k) mod (s - 1))).  A round is two phases: the rotations, then A <- J^T A J
// as disjoint 2 x 2 blocks (rows of pair k, columns of pair l; only blocks with
// k <= l are computed, each writing its mirror too, so A stays exactly symmetric)
// and V <- V J; a round in which no pair rotates skips its update.  A
// pair is rotated when |a_pq| > 1e-6 ||A||_F (the Frobenius norm is invariant
// under the rotations; FP32 rounding leaves off-diagonal noise near 6e-8 ||A||,
// so a threshold relative to the diagonal would never be met); a sweep that
// rotates nothing ends the iteration (at most `max_sweeps`).  Outputs the eigenvalues in
// decreasing order and the eigenvectors as columns of a row-major s x s matrix.
// ---------------------------------------------------------------------------
constexpr int kRlJacThreads = 1024;

__global__ void __launch_bounds__(kRlJacThreads) rl_jacobi_kernel(const float* __restrict__ Cin, int s, int max_sweeps,
                                                                  float* __restrict__ evals,
                                                                  float* __restrict__ evecs,
                                                                  const int* __restrict__ info) {
  extern __shared__ float sh[];
  const int ld = s + 1;
  float* A = sh;              // s x ld
  float* V = sh + s * ld;     // s x ld (2 s ld floats: a multiple of 16 bytes for even s)
  float4* ROT = reinterpret_cast<float4*>(V + s * ld);  // s / 2 pairs: (head, tail) as int bits, (cos, sin)
  __shared__ int rotated;
  __shared__ int round_rotated[2];  // round t's flag in [t & 1]
  __shared__ float red[kRlJacThreads / 32];
  if (*info != 0) return;
  float sq = 0.0f;
  for (int e = threadIdx.x; e < s * s; e += blockDim.x) {
    const int i = e / s, j = e % s;
    const float a = Cin[e];
    A[i * ld + j] = a;
    V[i * ld + j] = i == j ? 1.0f : 0.0f;
    sq += a * a;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
  __syncthreads();
  float fro2 = 0.0f;
  for (int w = 0; w < kRlJacThreads / 32; ++w) fro2 += red[w];
  const float thresh = 1e-6f * sqrtf(fro2);
  const int half = s / 2;
  // This thread's share of each round's update, the same in every round: 2 x 2 blocks (k, l), k <= l,
  // of A (A stays exactly symmetric: block (k, l) also writes its mirror, block (l, k)) and entries
  // (pair l, row i) of V, packed as k | l << 8 and l | i << 8 (s <= 128), computed once here rather
  // than by a division per item and round.
  constexpr int kItA = ((kRlMaxS / 2) * (kRlMaxS / 2 + 1) / 2 + kRlJacThreads - 1) / kRlJacThreads;
  constexpr int kItV = (kRlMaxS / 2) * kRlMaxS / kRlJacThreads;
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  uint32_t it_a[kItA], it_v[kItV];
#pragma unroll
  for (int j = 0; j < kItA; ++j) {
    int e = threadIdx.x + j * kRlJacThreads;
    it_a[j] = kNone;
    if (e < half * (half + 1) / 2) {  // row k of the upper triangle holds half - k blocks
      int k = 0;
      while (e >= half - k) e -= half - k, ++k;
      it_a[j] = (uint32_t)k | ((uint32_t)(k + e) << 8);
    }
  }
#pragma unroll
  for (int j = 0; j < kItV; ++j) {
    const int f = threadIdx.x + j * kRlJacThreads;
    it_v[j] = f < half * s ? (uint32_t)(f / s) | ((uint32_t)(f % s) << 8) : kNone;
  }
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    if (threadIdx.x == 0) rotated = round_rotated[0] = round_rotated[1] = 0;
    __syncthreads();
    for (int round = 0; round < s - 1; ++round) {
      for (int k = threadIdx.x; k < half; k += blockDim.x) {
        // round-robin pairs: (s - 1, round) and ((round + k) mod (s - 1), (round - k) mod (s - 1))
        int p = round + k, q = round - k;
        if (p >= s - 1) p -= s - 1;
        if (q < 0) q += s - 1;
        if (k == 0) p = s - 1;
        const float apq = A[p * ld + q], app = A[p * ld + p], aqq = A[q * ld + q];
        float c = 1.0f, t = 0.0f;
        if (fabsf(apq) > thresh) {
          const float tau = (aqq - app) / (2.0f * apq);
          t = (tau >= 0.0f ? 1.0f : -1.0f) / (fabsf(tau) + sqrtf(1.0f + tau * tau));
          c = rsqrtf(1.0f + t * t);
          round_rotated[round & 1] = 1;
          rotated = 1;
        }
        ROT[k] = make_float4(__int_as_float(p), __int_as_float(q), c, t * c);
      }
      // the next round's flag: every read of it (last round) came before this round's first barrier
      if (threadIdx.x == 0) round_rotated[(round + 1) & 1] = 0;
      __syncthreads();
      // a round without a rotation changes nothing: no update, and no second barrier (its pairs and
      // rotations are not read, and A is not written)
      if (!round_rotated[round & 1]) continue;
      // A <- J^T A J as 2 x 2 blocks (k <= l, each written with its mirror); V <- V J
#pragma unroll
      for (int j = 0; j < kItA; ++j) {
        if (it_a[j] == kNone) continue;
        const int k = it_a[j] & 0xFFu, l = it_a[j] >> 8;
        const float4 rk = ROT[k], rl = ROT[l];
        const int pk = __float_as_int(rk.x), qk = __float_as_int(rk.y), pl = __float_as_int(rl.x),
                  ql = __float_as_int(rl.y);
        const float ck = rk.z, sk = rk.w, cl = rl.z, sl = rl.w;
        const float xpp = A[pk * ld + pl], xpq = A[pk * ld + ql], xqp = A[qk * ld + pl], xqq = A[qk * ld + ql];
        const float rpp = ck * xpp - sk * xqp, rpq = ck * xpq - sk * xqq;  // rows of pair k
        const float rqp = sk * xpp + ck * xqp, rqq = sk * xpq + ck * xqq;
        const float npp = cl * rpp - sl * rpq, npq = sl * rpp + cl * rpq;  // columns of pair l
        const float nqp = cl * rqp - sl * rqq, nqq = sl * rqp + cl * rqq;
        if (k == l) {  // a diagonal block: its two off-diagonal entries are one value
          A[pk * ld + pk] = npp;
          A[pk * ld + qk] = npq;
          A[qk * ld + pk] = npq;
          A[qk * ld + qk] = nqq;
        } else {
          A[pk * ld + pl] = npp;
          A[pk * ld + ql] = npq;
          A[qk * ld + pl] = nqp;
          A[qk * ld + ql] = nqq;
          A[pl * ld + pk] = npp;
          A[ql * ld + pk] = npq;
          A[pl * ld + qk] = nqp;
          A[ql * ld + qk] = nqq;
        }
      }
#pragma unroll
      for (int j = 0; j < kItV; ++j) {
        if (it_v[j] == kNone) continue;
        const int l = it_v[j] & 0xFFu, i = it_v[j] >> 8;
        const float4 rl = ROT[l];
        const int pl = __float_as_int(rl.x), ql = __float_as_int(rl.y);
        const float cl = rl.z, sl = rl.w;
        const float vp = V[i * ld + pl], vq = V[i * ld + ql];
        V[i * ld + pl] = cl * vp - sl * vq;
        V[i * ld + ql] = sl * vp + cl * vq;
      }
      __syncthreads();
    }
    const int any = rotated;  // read after the last round's barrier
    __syncthreads();          // every thread has read it before thread 0 resets it
    if (!any) break;
  }
  // decreasing order (selection by one thread; s <= 128), then the permuted output
  int* order = reinterpret_cast<int*>(ROT);  // reuse: s entries fit in the s / 2 pairs
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < s; ++i) order[i] = i;
    for (int i = 0; i < s; ++i) {
      int best = i;
      for (int j = i + 1; j < s; ++j)
        if (A[order[j] * ld + order[j]] > A[order[best] * ld + order[best]]) best = j;
      const int tmp = order[i];
      order[i] = order[best];
      order[best] = tmp;
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < s; j += blockDim.x) evals[j] = A[order[j] * ld + order[j]];
  for (int e = threadIdx.x; e < s * s; e += blockDim.x) {
    const int i = e / s, j = e % s;
    evecs[e] = V[i * ld + order[j]];
  }
}

// Row j of T1 (r x K): the sign of its largest-magnitude entry (first index on ties)
// fixes the pair's sign; rs[j] = flip / sigma_j (L1 rows), cs[j] = flip sigma_j / beta
// (L2 columns), sigma_j = sqrt(max(lambda_j, 0)); a zero sigma gives zero scales.
__global__ void __launch_bounds__(kRlThreads) rl_sign_scale_kernel(const float* __restrict__ T1, int64_t K,
                                                                   const float* __restrict__ evals, float beta,
                                                                   float* __restrict__ rs, float* __restrict__ cs,
                                                                   const int* __restrict__ info) {
  __shared__ float bv[kRlThreads];
  __shared__ int64_t bi[kRlThreads];
  if (*info != 0) return;
  const int j = blockIdx.x;
  const float* row = T1 + j * K;
  float best = -1.0f;
  int64_t idx = 0;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
    const float a = fabsf(row[k]);
    if (a > best) {
      best = a;
      idx = k;
    }
  }
  bv[threadIdx.x] = best;
  bi[threadIdx.x] = idx;
  __syncthreads();
  for (int o = kRlThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      const float ov = bv[threadIdx.x + o];
      const int64_t oi = bi[threadIdx.x + o];
      if (ov > bv[threadIdx.x] || (ov == bv[threadIdx.x] && oi < bi[threadIdx.x])) {
        bv[threadIdx.x] = ov;
        bi[threadIdx.x] = oi;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float flip = row[bi[0]] < 0.0f ? -1.0f : 1.0f;
    const float sigma = sqrtf(fmaxf(evals[j], 0.0f));
    rs[j] = sigma > 0.0f ? flip / sigma : 0.0f;
    cs[j] = flip * sigma / beta;
  }
}

// ---------------------------------------------------------------------------
// Orchestration
// ---------------------------------------------------------------------------
namespace {

struct Rl {
  cudaStream_t s;
  int num_sms;
  float* split;  // kRlSplitFloats of split-K scratch
  cudaError_t err = cudaSuccess;

  // Row-major C (m x n, ldc) = alpha op(A) op(B) + beta C, op(A) m x k, op(B) k x n.  An output
  // of fewer tiles than two per SM is split over K (slices of at least 128) into the scratch, as
  // far as it holds the slices.
  void gemm(bool ta, bool tb, int64_t m, int64_t n, int64_t k, float alpha, const float* A, int64_t lda,
            const float* B, int64_t ldb, float beta, float* C, int64_t ldc) {
    if (err != cudaSuccess) return;
    // the tile shape that pads the output least (ties: the earlier in this list)
    const int64_t shapes[5][2] = {{128, 80}, {80, 128}, {64, 64}, {128, 32}, {32, 128}};
    int pick = 0;
    int64_t best = -1;
    for (int i = 0; i < 5; ++i) {
      const int64_t bm = shapes[i][0], bn = shapes[i][1];
      const int64_t area = ((m + bm - 1) / bm) * bm * ((n + bn - 1) / bn) * bn;
      if (best < 0 || area < best) best = area, pick = i;
    }
    const int64_t BM = shapes[pick][0], BN = shapes[pick][1];
    const int64_t tiles = ((m + BM - 1) / BM) * ((n + BN - 1) / BN);
    int64_t splits = 1;
    const int64_t want = 2 * static_cast<int64_t>(num_sms);
    if (tiles < want) {
      splits = (want + tiles - 1) / tiles;
      const int64_t by_k = (k + 127) / 128;
      if (splits > by_k) splits = by_k;
      const int64_t by_ws = kRlSplitFloats / (m * n);
      if (splits > by_ws) splits = by_ws;
      if (splits > 256) splits = 256;
      if (splits < 1) splits = 1;
    }
    int64_t kslice = (k + splits - 1) / splits;
    kslice = (kslice + rg::BK - 1) / rg::BK * rg::BK;
    splits = (k + kslice - 1) / kslice;
    const dim3 grid(static_cast<unsigned>((n + BN - 1) / BN), static_cast<unsigned>((m + BM - 1) / BM),
                    static_cast<unsigned>(splits));
    float* part = splits > 1 ? split : nullptr;
    launch_tile(pick, ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return;
    if (part) {
      rl_sgemm_reduce<<<this->grid(m * n), kRlThreads, 0, s>>>(m, n, static_cast<int>(splits), alpha, part, beta, C, ldc);
      count_launch();
      err = cudaGetLastError();
    }
  }
  template <int BM, int BN>
  void launch_t(bool ta, bool tb, dim3 grid, int64_t m, int64_t n, int64_t k, int64_t kslice, float alpha,
                const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                float* part) {
    constexpr int TM = BM == 128 && BN == 80 ? 8 : BM == 80 ? 5 : 4;
    constexpr int TN = BM == 128 && BN == 80 ? 5 : BM == 80 ? 8 : 4;
    if (ta && tb) rl_sgemm_kernel<true, true, BM, BN, TM, TN><<<grid, rg::THREADS, 0, s>>>(m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else if (ta) rl_sgemm_kernel<true, false, BM, BN, TM, TN><<<grid, rg::THREADS, 0, s>>>(m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else if (tb) rl_sgemm_kernel<false, true, BM, BN, TM, TN><<<grid, rg::THREADS, 0, s>>>(m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else rl_sgemm_kernel<false, false, BM, BN, TM, TN><<<grid, rg::THREADS, 0, s>>>(m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
  }
  void launch_tile(int pick, bool ta, bool tb, dim3 grid, int64_t m, int64_t n, int64_t k, int64_t kslice,
                   float alpha, const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                   int64_t ldc, float* part) {
    if (pick == 0) launch_t<128, 80>(ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else if (pick == 1) launch_t<80, 128>(ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else if (pick == 3) launch_t<128, 32>(ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else if (pick == 4) launch_t<32, 128>(ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
    else launch_t<64, 64>(ta, tb, grid, m, n, k, kslice, alpha, A, lda, B, ldb, beta, C, ldc, part);
  }
  // out (m x n, pitch n) = A X with A m x kc (pitch kc) and X kc x n (pitch n), on the tensor
  // cores (rl_tf32x3_kernel) when the shapes suit its tiles and TMA (m >= 128, kc >= 32 and a
  // multiple of 4, n a multiple of 16 up to 128), else on the tiled FP32 GEMM.  bsplit: 2 n x kc
  // floats of scratch for X^T split into its TF32 high and low parts.  Outputs with fewer
  // 128-row tiles than SMs are split over K, as far as the split-K scratch holds the slices.
  void tc(const float* A, int64_t m, int64_t kc, const float* X, int n, float* bsplit, float* out) {
    if (err != cudaSuccess) return;
    if (m < rt::BM || kc < rt::BK || kc % 4 != 0 || n % 16 != 0 || n > 128) {
      gemm(false, false, m, n, kc, 1.0f, A, kc, X, n, 0.0f, out, n);
      return;
    }
    rl_transpose_kernel<true><<<dim3(static_cast<unsigned>((n + 31) / 32), static_cast<unsigned>((kc + 31) / 32)),
                                dim3(32, 8), 0, s>>>(X, kc, n, bsplit);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return;
    CUtensorMap ta, tb;
    if (!make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, kc, m, kc * 4, rt::BK, rt::BM,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, bsplit, kc, 2 * n, kc * 4, rt::BK, n,
                      CU_TENSOR_MAP_SWIZZLE_128B)) {
      err = cudaErrorInvalidValue;
      return;
    }
    const int64_t tiles = (m + rt::BM - 1) / rt::BM, stages = (kc + rt::BK - 1) / rt::BK;
    int64_t splits = tiles < num_sms ? num_sms / tiles : 1;  // one CTA per SM: at most one wave
    if (splits > stages / 8) splits = stages / 8;             // slices of at least 8 stages
    if (splits > kRlSplitFloats / (m * n)) splits = kRlSplitFloats / (m * n);
    if (splits < 1) splits = 1;
    const int64_t kss = (stages + splits - 1) / splits;
    splits = (stages + kss - 1) / kss;
    rl_tf32x3_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(splits)), rt::NUM_THREADS,
                       rt::smem_bytes(static_cast<uint32_t>(n)), s>>>(ta, tb, static_cast<uint32_t>(m), static_cast<uint32_t>(n),
                                            static_cast<uint32_t>(kc), static_cast<uint32_t>(kss),
                                            splits > 1 ? split : out);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return;
    if (splits > 1) {
      rl_sgemm_reduce<<<grid(m * n), kRlThreads, 0, s>>>(m, n, static_cast<int>(splits), 1.0f, split, 0.0f, out, n);
      count_launch();
      err = cudaGetLastError();
    }
  }
  // out (cols x rows, pitch rows) = in^T, in rows x cols (pitch cols)
  void transpose(const float* in, int64_t rows, int64_t cols, float* out) {
    if (err != cudaSuccess) return;
    rl_transpose_kernel<false><<<dim3(static_cast<unsigned>((cols + 31) / 32), static_cast<unsigned>((rows + 31) / 32)),
                                 dim3(32, 8), 0, s>>>(in, rows, cols, out);
    count_launch();
    err = cudaGetLastError();
  }
  int grid(int64_t n) const {
    const int64_t b = (n + kRlThreads - 1) / kRlThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<int>(b < 1 ? 1 : (b < cap ? b : cap));
  }
  void to_f32(const void* in, int64_t ld, float* out, int64_t ldo, int64_t rows, int64_t cols) {
    if (err != cudaSuccess) return;
    rl_bf16_to_f32<<<grid(rows * cols), kRlThreads, 0, s>>>(static_cast<const uint16_t*>(in), ld, out, ldo, rows,
                                                            cols);
    count_launch();
    err = cudaGetLastError();
  }
  void to_bf16(const float* in, int64_t ld, void* out, int64_t ldo, int64_t rows, int64_t cols, const float* rs,
               const float* cs, const int* info) {
    if (err != cudaSuccess) return;
    rl_f32_to_bf16<<<grid(rows * cols), kRlThreads, 0, s>>>(in, ld, static_cast<uint16_t*>(out), ldo, rows, cols,
                                                            rs, cs, info);
    count_launch();
    err = cudaGetLastError();
  }
  // A basis of Y's columns (n x sc, pitch sc) by Cholesky-QR, Y^T Y = L L^T and Y <- Y L^-T:
  // two passes (orthonormal to FP32 precision; the result back in Y), or one (a well-conditioned
  // basis of the same span, left in tmp; enough between the products of the subspace iteration,
  // which depend on the span only).  Returns the buffer holding the result.
  float* orth(float* Y, float* tmp, int64_t n, int sc, float* G, float* M, int* info, int stage, int passes) {
    float* src = Y;
    float* dst = tmp;
    for (int pass = 0; pass < passes && err == cudaSuccess; ++pass) {
      gemm(true, false, sc, sc, n, 1.0f, src, sc, src, sc, 0.0f, G, sc);
      if (err != cudaSuccess) return src;
      if ((err = launch_cholesky(sc, G, pass == 0 ? 1e-6f : 0.0f, M, info, 2 * stage + pass, s)) != cudaSuccess)
        return src;
      gemm(false, true, n, sc, sc, 1.0f, src, sc, M, sc, 0.0f, dst, sc);
      float* t = src;
      src = dst;
      dst = t;
    }
    return src;
  }
};

}  // namespace

size_t realign_workspace_floats(int64_t N, int64_t K, int r, int s) {
  return static_cast<size_t>(N * K)                       // W
         + static_cast<size_t>(N * s) + static_cast<size_t>(K * s)  // Y, Z
         + static_cast<size_t>((N > K ? N : K) * s)         // orth() scratch
         + static_cast<size_t>(s * K)                       // B
         + static_cast<size_t>(K * s)                       // Omega
         + 5 * static_cast<size_t>(s) * s + 4 * static_cast<size_t>(s)  // G, M, C, evecs, spare; evals, rs, cs, spare
         + static_cast<size_t>(r * K) + static_cast<size_t>(N * r)      // T1, T2
         + static_cast<size_t>(r * K) + static_cast<size_t>(N * r)      // L1, L2 (FP32)
         + static_cast<size_t>(kRlSplitFloats)                          // split-K partial sums
         + 64 + static_cast<size_t>(N * K)                              // W^T (64: alignment)
         + 64 + 2 * static_cast<size_t>(s) * static_cast<size_t>(N > K ? N : K);  // split small operand
}

cudaError_t launch_lora_realign(const void* W_res, int64_t N, int64_t K, int64_t ldw, const void* L1, const void* L2,
                                int r, float beta, const void* Omega, int s_cols, int q, void* W_res_out,
                                void* L1_out, void* L2_out, int* info, float* ws, int num_sms, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  static std::atomic<int> attr_done{0};
  if (!attr_done.load()) {
    const int jac = (2 * kRlMaxS * (kRlMaxS + 1) + 2 * kRlMaxS) * 4;
    if ((e = cudaFuncSetAttribute(rl_jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, jac))) return e;
    if ((e = cudaFuncSetAttribute(rl_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, rt::SMEM_MAX)))
      return e;
    attr_done.store(1);
  }
  const int sc = s_cols;
  float* W = ws;
  float* Y = W + N * K;
  float* Z = Y + N * sc;
  float* T = Z + K * sc;  // orth() scratch
  float* B = T + (N > K ? N : K) * sc;
  float* Om = B + static_cast<int64_t>(sc) * K;
  float* G = Om + K * sc;
  float* L = G + sc * sc;
  float* C = L + sc * sc;
  float* Ub = C + sc * sc;
  float* evals = Ub + 2 * sc * sc;  // one spare s x s block before the vectors
  float* rs = evals + sc;
  float* cs = rs + sc;
  float* T1 = cs + 2 * sc;
  float* T2 = T1 + static_cast<int64_t>(r) * K;
  float* L1f = T2 + N * r;
  float* L2f = L1f + static_cast<int64_t>(r) * K;
  float* split = L2f + N * r;
  const auto aligned = [](float* p) {  // 256-byte aligned (TMA wants 16)
    return reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(p) + 255) & ~uintptr_t(255));
  };
  float* Wt = aligned(split + kRlSplitFloats);  // K x N
  float* Bs = aligned(Wt + N * K);             // 2 sc x max(N, K)

  if ((e = cudaMemsetAsync(info, 0, sizeof(int), st)) != cudaSuccess) return e;
  pdl_chain_break();
  Rl rl{st, num_sms, split};
  // W = W_res + beta L2 L1 (FP32)
  rl.to_f32(W_res, ldw, W, K, N, K);
  rl.to_f32(L1, K, L1f, K, r, K);
  rl.to_f32(L2, r, L2f, r, N, r);
  rl.gemm(false, false, N, K, r, beta, L2f, r, L1f, K, 1.0f, W, K);
  rl.transpose(W, N, K, Wt);
  // range finder with q power iterations (the products with W and W^T on the tensor cores)
  rl.to_f32(Omega, sc, Om, sc, K, sc);
  rl.tc(W, N, K, Om, sc, Bs, Y);
  for (int it = 0; it < q; ++it) {
    const float* Yb = rl.orth(Y, T, N, sc, G, L, info, 2 * it, 1);
    rl.tc(Wt, K, N, Yb, sc, Bs, Z);
    const float* Zb = rl.orth(Z, T, K, sc, G, L, info, 2 * it + 1, 1);
    rl.tc(W, N, K, Zb, sc, Bs, Y);
  }
  rl.orth(Y, T, N, sc, G, L, info, 2 * q, 2);  // the final basis, orthonormal, back in Y
  // B^T = W^T Q (K x sc, in B's place), C = B B^T = Ub Lambda Ub^T
  rl.tc(Wt, K, N, Y, sc, Bs, B);
  rl.gemm(true, false, sc, sc, K, 1.0f, B, sc, B, sc, 0.0f, C, sc);
  if (rl.err != cudaSuccess) return rl.err;
  {
    const size_t smem = (2 * static_cast<size_t>(sc) * (sc + 1) + 2 * sc) * sizeof(float);
    rl_jacobi_kernel<<<1, kRlJacThreads, smem, st>>>(C, sc, 15, evals, Ub, info);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // T1 = Ub_r^T B (r x K), T2 = Q Ub_r (N x r); signs and scales; BF16 factors
  rl.gemm(true, true, r, K, sc, 1.0f, Ub, sc, B, sc, 0.0f, T1, K);
  rl.gemm(false, false, N, r, sc, 1.0f, Y, sc, Ub, sc, 0.0f, T2, r);
  if (rl.err != cudaSuccess) return rl.err;
  rl_sign_scale_kernel<<<r, kRlThreads, 0, st>>>(T1, K, evals, beta, rs, cs, info);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  rl.to_bf16(T1, K, L1_out, K, r, K, rs, nullptr, info);
  rl.to_bf16(T2, r, L2_out, r, N, r, nullptr, cs, info);
  // W_res = bf16(W - beta bf16(L2) bf16(L1))
  rl.to_f32(L1_out, K, L1f, K, r, K);
  rl.to_f32(L2_out, r, L2f, r, N, r);
  rl.gemm(false, false, N, K, r, -beta, L2f, r, L1f, K, 1.0f, W, K);
  rl.to_bf16(W, K, W_res_out, ldw, N, K, nullptr, nullptr, info);
  return rl.err;
}

}  // namespace nvfp4
