// Periodic realignment of the LoRA-SVD subspace by a randomized SVD ("Full-Stack
// FP4", section 2.1, Realignment: the subspace is reset with a randomized SVD so
// that the BF16 branch stays optimal).  The method is the randomized subspace
// iteration and direct SVD of Halko, Martinsson and Tropp (SIAM Review 2011,
// Algorithms 4.4 and 5.1) on W = W_res + beta L2 L1:
//   Y = W Omega;  q times: Y = W basis(W^T basis(Y));  Q = orth(Y);  B = Q^T W;
//   B B^T = Ub Lambda Ub^T (Jacobi);  L2 = Q Ub_r Sigma_r / beta;  L1 = Ub_r^T B / Sigma_r;
//   W_res = W - beta bf16(L2) bf16(L1).
// FP32 throughout.  The plain products run in this file's own tiled FP32 GEMM
// (rl_sgemm_kernel: 64 x 64 output tiles, split over K into a fixed-order sum
// when the output has few tiles); orth() is Cholesky-QR (the factor and its
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
// Cholesky of an S x S Gram matrix (S <= 128, a multiple of 16) in one CTA, and
// the inverse of the factor: G + shift * mean(diag) I = L L^T (right-looking on
// the unscaled columns, one barrier per column: with d_j the pivot,
// G_ik -= G_ij G_kj / d_j, and L_ij = G_ij / sqrt(d_j) at the end), then
// M = L^-1 with thread c holding column c in registers: x_i = (delta_ic -
// sum_{k < i} L_ik x_k) / L_ii, every lane reading the same L_ik (a shared-memory
// broadcast).  Writes M (lower, row-major S x S); a non-positive pivot sets *info
// (if still 0) to 1000 * stage + its order.
// ---------------------------------------------------------------------------
constexpr int kRlCholThreads = 256;

template <int S>
__global__ void __launch_bounds__(kRlCholThreads) rl_cholesky_kernel(const float* __restrict__ Gin, float shift,
                                                                     float* __restrict__ Mout, int* __restrict__ info,
                                                                     int stage) {
  constexpr int ld = S + 1;
  extern __shared__ float G[];  // S x ld: G, then L
  __shared__ float mean_diag;
  for (int e = threadIdx.x; e < S * S; e += blockDim.x) G[(e / S) * ld + e % S] = Gin[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int i = 0; i < S; ++i) t += G[i * ld + i];
    mean_diag = t / S;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < S; i += blockDim.x) G[i * ld + i] += shift * mean_diag;
  __syncthreads();
  int bad = 0;
  for (int j = 0; j < S; ++j) {
    const float d = G[j * ld + j];  // every thread reads the same pivot: the test is uniform
    if (!(d > 0.0f)) {
      bad = j + 1;
      break;
    }
    const float inv = 1.0f / d;
    // lower triangle of the trailing block: warp w takes rows j + 1 + w, j + 1 + w + 8, ...
    for (int i = j + 1 + (threadIdx.x >> 5); i < S; i += blockDim.x >> 5) {
      const float gij = G[i * ld + j] * inv;
      for (int k = j + 1 + (threadIdx.x & 31); k <= i; k += 32) G[i * ld + k] -= gij * G[k * ld + j];
    }
    __syncthreads();
  }
  if (bad) {
    if (threadIdx.x == 0) atomicCAS(info, 0, 1000 * stage + bad);
    return;
  }
  for (int e = threadIdx.x; e < S * S; e += blockDim.x) {
    const int i = e / S, k = e % S;
    if (k < i) G[i * ld + k] *= rsqrtf(G[k * ld + k]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < S; i += blockDim.x) G[i * ld + i] = sqrtf(G[i * ld + i]);
  __syncthreads();
  if (threadIdx.x < S) {
    const int c = threadIdx.x;
    float x[S];
#pragma unroll
    for (int i = 0; i < S; ++i) {
      float acc = i == c ? 1.0f : 0.0f;
#pragma unroll
      for (int k = 0; k < i; ++k) acc = fmaf(-G[i * ld + k], x[k], acc);  // x_k = 0 for k < c
      x[i] = i < c ? 0.0f : acc / G[i * ld + i];
    }
#pragma unroll
    for (int i = 0; i < S; ++i) Mout[i * S + c] = x[i];
  }
}

template <int S>
static cudaError_t cholesky_launch(const float* G, float shift, float* M, int* info, int stage, cudaStream_t st) {
  const int smem = S * (S + 1) * static_cast<int>(sizeof(float));
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
// as disjoint 2 x 2 blocks (rows of pair k, columns of pair l) and V <- V J.  A
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
  float* V = sh + s * ld;     // s x ld (2 s ld floats: a multiple of 8 bytes)
  float2* CSN = reinterpret_cast<float2*>(V + s * ld);  // s / 2 (cosine, sine) pairs
  int2* PQ = reinterpret_cast<int2*>(CSN + s / 2);      // s / 2 (head, tail) pairs
  __shared__ int rotated;
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
  // This thread's share of each round's update, the same in every round: 2 x 2 blocks (k, l) of A
  // and entries (pair l, row i) of V, packed as k | l << 8 and l | i << 8 (s <= 128), computed once
  // here rather than by a division per item and round.
  constexpr int kItA = (kRlMaxS / 2) * (kRlMaxS / 2) / kRlJacThreads;
  constexpr int kItV = (kRlMaxS / 2) * kRlMaxS / kRlJacThreads;
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  uint32_t it_a[kItA], it_v[kItV];
#pragma unroll
  for (int j = 0; j < kItA; ++j) {
    const int e = threadIdx.x + j * kRlJacThreads;
    it_a[j] = e < half * half ? (uint32_t)(e / half) | ((uint32_t)(e % half) << 8) : kNone;
  }
#pragma unroll
  for (int j = 0; j < kItV; ++j) {
    const int f = threadIdx.x + j * kRlJacThreads;
    it_v[j] = f < half * s ? (uint32_t)(f / s) | ((uint32_t)(f % s) << 8) : kNone;
  }
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    if (threadIdx.x == 0) rotated = 0;
    __syncthreads();
    for (int round = 0; round < s - 1; ++round) {
      for (int k = threadIdx.x; k < half; k += blockDim.x) {
        const int p = k == 0 ? s - 1 : (round + k) % (s - 1);
        const int q = k == 0 ? round : (round - k + (s - 1)) % (s - 1);
        const float apq = A[p * ld + q], app = A[p * ld + p], aqq = A[q * ld + q];
        float c = 1.0f, t = 0.0f;
        if (fabsf(apq) > thresh) {
          const float tau = (aqq - app) / (2.0f * apq);
          t = (tau >= 0.0f ? 1.0f : -1.0f) / (fabsf(tau) + sqrtf(1.0f + tau * tau));
          c = rsqrtf(1.0f + t * t);
          rotated = 1;
        }
        PQ[k] = make_int2(p, q);
        CSN[k] = make_float2(c, t * c);
      }
      __syncthreads();
      // A <- J^T A J as 2 x 2 blocks; V <- V J
#pragma unroll
      for (int j = 0; j < kItA; ++j) {
        if (it_a[j] == kNone) continue;
        const int k = it_a[j] & 0xFFu, l = it_a[j] >> 8;
        const int2 qk2 = PQ[k], ql2 = PQ[l];
        const float2 rk = CSN[k], rl = CSN[l];
        const int pk = qk2.x, qk = qk2.y, pl = ql2.x, ql = ql2.y;
        const float ck = rk.x, sk = rk.y, cl = rl.x, sl = rl.y;
        const float xpp = A[pk * ld + pl], xpq = A[pk * ld + ql], xqp = A[qk * ld + pl], xqq = A[qk * ld + ql];
        const float rpp = ck * xpp - sk * xqp, rpq = ck * xpq - sk * xqq;  // rows of pair k
        const float rqp = sk * xpp + ck * xqp, rqq = sk * xpq + ck * xqq;
        A[pk * ld + pl] = cl * rpp - sl * rpq;  // columns of pair l
        A[pk * ld + ql] = sl * rpp + cl * rpq;
        A[qk * ld + pl] = cl * rqp - sl * rqq;
        A[qk * ld + ql] = sl * rqp + cl * rqq;
      }
#pragma unroll
      for (int j = 0; j < kItV; ++j) {
        if (it_v[j] == kNone) continue;
        const int l = it_v[j] & 0xFFu, i = it_v[j] >> 8;
        const int2 ql2 = PQ[l];
        const float2 rl = CSN[l];
        const int pl = ql2.x, ql = ql2.y;
        const float cl = rl.x, sl = rl.y;
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
  int* order = reinterpret_cast<int*>(PQ);  // reuse: s entries fit in the s / 2 int2
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
  // of fewer tiles than two per SM is split over K (slices of at least 512) into the scratch, as
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
      const int64_t by_k = (k + 511) / 512;
      if (splits > by_k) splits = by_k;
      const int64_t by_ws = kRlSplitFloats / (m * n);
      if (splits > by_ws) splits = by_ws;
      if (splits > 64) splits = 64;
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
         + static_cast<size_t>(kRlSplitFloats);                         // split-K partial sums
}

cudaError_t launch_lora_realign(const void* W_res, int64_t N, int64_t K, int64_t ldw, const void* L1, const void* L2,
                                int r, float beta, const void* Omega, int s_cols, int q, void* W_res_out,
                                void* L1_out, void* L2_out, int* info, float* ws, int num_sms, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  static std::atomic<int> attr_done{0};
  if (!attr_done.load()) {
    const int jac = (2 * kRlMaxS * (kRlMaxS + 1) + 2 * kRlMaxS) * 4;
    if ((e = cudaFuncSetAttribute(rl_jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, jac))) return e;
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

  if ((e = cudaMemsetAsync(info, 0, sizeof(int), st)) != cudaSuccess) return e;
  Rl rl{st, num_sms, split};
  // W = W_res + beta L2 L1 (FP32)
  rl.to_f32(W_res, ldw, W, K, N, K);
  rl.to_f32(L1, K, L1f, K, r, K);
  rl.to_f32(L2, r, L2f, r, N, r);
  rl.gemm(false, false, N, K, r, beta, L2f, r, L1f, K, 1.0f, W, K);
  // range finder with q power iterations
  rl.to_f32(Omega, sc, Om, sc, K, sc);
  rl.gemm(false, false, N, sc, K, 1.0f, W, K, Om, sc, 0.0f, Y, sc);
  for (int it = 0; it < q; ++it) {
    const float* Yb = rl.orth(Y, T, N, sc, G, L, info, 2 * it, 1);
    rl.gemm(true, false, K, sc, N, 1.0f, W, K, Yb, sc, 0.0f, Z, sc);
    const float* Zb = rl.orth(Z, T, K, sc, G, L, info, 2 * it + 1, 1);
    rl.gemm(false, false, N, sc, K, 1.0f, W, K, Zb, sc, 0.0f, Y, sc);
  }
  rl.orth(Y, T, N, sc, G, L, info, 2 * q, 2);  // the final basis, orthonormal, back in Y
  // B = Q^T W, C = B B^T = Ub Lambda Ub^T
  rl.gemm(true, false, sc, K, N, 1.0f, Y, sc, W, K, 0.0f, B, K);
  rl.gemm(false, true, sc, sc, K, 1.0f, B, K, B, K, 0.0f, C, sc);
  if (rl.err != cudaSuccess) return rl.err;
  {
    const size_t smem = (2 * static_cast<size_t>(sc) * (sc + 1) + 2 * sc) * sizeof(float);
    rl_jacobi_kernel<<<1, kRlJacThreads, smem, st>>>(C, sc, 15, evals, Ub, info);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // T1 = Ub_r^T B (r x K), T2 = Q Ub_r (N x r); signs and scales; BF16 factors
  rl.gemm(true, false, r, K, sc, 1.0f, Ub, sc, B, K, 0.0f, T1, K);
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
