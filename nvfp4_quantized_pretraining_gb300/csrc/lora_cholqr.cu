// Cholesky-QR step of the LoRA-SVD branch ("Full-Stack FP4", section 2.1: the
// backward pass is restricted to the subspace under a Cholesky-QR constraint).
// Reading: the rows of L1 (r x K) are re-orthonormalised through the Cholesky
// factor of their Gram matrix, L1 L1^T = L L^T, L1 <- L^-1 L1, and L2 (N x r)
// takes the factor, L2 <- L2 L, so beta L2 L1 is unchanged.
//
// Three launches, FP32 arithmetic (the BF16 products are exact in FP32):
//   1. Gram partials: CTA s (of at most 32) sums the 128-column chunks s, s + 32,
//      ... of L1 into an r x r FP32 partial;
//   2. one CTA adds the partials in a fixed order, factors G = L L^T
//      (right-looking, lower triangle) and reports a non-positive pivot in *info
//      (LAPACK convention: the order of the failing leading minor);
//   3. the update: one thread per column of L1 (forward substitution with L)
//      and one per row of L2 (the row times L), BF16 results; nothing is written
//      when *info != 0.  Each thread reads its whole column or row before writing
//      it, so the update may be in place.
#include "bf16_convert.cuh"
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kCqrChunk = 128;   // columns of L1 per Gram step
constexpr int kCqrMaxParts = 32; // Gram CTAs (partials)
constexpr int kCqrThreads = 256;

// r x r partial Gram matrix of the 128-column chunks blockIdx.x, blockIdx.x + gridDim.x, ...
// Thread t owns row i = t / 4 and columns j = t % 4 + 4 u (u < r / 4) of the partial.
template <int R>
__global__ void __launch_bounds__(kCqrThreads) cholqr_gram_kernel(const uint16_t* L1, int64_t K,
                                                                  int64_t ld, float* partial) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[R][kCqrChunk + 1];
  constexpr int kCols = R / 4;
  const int i = threadIdx.x / 4, j0 = threadIdx.x % 4;
  float acc[kCols];
#pragma unroll
  for (int u = 0; u < kCols; ++u) acc[u] = 0.0f;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kCqrChunk;
  for (int64_t k0 = static_cast<int64_t>(blockIdx.x) * kCqrChunk; k0 < K; k0 += step) {
    __syncthreads();  // the previous chunk's reads are done
    // a fixed trip count, unrolled: every load of the chunk is in flight before the first store
    static_assert(R * kCqrChunk % kCqrThreads == 0, "whole loads per thread");
    uint16_t v[R * kCqrChunk / kCqrThreads];
#pragma unroll
    for (int u = 0; u < R * kCqrChunk / kCqrThreads; ++u) {
      const int e = threadIdx.x + u * kCqrThreads;
      const int64_t k = k0 + e % kCqrChunk;
      v[u] = k < K ? L1[(e / kCqrChunk) * ld + k] : static_cast<uint16_t>(0);
    }
#pragma unroll
    for (int u = 0; u < R * kCqrChunk / kCqrThreads; ++u) {
      const int e = threadIdx.x + u * kCqrThreads;
      tile[e / kCqrChunk][e % kCqrChunk] = __uint_as_float(static_cast<uint32_t>(v[u]) << 16);
    }
    __syncthreads();
    if (i < R) {
      for (int k = 0; k < kCqrChunk; ++k) {
        const float a = tile[i][k];
#pragma unroll
        for (int u = 0; u < kCols; ++u) acc[u] = fmaf(a, tile[j0 + 4 * u][k], acc[u]);
      }
    }
  }
  if (i < R) {
    float* out = partial + static_cast<int64_t>(blockIdx.x) * R * R + i * R;
#pragma unroll
    for (int u = 0; u < kCols; ++u) out[j0 + 4 * u] = acc[u];
  }
}

// One CTA of 256 threads: G = sum of the partials (fixed order), G = L L^T (right-looking).  The
// threads hold G as a 16 x 16 grid of (R/16) x (R/16) register blocks (thread (ty, tx) has rows
// ty + 16a and columns tx + 16b).  Step j: the owners of column j publish it in shared memory,
// one barrier, then every thread reads the pivot d_j, scales the column, l_i = G_ij (1 / sqrt(d_j)),
// and updates its own trailing elements, G_ik -= l_i l_k (k <= i).  A non-positive pivot is seen
// by every thread at once.  Writes L (lower, zeros above) and the reciprocals of its diagonal.
template <int R>
__global__ void __launch_bounds__(kCqrThreads) cholqr_factor_kernel(const float* partial, int nparts,
                                                                    float* Lout, float* inv_diag,
                                                                    int* info) {
  constexpr int B = R / 16;
  __shared__ float col[2][R];
  __shared__ float piv[R];
  pdl_trigger();
  pdl_wait();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float g[B][B];
#pragma unroll
  for (int a = 0; a < B; ++a)
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int e = (ty + 16 * a) * R + tx + 16 * b;
      float v[kCqrMaxParts];
#pragma unroll
      for (int p = 0; p < kCqrMaxParts; ++p) v[p] = p < nparts ? partial[p * R * R + e] : 0.0f;
      float s = 0.0f;
#pragma unroll
      for (int p = 0; p < kCqrMaxParts; ++p) s += v[p];
      g[a][b] = s;
    }
  int bad = 0;
#pragma unroll
  for (int bj = 0; bj < B; ++bj) {
    for (int jj = 0; jj < 16 && !bad; ++jj) {
      const int j = 16 * bj + jj;
      float* cj = col[j & 1];
      if (tx == jj) {  // the owners of column j publish rows j.. of it
#pragma unroll
        for (int a = 0; a < B; ++a)
          if (ty + 16 * a >= j) cj[ty + 16 * a] = g[a][bj];
      }
      __syncthreads();  // column j visible; every read of column j - 2's buffer is done
      const float d = cj[j];  // the same pivot for every thread: the test is uniform
      if (!(d > 0.0f)) {
        bad = j + 1;
        break;
      }
      if (threadIdx.x == 0) piv[j] = d;
      const float rdjj = 1.0f / sqrtf(d);  // one reciprocal per column; the column is scaled by it
      float li[B], lk[B];
#pragma unroll
      for (int a = 0; a < B; ++a) li[a] = ty + 16 * a > j ? cj[ty + 16 * a] * rdjj : 0.0f;
#pragma unroll
      for (int b = 0; b < B; ++b) lk[b] = tx + 16 * b > j ? cj[tx + 16 * b] * rdjj : 0.0f;
#pragma unroll
      for (int a = 0; a < B; ++a)
#pragma unroll
        for (int b = 0; b < B; ++b)
          if (tx + 16 * b > j && tx + 16 * b <= ty + 16 * a) g[a][b] = fmaf(-li[a], lk[b], g[a][b]);
    }
  }
  if (threadIdx.x == 0) *info = bad;
  if (bad) return;  // uniform
  __syncthreads();  // every pivot written
#pragma unroll
  for (int a = 0; a < B; ++a)
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int i = ty + 16 * a, k = tx + 16 * b;
      Lout[i * R + k] = k < i ? g[a][b] * (1.0f / sqrtf(piv[k])) : k == i ? sqrtf(piv[k]) : 0.0f;
    }
  if (threadIdx.x < R) inv_diag[threadIdx.x] = 1.0f / sqrtf(piv[threadIdx.x]);
}


// Blocks [0, ncolblocks): columns of L1 (L1' = L^-1 L1 by forward substitution, right-looking:
// once x_i is known every later row takes its term, in the same order per row as the
// left-looking sum); the rest: rows of L2 (L2' = L2 L, y_j = sum_{i >= j} x_i L_ij with the
// terms added in increasing i).  Both run a runtime loop over the R steps with the per-thread
// values in registers that shift down by one each step (so every register index is a
// compile-time one and the loop body stays small: a fully unrolled triangle of R^2 / 2
// multiply-adds outgrew the instruction cache), reading each step's coefficients from a
// zero-padded shared-memory row, 16 bytes at a time.
constexpr int kCqrApplyThreads = 128;

template <int R>
__global__ void __launch_bounds__(kCqrApplyThreads) cholqr_apply_kernel(
    const uint16_t* L1, int64_t K, int64_t ld1, uint16_t* L1_out, const uint16_t* L2, int64_t N, uint16_t* L2_out,
    const float* Lmat, const float* inv_diag, const int* info, int ncolblocks) {
  constexpr int ldl = R + 4;
  __shared__ __align__(16) float LS[R][ldl];   // LS[i][t] = L_{i+1+t, i} (below the diagonal), 0 past R - 2 - i
  __shared__ __align__(16) float LR[R][ldl];   // LR[i][j] = L_ij, 0 above the diagonal
  __shared__ float dinv[R];
  pdl_trigger();
  pdl_wait();
  if (*info != 0) return;
  for (int e = threadIdx.x; e < R * ldl; e += blockDim.x) {
    (&LS[0][0])[e] = 0.0f;
    (&LR[0][0])[e] = 0.0f;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < R * R; e += blockDim.x) {
    const int i = e / R, k = e % R;
    if (k <= i) {
      const float v = Lmat[e];
      LR[i][k] = v;
      if (k < i) LS[k][i - k - 1] = v;
    }
  }
  if (threadIdx.x < R) dinv[threadIdx.x] = inv_diag[threadIdx.x];
  __syncthreads();
  if (static_cast<int>(blockIdx.x) < ncolblocks) {
    const int64_t k = static_cast<int64_t>(blockIdx.x) * kCqrApplyThreads + threadIdx.x;
    if (k >= K) return;
    // r[t]: the partial sum of row i + t at step i
    float r[R];
#pragma unroll
    for (int c = 0; c < R; ++c) r[c] = __uint_as_float(static_cast<uint32_t>(L1[c * ld1 + k]) << 16);
    for (int i = 0; i < R; ++i) {
      const float x = r[0] * dinv[i];
      L1_out[i * ld1 + k] = static_cast<uint16_t>(bf16_rn_bits(x));
      const float4* row = reinterpret_cast<const float4*>(&LS[i][0]);
#pragma unroll
      for (int q = 0; q < R / 4; ++q) {
        const float4 l = row[q];
        r[4 * q] = fmaf(-l.x, x, r[4 * q + 1]);
        r[4 * q + 1] = fmaf(-l.y, x, r[4 * q + 2]);
        r[4 * q + 2] = fmaf(-l.z, x, r[4 * q + 3]);
        if (4 * q + 4 < R) r[4 * q + 3] = fmaf(-l.w, x, r[4 * q + 4]);
      }
    }
  } else {
    const int64_t n = static_cast<int64_t>(blockIdx.x - ncolblocks) * kCqrApplyThreads + threadIdx.x;
    if (n >= N) return;
    // xr[t] = x_{i + t} at step i
    float xr[R];
    const uint4* src = reinterpret_cast<const uint4*>(L2 + n * R);
#pragma unroll
    for (int q = 0; q < R / 8; ++q) {
      const uint4 w = src[q];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        xr[8 * q + 2 * h] = __uint_as_float(ws[h] << 16);
        xr[8 * q + 2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
      }
    }
    float y[R];
#pragma unroll
    for (int j = 0; j < R; ++j) y[j] = 0.0f;
    for (int i = 0; i < R; ++i) {
      const float xi = xr[0];
      const float4* row = reinterpret_cast<const float4*>(&LR[i][0]);
      // L_ij = 0 for j > i: those y_j stay +0 until their first term (i = j)
#pragma unroll
      for (int q = 0; q < R / 4; ++q) {
        const float4 l = row[q];
        y[4 * q] = fmaf(xi, l.x, y[4 * q]);
        y[4 * q + 1] = fmaf(xi, l.y, y[4 * q + 1]);
        y[4 * q + 2] = fmaf(xi, l.z, y[4 * q + 2]);
        y[4 * q + 3] = fmaf(xi, l.w, y[4 * q + 3]);
      }
#pragma unroll
      for (int t = 0; t + 1 < R; ++t) xr[t] = xr[t + 1];
    }
    uint4* out = reinterpret_cast<uint4*>(L2_out + n * R);
#pragma unroll
    for (int q = 0; q < R / 8; ++q) {
      uint32_t packed[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) packed[h] = bf16_rn_bits(y[8 * q + 2 * h]) | (bf16_rn_bits(y[8 * q + 2 * h + 1]) << 16);
      out[q] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
  }
}

int cholqr_parts(int64_t K) {
  const int64_t chunks = (K + kCqrChunk - 1) / kCqrChunk;
  return static_cast<int>(chunks < kCqrMaxParts ? chunks : kCqrMaxParts);
}

template <int R>
static cudaError_t cholqr_launch(const void* L1, int64_t K, int64_t ld1, const void* L2, int64_t N, void* L1_out,
                                 void* L2_out, int* info, float* ws, cudaStream_t s) {
  const int parts = cholqr_parts(K);
  float* partial = ws;
  float* Lmat = ws + static_cast<int64_t>(parts) * R * R;
  float* inv_diag = Lmat + R * R;
  // programmatic dependent launches: each kernel's set-up overlaps the previous one's tail, and
  // each waits (griddepcontrol.wait) before its first global read
  cudaError_t e = launch_pdl(cholqr_gram_kernel<R>, dim3(parts), dim3(kCqrThreads), 0, s,
                             static_cast<const uint16_t*>(L1), K, ld1, partial);
  count_launch();
  if (e != cudaSuccess) return e;
  e = launch_pdl(cholqr_factor_kernel<R>, dim3(1), dim3(kCqrThreads), 0, s, static_cast<const float*>(partial), parts,
                 Lmat, inv_diag, info);
  count_launch();
  if (e != cudaSuccess) return e;
  const int colblocks = static_cast<int>((K + kCqrApplyThreads - 1) / kCqrApplyThreads);
  const int rowblocks = static_cast<int>((N + kCqrApplyThreads - 1) / kCqrApplyThreads);
  e = launch_pdl(cholqr_apply_kernel<R>, dim3(colblocks + rowblocks), dim3(kCqrApplyThreads), 0, s,
                 static_cast<const uint16_t*>(L1), K, ld1, static_cast<uint16_t*>(L1_out),
                 static_cast<const uint16_t*>(L2), N, static_cast<uint16_t*>(L2_out), static_cast<const float*>(Lmat),
                 static_cast<const float*>(inv_diag), static_cast<const int*>(info), colblocks);
  count_launch();
  return e;
}

cudaError_t launch_lora_cholqr(const void* L1, int64_t K, int64_t ld1, const void* L2, int64_t N, int r,
                               void* L1_out, void* L2_out, int* info, float* ws, cudaStream_t s) {
  switch (r) {
    case 16: return cholqr_launch<16>(L1, K, ld1, L2, N, L1_out, L2_out, info, ws, s);
    case 32: return cholqr_launch<32>(L1, K, ld1, L2, N, L1_out, L2_out, info, ws, s);
    case 48: return cholqr_launch<48>(L1, K, ld1, L2, N, L1_out, L2_out, info, ws, s);
    case 64: return cholqr_launch<64>(L1, K, ld1, L2, N, L1_out, L2_out, info, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4
