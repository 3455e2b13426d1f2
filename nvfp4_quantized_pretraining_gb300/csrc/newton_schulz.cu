// Elementwise kernels of the Q-Root Newton-Schulz iteration with NVFP4 products
// ("Full-Stack FP4", section 2.3, NVFP4 Root optimizer).  The three products of a
// step run through the quantizer and the block-scaled GEMM; what remains is HBM-bound
// elementwise work, done here:
//   - X_0 = bf16(G / ||G||_F): a sum of squares (fixed-order reduction), then the
//     scaled copy, which also histograms |X_0| for the first clip;
//   - the p99 clip: the k-th smallest |x| of the iterate read off a 32768-bin
//     histogram of the BF16 magnitude patterns (integer, exact); the clip itself
//     is applied by the iterate's two readers (the quantizer as it stages a
//     tile, and the step's final linear combination), so the iterate is never
//     rewritten;
//   - the linear combinations out = bf16(fl32(p x) + fl32(q y)), fused either with
//     the amax of the output (for its quantization) or with the histogram of the
//     output (the next step's clip).
// All kernels are grid-stride loops over 16-byte chunks (8 BF16) of row-major
// matrices with a row pitch; the grid is sized in multiples of the SM count.
#include "bf16_convert.cuh"
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kNsThreads = 512;
constexpr int kNsHistThreads = 1024;  // kernels with a 128 KB shared histogram: one CTA per SM
constexpr int kHistBins = kNsHistBins;  // one bin per BF16 magnitude pattern (sign cleared)
constexpr size_t kHistSmem = kHistBins * sizeof(uint32_t);

__device__ __forceinline__ const uint16_t* chunk_ptr(const uint16_t* base, uint32_t c, uint32_t cpr, int64_t ld) {
  const uint32_t row = c / cpr;
  return base + static_cast<int64_t>(row) * ld + static_cast<int64_t>(c - row * cpr) * 8;
}


// Round a double to the nearest BF16 pattern, ties to even, directly (rounding to
// binary32 first would round twice).  Normal range: keep the top 7 of the 52
// fraction bits with round-half-even on the integer pattern, then rebias the
// exponent (1023 -> 127); a carry out of the fraction steps the exponent, up to
// the infinity pattern.  Below 2^-126 the BF16 spacing is 2^-133, so the pattern
// is the value in units of 2^-133 rounded half-even (128 is the smallest normal's
// pattern, so the carry is right there too).
__device__ __forceinline__ uint32_t bf16_from_f64_rn(double v) {
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(v));
  const uint32_t sign = static_cast<uint32_t>(bits >> 48) & 0x8000u;
  const uint64_t u = bits & 0x7FFFFFFFFFFFFFFFull;
  if (u > 0x7FF0000000000000ull) return 0x7FC0u;               // NaN
  const double a = __longlong_as_double(static_cast<long long>(u));
  if (a >= 0x1.FEp127) return sign | 0x7F80u;                 // rounds to infinity
  if (a < 0x1p-126) return sign | static_cast<uint32_t>(rint(a * 0x1p133));
  const uint64_t r = (u + 0xFFFFFFFFFFFull + ((u >> 45) & 1u)) >> 45;  // 11-bit exponent : 7-bit fraction
  return sign | static_cast<uint32_t>(r - (uint64_t(896) << 7));
}

// The exact FP64 value of a BF16 pattern.
__device__ __forceinline__ double bf16_to_f64(uint32_t h) { return static_cast<double>(__uint_as_float(h << 16)); }

// bf16(g * inv) for a BF16 g and inv = 1 / ||G||, rounded as the FP64 quotient
// would be.  p = fl32(g * inv32) is within 2 binary32 ulps of the FP64 quotient
// (inv32 and the product each round once), so the BF16 rounding of p is that of
// the quotient unless p lies within 4 ulps of a BF16 midpoint (low 16 bits near
// 0x8000) or is tiny; those elements, and all of them when inv32 itself is tiny
// (`wide`), are recomputed in FP64.
__device__ __forceinline__ uint32_t scaled_bf16(uint32_t h, float inv32, double inv64, bool wide) {
  const float p = __fmul_rn(__uint_as_float(h << 16), inv32);
  const uint32_t pb = __float_as_uint(p);
  const uint32_t low = pb & 0xFFFFu;
  const bool near_mid = (low > 0x8000u - 5u) && (low < 0x8000u + 5u);
  const bool tiny = (pb & 0x7F800000u) < (27u << 23) && (pb & 0x7FFFFFFFu) != 0;  // |p| < 2^-100
  if (near_mid || tiny || wide) return bf16_from_f64_rn(bf16_to_f64(h) * inv64);
  return bf16_rn_bits(p);
}

// ---------------------------------------------------------------------------
// Histogram helpers: a 32768-bin shared histogram per CTA, flushed into the
// global histogram with one atomic add per non-empty bin.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void hist_zero(uint32_t* sh) {
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
}
__device__ __forceinline__ void hist_add8(uint32_t* sh, const uint32_t (&w)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    atomicAdd(&sh[w[j] & 0x7FFFu], 1u);
    atomicAdd(&sh[(w[j] >> 16) & 0x7FFFu], 1u);
  }
}
__device__ __forceinline__ void hist_flush(const uint32_t* sh, uint32_t* __restrict__ hist) {
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    const uint32_t h = sh[i];
    if (h) atomicAdd(&hist[i], h);
  }
}

// ---------------------------------------------------------------------------
// Sum of squares of a BF16 matrix.  For 2^-50 <= |g| < 2^50 the square is exact
// in binary32 (8-bit significands) and far from its range limits, so every
// thread sums those with a compensated (two-sum) binary32 pair; the rare larger
// or smaller magnitudes go to an FP64 accumulator.  The per-thread sums are
// combined in FP64 in a fixed order: one FP64 partial per CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kNsThreads) ns_sumsq_kernel(const uint16_t* __restrict__ g, uint32_t cpr,
                                                              uint32_t nchunks, int64_t ld,
                                                              double* __restrict__ partial) {
  float s = 0.f, comp = 0.f;
  double wide = 0.0;
  for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < nchunks; c += gridDim.x * blockDim.x) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(chunk_ptr(g, c, cpr, ld)));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float f = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
      const uint32_t e = __float_as_uint(f) & 0x7F800000u;
      if (e < (77u << 23) || e >= (177u << 23)) {  // |f| < 2^-50 or >= 2^50 (zeros add nothing)
        if (e != 0 || (__float_as_uint(f) & 0x7FFFFFu) != 0) wide = fma(static_cast<double>(f), static_cast<double>(f), wide);
        continue;
      }
      const float x = __fmul_rn(f, f);
      const float t = __fadd_rn(s, x);
      const float bp = __fsub_rn(t, s);
      const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(x, bp));
      s = t;
      comp = __fadd_rn(comp, err);
    }
  }
  double d = (static_cast<double>(s) + static_cast<double>(comp)) + wide;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
  __shared__ double red[kNsThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = d;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < kNsThreads / 32; ++w) t += red[w];
    partial[blockIdx.x] = t;
  }
}

// The total of the partials in a fixed order (every CTA computes the same value).
__device__ __forceinline__ double sum_partials(const double* __restrict__ partial, int n) {
  __shared__ double total;
  if (threadIdx.x < 32) {
    double t = 0.0;
    for (int i = threadIdx.x; i < n; i += 32) t += partial[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (threadIdx.x == 0) total = t;
  }
  __syncthreads();
  return total;
}

// X = bf16(G / max(||G||_F, 1e-7)); HIST: also histogram |X| into `hist`.
// G and X may be the same matrix (each element is read, then written, by one thread).
template <bool HIST>
__global__ void __launch_bounds__(HIST ? kNsHistThreads : kNsThreads) ns_normalize_kernel(const uint16_t* g, int64_t ldg,
                                                                  uint16_t* x, int64_t ldx, uint32_t cpr,
                                                                  uint32_t nchunks, const double* __restrict__ partial,
                                                                  int npartial, uint32_t* __restrict__ hist) {
  extern __shared__ uint32_t sh_hist[];
  if (HIST) hist_zero(sh_hist);
  const double norm = sqrt(sum_partials(partial, npartial));
  const double inv64 = 1.0 / fmax(norm, 1e-7);
  const float inv32 = __double2float_rn(inv64);
  const bool wide = inv64 < 0x1p-100;
  // two chunks per iteration, both loads issued before either is used
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t c0 = blockIdx.x * blockDim.x + threadIdx.x; c0 < nchunks; c0 += 2 * stride) {
    const uint32_t c1 = c0 + stride;
    const uint4 v0 = *reinterpret_cast<const uint4*>(chunk_ptr(g, c0, cpr, ldg));
    uint4 v1 = make_uint4(0, 0, 0, 0);
    if (c1 < nchunks) v1 = *reinterpret_cast<const uint4*>(chunk_ptr(g, c1, cpr, ldg));
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t c = u ? c1 : c0;
      if (c >= nchunks) break;
      const uint4 v = u ? v1 : v0;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = scaled_bf16(w[j] & 0xFFFFu, inv32, inv64, wide) | (scaled_bf16(w[j] >> 16, inv32, inv64, wide) << 16);
      *reinterpret_cast<uint4*>(const_cast<uint16_t*>(chunk_ptr(x, c, cpr, ldx))) = make_uint4(o[0], o[1], o[2], o[3]);
      if (HIST) hist_add8(sh_hist, o);
    }
  }
  if (HIST) hist_flush(sh_hist, hist);
}

// The k-th smallest magnitude pattern (k >= 1) from the histogram: one CTA of
// 1024 threads; warp w owns bins [1024 w, 1024 w + 1024) and reads them in 32
// coalesced rounds (round j, lane l: bin 1024 w + 32 j + l), so each round is a
// run of 32 consecutive bins.  The warp totals are scanned across the CTA; the
// warp whose range holds the k-th element then scans its rounds in order.
// Writes the pattern to clip_out[0], its binary32 value to amax_out (the
// clipped tensor's max |x|) and zeroes the histogram for its next use.
__global__ void __launch_bounds__(1024) ns_select_kernel(uint32_t* __restrict__ hist, uint32_t k,
                                                         uint32_t* __restrict__ clip_out, float* __restrict__ amax_out) {
  constexpr int kRounds = kHistBins / 1024;
  __shared__ uint32_t warp_excl[32];
  __shared__ uint32_t found;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  uint32_t* base = hist + wid * 1024 + lane;
  uint32_t h[kRounds];
  uint32_t wsum = 0;
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    h[j] = base[32 * j];
    wsum += h[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, o);  // counts < 2^32
  if (lane == 0) warp_excl[wid] = wsum;
  if (t == 0) found = 0xFFFFFFFFu;
  __syncthreads();
  if (wid == 0) {
    const uint32_t mine = warp_excl[lane];
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += n;
    }
    warp_excl[lane] = incl - mine;
  }
  __syncthreads();
  const uint32_t excl = warp_excl[wid];
  if (excl < k && k - excl <= wsum) {  // exactly one warp (uniform branch)
    uint32_t run = excl;
#pragma unroll
    for (int j = 0; j < kRounds; ++j) {
      uint32_t incl = h[j];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, run + incl >= k);
      if (hit) {
        if (lane == 0) found = static_cast<uint32_t>(wid * 1024 + 32 * j + __ffs(hit) - 1);
        break;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
#pragma unroll
  for (int j = 0; j < kRounds; ++j) base[32 * j] = 0;
  __syncthreads();
  if (t == 0) {
    const uint32_t v = found == 0xFFFFFFFFu ? 0x7FFFu : found;
    clip_out[0] = v;
    *amax_out = __uint_as_float(v << 16);
  }
}

// out = bf16(fl32(p x') + fl32(q y)) (no contraction); without y: bf16(fl32(p x')),
// where x' is x with |x| clipped to *clip_x (when given).
// EPI 1: max |out| into *amax (float bits, the slot zeroed beforehand);
// EPI 2: |out| histogram into `hist`.  out may alias x or y (same index only).
template <bool HAS_Y, int EPI>
__global__ void __launch_bounds__(EPI == 2 ? kNsHistThreads : kNsThreads) ns_lincomb_kernel(const uint16_t* x, int64_t ldx, float p,
                                                                const uint16_t* y, int64_t ldy, float q, uint16_t* out,
                                                                int64_t ldo, uint32_t cpr, uint32_t nchunks,
                                                                const uint32_t* __restrict__ clip_x,
                                                                unsigned int* __restrict__ amax,
                                                                uint32_t* __restrict__ hist) {
  extern __shared__ uint32_t sh_hist[];
  if (EPI == 2) hist_zero(sh_hist);
  // min with 0x7FFF leaves every magnitude pattern as it is
  const uint32_t clip2 = clip_x ? *clip_x * 0x10001u : 0x7FFF7FFFu;
  uint32_t m2 = 0;
  // two chunks per iteration, all loads issued before any is used
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t c0 = blockIdx.x * blockDim.x + threadIdx.x; c0 < nchunks; c0 += 2 * stride) {
    const uint32_t c1 = c0 + stride;
    const bool two = c1 < nchunks;
    uint4 vx[2], vy[2];
    vx[0] = *reinterpret_cast<const uint4*>(chunk_ptr(x, c0, cpr, ldx));
    vx[1] = two ? *reinterpret_cast<const uint4*>(chunk_ptr(x, c1, cpr, ldx)) : make_uint4(0, 0, 0, 0);
    vy[0] = vy[1] = make_uint4(0, 0, 0, 0);
    if (HAS_Y) {
      vy[0] = *reinterpret_cast<const uint4*>(chunk_ptr(y, c0, cpr, ldy));
      if (two) vy[1] = *reinterpret_cast<const uint4*>(chunk_ptr(y, c1, cpr, ldy));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !two) break;
      uint32_t wx[4] = {vx[u].x, vx[u].y, vx[u].z, vx[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) wx[j] = (wx[j] & 0x80008000u) | __vminu2(wx[j] & 0x7FFF7FFFu, clip2);
      const uint32_t wy[4] = {vy[u].x, vy[u].y, vy[u].z, vy[u].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo = __fmul_rn(p, bf16_lo(wx[j]));
        float hi = __fmul_rn(p, bf16_hi(wx[j]));
        if (HAS_Y) {
          lo = __fadd_rn(lo, __fmul_rn(q, bf16_lo(wy[j])));
          hi = __fadd_rn(hi, __fmul_rn(q, bf16_hi(wy[j])));
        }
        o[j] = bf16_rn_bits(lo) | (bf16_rn_bits(hi) << 16);
        if (EPI == 1) m2 = __vmaxu2(m2, o[j] & 0x7FFF7FFFu);
      }
      *reinterpret_cast<uint4*>(const_cast<uint16_t*>(chunk_ptr(out, u ? c1 : c0, cpr, ldo))) =
          make_uint4(o[0], o[1], o[2], o[3]);
      if (EPI == 2) hist_add8(sh_hist, o);
    }
  }
  if (EPI == 1) {
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax, m << 16);
  }
  if (EPI == 2) hist_flush(sh_hist, hist);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int ns_grid(uint32_t nchunks, int num_sms, int per_sm) {
  const uint64_t need = (static_cast<uint64_t>(nchunks) + kNsThreads - 1) / kNsThreads;
  const uint64_t cap = static_cast<uint64_t>(num_sms) * per_sm;
  return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

static cudaError_t hist_attr(const void* fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kHistSmem));
}

int ns_sumsq_blocks(int num_sms) { return num_sms * 4; }

cudaError_t launch_ns_normalize(const void* G, int64_t rows, int64_t cols, int64_t ldg, void* X, int64_t ldx,
                                double* partial, uint32_t* hist, int num_sms, cudaStream_t s) {
  const uint32_t cpr = static_cast<uint32_t>(cols / 8);
  const uint32_t nchunks = static_cast<uint32_t>(rows) * cpr;
  // the partials are indexed by CTA: a fixed grid keeps the reduction order fixed
  const int nb = ns_sumsq_blocks(num_sms);
  ns_sumsq_kernel<<<nb, kNsThreads, 0, s>>>(static_cast<const uint16_t*>(G), cpr, nchunks, ldg, partial);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (hist) {
    static cudaError_t attr = hist_attr(reinterpret_cast<const void*>(ns_normalize_kernel<true>));
    if (attr != cudaSuccess) return attr;
    ns_normalize_kernel<true><<<num_sms, kNsHistThreads, kHistSmem, s>>>(
        static_cast<const uint16_t*>(G), ldg, static_cast<uint16_t*>(X), ldx, cpr, nchunks, partial, nb, hist);
  } else {
    ns_normalize_kernel<false><<<ns_grid(nchunks, num_sms, 4), kNsThreads, 0, s>>>(
        static_cast<const uint16_t*>(G), ldg, static_cast<uint16_t*>(X), ldx, cpr, nchunks, partial, nb, nullptr);
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_ns_select(uint32_t* hist, uint32_t k, uint32_t* clip_slot, float* amax_out, cudaStream_t s) {
  ns_select_kernel<<<1, 1024, 0, s>>>(hist, k, clip_slot, amax_out);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_ns_lincomb(const void* x, int64_t ldx, float p, const void* y, int64_t ldy, float q, void* out,
                              int64_t ldo, int64_t rows, int64_t cols, const uint32_t* clip_x, float* amax_out,
                              uint32_t* hist, int num_sms, cudaStream_t s) {
  const uint32_t cpr = static_cast<uint32_t>(cols / 8);
  const uint32_t nchunks = static_cast<uint32_t>(rows) * cpr;
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const uint16_t* yy = static_cast<const uint16_t*>(y);
  uint16_t* oo = static_cast<uint16_t*>(out);
  unsigned int* am = reinterpret_cast<unsigned int*>(amax_out);
  if (amax_out) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), s);
    pdl_chain_break();
    if (e != cudaSuccess) return e;
  }
  const int g4 = ns_grid(nchunks, num_sms, 4), g1 = num_sms;  // the histogram kernels: one CTA per SM
#define NS_LINCOMB_ARGS xx, ldx, p, yy, ldy, q, oo, ldo, cpr, nchunks, clip_x
  if (hist) {
    if (y) {
      static cudaError_t attr = hist_attr(reinterpret_cast<const void*>(ns_lincomb_kernel<true, 2>));
      if (attr != cudaSuccess) return attr;
      ns_lincomb_kernel<true, 2><<<g1, kNsHistThreads, kHistSmem, s>>>(NS_LINCOMB_ARGS, nullptr, hist);
    } else {
      static cudaError_t attr = hist_attr(reinterpret_cast<const void*>(ns_lincomb_kernel<false, 2>));
      if (attr != cudaSuccess) return attr;
      ns_lincomb_kernel<false, 2><<<g1, kNsHistThreads, kHistSmem, s>>>(NS_LINCOMB_ARGS, nullptr, hist);
    }
  } else if (amax_out) {
    if (y)
      ns_lincomb_kernel<true, 1><<<g4, kNsThreads, 0, s>>>(NS_LINCOMB_ARGS, am, nullptr);
    else
      ns_lincomb_kernel<false, 1><<<g4, kNsThreads, 0, s>>>(NS_LINCOMB_ARGS, am, nullptr);
  } else {
    if (y)
      ns_lincomb_kernel<true, 0><<<g4, kNsThreads, 0, s>>>(NS_LINCOMB_ARGS, nullptr, nullptr);
    else
      ns_lincomb_kernel<false, 0><<<g4, kNsThreads, 0, s>>>(NS_LINCOMB_ARGS, nullptr, nullptr);
  }
#undef NS_LINCOMB_ARGS
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
