// Q-AdamW second-moment codec ("Full-Stack FP4", section 2.2, Quantized-state
// AdamW): v_t is stored in NVFP4 after three transforms, the square root (which
// shortens the heavy tail), a tile mean kept in BF16 (the common positive part),
// and a Hadamard transform of the zero-mean residual; the decoder inverts the
// transform and the mean separation and squares.
//
// Reading of the sizes the pages leave open: the tile and the Hadamard both span
// one 16-element NVFP4 block along a row, so one thread owns one block end to end:
//   u = sqrt(v); mean = bf16(pairwise-tree sum of u / 16); r = u - mean;
//   h = WHT16(r) / 4 (natural-order butterfly, orthonormal, its own inverse);
//   codes, block scale = NVFP4 RTN of h with one tensor scale from max |h|.
// Every operation is a single FP32 operation in a fixed order (no contraction).
// The encoder makes two passes over v (max |h|, then the codes), since the tensor
// scale needs the whole tensor; both recompute h from v instead of storing it.
#include "bf16_convert.cuh"
#include "common.cuh"
#include "kernels.h"
#include "scale_layout.cuh"

namespace nvfp4 {

constexpr int kVtThreads = 256;


// In-place unnormalised Walsh-Hadamard transform of 16 values, natural order.
__device__ __forceinline__ void wht16(float (&x)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i += 2 * h) {
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float a = x[j], b = x[j + h];
        x[j] = __fadd_rn(a, b);
        x[j + h] = __fsub_rn(a, b);
      }
    }
  }
}

__device__ __forceinline__ void load_block(const float* __restrict__ v, float4 (&f)[4]) {
  const float4* p = reinterpret_cast<const float4*>(v);
#pragma unroll
  for (int q = 0; q < 4; ++q) f[q] = __ldcs(p + q);
}

// h (16 values) and the BF16 mean pattern of one block of v (loaded into f).
__device__ __forceinline__ uint32_t vt_forward(const float4 (&fv)[4], float (&h)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = fv[q];
    h[4 * q + 0] = __fsqrt_rn(f.x);
    h[4 * q + 1] = __fsqrt_rn(f.y);
    h[4 * q + 2] = __fsqrt_rn(f.z);
    h[4 * q + 3] = __fsqrt_rn(f.w);
  }
  float t[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) t[i] = __fadd_rn(h[2 * i], h[2 * i + 1]);
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
#pragma unroll
  for (int i = 0; i < 2; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
  const uint32_t mean = bf16_rn_bits(__fmul_rn(__fadd_rn(t[0], t[1]), 0.0625f));
  const float mu = __uint_as_float(mean << 16);
#pragma unroll
  for (int i = 0; i < 16; ++i) h[i] = __fsub_rn(h[i], mu);
  wht16(h);
#pragma unroll
  for (int i = 0; i < 16; ++i) h[i] = __fmul_rn(h[i], 0.25f);
  return mean;
}

__device__ __forceinline__ const float* block_src(const float* v, uint32_t b, uint32_t kbpr, int64_t ldv) {
  const uint32_t row = b / kbpr;
  return v + static_cast<int64_t>(row) * ldv + static_cast<int64_t>(b - row * kbpr) * 16;
}

// Pass 1: max |h| over the tensor into *amax (float bits, zeroed beforehand).
__global__ void __launch_bounds__(kVtThreads) vt_amax_kernel(const float* __restrict__ v, int64_t ldv, uint32_t kbpr,
                                                             uint32_t nblocks, unsigned int* __restrict__ amax) {
  uint32_t m = 0;
  // the next block's loads are issued before the current block's arithmetic
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  float4 cur[4];
  if (b < nblocks) load_block(block_src(v, b, kbpr, ldv), cur);
  for (; b < nblocks; b += stride) {
    float4 nxt[4];
    if (b + stride < nblocks) load_block(block_src(v, b + stride, kbpr, ldv), nxt);
    float h[16];
    vt_forward(cur, h);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max(m, __float_as_uint(h[i]) & 0x7FFFFFFFu);
#pragma unroll
    for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax, m);
}

// Pass 2: codes (8 bytes per block), the block scale in the MMA layout and the
// BF16 mean; the tensor scale from the pass-1 amax (amax is scale_out + 1: one
// thread writes back the value every thread read).
__global__ void __launch_bounds__(kVtThreads) vt_encode_kernel(const float* __restrict__ v, int64_t ldv, uint32_t kbpr,
                                                               uint32_t nblocks, const float* amax,
                                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                               uint32_t atoms_k, float* scale_out,
                                                               uint16_t* __restrict__ mean_out) {
  const float a = *amax;
  const float S_t = tensor_scale(a);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    scale_out[0] = S_t;
    scale_out[1] = a;
  }
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  float4 cur[4];
  if (b < nblocks) load_block(block_src(v, b, kbpr, ldv), cur);
  for (; b < nblocks; b += stride) {
    float4 nxt[4];
    if (b + stride < nblocks) load_block(block_src(v, b + stride, kbpr, ldv), nxt);
    float h[16];
    const uint32_t mean = vt_forward(cur, h);
#pragma unroll
    for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
    float amax_b = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(h[i]));
    const BlockScale bs = block_scale(amax_b, S_t);
    float y0[8], y1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y0[i] = __fmul_rn(h[i], bs.inv);
      y1[i] = __fmul_rn(h[8 + i], bs.inv);
    }
    *reinterpret_cast<uint2*>(codes + static_cast<uint64_t>(b) * 8) = make_uint2(e2m1x8(y0), e2m1x8(y1));
    const uint32_t row = b / kbpr;
    scales[sf_offset(row, b - row * kbpr, atoms_k)] = static_cast<uint8_t>(bs.sb);
    mean_out[b] = static_cast<uint16_t>(mean);
  }
}

// E2M1 code (sign in bit 3) to its value.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const uint32_t mag = e == 0 ? (m ? 0x3F000000u : 0u) : (((126u + e) << 23) | (m << 22));
  return __uint_as_float(mag | ((c & 8u) << 28));
}

// Decode: v = (WHT16(deq) / 4 + mean)^2, deq = fl32(e2m1 * e4m3 * S_t) (the first
// product is exact, so one rounding).
__global__ void __launch_bounds__(kVtThreads) vt_decode_kernel(const uint8_t* __restrict__ codes,
                                                               const uint8_t* __restrict__ scales, uint32_t atoms_k,
                                                               const float* __restrict__ scale_in,
                                                               const uint16_t* __restrict__ mean_in, uint32_t kbpr,
                                                               uint32_t nblocks, float* __restrict__ out, int64_t ldo) {
  const float S_t = scale_in[0];
  // Each warp decodes 32 consecutive blocks (one per lane), stages the 2 KB of results in shared
  // memory and stores them lane-consecutively (512 contiguous bytes per instruction instead of 32
  // pieces of 16 bytes at a 64-byte stride).  The next blocks' codes, scale byte and mean are
  // loaded before the current ones' arithmetic.
  __shared__ float4 stg[kVtThreads / 32][128];
  const uint32_t lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  uint2 cn = make_uint2(0, 0);
  uint32_t sn = 0, mn = 0;
  auto fetch = [&](uint32_t bb) {
    const uint32_t row = bb / kbpr;
    cn = __ldcs(reinterpret_cast<const uint2*>(codes + static_cast<uint64_t>(bb) * 8));
    sn = scales[sf_offset(row, bb - row * kbpr, atoms_k)];
    mn = mean_in[bb];
  };
  if (b < nblocks) fetch(b);
  for (; b - lane < nblocks; b += stride) {  // while the warp's first block exists (warp-uniform)
    long long off = 0;  // this lane's block: offset of its 16 outputs
    if (b < nblocks) {
      const uint2 c = cn;
      const uint32_t row = b / kbpr, kb = b - row * kbpr;
      off = static_cast<long long>(row) * ldo + static_cast<long long>(kb) * 16;
      const float sv = e4m3_value(sn);
      const float mu = __uint_as_float(mn << 16);
      if (b + stride < nblocks) fetch(b + stride);
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = __fmul_rn(__fmul_rn(e2m1_value(c.x >> (4 * i)), sv), S_t);
        x[8 + i] = __fmul_rn(__fmul_rn(e2m1_value(c.y >> (4 * i)), sv), S_t);
      }
      wht16(x);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float u[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float w = __fadd_rn(__fmul_rn(x[4 * q + j], 0.25f), mu);
          u[j] = __fmul_rn(w, w);
        }
        stg[wib][lane * 4 + q] = make_float4(u[0], u[1], u[2], u[3]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t j = i * 32 + lane;  // float4 j of the warp's 128: block j / 4, quarter j % 4
      const long long o = __shfl_sync(0xFFFFFFFFu, off, j >> 2);
      if (b - lane + (j >> 2) < nblocks) __stcs(reinterpret_cast<float4*>(out + o) + (j & 3), stg[wib][j]);
    }
    __syncwarp();
  }
}

static int vt_grid(uint32_t nblocks, int num_sms) {
  const uint64_t need = (static_cast<uint64_t>(nblocks) + kVtThreads - 1) / kVtThreads;
  const uint64_t cap = static_cast<uint64_t>(num_sms) * 8;
  return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

cudaError_t launch_vt_encode(const float* v, int64_t rows, int64_t cols, int64_t ldv, const QOut& out,
                             uint16_t* mean, int num_sms, cudaStream_t s) {
  const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
  const uint32_t nblocks = static_cast<uint32_t>(rows) * kbpr;
  const uint32_t atoms_k = (kbpr + 3) / 4;
  float* amax = &out.scale[1];
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  const int grid = vt_grid(nblocks, num_sms);
  vt_amax_kernel<<<grid, kVtThreads, 0, s>>>(v, ldv, kbpr, nblocks, reinterpret_cast<unsigned int*>(amax));
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  vt_encode_kernel<<<grid, kVtThreads, 0, s>>>(v, ldv, kbpr, nblocks, amax, static_cast<uint8_t*>(out.codes),
                                               static_cast<uint8_t*>(out.scales), atoms_k, out.scale, mean);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_vt_decode(const void* codes, const void* scales, const float* scale, const uint16_t* mean,
                             int64_t rows, int64_t cols, float* out, int64_t ldo, int num_sms, cudaStream_t s) {
  const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
  const uint32_t nblocks = static_cast<uint32_t>(rows) * kbpr;
  const uint32_t atoms_k = (kbpr + 3) / 4;
  vt_decode_kernel<<<vt_grid(nblocks, num_sms), kVtThreads, 0, s>>>(
      static_cast<const uint8_t*>(codes), static_cast<const uint8_t*>(scales), atoms_k, scale, mean, kbpr, nblocks,
      out, ldo);
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
