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


// A block's 16 values are held as eight FP32 pairs p[k] = (x[k], x[k + 8]), so that most of the
// per-block arithmetic runs as packed FP32x2 operations (each lane exactly the scalar operation).
__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b) {  // a - b: b * -1 is exact, one rounding
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

// In-place unnormalised Walsh-Hadamard transform of 16 values, natural order: levels h = 1, 2, 4
// pair x[j] with x[j + h] inside each half, i.e. p[j] with p[j + h] in both lanes at once; level 8
// pairs the two lanes of each p[k].
__device__ __forceinline__ void wht16(float2 (&p)[8]) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; i += 2 * h) {
#pragma unroll
      for (int j = i; j < i + h; ++j) {
        const float2 a = p[j], b = p[j + h];
        p[j] = __fadd2_rn(a, b);
        p[j + h] = sub2_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) p[k] = make_float2(__fadd_rn(p[k].x, p[k].y), __fsub_rn(p[k].x, p[k].y));
}

__device__ __forceinline__ void load_block(const float* __restrict__ v, float4 (&f)[4]) {
  const float4* p = reinterpret_cast<const float4*>(v);
#pragma unroll
  for (int q = 0; q < 4; ++q) f[q] = __ldcs(p + q);
}

// h (16 values, as pairs h[k] = (h_k, h_k+8)) and the BF16 mean pattern of one block of v (loaded
// into f).  The mean's pairwise tree adds (h_2i, h_2i+1) for i = 0..7, then neighbours twice more,
// then the last two: in the pair layout the first three levels are packed additions of the same
// operands, (t_i, t_i+4) = h[2i] + h[2i+1] and so on.
__device__ __forceinline__ uint32_t vt_forward(const float4 (&fv)[4], float2 (&h)[8]) {
  const float* f = reinterpret_cast<const float*>(fv);
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = make_float2(__fsqrt_rn(f[k]), __fsqrt_rn(f[k + 8]));
  float2 t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = __fadd2_rn(h[2 * i], h[2 * i + 1]);  // (t_i, t_i+4)
#pragma unroll
  for (int i = 0; i < 2; ++i) t[i] = __fadd2_rn(t[2 * i], t[2 * i + 1]);  // (t0+t1, t4+t5), (t2+t3, t6+t7)
  t[0] = __fadd2_rn(t[0], t[1]);
  const uint32_t mean = bf16_rn_bits(__fmul_rn(__fadd_rn(t[0].x, t[0].y), 0.0625f));
  const float mu = __uint_as_float(mean << 16);
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = __fadd2_rn(h[k], make_float2(-mu, -mu));
  wht16(h);
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = __fmul2_rn(h[k], make_float2(0.25f, 0.25f));
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
    float2 h[8];
    vt_forward(cur, h);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      m = max(m, max(__float_as_uint(h[k].x) & 0x7FFFFFFFu, __float_as_uint(h[k].y) & 0x7FFFFFFFu));
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
    float2 h[8];
    const uint32_t mean = vt_forward(cur, h);
#pragma unroll
    for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
    float amax_b = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax_b = fmaxf(amax_b, fmaxf(fabsf(h[k].x), fabsf(h[k].y)));
    const BlockScale bs = block_scale(amax_b, S_t);
    float y0[8], y1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 y = __fmul2_rn(h[k], make_float2(bs.inv, bs.inv));
      y0[k] = y.x;
      y1[k] = y.y;
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
      float2 x[8];  // (x_k, x_k+8)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        x[k] = __fmul2_rn(__fmul2_rn(make_float2(e2m1_value(c.x >> (4 * k)), e2m1_value(c.y >> (4 * k))),
                                     make_float2(sv, sv)),
                          make_float2(S_t, S_t));
      wht16(x);
      float2 u[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 w = __fadd2_rn(__fmul2_rn(x[k], make_float2(0.25f, 0.25f)), make_float2(mu, mu));
        u[k] = __fmul2_rn(w, w);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        stg[wib][lane * 4 + q] = make_float4(u[4 * q].x, u[4 * q + 1].x, u[4 * q + 2].x, u[4 * q + 3].x);
        stg[wib][lane * 4 + 2 + q] = make_float4(u[4 * q].y, u[4 * q + 1].y, u[4 * q + 2].y, u[4 * q + 3].y);
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
  pdl_chain_break();
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
