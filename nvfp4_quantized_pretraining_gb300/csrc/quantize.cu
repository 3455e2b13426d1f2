// NVFP4 quantize kernels (sm_103a): the tensor amax and one tiled kernel that
// produces the row-wise form, the column-wise (transposed) form, or both from
// one read.
//
// Both stream BF16 with 16-byte coalesced loads.  Block maxima are integer
// maxima of |bf16| patterns; E2M1 codes are written 8 or 16 bytes at a time and
// the UE4M3 scales straight into the layout the block-scaled MMA reads.
//
// Format reading (the Full-Stack FP4 pages name NVFP4, section 1, and
// "standard NVFP4", section 3, without defining it): see block_scale() and
// tensor_scale() in common.cuh.
#include <atomic>
#include <mutex>

#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "scale_layout.cuh"
#include "sr.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// amax: max |x| over a BF16 tensor.  |x| ordering equals the ordering of the
// BF16 bit patterns with the sign cleared, so the reduction is integer
// (two elements per 32-bit word with __vmaxu2).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* x, uint32_t cpr, uint32_t nchunks,
                                                   int64_t ld, unsigned int* out) {
  pdl_trigger();
  pdl_wait();
  uint32_t m = 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
  for (; g + 3 * stride < nchunks; g += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t gg = g + u * stride;
      const uint32_t row = gg / cpr, c8 = gg - row * cpr;
      v[u] = __ldcs(reinterpret_cast<const uint4*>(x + row * ld + c8 * 8));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m = __vmaxu2(m, v[u].x & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].y & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].z & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; g < nchunks; g += stride) {
    const uint32_t row = g / cpr, c8 = g - row * cpr;
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(x + row * ld + c8 * 8));
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) b = max(b, red[w]);
    if (b != 0) atomicMax(out, b << 16);  // float bits of the BF16 amax; ordered as unsigned
  }
}

// ---------------------------------------------------------------------------
// Column-wise (transposed) quantization, optionally with the row-wise output
// from the same read.  A CTA of 128 threads stages a 64-row x 128-column BF16
// tile in shared memory (8 coalesced 16-byte loads per thread in flight; small
// CTAs, nine per SM for RTN (56 registers; ten would spill) and six for SR, so
// that the load phase of some overlaps the arithmetic of others).  Both forms
// are then produced from the staged tile: the row form by one thread per 16-element
// block, the column form by threads that own two adjacent columns (one 4-byte
// shared load per row yields both, their block maxima in one packed register)
// and 32 rows, i.e. two 16-row blocks per column.  SR random bits of the column
// form are drawn in the row-chunk mapping (one Philox call per 8 source
// elements) and staged beside the tile.
// ---------------------------------------------------------------------------
struct DualQuantArgs {
  const uint16_t* x;
  int64_t ld;
  uint32_t rows, cols, cpr;
  const float* amax;
  // row-wise output (rows x cols)
  uint8_t* codes_r;
  uint8_t* scales_r;
  float* scale_out_r;
  uint32_t atoms_k_r;
  // column-wise output (cols x rows)
  uint8_t* codes_c;
  uint8_t* scales_c;
  float* scale_out_c;
  uint32_t atoms_k_c;
  PhiloxKeys keys;  // SR: the round keys of the seed (read from the parameter bank, no registers held)
  uint32_t stream_r, stream_c;
  const uint32_t* clip;  // CLIP: |x| is clipped to this BF16 magnitude pattern as the tile is staged
  // Optional, for the GEMM that consumes the row form: its BF16 branch factor P (rows x fold_r,
  // pitch fold_r) rewritten in place as P~ = bf16(fl32(P * fl32(beta / alpha))), alpha =
  // fl32(S_t * the GEMM's other operand's S_t) (1 when 0), the branch fold of the block-scaled
  // GEMM, done here because this kernel knows S_t.  The CTAs of the first tile column each take
  // their tile's rows.
  uint16_t* fold_p;
  const float* fold_other;
  float fold_beta;
  uint32_t fold_r;
};

// The block-scale arithmetic of block_scale() (common.cuh) with its per-tensor parts set up
// once per CTA.  s_b = E4M3_rn_sat(fl32(amax_b / D)), D = fl32(6 S_t).  The quotient comes from
// Markstein's division: with D scaled by a power of two pw into [1, 2) (exact; also for a
// subnormal D), a = amax_b pw, R = fl32(1 / (D pw)), q0 = fl32(a R), then one correction step
// with the exact residual, q = fl32(q0 + fl32(a - q0 D pw) R): four FMA-pipe operations instead
// of a full division per block.  Equality of the resulting scale byte with the one from the
// IEEE division was checked on the CPU for every BF16 amax and every BF16 block maximum up to
// it (the library's own amax values are BF16 magnitudes), and for 20000 random FP32 amax values.
// The element multiplier 1/(s_b S_t) depends on s_b alone, so it is read from a 128-entry table
// built with block_scale()'s own expression (fl32 reciprocal capped at FLT_MAX; 0 for s_b = 0).
struct ScaleCtx {
  float pw, Dp, R;  // pw = 2^k with D pw in [1, 2); Dp = D pw; R = fl32(1 / Dp)
  bool zero;        // S_t == 0: every scale and multiplier is 0
};
__device__ __forceinline__ ScaleCtx scale_ctx(float S_t) {
  ScaleCtx c;
  c.zero = !(S_t > 0.0f);
  const float D = __fmul_rn(6.0f, S_t);
  const uint32_t e = (__float_as_uint(D) >> 23) & 0xFFu;  // 1..245 for a normal D, 0 for a subnormal one
  c.pw = e == 0 ? 0x1p127f : __uint_as_float((254u - e) << 23);
  c.Dp = __fmul_rn(D, c.pw);
  c.R = c.zero ? 0.0f : __frcp_rn(c.Dp);
  return c;
}
__device__ __forceinline__ uint32_t block_sb(float amax_b, const ScaleCtx& c) {
  if (c.zero) return 0u;
  const float a = __fmul_rn(amax_b, c.pw);
  const float q0 = __fmul_rn(a, c.R);
  const float q = __fmaf_rn(__fmaf_rn(-q0, c.Dp, a), c.R, q0);
  return e4m3_rn_sat(q);
}
// tile row r, 16-byte chunk c (0..15) of a 256-byte row: stored at chunk c ^ (bit 3 of c), so
// that the eight chunks 2b (or 2b + 1), b = 0..7, of one row read by eight lanes fall on
// distinct banks
__device__ __forceinline__ uint32_t swz(uint32_t c) { return c ^ ((c >> 3) & 1u); }

constexpr int kTileR = 64, kTileC = 128;  // 64 x 128 BF16 tiles: 16 KB staged per CTA
constexpr int kDualThreads = 128;

// J32: every element group index j = row * cpr + c8 of the tensor is below 2^32 (chosen by the host).
template <bool ROW, bool COL, bool SR, bool CLIP = false, bool J32 = false>
__global__ void __launch_bounds__(kDualThreads, SR ? 6 : 9) quantize_dual_kernel(const DualQuantArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint16_t(*tile)[kTileC] = reinterpret_cast<uint16_t(*)[kTileC]>(dsm);
  uint16_t(*rtile)[kTileC] = reinterpret_cast<uint16_t(*)[kTileC]>(dsm + kTileR * kTileC * 2);
  pdl_trigger();
  pdl_wait();
  const uint32_t r0 = blockIdx.y * kTileR, c0 = blockIdx.x * kTileC;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  constexpr int kLoads = kTileR * (kTileC / 8) / kDualThreads;  // 8
  // the tile's loads first: the tensor amax, the scale set-up below and (SR) the column form's random
  // bits run while they are in flight
  uint4 w[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const int q = tid + i * kDualThreads;
    const uint32_t row = r0 + (q >> 4), c8 = (c0 >> 3) + (q & 15);
    w[i] = make_uint4(0, 0, 0, 0);
    if (row < a.rows && c8 < a.cpr) w[i] = __ldcs(reinterpret_cast<const uint4*>(a.x + row * a.ld + c8 * 8));
  }
  const float amax = *a.amax;
  const float S_t = tensor_scale(amax);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (ROW && a.scale_out_r) { a.scale_out_r[0] = S_t; a.scale_out_r[1] = amax; }
    if (COL && a.scale_out_c) { a.scale_out_c[0] = S_t; a.scale_out_c[1] = amax; }
  }
  const bool pack4 = (a.cols & 63u) == 0;
  __shared__ float inv_tab[128];
  const ScaleCtx sc = scale_ctx(S_t);
  if (tid < 128)
    inv_tab[tid] = (tid == 0 || sc.zero) ? 0.0f : fminf(__frcp_rn(__fmul_rn(e4m3_value(tid), S_t)), 3.402823466e38f);
  if (a.fold_p && blockIdx.x == 0) {  // (overlaps the tile's loads in flight)
    float alpha = __fmul_rn(S_t, *a.fold_other);
    if (alpha == 0.0f) alpha = 1.0f;
    const float g = __fdiv_rn(a.fold_beta, alpha);
    const uint32_t nrow = a.rows - r0 < (uint32_t)kTileR ? a.rows - r0 : (uint32_t)kTileR;
    uint32_t* P = reinterpret_cast<uint32_t*>(a.fold_p + (size_t)r0 * a.fold_r);
    for (uint32_t i = tid; i < nrow * a.fold_r / 2; i += kDualThreads) {
      const uint32_t v = P[i];
      __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(bf16_lo(v), g), __fmul_rn(bf16_hi(v), g));
      P[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
  }
  if (COL && SR) {
    // the column form's random bits first: their ALU work overlaps the global loads in flight.
    // Element e of a chunk takes word e/2, low half for even e: in element order the eight
    // 16-bit draws are exactly the four words as stored
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int q = tid + i * kDualThreads;
      const uint32_t row = r0 + (q >> 4), c8 = (c0 >> 3) + (q & 15);
      *reinterpret_cast<uint4*>(&rtile[q >> 4][(q & 15) * 8]) =
          J32 ? sr_random32(a.keys, a.stream_c, row * a.cpr + c8) : sr_random(a.keys, a.stream_c, (uint64_t)row * a.cpr + c8);
    }
  }
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const int q = tid + i * kDualThreads;
    if (CLIP) {
      const uint32_t v2 = *a.clip * 0x10001u;
      w[i].x = (w[i].x & 0x80008000u) | __vminu2(w[i].x & 0x7FFF7FFFu, v2);
      w[i].y = (w[i].y & 0x80008000u) | __vminu2(w[i].y & 0x7FFF7FFFu, v2);
      w[i].z = (w[i].z & 0x80008000u) | __vminu2(w[i].z & 0x7FFF7FFFu, v2);
      w[i].w = (w[i].w & 0x80008000u) | __vminu2(w[i].w & 0x7FFF7FFFu, v2);
    }
    *reinterpret_cast<uint4*>(&tile[q >> 4][swz(q & 15) * 8]) = w[i];
  }
  __syncthreads();

  if (ROW) {
    // row phase: one thread per 16-element block (block b = tid + 256 i: tile row b / 8, block b % 8),
    // so each block scale is computed once.  With the chunk swizzle, the 128-bit shared reads of
    // each 8-lane phase (one row, blocks 0..7) fall on distinct banks.
#pragma unroll 2
    for (int i = 0; i < kTileR * (kTileC / 16) / kDualThreads; ++i) {
      const int b = tid + i * kDualThreads;
      const int tr = b >> 3, blk = b & 7;
      const uint32_t row = r0 + tr, c16 = (c0 >> 4) + blk;
      const uint4 wl = *reinterpret_cast<const uint4*>(&tile[tr][swz(2 * blk) * 8]);      // elements 0..7
      const uint4 wh = *reinterpret_cast<const uint4*>(&tile[tr][swz(2 * blk + 1) * 8]);  // elements 8..15
      const uint32_t wd[8] = {wl.x, wl.y, wl.z, wl.w, wh.x, wh.y, wh.z, wh.w};
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = __vmaxu2(m, wd[e] & 0x7FFF7FFFu);
      m = max(m & 0xFFFFu, m >> 16);
      BlockScale bs;
      bs.sb = block_sb(__uint_as_float(m << 16), sc);
      bs.inv = inv_tab[bs.sb];
      float2 y2[2][4];  // element pairs (2q, 2q+1) of elements 0..7 and 8..15, the two halves of word q
      const float2 inv2 = make_float2(bs.inv, bs.inv);
#pragma unroll
      for (int e = 0; e < 8; ++e) y2[e >> 2][e & 3] = __fmul2_rn(make_float2(bf16_lo(wd[e]), bf16_hi(wd[e])), inv2);
      if (SR) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint4 rr = J32 ? sr_random32(a.keys, a.stream_r, row * a.cpr + 2 * c16 + hh)
                               : sr_random(a.keys, a.stream_r, (uint64_t)row * a.cpr + 2 * c16 + hh);
          const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) y2[hh][q] = sr_round2(y2[hh][q], sr_bias_lo(rw[q]), sr_bias_hi(rw[q]));
        }
      }
      float y[2][8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y[e >> 2][2 * (e & 3)] = y2[e >> 2][e & 3].x;
        y[e >> 2][2 * (e & 3) + 1] = y2[e >> 2][e & 3].y;
      }
      const uint32_t lo = e2m1x8(y[0]), hi = e2m1x8(y[1]);
      const bool valid = row < a.rows && 16 * c16 < a.cols;
      if (valid) *reinterpret_cast<uint2*>(a.codes_r + (size_t)row * (a.cols >> 1) + c16 * 8) = make_uint2(lo, hi);
      if (pack4) {
        // lanes 4k .. 4k+3 hold four consecutive scales of one row
        const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, bs.sb, 1);
        const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, bs.sb, 2);
        const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, bs.sb, 3);
        if (valid && (lane & 3) == 0)
          *reinterpret_cast<uint32_t*>(a.scales_r + sf_offset(row, c16, a.atoms_k_r)) =
              bs.sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
      } else if (valid) {
        a.scales_r[sf_offset(row, c16, a.atoms_k_r)] = static_cast<uint8_t>(bs.sb);
      }
    }
  }
  if (!COL) return;

  // column phase: columns c0 + 2cp, c0 + 2cp + 1; rows r0 + 32rq .. +31 (blocks 2rq .. 2rq+1 of 16)
  const uint32_t cp = tid & 63, rq = tid >> 6;
  const uint32_t col = c0 + 2 * cp;
  if (col >= a.cols) return;
  const bool has2 = col + 1 < a.cols;
  uint32_t sbits[2] = {0, 0};
  uint4 cbuf[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t rb = 2 * rq + h;  // 16-row block within the tile
    float va[16], vb[16];
    uint32_t m2 = 0;  // both columns' |bf16| maxima, one per half-word
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t pr = *reinterpret_cast<const uint32_t*>(&tile[rb * 16 + i][swz(cp >> 2) * 8 + 2 * (cp & 3)]);
      m2 = __vmaxu2(m2, pr & 0x7FFF7FFFu);
      va[i] = bf16_lo(pr);
      vb[i] = bf16_hi(pr);
    }
    BlockScale sa, sb;
    sa.sb = block_sb(__uint_as_float(m2 << 16), sc);
    sa.inv = inv_tab[sa.sb];
    sb.sb = block_sb(__uint_as_float(m2 & 0xFFFF0000u), sc);
    sb.inv = inv_tab[sb.sb];
    const float2 inv2 = make_float2(sa.inv, sb.inv);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float2 v = __fmul2_rn(make_float2(va[i], vb[i]), inv2);
      if (SR) {
        const uint32_t rp = *reinterpret_cast<const uint32_t*>(&rtile[rb * 16 + i][2 * cp]);
        v = sr_round2(v, sr_bias_lo(rp), sr_bias_hi(rp));
      }
      va[i] = v.x;
      vb[i] = v.y;
    }
    float t8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = va[i];
    const uint32_t a0 = e2m1x8(t8);
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = va[8 + i];
    const uint32_t a1 = e2m1x8(t8);
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = vb[i];
    const uint32_t b0 = e2m1x8(t8);
#pragma unroll
    for (int i = 0; i < 8; ++i) t8[i] = vb[8 + i];
    const uint32_t b1 = e2m1x8(t8);
    if (h == 0) {
      cbuf[0].x = a0; cbuf[0].y = a1; cbuf[1].x = b0; cbuf[1].y = b1;
    } else {
      cbuf[0].z = a0; cbuf[0].w = a1; cbuf[1].z = b0; cbuf[1].w = b1;
    }
    sbits[0] |= sa.sb << (8 * h);
    sbits[1] |= sb.sb << (8 * h);
  }
  const uint32_t rowb = r0 + 32 * rq;  // first source row of this thread's 32
  const uint32_t kb = rowb >> 4;       // even: kb and kb+1 share one 32-bit scale group
  if (rowb < a.rows) {
    const bool two = rowb + 16 < a.rows;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j == 1 && !has2) break;
      uint8_t* cdst = a.codes_c + (size_t)(col + j) * (a.rows >> 1) + (rowb >> 1);
      if (two && (((a.rows >> 1) & 15u) == 0)) {
        *reinterpret_cast<uint4*>(cdst) = cbuf[j];
      } else {
        *reinterpret_cast<uint2*>(cdst) = make_uint2(cbuf[j].x, cbuf[j].y);
        if (two) *reinterpret_cast<uint2*>(cdst + 8) = make_uint2(cbuf[j].z, cbuf[j].w);
      }
      uint8_t* sdst = a.scales_c + sf_offset(col + j, kb, a.atoms_k_c);
      if (two) *reinterpret_cast<uint16_t*>(sdst) = static_cast<uint16_t>(sbits[j]);
      else *sdst = static_cast<uint8_t>(sbits[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Diagnostic conversion kernel: the quantizer's own E2M1 and E4M3 routines.
// ---------------------------------------------------------------------------
__global__ void debug_convert_kernel(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ e2m1,
                                     uint8_t* __restrict__ e4m3) {
  const int64_t i8 = (int64_t)(blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i8 >= n) return;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = (i8 + i < n) ? in[i8 + i] : 0.0f;
  const uint32_t c = e2m1x8(v);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i8 + i < n) {
      e2m1[i8 + i] = (c >> (4 * i)) & 0xFu;
      e4m3[i8 + i] = static_cast<uint8_t>(e4m3_rn_sat(v[i]));
    }
}

// Diagnostic stochastic rounding: the quantizer's own sr_round on given random bits.
__global__ void debug_sr_round_kernel(const float* __restrict__ in, const uint16_t* __restrict__ rnd, int64_t n,
                                      uint8_t* __restrict__ e2m1) {
  const int64_t i8 = (int64_t)(blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i8 >= n) return;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = (i8 + i < n) ? sr_round(in[i8 + i], sr_bias_lo(rnd[i8 + i])) : 0.0f;
  const uint32_t c = e2m1x8(v);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i8 + i < n) e2m1[i8 + i] = (c >> (4 * i)) & 0xFu;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
// Diagnostic switch (fp4_debug_force_counter64): the SR kernels take their general 64-bit counter
// form whatever the tensor's size, so that tests reach the form that tensors of 2^35 or more
// elements take.
static std::atomic<int> g_force_counter64{0};
void set_force_counter64(bool on) { g_force_counter64.store(on ? 1 : 0); }

static int grid_for(uint64_t work_items, int per_block, int max_blocks) {
  uint64_t b = (work_items + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > (uint64_t)max_blocks) b = max_blocks;
  return static_cast<int>(b);
}

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* out, int num_sms,
                        cudaStream_t s) {
  const uint32_t cpr = static_cast<uint32_t>(cols / 8);
  const uint32_t nchunks = static_cast<uint32_t>(rows) * cpr;
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), s);
  pdl_chain_break();
  if (e != cudaSuccess) return e;
  const int grid = grid_for(nchunks, 256 * 4, num_sms * 8);
  e = launch_pdl(amax_kernel, dim3(grid), dim3(256), 0, s, static_cast<const uint16_t*>(x), cpr, nchunks, ld,
                 reinterpret_cast<unsigned int*>(out));
  count_launch();
  return e;
}

cudaError_t launch_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, bool sr, uint64_t seed,
                                 uint32_t stream_r, uint32_t stream_c, const float* amax, const QOut* row_out,
                                 const QOut* col_out, cudaStream_t s, const uint32_t* clip, const BranchFold* fold) {
  DualQuantArgs a{};
  a.clip = clip;
  if (fold) {
    a.fold_p = static_cast<uint16_t*>(fold->P);
    a.fold_other = fold->other_scale;
    a.fold_beta = fold->beta;
    a.fold_r = static_cast<uint32_t>(fold->r);
  }
  a.x = static_cast<const uint16_t*>(x);
  a.ld = ld;
  a.rows = static_cast<uint32_t>(rows);
  a.cols = static_cast<uint32_t>(cols);
  a.cpr = static_cast<uint32_t>(cols / 8);
  a.amax = amax;
  if (row_out) {
    a.codes_r = static_cast<uint8_t*>(row_out->codes);
    a.scales_r = static_cast<uint8_t*>(row_out->scales);
    a.scale_out_r = row_out->scale;
    a.atoms_k_r = static_cast<uint32_t>((cols / 16 + 3) / 4);
  }
  if (col_out) {
    a.codes_c = static_cast<uint8_t*>(col_out->codes);
    a.scales_c = static_cast<uint8_t*>(col_out->scales);
    a.scale_out_c = col_out->scale;
    a.atoms_k_c = static_cast<uint32_t>((rows / 16 + 3) / 4);
  }
  a.keys = philox_keys(seed);
  a.stream_r = stream_r;
  a.stream_c = stream_c;
  dim3 grid(static_cast<unsigned>((cols + kTileC - 1) / kTileC), static_cast<unsigned>((rows + kTileR - 1) / kTileR));
  const bool R = row_out != nullptr, C = col_out != nullptr;
  // the BF16 tile is staged for both forms; the SR column form also stages its random bits
  const int smem = kTileR * kTileC * 2 * ((C && sr) ? 2 : 1);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    for (auto k : {quantize_dual_kernel<true, true, true>, quantize_dual_kernel<false, true, true>,
                   quantize_dual_kernel<true, true, true, false, true>, quantize_dual_kernel<false, true, true, false, true>})
      if (attr == cudaSuccess)
        attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kTileR * kTileC * 2);
  });
  // every element group index row * cpr + c8 below 2^32: the SR kernels' 32-bit counter form
  const bool j32 = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols / 8) <= 0xFFFFFFFFull &&
                   !g_force_counter64.load(std::memory_order_relaxed);
  if (attr != cudaSuccess) return attr;
  cudaError_t e = cudaSuccess;
  if (clip) {  // the clipped form: both orientations, RTN
    if (!(R && C) || sr) return cudaErrorInvalidValue;
    e = launch_pdl(quantize_dual_kernel<true, true, false, true>, grid, dim3(kDualThreads), smem, s, a);
  } else if (R && C) {
    if (sr && j32)
      e = launch_pdl(quantize_dual_kernel<true, true, true, false, true>, grid, dim3(kDualThreads), smem, s, a);
    else if (sr) e = launch_pdl(quantize_dual_kernel<true, true, true>, grid, dim3(kDualThreads), smem, s, a);
    else e = launch_pdl(quantize_dual_kernel<true, true, false>, grid, dim3(kDualThreads), smem, s, a);
  } else if (C) {
    if (sr && j32)
      e = launch_pdl(quantize_dual_kernel<false, true, true, false, true>, grid, dim3(kDualThreads), smem, s, a);
    else if (sr) e = launch_pdl(quantize_dual_kernel<false, true, true>, grid, dim3(kDualThreads), smem, s, a);
    else e = launch_pdl(quantize_dual_kernel<false, true, false>, grid, dim3(kDualThreads), smem, s, a);
  } else {
    if (sr && j32)
      e = launch_pdl(quantize_dual_kernel<true, false, true, false, true>, grid, dim3(kDualThreads), smem, s, a);
    else if (sr) e = launch_pdl(quantize_dual_kernel<true, false, true>, grid, dim3(kDualThreads), smem, s, a);
    else e = launch_pdl(quantize_dual_kernel<true, false, false>, grid, dim3(kDualThreads), smem, s, a);
  }
  count_launch();
  return e;
}

cudaError_t launch_debug_convert(const float* in, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t s) {
  const int64_t threads = (n + 7) / 8;
  const int grid = static_cast<int>((threads + 255) / 256);
  debug_convert_kernel<<<grid, 256, 0, s>>>(in, n, e2m1, e4m3);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_debug_sr_round(const float* in, const uint16_t* rnd, int64_t n, uint8_t* e2m1, cudaStream_t s) {
  const int64_t threads = (n + 7) / 8;
  const int grid = static_cast<int>((threads + 255) / 256);
  debug_sr_round_kernel<<<grid, 256, 0, s>>>(in, rnd, n, e2m1);
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
