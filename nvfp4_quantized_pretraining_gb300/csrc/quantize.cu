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
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "scale_layout.cuh"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// amax: max |x| over a BF16 tensor.  |x| ordering equals the ordering of the
// BF16 bit patterns with the sign cleared, so the reduction is integer
// (two elements per 32-bit word with __vmaxu2).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, uint32_t cpr, uint32_t nchunks,
                                                   int64_t ld, unsigned int* __restrict__ out) {
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
// Dual quantizer: the row-wise form, the column-wise (transposed) form, or both
// from one read of x.  Persistent CTAs walk the 128 x 128 BF16 tiles of x; a
// producer warp streams each tile into a ring of shared-memory stages with TMA
// (two 128-row x 64-column boxes, 128-byte swizzle: the 16-byte chunk c of
// tile row r sits at chunk c ^ (r & 7) of its box row), so loads of the next
// tiles overlap the work on the current one.  Eight compute warps produce
// both forms from the staged tile:
//   * row form: one thread per 16-element block (block scale computed once);
//   * column form: one thread per 8-column x 8-row task, the two tasks of a
//     16-row block in lanes l and l ^ 16 (block maxima combined by a shuffle).
//     A task's eight columns share, in every row, one Philox counter (the 8
//     source elements of one group j), so its SR draws are made in registers.
// ---------------------------------------------------------------------------
struct DualQuantArgs {
  uint32_t rows, cols, cpr;  // cpr = cols / 8
  uint32_t tiles_c, num_tiles;
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
  PhiloxKeys keys;  // SR: the round keys of the seed
  uint32_t stream_r, stream_c;
  const uint32_t* clip;  // CLIP: |x| is clipped to this BF16 magnitude pattern as the tile is read
};

namespace qd {
constexpr int TILE = 128;
constexpr int BOX_C = 64;                     // TMA box: 128 rows x 64 BF16 columns (128-byte rows)
constexpr int BOX_BYTES = TILE * BOX_C * 2;   // 16 KB
constexpr int TILE_BYTES = 2 * BOX_BYTES;     // 32 KB
constexpr int STAGES = 3;
constexpr int COMPUTE_WARPS = 8;
constexpr int COMPUTE_THREADS = COMPUTE_WARPS * 32;
constexpr int THREADS = COMPUTE_THREADS + 32;  // + the TMA producer warp
constexpr int CTAS_PER_SM = 2;
constexpr int SMEM_BYTES = STAGES * TILE_BYTES + 1024 /*align*/ + 128 /*barriers*/;
}  // namespace qd

// Shared-memory byte offset of the 16-byte chunk holding tile columns 8c .. 8c + 7 (c = 0..15) of tile row r.
__device__ __forceinline__ uint32_t qd_chunk(uint32_t r, uint32_t c) {
  return (c >> 3) * qd::BOX_BYTES + r * 128u + ((((c & 7u) ^ (r & 7u))) << 4);
}

__device__ __forceinline__ uint32_t clip_word(uint32_t w, uint32_t v2) {
  return (w & 0x80008000u) | __vminu2(w & 0x7FFF7FFFu, v2);
}

template <bool ROW, bool COL, bool SR, bool CLIP>
__global__ void __launch_bounds__(qd::THREADS, qd::CTAS_PER_SM)
    quantize_dual_kernel(const __grid_constant__ CUtensorMap tmap_x, const DualQuantArgs a) {
  using namespace qd;
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * TILE_BYTES);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], COMPUTE_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const float amax = *a.amax;
  const float S_t = tensor_scale(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (ROW && a.scale_out_r) { a.scale_out_r[0] = S_t; a.scale_out_r[1] = amax; }
    if (COL && a.scale_out_c) { a.scale_out_c[0] = S_t; a.scale_out_c[1] = amax; }
  }

  if (warp == COMPUTE_WARPS) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmap_x);
      uint32_t stage = 0, phase = 0;
      int armed[STAGES];
      uint32_t armed_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) {
          ok = false;
          break;
        }
        armed[stage] = 0;
        const int32_t r0 = (int32_t)((t / a.tiles_c) * TILE), c0 = (int32_t)((t % a.tiles_c) * TILE);
        uint8_t* dst = smem + stage * TILE_BYTES;
        mbar_arrive_expect_tx(&full[stage], TILE_BYTES);  // out-of-range parts arrive zero-filled
        tma_load_2d(dst, &tmap_x, &full[stage], c0, r0);
        tma_load_2d(dst + BOX_BYTES, &tmap_x, &full[stage], c0 + BOX_C, r0);
        armed[stage] = 1;
        armed_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        for (int s = 0; s < STAGES; ++s)  // copies already issued land before the CTA may exit
          if (armed[s]) mbar_wait(&full[s], armed_phase[s]);
      }
    }
  } else {
    // ---------------- compute warps ----------------
    const uint32_t tid = threadIdx.x;  // 0 .. COMPUTE_THREADS - 1
    const bool pack4 = (a.cols & 63u) == 0;
    const uint32_t clip2 = CLIP ? *a.clip * 0x10001u : 0u;
    uint32_t stage = 0, phase = 0;
    for (uint32_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
      if (*abort_flag || !mbar_wait(&full[stage], phase)) {
        *abort_flag = 1;
        break;
      }
      const uint8_t* tile = smem + stage * TILE_BYTES;
      const uint32_t r0 = (t / a.tiles_c) * TILE, c0 = (t % a.tiles_c) * TILE;

      if (ROW) {
        // row form: block b = tid + 256 i covers tile row b / 8, columns 16 (b % 8) .. + 15.  Lanes
        // 4..7 of every 8 read their second chunk first, so each 8-lane phase of the 128-bit shared
        // loads touches 8 distinct chunk positions (the two boxes share banks).
        const int first = (lane >> 2) & 1;
#pragma unroll(SR ? 1 : 2)
        for (int i = 0; i < TILE * (TILE / 16) / COMPUTE_THREADS; ++i) {
          const uint32_t b = tid + COMPUTE_THREADS * i;
          const uint32_t tr = b >> 3, blk = b & 7;
          const uint32_t row = r0 + tr, c16 = (c0 >> 4) + blk;
          const uint4 h0 = *reinterpret_cast<const uint4*>(tile + qd_chunk(tr, 2 * blk + first));
          const uint4 h1 = *reinterpret_cast<const uint4*>(tile + qd_chunk(tr, 2 * blk + (first ^ 1)));
          const uint4 wl = first ? h1 : h0, wh = first ? h0 : h1;  // elements 0..7, 8..15
          uint32_t wd[8] = {wl.x, wl.y, wl.z, wl.w, wh.x, wh.y, wh.z, wh.w};
          if (CLIP) {
#pragma unroll
            for (int e = 0; e < 8; ++e) wd[e] = clip_word(wd[e], clip2);
          }
          uint32_t m = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) m = __vmaxu2(m, wd[e] & 0x7FFF7FFFu);
          m = max(m & 0xFFFFu, m >> 16);
          const BlockScale bs = block_scale(__uint_as_float(m << 16), S_t);
          float y[2][8];  // elements 0..7 and 8..15
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            y[e >> 2][2 * (e & 3)] = __fmul_rn(bf16_lo(wd[e]), bs.inv);
            y[e >> 2][2 * (e & 3) + 1] = __fmul_rn(bf16_hi(wd[e]), bs.inv);
          }
          if (SR) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint4 rr = sr_random(a.keys, a.stream_r, (uint64_t)row * a.cpr + 2 * c16 + hh);
              const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                y[hh][e] = sr_round(y[hh][e], (e & 1) ? sr_draw_hi(rw[e >> 1]) : sr_draw_lo(rw[e >> 1]));
            }
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

      if (COL) {
        // column form: task (cg, rb8) = tile columns 8cg .. 8cg+7, tile rows 8rb8 .. 8rb8+7; lanes
        // 0..15 take cg = 0..15 of one row group, so each 8-lane phase reads 8 distinct chunks of one row
        const uint32_t cg = lane & 15, hsel = (uint32_t)lane >> 4, rb8 = 2 * warp + hsel;
        const uint32_t col0 = c0 + 8 * cg, rowbase = r0 + 8 * rb8;
        // pass 1: block maxima of the 8 columns over this task's 8 rows, then over the 16-row block
        uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 q = *reinterpret_cast<const uint4*>(tile + qd_chunk(8 * rb8 + i, cg));
          uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (CLIP) w[e] = clip_word(w[e], clip2);
            m[e] = __vmaxu2(m[e], w[e] & 0x7FFF7FFFu);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = __vmaxu2(m[e], __shfl_xor_sync(0xFFFFFFFFu, m[e], 16));
        // this lane scales columns 4 hsel .. 4 hsel + 3 and takes the partner's multipliers for the rest
        float inv_mine[4];
        uint32_t sb_mine[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t mw = m[2 * hsel + (kk >> 1)];  // columns 4 hsel + kk
          const uint32_t mb = (kk & 1) ? (mw & 0xFFFF0000u) : (mw << 16);
          const BlockScale bs = block_scale(__uint_as_float(mb), S_t);
          inv_mine[kk] = bs.inv;
          sb_mine[kk] = bs.sb;
        }
        float inv[8];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float other = __shfl_xor_sync(0xFFFFFFFFu, inv_mine[kk], 16);
          inv[kk] = hsel ? other : inv_mine[kk];
          inv[4 + kk] = hsel ? inv_mine[kk] : other;
        }
        // pass 2, two rows at a time: codes of rows (2p, 2p + 1) of each column go to byte p of its word
        uint32_t out[8];
#pragma unroll(SR ? 1 : 4)
        for (int p = 0; p < 4; ++p) {
          float y[2][8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t i = 2 * p + h;
            const uint4 q = *reinterpret_cast<const uint4*>(tile + qd_chunk(8 * rb8 + i, cg));
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (CLIP) w[e] = clip_word(w[e], clip2);
              y[h][2 * e] = __fmul_rn(bf16_lo(w[e]), inv[2 * e]);
              y[h][2 * e + 1] = __fmul_rn(bf16_hi(w[e]), inv[2 * e + 1]);
            }
            if (SR) {
              // source elements (rowbase + i, col0 .. col0 + 7): one Philox group
              const uint4 rr = sr_random(a.keys, a.stream_c, (uint64_t)(rowbase + i) * a.cpr + (col0 >> 3));
              const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
              for (int k = 0; k < 8; ++k)
                y[h][k] = sr_round(y[h][k], (k & 1) ? sr_draw_hi(rw[k >> 1]) : sr_draw_lo(rw[k >> 1]));
            }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t b = e2m1x2(y[0][k], y[1][k]);  // row 2p in the low nibble
            // byte p of the word <- byte 0 of b (selector 0x3210 with nibble p replaced by 4)
            out[k] = p == 0 ? b : __byte_perm(out[k], b, (0x3210u & ~(0xFu << (4 * p))) | (4u << (4 * p)));
          }
        }
        if (col0 < a.cols && rowbase < a.rows) {
          uint8_t* cdst = a.codes_c + (size_t)col0 * (a.rows >> 1) + (rowbase >> 1);
#pragma unroll
          for (int k = 0; k < 8; ++k) *reinterpret_cast<uint32_t*>(cdst + (size_t)k * (a.rows >> 1)) = out[k];
          const uint32_t kb = rowbase >> 4;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            a.scales_c[sf_offset(col0 + 4 * hsel + kk, kb, a.atoms_k_c)] = static_cast<uint8_t>(sb_mine[kk]);
        }
      }

      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == STAGES) stage = 0, phase ^= 1;
    }
  }
  __syncthreads();
  if (*abort_flag) {  // a wait expired: let copies still in flight land first
    if (threadIdx.x == 0) drain_pause();
    __syncthreads();
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
  for (int i = 0; i < 8; ++i) v[i] = (i8 + i < n) ? sr_round(in[i8 + i], 0x47800000u | rnd[i8 + i]) : 0.0f;
  const uint32_t c = e2m1x8(v);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i8 + i < n) e2m1[i8 + i] = (c >> (4 * i)) & 0xFu;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
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
  if (e != cudaSuccess) return e;
  const int grid = grid_for(nchunks, 256 * 4, num_sms * 8);
  amax_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), cpr, nchunks, ld,
                                   reinterpret_cast<unsigned int*>(out));
  count_launch();
  return cudaGetLastError();
}

template <bool ROW, bool COL, bool SR, bool CLIP>
static cudaError_t launch_qd(const CUtensorMap& tm, const DualQuantArgs& a, int num_sms, cudaStream_t s) {
  using namespace qd;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(quantize_dual_kernel<ROW, COL, SR, CLIP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_BYTES);
  });
  if (attr != cudaSuccess) return attr;
  const uint32_t slots = (uint32_t)num_sms * CTAS_PER_SM;
  const uint32_t grid = a.num_tiles < slots ? a.num_tiles : slots;
  quantize_dual_kernel<ROW, COL, SR, CLIP><<<grid, THREADS, SMEM_BYTES, s>>>(tm, a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ld, bool sr, uint64_t seed,
                                 uint32_t stream_r, uint32_t stream_c, const float* amax, const QOut* row_out,
                                 const QOut* col_out, cudaStream_t s, const uint32_t* clip, int num_sms) {
  DualQuantArgs a{};
  a.clip = clip;
  a.rows = static_cast<uint32_t>(rows);
  a.cols = static_cast<uint32_t>(cols);
  a.cpr = static_cast<uint32_t>(cols / 8);
  a.tiles_c = static_cast<uint32_t>((cols + qd::TILE - 1) / qd::TILE);
  a.num_tiles = a.tiles_c * static_cast<uint32_t>((rows + qd::TILE - 1) / qd::TILE);
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
  // x as 128-row x 64-column boxes with the 128-byte swizzle
  CUtensorMap tm;
  if (!make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)cols, (uint64_t)rows, (uint64_t)ld * 2,
                    qd::BOX_C, qd::TILE, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const bool R = row_out != nullptr, C = col_out != nullptr;
  cudaError_t e;
  if (clip) {  // the clipped form: both orientations, RTN
    if (!(R && C) || sr) return cudaErrorInvalidValue;
    e = launch_qd<true, true, false, true>(tm, a, num_sms, s);
  } else if (R && C) {
    e = sr ? launch_qd<true, true, true, false>(tm, a, num_sms, s) : launch_qd<true, true, false, false>(tm, a, num_sms, s);
  } else if (C) {
    e = sr ? launch_qd<false, true, true, false>(tm, a, num_sms, s) : launch_qd<false, true, false, false>(tm, a, num_sms, s);
  } else {
    e = sr ? launch_qd<true, false, true, false>(tm, a, num_sms, s) : launch_qd<true, false, false, false>(tm, a, num_sms, s);
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
