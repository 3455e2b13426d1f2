// The branch factor of the LoRA-SVD split (Full-Stack FP4, section 2.1, "Mechanism": the
// subspace kept in BF16): P = bf16(X L^T), the skinny BF16 product (M x r, r <= 64) that feeds the
// block-scaled GEMM's branch, with max |X| taken from the same read of X; and the BF16 transpose of
// the small factor matrices.
//
// branch_factor_kernel is warp-specialised like the GEMMs: a TMA producer warp fills a ring of
// shared-memory stages, one thread issues tcgen05.mma (kind::f16, accumulator in TMEM), four warps
// fold the landed X tiles into max |X| and then drain the accumulator.  Every mbarrier wait is
// bounded (FP4_ERR_TIMEOUT in the status word on expiry).
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Branch factor P = bf16(X L^T), BF16 tcgen05 GEMM with N = r.
// ---------------------------------------------------------------------------
namespace bf {
constexpr int BM = 128;
constexpr int BOX = 64;                 // BF16 columns per TMA box (128-byte rows, 128-byte swizzle)
constexpr int BOXES = 2;                // boxes per stage, adjacent in K: 256 contiguous bytes per row
constexpr int BK = BOX * BOXES;         // BF16 elements of K per stage
constexpr int STAGES = 4;               // one CTA per SM
constexpr int SPLIT_STAGES = 2;         // two CTAs per SM (K split over a CTA pair)
constexpr int XBOX_BYTES = BM * BOX * 2;  // 16 KB
constexpr int LBOX_BYTES = 64 * BOX * 2;  // 8 KB (r <= 64 rows)
constexpr int A_BYTES = BOXES * XBOX_BYTES;
constexpr int STAGE_BYTES = A_BYTES + BOXES * LBOX_BYTES;  // 48 KB
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
}  // namespace bf

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Without SPLIT, CTA i takes the h rows [i h, i h + h) of X (h <= 128; the X tensor map's box is h
// rows high): with h = ceil(M / SMs) every SM streams the same share of X, one CTA each.  The MMA
// still runs M = 128: rows h..127 of a stage hold whatever an earlier stage left there, and the
// results of those rows are neither stored nor folded into max |X|.
// SPLIT: a cluster of two CTAs shares one 128-row block, each taking half of the K stages
// (for M too small for h >= 48 rows per SM; 4 stages so that two CTAs fit per SM).  Rank 1
// hands its FP32 partial sum to rank 0 through distributed shared memory and rank 0 writes
// P = bf16(partial_0 + partial_1): a fixed order, so the result is deterministic.
template <bool SPLIT>
__global__ void __launch_bounds__(bf::NUM_THREADS, 1)
    branch_factor_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_l,
                         uint32_t M, uint32_t K, uint32_t h, int r, __nv_bfloat16* P,
                         unsigned int* amax_out) {
  using namespace bf;
  pdl_trigger();
  constexpr int NST = SPLIT ? SPLIT_STAGES : STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * STAGE_BYTES);
  uint64_t* empty = full + NST;
  uint64_t* acc_full = empty + NST;
  uint64_t* done_bar = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = SPLIT ? cluster_ctarank() : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], amax_out ? 1 + 4 : 1);  // the MMA commit (+ the 4 amax warps)
    }
    mbar_init(acc_full, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // (the set-up above touches no global data)
  const uint32_t num_k_all = (K + BK - 1) / BK;
  const uint32_t kh = SPLIT ? (num_k_all + 1) / 2 : num_k_all;
  const uint32_t k_begin = rank * kh;                 // this CTA's first K stage
  const uint32_t num_k = SPLIT ? min(kh, num_k_all - k_begin) : num_k_all;  // >= 1: the host splits only K >= 2 stages
  const uint32_t m0 = SPLIT ? (blockIdx.x >> 1) * BM : blockIdx.x * h;
  const uint32_t l_bytes = (uint32_t)r * BOX * 2;  // one L box
  const uint32_t x_bytes = h * BOX * 2;            // one X box (h rows; rows past M arrive zero-filled)

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int armed[NST];
      uint32_t armed_phase[NST];
      for (int s = 0; s < NST; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        uint8_t* sB = sA + A_BYTES;
        // both boxes of X back to back (256 contiguous bytes of each row), then both of L;
        // a box past K arrives zero-filled
        mbar_arrive_expect_tx(&full[stage], BOXES * (x_bytes + l_bytes));
        const int32_t kx = (int32_t)((k_begin + it) * BK);
#pragma unroll
        for (int b = 0; b < BOXES; ++b)
          tma_load_2d(sA + b * XBOX_BYTES, &tmap_x, &full[stage], kx + b * BOX, (int32_t)m0);
#pragma unroll
        for (int b = 0; b < BOXES; ++b) tma_load_2d(sB + b * LBOX_BYTES, &tmap_l, &full[stage], kx + b * BOX, 0);
        armed[stage] = 1;
        armed_phase[stage] = phase;
        if (++stage == NST) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        for (int s = 0; s < NST; ++s)
          if (armed[s]) mbar_wait(&full[s], armed_phase[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, (uint32_t)r);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait(&full[stage], phase)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sB = sA + A_BYTES;
        const uint32_t krem = K - (k_begin + it) * BK;
        const uint32_t nk = krem >= (uint32_t)BK ? BK / 16 : krem / 16;
        for (uint32_t kk = 0; kk < nk; ++kk) {  // K step kk: box kk / 4, +32 bytes per step inside it
          const uint32_t b = kk >> 2, o = (kk & 3) * 32;
          mma_bf16(tmem, smem_desc(sA + b * XBOX_BYTES + o, 16, 1024, kSwizzle128B),
                   smem_desc(sB + b * LBOX_BYTES + o, 16, 1024, kSwizzle128B), idesc, (it | kk) != 0);
        }
        tc_commit(&empty[stage]);
        if (++stage == NST) stage = 0, phase ^= 1;
      }
      if (ok) tc_commit(acc_full);
      else *abort_flag = 1;
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
  }
  // warps 2..5: amax of the landed tiles, then the accumulator
  uint32_t accr[4][16];  // SPLIT: this CTA's partial sum, row quad * 32 + lane, columns 16j .. 16j + 15
  const uint32_t quad = warp & 3;
  if (warp >= 2) {
    if (amax_out) {
      // fold every landed X tile into max |x| while the MMAs consume it: the tensor scale of X
      // comes out of this read of X (integer max of the |bf16| patterns, as the standalone
      // amax kernel takes it; zero padding past K does not change it)
      const int t = (warp - 2) * 32 + lane;
      uint32_t m = 0, stage = 0, phase = 0;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait_warp(&full[stage], phase)) {
          *abort_flag = 1;
          break;
        }
        const uint4* tile = reinterpret_cast<const uint4*>(smem + stage * STAGE_BYTES);
#pragma unroll
        for (int i = 0; i < A_BYTES / 16 / 128; ++i) {  // both X boxes, the h rows landed in each
          const int u = t + 128 * i;  // 16-byte unit: box u / 1024, row (u % 1024) / 8
          if ((uint32_t)((u & 1023) >> 3) >= h) continue;
          const uint4 v = tile[u];
          m = __vmaxu2(m, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                   __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == NST) stage = 0, phase ^= 1;
      }
      m = max(m & 0xFFFFu, m >> 16);
      m = __reduce_max_sync(0xFFFFFFFFu, m);
      if (lane == 0 && m != 0) atomicMax(amax_out, m << 16);
    }
    if (!*abort_flag && mbar_wait_warp(acc_full, 0)) {
      tc_fence_after();
      const uint32_t row = m0 + quad * 32 + lane;
      const bool mine = quad * 32 + lane < h && row < M;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (16 * j < r) {
          tmem_ld_32x32b_x16(tmem + ((quad * 32) << 16) + 16 * j, accr[j]);
          tmem_ld_wait16(accr[j]);
        }
      }
      tc_fence_before();
      if (!SPLIT && mine) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (16 * j >= r) break;
          uint32_t w[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            __nv_bfloat162 b2 =
                __floats2bfloat162_rn(__uint_as_float(accr[j][2 * h]), __uint_as_float(accr[j][2 * h + 1]));
            w[h] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(P + (size_t)row * r + 16 * j);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    } else {
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (SPLIT) {
    // rank 0's stages are idle once both pipelines are done: rank 1 writes its partial there
    // (row-major, rows padded to r + 4 floats so that 16-byte stores of 8 lanes hit distinct banks)
    const uint32_t pitch = (uint32_t)r + 4;
    float* partial = reinterpret_cast<float*>(smem);
    cluster_sync();
    if (rank == 1 && warp >= 2 && !*abort_flag) {
      const uint32_t rl = quad * 32 + lane;
      const uint32_t dst0 = mapa_shared(smem_u32(partial + rl * pitch), 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (16 * j < r) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst0 + (16 * j + 4 * q) * 4),
                         "r"(accr[j][4 * q]), "r"(accr[j][4 * q + 1]), "r"(accr[j][4 * q + 2]),
                         "r"(accr[j][4 * q + 3])
                         : "memory");
        }
      }
    }
    cluster_sync();  // release / acquire: rank 1's partial is visible to rank 0
    if (rank == 0 && warp >= 2 && !*abort_flag) {
      const uint32_t rl = quad * 32 + lane;
      const uint32_t row = m0 + rl;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (16 * j >= r) break;
        uint32_t w[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 o = *reinterpret_cast<const float4*>(partial + rl * pitch + 16 * j + 4 * q);
          const float s0 = __fadd_rn(__uint_as_float(accr[j][4 * q]), o.x);
          const float s1 = __fadd_rn(__uint_as_float(accr[j][4 * q + 1]), o.y);
          const float s2 = __fadd_rn(__uint_as_float(accr[j][4 * q + 2]), o.z);
          const float s3 = __fadd_rn(__uint_as_float(accr[j][4 * q + 3]), o.w);
          __nv_bfloat162 b0 = __floats2bfloat162_rn(s0, s1), b1 = __floats2bfloat162_rn(s2, s3);
          w[2 * q] = *reinterpret_cast<uint32_t*>(&b0);
          w[2 * q + 1] = *reinterpret_cast<uint32_t*>(&b1);
        }
        uint4* dst = reinterpret_cast<uint4*>(P + (size_t)row * r + 16 * j);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
  if (*abort_flag) {  // a wait expired: let copies still in flight land first
    if (threadIdx.x == 0) drain_pause();
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------
// BF16 transpose (small factor matrices)
// ---------------------------------------------------------------------------
__global__ void transpose_bf16_kernel(const uint16_t* in, uint32_t rows, uint32_t cols,
                                      uint16_t* out) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint16_t t[32][33];
  const uint32_t c = blockIdx.x * 32 + threadIdx.x;
  for (uint32_t i = threadIdx.y; i < 32; i += blockDim.y) {
    const uint32_t r = blockIdx.y * 32 + i;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[(size_t)r * cols + c];
  }
  __syncthreads();
  const uint32_t r2 = blockIdx.y * 32 + threadIdx.x;
  for (uint32_t i = threadIdx.y; i < 32; i += blockDim.y) {
    const uint32_t c2 = blockIdx.x * 32 + i;
    if (r2 < rows && c2 < cols) out[(size_t)c2 * rows + r2] = t[threadIdx.x][i];
  }
}

cudaError_t launch_branch_factor(const void* X, int64_t M, int64_t K, int64_t ldx, const void* L, int r, void* P,
                                 float* amax_out, int num_sms, cudaStream_t s) {
  using namespace bf;
  constexpr int kSmemSplit = SPLIT_STAGES * STAGE_BYTES + 1024 + 256;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(branch_factor_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(branch_factor_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemSplit);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int blocks = (int)(M / BM);
  const int num_k = (int)((K + BK - 1) / BK);
  // rows per CTA with one CTA per SM; below 48 the re-read of L (r rows per stage, from L2) would
  // outweigh X in each SM's intake, and the K split over CTA pairs takes over
  const uint32_t h_rows = (uint32_t)((M + num_sms - 1) / num_sms);
  const bool by_rows = h_rows >= 48 && h_rows <= (uint32_t)BM;
  const bool split = !by_rows && blocks < num_sms && num_k >= 2;
  const uint32_t h = by_rows ? h_rows : (uint32_t)BM;
  CUtensorMap tx, tl;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, (uint64_t)ldx * 2, BOX, h,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L, K, r, (uint64_t)K * 2, BOX, (uint32_t)r,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (amax_out) {
    const cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), s);
    pdl_chain_break();
    if (e != cudaSuccess) return e;
  }
  __nv_bfloat16* Pb = static_cast<__nv_bfloat16*>(P);
  unsigned int* am = reinterpret_cast<unsigned int*>(amax_out);
  cudaError_t e;
  if (split) {
    // fewer row blocks than SMs: two CTAs (a cluster) per row block, half of K each
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    cfg.gridDim = dim3(2 * blocks);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = kSmemSplit;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = g_pdl_chain ? 2 : 1;  // programmatic launch only after one of the library's kernels
    e = cudaLaunchKernelEx(&cfg, branch_factor_kernel<true>, tx, tl, (uint32_t)M, (uint32_t)K, (uint32_t)BM, r, Pb,
                           am);
    g_pdl_chain = e == cudaSuccess;
  } else {
    const unsigned grid = (unsigned)((M + h - 1) / h);
    e = launch_pdl(branch_factor_kernel<false>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, tx, tl, (uint32_t)M,
                   (uint32_t)K, h, r, Pb, am);
  }
  count_launch();
  return e;
}

cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, void* out, cudaStream_t s) {
  dim3 block(32, 8);
  dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  const cudaError_t e = launch_pdl(transpose_bf16_kernel, grid, block, 0, s, static_cast<const uint16_t*>(in),
                                   (uint32_t)rows, (uint32_t)cols, static_cast<uint16_t*>(out));
  count_launch();
  return e;
}

}  // namespace nvfp4
