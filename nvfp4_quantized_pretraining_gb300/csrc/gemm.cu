// Tensor-core GEMMs for the NVFP4 linear projection (sm_103a, tcgen05):
//
//  * gemm_nvf4_kernel: C = S_tA S_tB * (A . SFA)(B . SFB)^T + beta * P Q^T.
//    The NVFP4 residual product and the BF16 low-rank branch of the LoRA-SVD
//    weight split (Full-Stack FP4, section 2.1, "Mechanism":
//    W = W_res + beta L2 L1, the subspace in BF16, the residual in NVFP4) are
//    accumulated in two tensor-memory accumulators of the same output tile and
//    combined in the epilogue.
//  * branch_factor_kernel: P = bf16(X L^T), the skinny BF16 product that
//    feeds the branch (M x r, r <= 64).
//
// Both are warp-specialised: warp 0 issues TMA loads into a ring of shared
// memory stages, warp 1 issues tcgen05.mma from one thread (accumulators in
// TMEM), warps 2..5 drain TMEM with tcgen05.ld and write the output.  Every
// mbarrier wait is bounded (FP4_ERR_TIMEOUT in the status word on expiry).
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Block-scaled NVFP4 GEMM
// ---------------------------------------------------------------------------
namespace g4 {
constexpr int BM = 128;             // rows of A per tile (one tcgen05 M=128 MMA)
constexpr int BN = 128;             // rows of B per tile (MMA N)
constexpr int BK = 256;             // K elements per stage (128 bytes of E2M1 per row)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK / 2;              // 16 KB
constexpr int B_BYTES = BN * BK / 2;              // 16 KB
constexpr int SF_ATOM = 512;                      // 128 rows x 4 scales
constexpr int SFA_BYTES = (BM / 128) * (BK / 64) * SF_ATOM;  // 2 KB
constexpr int SFB_BYTES = (BN / 128) * (BK / 64) * SF_ATOM;  // 2 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int BR_K = 64;                          // branch rank padded to 64 (128-byte BF16 rows)
constexpr int P_BYTES = BM * BR_K * 2;            // 16 KB, fits the A slot
constexpr int Q_BYTES = BN * BR_K * 2;            // 16 KB, fits the B slot
// tensor memory columns
constexpr uint32_t TM_ACC = 0;                    // 2 x BN accumulators (double buffered)
constexpr uint32_t TM_BR = 2 * BN;                // BN branch accumulator
constexpr uint32_t TM_SF = 3 * BN;                // STAGES x (SFA 16 + SFB 16) scale columns
constexpr uint32_t TM_COLS = 512;
static_assert(TM_SF + STAGES * (4 * (BK / 64) * (BM / 128) + 4 * (BK / 64) * (BN / 128)) <= TM_COLS, "TMEM");
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
}  // namespace g4

struct GemmParams {
  const uint8_t* a_scales;
  const uint8_t* b_scales;
  const float* a_scale;
  const float* b_scale;
  uint32_t M, N, K;
  uint32_t atoms_k;  // K / 64
  uint32_t num_m, num_n;
  int r;
  float beta;
  void* C;
  int c_f32;
  int64_t ldc;
};

__global__ void __launch_bounds__(g4::NUM_THREADS, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_p, const __grid_constant__ CUtensorMap tmap_q,
                     const GemmParams p) {
  using namespace g4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* br_empty = acc_empty + 2;
  uint64_t* done_bar = br_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(br_empty, 4);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    if (p.r > 0) {
      prefetch_tmap(&tmap_p);
      prefetch_tmap(&tmap_q);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t num_tiles = p.num_m * p.num_n;
  const uint32_t num_k = (p.K + BK - 1) / BK;
  const bool has_branch = p.r > 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      int armed[STAGES];
      uint32_t armed_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const uint32_t mb = tile % p.num_m, nb = tile / p.num_m;
        const uint32_t n_iter = num_k + (has_branch ? 1 : 0);
        for (uint32_t it = 0; it < n_iter; ++it) {
          if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) {
            ok = false;
            break;
          }
          armed[stage] = 0;
          uint8_t* sA = smem + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sSFA = sB + B_BYTES;
          uint8_t* sSFB = sSFA + SFA_BYTES;
          if (it < num_k) {
            const uint32_t krem = p.K - it * BK;
            const uint32_t nk = krem >= (uint32_t)BK ? BK / 64 : krem / 64;
            mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + 2 * nk * SF_ATOM);
            tma_load_2d(sA, &tmap_a, &full[stage], (int32_t)(it * (BK / 2)), (int32_t)(mb * BM));
            tma_load_2d(sB, &tmap_b, &full[stage], (int32_t)(it * (BK / 2)), (int32_t)(nb * BN));
            bulk_load(sSFA, p.a_scales + ((size_t)mb * p.atoms_k + it * (BK / 64)) * SF_ATOM, nk * SF_ATOM,
                      &full[stage]);
            bulk_load(sSFB, p.b_scales + ((size_t)nb * p.atoms_k + it * (BK / 64)) * SF_ATOM, nk * SF_ATOM,
                      &full[stage]);
          } else {
            mbar_arrive_expect_tx(&full[stage], P_BYTES + Q_BYTES);
            tma_load_2d(sA, &tmap_p, &full[stage], 0, (int32_t)(mb * BM));
            tma_load_2d(sB, &tmap_q, &full[stage], 0, (int32_t)(nb * BN));
          }
          armed[stage] = 1;
          armed_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // let copies already in flight land before the CTA may exit
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) mbar_wait(&full[s], armed_phase[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_nvf4(BM, BN);
      const uint32_t idesc_br = idesc_bf16(BM, BN);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      uint32_t t = 0;
      for (uint32_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++t) {
        const uint32_t buf = t & 1;
        if (!mbar_wait(&acc_empty[buf], ((t >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + TM_ACC + buf * BN;
        for (uint32_t it = 0; it < num_k; ++it) {
          if (*abort_flag || !mbar_wait(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sB = sA + A_BYTES;
          const uint32_t sSFA = sB + B_BYTES;
          const uint32_t sSFB = sSFA + SFA_BYTES;
          const uint32_t krem = p.K - it * BK;
          const uint32_t nk = krem >= (uint32_t)BK ? BK / 64 : krem / 64;
          const uint32_t tsfa = tmem + TM_SF + stage * 32;
          const uint32_t tsfb = tsfa + 16;
          for (uint32_t kk = 0; kk < nk; ++kk) {
            tc_cp_32x128b_warpx4(tsfa + kk * 4, smem_desc(sSFA + kk * SF_ATOM, 0, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4(tsfb + kk * 4, smem_desc(sSFB + kk * SF_ATOM, 0, 128, kSwizzleNone));
          }
          for (uint32_t kk = 0; kk < nk; ++kk) {
            mma_nvf4(d_tmem, smem_desc(sA + kk * 32, 16, 1024, kSwizzle128B),
                     smem_desc(sB + kk * 32, 16, 1024, kSwizzle128B), idesc, tsfa + kk * 4, tsfb + kk * 4,
                     (it | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        if (has_branch) {
          if (!mbar_wait(br_empty, (t & 1) ^ 1)) { ok = false; break; }
          if (*abort_flag || !mbar_wait(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sB = sA + A_BYTES;
          const uint32_t nkb = (uint32_t)(p.r + 15) / 16;
          for (uint32_t kk = 0; kk < nkb; ++kk)
            mma_bf16(tmem + TM_BR, smem_desc(sA + kk * 32, 16, 1024, kSwizzle128B),
                     smem_desc(sB + kk * 32, 16, 1024, kSwizzle128B), idesc_br, kk != 0);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        tc_commit(&acc_full[buf]);
      }
      if (!ok) *abort_flag = 1;
      // every tcgen05 operation issued above completes before TMEM is released
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const uint32_t quad = warp & 3;  // TMEM lanes this warp may access
    const float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
    const float beta = p.beta;
    uint32_t t = 0;
    for (uint32_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t) {
      const uint32_t mb = tile % p.num_m, nb = tile / p.num_m;
      const uint32_t buf = t & 1;
      if (*abort_flag || !mbar_wait(&acc_full[buf], (t >> 1) & 1)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t row = mb * BM + quad * 32 + lane;
      const uint32_t lane_off = (quad * 32) << 16;
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t acc[32], br[32];
        tmem_ld_32x32b_x32(tmem + lane_off + TM_ACC + buf * BN + j * 32, acc);
        if (has_branch) tmem_ld_32x32b_x32(tmem + lane_off + TM_BR + j * 32, br);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = __fmul_rn(alpha, __uint_as_float(acc[i]));
          if (has_branch) v[i] = __fadd_rn(v[i], __fmul_rn(beta, __uint_as_float(br[i])));
        }
        const size_t col = (size_t)nb * BN + j * 32;
        if (p.c_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.C) + row * p.ldc + col);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) + row * p.ldc + col);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * h], v[8 * i + 2 * h + 1]);
              w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acc_empty[buf]);
        if (has_branch) mbar_arrive(br_empty);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Branch factor P = bf16(X L^T), BF16 tcgen05 GEMM with N = r.
// ---------------------------------------------------------------------------
namespace bf {
constexpr int BM = 128;
constexpr int BK = 64;              // BF16 elements per stage (128-byte rows)
constexpr int STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = 64 * BK * 2;  // 8 KB (r <= 64 rows)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
}  // namespace bf

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__global__ void __launch_bounds__(bf::NUM_THREADS, 1)
    branch_factor_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_l,
                         uint32_t K, int r, __nv_bfloat16* __restrict__ P) {
  using namespace bf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* done_bar = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
  const uint32_t num_k = (K + BK - 1) / BK;
  const uint32_t m0 = blockIdx.x * BM;
  const uint32_t l_bytes = (uint32_t)r * BK * 2;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int armed[STAGES];
      uint32_t armed_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t it = 0; it < num_k; ++it) {
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        uint8_t* sB = sA + A_BYTES;
        mbar_arrive_expect_tx(&full[stage], A_BYTES + l_bytes);
        tma_load_2d(sA, &tmap_x, &full[stage], (int32_t)(it * BK), (int32_t)m0);
        tma_load_2d(sB, &tmap_l, &full[stage], (int32_t)(it * BK), 0);
        armed[stage] = 1;
        armed_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        for (int s = 0; s < STAGES; ++s)
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
        const uint32_t krem = K - it * BK;
        const uint32_t nk = krem >= (uint32_t)BK ? BK / 16 : krem / 16;
        for (uint32_t kk = 0; kk < nk; ++kk)
          mma_bf16(tmem, smem_desc(sA + kk * 32, 16, 1024, kSwizzle128B),
                   smem_desc(sB + kk * 32, 16, 1024, kSwizzle128B), idesc, (it | kk) != 0);
        tc_commit(&empty[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (ok) tc_commit(acc_full);
      else *abort_flag = 1;
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
  } else {
    const uint32_t quad = warp & 3;
    if (!*abort_flag && mbar_wait(acc_full, 0)) {
      tc_fence_after();
      const uint32_t row = m0 + quad * 32 + lane;
      for (int j = 0; j < r; j += 16) {
        uint32_t acc[16];
        tmem_ld_32x32b_x16(tmem + ((quad * 32) << 16) + j, acc);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(acc[2 * h]), __uint_as_float(acc[2 * h + 1]));
          w[h] = *reinterpret_cast<uint32_t*>(&b2);
        }
        uint4* dst = reinterpret_cast<uint4*>(P + (size_t)row * r + j);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      tc_fence_before();
    } else {
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------
// BF16 transpose (small factor matrices)
// ---------------------------------------------------------------------------
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ in, uint32_t rows, uint32_t cols,
                                      uint16_t* __restrict__ out) {
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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 2-D row-major tensor map: inner dimension `inner` elements, `outer` rows,
// row pitch `pitch_bytes`, box inner x outer, 128-byte swizzle.
static bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_nvf4(const GemmArgs& g, int num_sms, cudaStream_t s) {
  using namespace g4;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ta, tb, tp, tq;
  if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a_codes, g.K / 2, g.M, g.K / 2, BK / 2, BM) ||
      !make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b_codes, g.K / 2, g.N, g.K / 2, BK / 2, BN))
    return cudaErrorInvalidValue;
  if (g.r > 0) {
    if (!make_tmap(&tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.P, g.r, g.M, (uint64_t)g.r * 2, BR_K, BM) ||
        !make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.Q, g.r, g.N, (uint64_t)g.r * 2, BR_K, BN))
      return cudaErrorInvalidValue;
  } else {
    tp = ta;
    tq = tb;
  }
  GemmParams p;
  p.a_scales = static_cast<const uint8_t*>(g.a_scales);
  p.b_scales = static_cast<const uint8_t*>(g.b_scales);
  p.a_scale = g.a_scale;
  p.b_scale = g.b_scale;
  p.M = (uint32_t)g.M;
  p.N = (uint32_t)g.N;
  p.K = (uint32_t)g.K;
  p.atoms_k = (uint32_t)(g.K / 64);
  p.num_m = (uint32_t)(g.M / BM);
  p.num_n = (uint32_t)(g.N / BN);
  p.r = g.r;
  p.beta = g.beta;
  p.C = g.C;
  p.c_f32 = g.c_f32;
  p.ldc = g.ldc;
  const uint32_t tiles = p.num_m * p.num_n;
  const int grid = (int)(tiles < (uint32_t)num_sms ? tiles : (uint32_t)num_sms);
  gemm_nvf4_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, tp, tq, p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_branch_factor(const void* X, int64_t M, int64_t K, int64_t ldx, const void* L, int r, void* P,
                                 int num_sms, cudaStream_t s) {
  using namespace bf;
  (void)num_sms;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(branch_factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tx, tl;
  if (!make_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, (uint64_t)ldx * 2, BK, BM) ||
      !make_tmap(&tl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L, K, r, (uint64_t)K * 2, BK, (uint32_t)r))
    return cudaErrorInvalidValue;
  const int grid = (int)(M / BM);
  branch_factor_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tx, tl, (uint32_t)K, r,
                                                             static_cast<__nv_bfloat16*>(P));
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, void* out, cudaStream_t s) {
  dim3 block(32, 8);
  dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  transpose_bf16_kernel<<<grid, block, 0, s>>>(static_cast<const uint16_t*>(in), (uint32_t)rows, (uint32_t)cols,
                                               static_cast<uint16_t*>(out));
  count_launch();
  return cudaGetLastError();
}

cudaError_t gemm_status_read_clear(unsigned int* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace nvfp4
