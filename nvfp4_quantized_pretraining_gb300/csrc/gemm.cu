// Tensor-core GEMMs for the NVFP4 linear projection (sm_103a, tcgen05):
//
//  * gemm_nvf4_pair_kernel (M, N multiples of 256) and gemm_nvf4_kernel
//    (multiples of 128): C = alpha * (A B^T + P~ Q^T), alpha = S_tA S_tB, with
//    A, B NVFP4 (E2M1 codes, UE4M3 scales per 16 elements) and the BF16
//    low-rank branch of the LoRA-SVD weight split (Full-Stack FP4, section
//    2.1, "Mechanism": W = W_res + beta L2 L1, the subspace in BF16, the
//    residual in NVFP4) accumulated into the same tensor-memory accumulator
//    after rescaling P~ = bf16(P * beta / alpha), so C is rounded once.
//  (the branch factor P that feeds it is computed in branch.cu.)
//
// All are warp-specialised: a TMA producer warp fills a ring of shared-memory
// stages, one thread issues tcgen05.mma (accumulators in TMEM), "scale" warps
// stage block scales into TMEM, epilogue warps drain TMEM with tcgen05.ld.
// Every mbarrier wait is bounded (FP4_ERR_TIMEOUT in the status word on expiry).
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Block-scaled NVFP4 GEMM, one CTA per 128 x 128 tile (shapes whose M or N is
// an odd multiple of 128; multiples of 256 take the CTA-pair kernel below)
//
// 256 K elements per pipeline stage; each CTA loads its own A and B tiles and
// their block scales with plain TMA / bulk copies and walks its tiles
// persistently.  Block scales reach tensor memory through tcgen05.st from four
// "scale" warps (one per TMEM lane quadrant) instead of tcgen05.cp on the
// tensor pipe.  For output rows m in lane quadrant q = m / 32, the MMA reads
// the scales of A row m from lane m, column (base + q), and the scales of B
// row n from lane 32q + n % 32, column (base + n / 32); the byte is the
// 16-element block within the 64-wide K step.  So A scales are written once
// (the diagonal) and B scales once per quadrant.
// ---------------------------------------------------------------------------
namespace g4 {
constexpr int BM = 128;             // rows of A per tile (tcgen05 M=128)
constexpr int BN = 128;             // rows of B per tile (MMA N)
constexpr int BK = 256;             // K elements per stage (128 bytes of E2M1 per row)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK / 2;              // 16 KB
constexpr int B_BYTES = BN * BK / 2;              // 16 KB
constexpr int SF_ATOM = 512;                      // 128 rows x 4 scales
constexpr int SFA_BYTES = (BK / 64) * SF_ATOM;    // 2 KB (4 atoms)
constexpr int SFB_BYTES = (BK / 64) * SF_ATOM;    // 2 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int BR_K = 64;                          // branch rank padded to 64 (128-byte BF16 rows)
constexpr int P_BYTES = BM * BR_K * 2;            // 16 KB, fits the A slot
constexpr int Q_BYTES = BN * BR_K * 2;            // 16 KB, fits the B slot
// tensor memory columns
constexpr uint32_t TM_ACC = 0;                    // 2 x BN accumulators (double buffered)
constexpr uint32_t TM_SF = 2 * BN;                // per stage: SFA 16 + SFB 16 columns
constexpr uint32_t TM_SF_STAGE = 32;
constexpr uint32_t TM_COLS = 512;
static_assert(TM_SF + STAGES * TM_SF_STAGE <= TM_COLS, "TMEM budget");
// warps: 0 TMA producer, 1 MMA issuer, 2..5 scale stagers, 6..9 epilogue
constexpr int NUM_THREADS = 320;
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
  // 2-SM kernel tile order: 0 walks M fastest, 1 walks N fastest.  The larger operand is walked
  // slowest so that it streams from DRAM once while the smaller one stays resident in L2.
  int raster_n;
  // 2-SM kernel, split tail: tiles [0, dp_tiles) are computed whole, round-robin over the CTA
  // pairs; when sk_split = S > 0, each of the remaining tiles is cut into S pieces along K, one
  // per pair, whose FP32 partial accumulators go to sk_ws (256 x 256 floats per piece) for
  // gemm_splitk_reduce_kernel to sum.  sk_split = 0: every tile whole (dp_tiles unused).
  uint32_t dp_tiles;
  uint32_t sk_split;
  float* sk_ws;
  // 2-SM kernel: P holds P~ already (folded before the launch), so the branch stage is loaded by
  // TMA like any operand stage (P and Q both complete on the leader's barrier) and the scale
  // warps leave it alone; 0: they fold P into P~ in shared memory
  int p_folded;
  // 2-SM kernel: B's scales by one TMA box per stage (tmap_sfb); 0 (K < 256): two bulk copies
  int sfb_tma;
};

__global__ void __launch_bounds__(g4::NUM_THREADS, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_p, const __grid_constant__ CUtensorMap tmap_q,
                     const GemmParams p) {
  pdl_trigger();
  using namespace g4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_ready = empty + STAGES;
  uint64_t* acc_full = sf_ready + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
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
  pdl_wait();  // (the set-up above touches no global data)

  // 128 x 128 output tiles, M fastest; the CTAs walk them persistently
  const uint32_t num_tiles = p.num_m * p.num_n;
  const uint32_t num_k = (p.K + BK - 1) / BK;
  const bool has_branch = p.r > 0;
  const uint32_t n_iter = num_k + (has_branch ? 1 : 0);
  float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
  if (alpha == 0.0f) alpha = 1.0f;  // an all-zero operand contributes exact zeros

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      int armed[STAGES];
      uint32_t armed_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = 0, armed_phase[s] = 0;
      bool ok = true;
      for (uint32_t mt = blockIdx.x; mt < num_tiles && ok; mt += gridDim.x) {
        const uint32_t mb = mt % p.num_m, nb = mt / p.num_m;
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
            const uint32_t nk = krem >= (uint32_t)BK ? BK / 64 : krem / 64;  // 64-wide K steps in this stage
            mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + 2 * nk * SF_ATOM);
            const int32_t kx = (int32_t)(it * (BK / 2));
            tma_load_2d(sA, &tmap_a, &full[stage], kx, (int32_t)(mb * BM));
            tma_load_2d(sB, &tmap_b, &full[stage], kx, (int32_t)(nb * BN));
            // the scale atoms of this stage: nk consecutive 512-byte atoms per operand
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
      // One thread issues every MMA, so the loop is kept lean: descriptors are
      // a base plus a per-stage constant (the start-address field counts 16-byte
      // units), a full 256-wide stage is four unrolled MMAs at +32-byte K
      // offsets, and the abort flag is only consulted at tile boundaries.
      const uint32_t idesc = idesc_nvf4(BM, BN);
      const uint32_t idesc_br = idesc_bf16(BM, BN);
      const uint64_t adesc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
      const uint64_t bdesc0 = adesc0 + (A_BYTES >> 4);
      constexpr uint64_t kStageD = STAGE_BYTES >> 4;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      uint32_t t = 0;
      for (uint32_t mt = blockIdx.x; mt < num_tiles && ok; mt += gridDim.x, ++t) {
        const uint32_t buf = t & 1;
        if (*abort_flag || !mbar_wait(&acc_empty[buf], ((t >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + TM_ACC + buf * BN;
        for (uint32_t it = 0; it < num_k; ++it) {
          if (!mbar_wait(&full[stage], phase) || !mbar_wait(&sf_ready[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + stage * kStageD, bd = bdesc0 + stage * kStageD;
          const uint32_t tsf = tmem + TM_SF + stage * TM_SF_STAGE;
          const uint32_t krem = p.K - it * BK;
          if (krem >= (uint32_t)BK) {
            mma_nvf4(d_tmem, ad, bd, idesc, tsf, tsf + 16, it != 0);
            mma_nvf4(d_tmem, ad + 2, bd + 2, idesc, tsf + 4, tsf + 20, 1);
            mma_nvf4(d_tmem, ad + 4, bd + 4, idesc, tsf + 8, tsf + 24, 1);
            mma_nvf4(d_tmem, ad + 6, bd + 6, idesc, tsf + 12, tsf + 28, 1);
          } else {
            for (uint32_t kk = 0; kk < krem / 64; ++kk)
              mma_nvf4(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, tsf + kk * 4, tsf + 16 + kk * 4, (it | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        if (has_branch) {
          // P~ Q^T (P~ rescaled in shared memory by the scale warps) accumulates onto A B^T
          if (!mbar_wait(&full[stage], phase) || !mbar_wait(&sf_ready[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = adesc0 + stage * kStageD, bd = bdesc0 + stage * kStageD;
          const uint32_t nkb = (uint32_t)(p.r + 15) / 16;
          for (uint32_t kk = 0; kk < nkb; ++kk)
            mma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc_br, 1);
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
  } else if (warp < 6) {
    // ---------------- scale stagers (warps 2..5) ----------------
    const uint32_t quad = warp & 3;
    const uint32_t lane_off = (quad * 32) << 16;
    const float g = __fdiv_rn(p.beta, alpha);
    uint32_t stage = 0, phase = 0;
    for (uint32_t mt = blockIdx.x; mt < num_tiles; mt += gridDim.x) {
      bool ok = true;
      for (uint32_t it = 0; it < n_iter; ++it) {
        // every use of a stage (scale-carrying or not) waits for its data and
        // arrives once on sf_ready, so sf_ready's phase tracks full's
        if (*abort_flag || !mbar_wait_warp(&full[stage], phase)) {
          ok = false;
          break;
        }
        if (it < num_k) {
          const uint32_t krem = p.K - it * BK;
          const uint32_t nk = krem >= (uint32_t)BK ? BK / 64 : krem / 64;
          const uint8_t* sSFA = smem + stage * STAGE_BYTES + A_BYTES + B_BYTES;
          const uint8_t* sSFB = sSFA + SFA_BYTES;
          const uint32_t tsf = TM_SF + stage * TM_SF_STAGE;
          uint32_t wa[16], wb[16];
          // A row m = 32*quad + lane: its 4 scales of K step j sit in atom j at byte
          // (m % 32) * 16 + (m / 32) * 4; the MMA reads them at column tsf + 4j + quad
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t v = (uint32_t)j < nk
                                   ? *reinterpret_cast<const uint32_t*>(sSFA + j * SF_ATOM + lane * 16 + quad * 4)
                                   : 0u;
            wa[4 * j] = wa[4 * j + 1] = wa[4 * j + 2] = wa[4 * j + 3] = v;
          }
          tmem_st_32x32b_x16(tmem + lane_off + tsf, wa);
          // B row n = lane + 32c: its scales of K step j at column tsf + 16 + 4j + c.  The MMA reads
          // B scales for the rows of quadrant q from lanes 32q..32q+31, so every quadrant gets a copy.
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if ((uint32_t)j < nk) v = *reinterpret_cast<const uint4*>(sSFB + j * SF_ATOM + lane * 16);
            wb[4 * j] = v.x;
            wb[4 * j + 1] = v.y;
            wb[4 * j + 2] = v.z;
            wb[4 * j + 3] = v.w;
          }
          tmem_st_32x32b_x16(tmem + lane_off + tsf + 16, wb);
          tmem_st_wait(wb);
          tmem_st_wait(wa);
          tc_fence_before();
        } else if (!p.p_folded) {
          // branch stage: P~ = bf16(P * g) in place (an elementwise map, so the swizzle is irrelevant)
          uint4* tile = reinterpret_cast<uint4*>(smem + stage * STAGE_BYTES);
          const int tid = (warp - 2) * 32 + lane;
#pragma unroll 4
          for (int i = tid; i < P_BYTES / 16; i += 128) {
            uint4 v = tile[i];
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(bf16_lo(w[e]), g), __fmul_rn(bf16_hi(w[e]), g));
              w[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            tile[i] = v;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
  } else {
    // ---------------- epilogue (warps 6..9): C = alpha * acc ----------------
    const uint32_t quad = warp & 3;  // TMEM lanes this warp may access
    uint32_t t = 0;
    for (uint32_t mt = blockIdx.x; mt < num_tiles; mt += gridDim.x, ++t) {
      const uint32_t mb = mt % p.num_m, nb = mt / p.num_m;
      const uint32_t buf = t & 1;
      if (*abort_flag || !mbar_wait_warp(&acc_full[buf], (t >> 1) & 1)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t row = mb * BM + quad * 32 + lane;
      const uint32_t lane_off = (quad * 32) << 16;
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t acc[32];
        tmem_ld_32x32b_x32(tmem + lane_off + TM_ACC + buf * BN + j * 32, acc);
        tmem_ld_wait(acc);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(alpha, __uint_as_float(acc[i]));
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
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
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
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Block-scaled NVFP4 GEMM on CTA pairs (tcgen05 cta_group::2)
//
// A cluster of 2 CTAs on neighbouring SMs computes a 256 x 256 output tile
// with 2-SM MMAs (M=256, N=256, K=64 per instruction).  CTA r of the pair
// holds A rows [128r, 128r+128) and B rows [128r, 128r+128) of the tile in its
// shared memory and receives output rows [128r, 128r+128) x 256 columns in its
// tensor memory; the pair leader (r = 0) issues every MMA.  Each SM thus loads
// half of the B tile and no A rows of its partner: per SM, 38 KB of operands
// and scales per 256-wide K stage feed 16.8 MFLOP, half the bytes per FLOP of
// a 128 x 128 single-SM tile, which is what bounds this GEMM.
//
// The LoRA-SVD branch (Full-Stack FP4, section 2.1: W = W_res + beta L2 L1,
// subspace in BF16) is accumulated into the same TMEM accumulator: with
// alpha = S_tA S_tB (1 when 0), the scale warps rewrite the P tile in shared
// memory as P~ = bf16(P * (beta / alpha)) and BF16 MMAs add P~ Q^T, so that
// C = alpha * (A B^T + P~ Q^T) is rounded once.
// ---------------------------------------------------------------------------
namespace g2 {
constexpr int BK = 256;
constexpr int STAGES = 5;
constexpr int A_BYTES = 128 * BK / 2;            // 16 KB: this CTA's 128 A rows
constexpr int B_BYTES = 128 * BK / 2;            // 16 KB: this CTA's 128 B rows
constexpr int SF_ATOM = 512;
constexpr int SFA_BYTES = 4 * SF_ATOM;           // 2 KB: scales of this CTA's A rows
constexpr int SFB_BYTES = 8 * SF_ATOM;           // 4 KB: scales of all 256 B rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // 38 KB
constexpr int BR_K = 64;
constexpr int P_BYTES = 128 * BR_K * 2;          // 16 KB (A slot)
constexpr int Q_BYTES = 128 * BR_K * 2;          // 16 KB (B slot)
constexpr int EPI_WARPS = 8;                     // two per TMEM lane quadrant, 128 columns each
constexpr int CHUNK_BYTES = 32 * 64;             // 32 rows x 32 BF16 columns, 64-byte swizzled rows
constexpr int OUT_BYTES = EPI_WARPS * 2 * CHUNK_BYTES;  // 32 KB: two chunks in flight per epilogue warp
constexpr uint32_t TM_ACC = 0;                   // 256 columns
constexpr uint32_t TM_SF = 256;                  // per stage: SFA 16 + SFB 32 columns
constexpr uint32_t TM_SF_STAGE = 48;
constexpr uint32_t TM_COLS = 512;
static_assert(TM_SF + STAGES * TM_SF_STAGE <= TM_COLS, "TMEM budget");
// warps: 0 A/B producer, 1 MMA (leader) + TMEM allocator, 2 scale/P producer,
// 3..10 scale stagers (two per TMEM lane quadrant, two K steps each), 11..18 epilogue
constexpr int FIRST_EPI_WARP = 11;
// Split the tail wave only when K >= 48 * 256: the last wave's few pairs run with the L2 to
// themselves, faster than a full wave, so shorter pieces do not repay the partial stores and
// the reduction's launch (measured on the 3B block's GEMMs: a loss at K = 8192 and 9216, a gain
// of 2-5% at K = 16384).
constexpr uint32_t kSplitMinStages = 48;
constexpr int NUM_THREADS = (FIRST_EPI_WARP + EPI_WARPS) * 32;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + 256;
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
}  // namespace g2

// One unit of a CTA pair's work: a whole 256 x 256 tile, or K stages [kb, ke) of a tile of
// the split tail, whose FP32 partial goes to workspace slot `slot`.
struct PairWork {
  uint32_t mb2, nb2, kb, ke;
  int32_t slot;  // -1: the tile's result goes to C
  bool branch;   // this unit adds the BF16 branch stage (a split tile's last piece)
};

// Unit i of cluster cid (of ncl): the whole tiles cid, cid + ncl, ... (below dp_tiles when the
// tail is split), then, with a split tail, tail unit cid: tile dp_tiles + cid / S, K piece cid % S.
// Every role of the kernel walks the same sequence.
__device__ __forceinline__ bool pair_work(const GemmParams& p, uint32_t cid, uint32_t ncl, uint32_t i,
                                          uint32_t tiles_m, uint32_t tiles_n, uint32_t num_k, bool has_branch,
                                          PairWork& w) {
  const uint32_t num_tiles = tiles_m * tiles_n;
  uint32_t mt;
  w.kb = 0;
  w.ke = num_k;
  w.slot = -1;
  w.branch = has_branch;
  if (p.sk_split == 0) {
    mt = cid + i * ncl;
    if (mt >= num_tiles) return false;
  } else {
    const uint32_t ndp = p.dp_tiles / ncl, S = p.sk_split;
    if (i < ndp) {
      mt = cid + i * ncl;
    } else if (i == ndp && cid < (num_tiles - p.dp_tiles) * S) {
      const uint32_t piece = cid % S;
      mt = p.dp_tiles + cid / S;
      w.kb = piece * num_k / S;
      w.ke = (piece + 1) * num_k / S;
      w.slot = (int32_t)cid;
      w.branch = has_branch && piece == S - 1;
    } else {
      return false;
    }
  }
  w.mb2 = p.raster_n ? mt / tiles_n : mt % tiles_m;
  w.nb2 = p.raster_n ? mt % tiles_n : mt / tiles_m;
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(g2::NUM_THREADS, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_p, const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_sfb,
                          const GemmParams p) {
  using namespace g2;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sOut = smem + STAGES * STAGE_BYTES;
  // leader's full[s]: A/B (+Q) of both CTAs landed AND the scales are in TMEM (P~ in smem)
  // in both CTAs -- one wait per stage for the MMA warp
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + OUT_BYTES);
  uint64_t* sf_full = full + STAGES;        // each CTA: its scales (or P) landed
  uint64_t* empty = sf_full + STAGES;       // each CTA: the stage was consumed by the MMAs (both producers wait)
  uint64_t* peer_ready = empty + STAGES;    // peer CTA: its 8 stager warps are done with stage s
  uint64_t* acc_full = peer_ready + STAGES; // each CTA: accumulator complete
  uint64_t* acc_empty = acc_full + 1;       // leader: both CTAs drained the accumulator
  uint64_t* done_bar = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // leader: producer (expect_tx) + its 8 stager warps + one forwarded arrival for the peer's 8
      mbar_init(&full[s], 1 + 8 + 1);
      mbar_init(&sf_full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&peer_ready[s], 8);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * EPI_WARPS);  // every epilogue warp of both CTAs
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    if (p.sfb_tma) prefetch_tmap(&tmap_sfb);
    if (p.r > 0) {
      prefetch_tmap(&tmap_p);
      prefetch_tmap(&tmap_q);
    }
    if (!p.c_f32) prefetch_tmap(&tmap_c);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // (the set-up above touches no global data)

  const uint32_t cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
  const uint32_t tiles_m = p.M / 256, tiles_n = p.N / 256;
  const uint32_t num_k = (p.K + BK - 1) / BK;
  const bool has_branch = p.r > 0;
  float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
  if (alpha == 0.0f) alpha = 1.0f;  // an all-zero operand contributes exact zeros

  if (warp == 0 || warp == 2) {
    if (lane == 0) {
      // ---------------- producers (both CTAs): warp 0 operands (TMA), warp 2 scales / P ----------------
      const bool ab = warp == 0;
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);  // leader's full[] in the cluster window
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      PairWork w;
      for (uint32_t wi = 0; ok && pair_work(p, cluster_id, num_clusters, wi, tiles_m, tiles_n, num_k, has_branch, w);
           ++wi) {
        const uint32_t mb2 = w.mb2, nb2 = w.nb2;
        for (uint32_t it = w.kb; it < w.ke + (w.branch ? 1u : 0u); ++it) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sSFA = sB + B_BYTES;
          uint8_t* sSFB = sSFA + SFA_BYTES;
          const uint32_t full_l = full0 + stage * 8;
          if (it < w.ke) {
            if (ab) {
              if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (A_BYTES + B_BYTES));
              const int32_t kx = (int32_t)(it * (BK / 2));
              tma_load_2d_pair(sA, &tmap_a, full_l, kx, (int32_t)(mb2 * 256 + rank * 128));
              tma_load_2d_pair(sB, &tmap_b, full_l, kx, (int32_t)(nb2 * 256 + rank * 128));
            } else {
              const uint32_t krem = p.K - it * BK;
              const uint32_t nk = krem >= (uint32_t)BK ? 4 : krem / 64;
              // this CTA's A scale atoms by a bulk copy, the tile's two B row blocks (all 256 B rows)
              // by one 2 x 2 KB TMA box (atoms past K arrive zero-filled)
              mbar_arrive_expect_tx(&sf_full[stage], nk * SF_ATOM + (p.sfb_tma ? SFB_BYTES : 2 * nk * SF_ATOM));
              const size_t ka = (size_t)it * 4;
              bulk_load(sSFA, p.a_scales + ((size_t)(mb2 * 2 + rank) * p.atoms_k + ka) * SF_ATOM, nk * SF_ATOM,
                        &sf_full[stage]);
              if (p.sfb_tma) {
                tma_load_2d(sSFB, &tmap_sfb, &sf_full[stage], (int32_t)(ka * 64), (int32_t)(nb2 * 2));
              } else {
                bulk_load(sSFB, p.b_scales + ((size_t)(nb2 * 2) * p.atoms_k + ka) * SF_ATOM, nk * SF_ATOM,
                          &sf_full[stage]);
                bulk_load(sSFB + 4 * SF_ATOM, p.b_scales + ((size_t)(nb2 * 2 + 1) * p.atoms_k + ka) * SF_ATOM,
                          nk * SF_ATOM, &sf_full[stage]);
              }
            }
          } else if (p.p_folded) {
            // P~ and Q by TMA, both completing on the leader's barrier; the scale warps only pass
            if (ab) {
              if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (P_BYTES + Q_BYTES));
              tma_load_2d_pair(sA, &tmap_p, full_l, 0, (int32_t)(mb2 * 256 + rank * 128));
              tma_load_2d_pair(sB, &tmap_q, full_l, 0, (int32_t)(nb2 * 256 + rank * 128));
            } else {
              mbar_arrive(&sf_full[stage]);
            }
          } else {
            if (ab) {
              if (leader) mbar_arrive_expect_tx(&full[stage], 2 * Q_BYTES);
              tma_load_2d_pair(sB, &tmap_q, full_l, 0, (int32_t)(nb2 * 256 + rank * 128));
            } else {
              mbar_arrive_expect_tx(&sf_full[stage], P_BYTES);
              tma_load_2d(sA, &tmap_p, &sf_full[stage], 0, (int32_t)(mb2 * 256 + rank * 128));
            }
          }
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (pair leader) ----------------
      const uint32_t idesc = idesc_nvf4(256, 256);
      const uint32_t idesc_br = idesc_bf16(256, 256);
      const uint64_t adesc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
      const uint64_t bdesc0 = adesc0 + (A_BYTES >> 4);
      constexpr uint64_t kStageD = STAGE_BYTES >> 4;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      uint32_t t = 0;
      PairWork w;
      for (; ok && pair_work(p, cluster_id, num_clusters, t, tiles_m, tiles_n, num_k, has_branch, w); ++t) {
        if (*abort_flag || !mbar_wait(acc_empty, (t & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + TM_ACC;
        for (uint32_t it = w.kb; it < w.ke; ++it) {
          if (!mbar_wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + stage * kStageD, bd = bdesc0 + stage * kStageD;
          const uint32_t tsf = tmem + TM_SF + stage * TM_SF_STAGE;
          const uint32_t krem = p.K - it * BK;
          if (krem >= (uint32_t)BK) {
            mma_nvf4_pair(d_tmem, ad, bd, idesc, tsf, tsf + 16, it != w.kb);
            mma_nvf4_pair(d_tmem, ad + 2, bd + 2, idesc, tsf + 4, tsf + 24, 1);
            mma_nvf4_pair(d_tmem, ad + 4, bd + 4, idesc, tsf + 8, tsf + 32, 1);
            mma_nvf4_pair(d_tmem, ad + 6, bd + 6, idesc, tsf + 12, tsf + 40, 1);
          } else {
            for (uint32_t kk = 0; kk < krem / 64; ++kk)
              mma_nvf4_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, tsf + kk * 4, tsf + 16 + kk * 8,
                            it != w.kb || kk != 0);
          }
          tc_commit_pair_mc(&empty[stage], 3);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        if (w.branch) {
          if (!mbar_wait(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = adesc0 + stage * kStageD, bd = bdesc0 + stage * kStageD;
          const uint32_t nkb = (uint32_t)(p.r + 15) / 16;
          for (uint32_t kk = 0; kk < nkb; ++kk) mma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc_br, 1);
          tc_commit_pair_mc(&empty[stage], 3);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        tc_commit_pair_mc(acc_full, 3);
      }
      if (!ok) *abort_flag = 1;
      tc_commit_pair_mc(done_bar, 1);  // (a kernel may not mix cta_group::1 and ::2 forms)
      mbar_wait(done_bar, 0);
    } else if (lane == 0) {
      // ---------------- peer: forward its stagers' completion as one remote arrival per stage ----------------
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      PairWork w;
      for (uint32_t wi = 0; ok && pair_work(p, cluster_id, num_clusters, wi, tiles_m, tiles_n, num_k, has_branch, w);
           ++wi) {
        for (uint32_t it = w.kb; it < w.ke + (w.branch ? 1u : 0u); ++it) {
          if (*abort_flag || !mbar_wait(&peer_ready[stage], phase)) {
            ok = false;
            break;
          }
          // K stage: the TMEM stores are complete; a folded branch stage: nothing was written
          if (it < w.ke || p.p_folded) mbar_arrive_cluster_relaxed(full0 + stage * 8);
          else mbar_arrive_cluster(full0 + stage * 8);  // P~ was written through the generic proxy
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp < 11) {
    // ---------------- scale stagers (warps 3..10, both CTAs) ----------------
    // warp w serves TMEM lane quadrant w % 4 and the two K steps {2h, 2h+1}, h = (w - 3) / 4
    const uint32_t quad = warp & 3, h = (uint32_t)(warp - 3) >> 2;
    const uint32_t lane_off = (quad * 32) << 16;
    const float g = __fdiv_rn(p.beta, alpha);
    uint32_t stage = 0, phase = 0;
    PairWork w;
    for (uint32_t wi = 0; pair_work(p, cluster_id, num_clusters, wi, tiles_m, tiles_n, num_k, has_branch, w); ++wi) {
      bool ok = true;
      for (uint32_t it = w.kb; it < w.ke + (w.branch ? 1u : 0u); ++it) {
        if (*abort_flag || !mbar_wait_warp(&sf_full[stage], phase)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        if (it < w.ke) {
          const uint32_t krem = p.K - it * BK;
          const uint32_t nk = krem >= (uint32_t)BK ? 4 : krem / 64;
          const uint8_t* sSFA = sA + A_BYTES + B_BYTES;
          const uint8_t* sSFB = sSFA + SFA_BYTES;
          const uint32_t tsf = TM_SF + stage * TM_SF_STAGE;
          uint32_t wa[8], wb[16];
          // A row m = 32*quad + lane: scales of K step j at atom j, byte (m%32)*16 + (m/32)*4;
          // the MMA reads them at lane m, column tsf + 4j + quad
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint32_t j = 2 * h + jj;
            const uint32_t v =
                j < nk ? *reinterpret_cast<const uint32_t*>(sSFA + j * SF_ATOM + lane * 16 + quad * 4) : 0u;
            wa[4 * jj] = wa[4 * jj + 1] = wa[4 * jj + 2] = wa[4 * jj + 3] = v;
          }
          tmem_st_32x32b_x8(tmem + lane_off + tsf + 8 * h, wa);
          // B row n = 32c + lane (c = 0..7): scales of K step j at column tsf + 16 + 8j + c, every quadrant
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint32_t j = 2 * h + jj;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (j < nk) v = *reinterpret_cast<const uint4*>(sSFB + hh * 4 * SF_ATOM + j * SF_ATOM + lane * 16);
              wb[8 * jj + 4 * hh] = v.x;
              wb[8 * jj + 4 * hh + 1] = v.y;
              wb[8 * jj + 4 * hh + 2] = v.z;
              wb[8 * jj + 4 * hh + 3] = v.w;
            }
          }
          tmem_st_32x32b_x16(tmem + lane_off + tsf + 16 + 16 * h, wb);
          tmem_st_wait(wb);
          tmem_st_wait8(wa);
          tc_fence_before();
        } else if (!p.p_folded) {
          // branch stage: P~ = bf16(P * g) in place (an elementwise map, so the swizzle is irrelevant)
          uint4* tile = reinterpret_cast<uint4*>(sA);
          const int tid = (warp - 3) * 32 + lane;
#pragma unroll 4
          for (int i = tid; i < P_BYTES / 16; i += 256) {
            uint4 v = tile[i];
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __fmul_rn(bf16_lo(w[e]), g), hi = __fmul_rn(bf16_hi(w[e]), g);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
              w[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            tile[i] = v;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(leader ? &full[stage] : &peer_ready[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
  } else {
    // ---------------- epilogue (warps 11..18, both CTAs): C = alpha * acc ----------------
    // warp w reads TMEM lane quadrant w % 4 (rows 32q..32q+31 of this CTA's 128) and
    // columns [128h, 128h + 128), h = (w - 11) / 4, in four 32-column chunks
    const uint32_t quad = warp & 3, h = (uint32_t)(warp - FIRST_EPI_WARP) >> 2;
    const uint32_t lane_off = (quad * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    uint8_t* stg = sOut + (warp - FIRST_EPI_WARP) * 2 * CHUNK_BYTES;  // this warp's two staging chunks
    uint32_t t = 0;
    PairWork w;
    for (; pair_work(p, cluster_id, num_clusters, t, tiles_m, tiles_n, num_k, has_branch, w); ++t) {
      const uint32_t mb2 = w.mb2, nb2 = w.nb2;
      if (*abort_flag || !mbar_wait_warp(acc_full, t & 1)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t row0 = mb2 * 256 + rank * 128 + quad * 32;
      const uint32_t col0 = nb2 * 256 + h * 128;
      if (w.slot >= 0) {
        // a piece of a split tile: the raw FP32 accumulator to its slot, 256 x 256 row-major
        float* part = p.sk_ws + (size_t)w.slot * 65536 + (size_t)(rank * 128 + quad * 32 + lane) * 256 + h * 128;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t acc[32];
          tmem_ld_32x32b_x32(tmem + lane_off + TM_ACC + h * 128 + j * 32, acc);
          tmem_ld_wait(acc);
          float4* dst = reinterpret_cast<float4*>(part + j * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(acc[4 * i]), __uint_as_float(acc[4 * i + 1]),
                                 __uint_as_float(acc[4 * i + 2]), __uint_as_float(acc[4 * i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(acc_empty);
          else mbar_arrive_cluster_relaxed(acc_empty0);
        }
      } else if (!p.c_f32) {
        // TMEM -> registers -> BF16.  The accumulator is released as soon as all four chunks are in
        // registers or staged: chunks 0 and 1 go to this warp's two swizzled shared chunks, 2 and 3
        // stay packed in registers until the first two TMA stores have read their buffers.
        auto convert = [&](const uint32_t (&a32)[32], uint32_t (&pk)[16]) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(alpha, __uint_as_float(a32[2 * e])),
                                                      __fmul_rn(alpha, __uint_as_float(a32[2 * e + 1])));
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
        };
        // row = lane, 64 bytes; 16-byte unit u lands at u ^ ((row >> 1) & 3) (64-byte swizzle)
        auto stage_chunk = [&](uint8_t* chunk, const uint32_t (&pk)[16]) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(chunk + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        };
        uint8_t* buf0 = stg;
        uint8_t* buf1 = stg + CHUNK_BYTES;
        const uint32_t tacc = tmem + lane_off + TM_ACC + h * 128;
        uint32_t ra[32], rb[32], pk[16], pk2[16], pk3[16];
        // the previous tile's stores must have read both buffers before they are rewritten
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        tmem_ld_32x32b_x32(tacc, ra);
        tmem_ld_wait(ra);
        tmem_ld_32x32b_x32(tacc + 32, rb);
        convert(ra, pk);
        stage_chunk(buf0, pk);
        tmem_ld_wait(rb);
        tmem_ld_32x32b_x32(tacc + 64, ra);
        convert(rb, pk);
        stage_chunk(buf1, pk);
        tmem_ld_wait(ra);
        tmem_ld_32x32b_x32(tacc + 96, rb);
        convert(ra, pk2);
        tmem_ld_wait(rb);
        // every TMEM read of the accumulator is complete: release it to the MMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(acc_empty);
          else mbar_arrive_cluster_relaxed(acc_empty0);
        }
        convert(rb, pk3);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_c, buf0, (int32_t)col0, (int32_t)row0);
          tma_store_2d(&tmap_c, buf1, (int32_t)(col0 + 32), (int32_t)row0);
          bulk_commit_group();
          bulk_wait_read<0>();
        }
        __syncwarp();
        stage_chunk(buf0, pk2);
        stage_chunk(buf1, pk3);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_c, buf0, (int32_t)(col0 + 64), (int32_t)row0);
          tma_store_2d(&tmap_c, buf1, (int32_t)(col0 + 96), (int32_t)row0);
          bulk_commit_group();
        }
      } else {
        const size_t row = (size_t)row0 + lane;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t acc[32];
          tmem_ld_32x32b_x32(tmem + lane_off + TM_ACC + h * 128 + j * 32, acc);
          tmem_ld_wait(acc);
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.C) + row * p.ldc + col0 + j * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__fmul_rn(alpha, __uint_as_float(acc[4 * i])),
                                 __fmul_rn(alpha, __uint_as_float(acc[4 * i + 1])),
                                 __fmul_rn(alpha, __uint_as_float(acc[4 * i + 2])),
                                 __fmul_rn(alpha, __uint_as_float(acc[4 * i + 3])));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(acc_empty);
          else mbar_arrive_cluster_relaxed(acc_empty0);
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
    __syncwarp();
  }

  __syncthreads();
  if (*abort_flag) {  // a wait expired: let copies still in flight land first
    if (threadIdx.x == 0) drain_pause();
    __syncthreads();
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TM_COLS);
  }
  cluster_sync();
}

// The split tail's result: C = round_c(fl32(alpha * acc)) with acc the FP32 sum of a tile's
// S partial accumulators taken in piece order (so the result does not depend on which pair
// finished first).  One thread per 4 consecutive columns of one row of one tail tile.
__global__ void __launch_bounds__(256) gemm_splitk_reduce_kernel(const GemmParams p, uint32_t tail_tiles) {
  pdl_trigger();
  pdl_wait();
  const uint32_t idx = blockIdx.x * 256 + threadIdx.x;
  const uint32_t tt = idx >> 14;  // 16384 float4 per 256 x 256 tile
  if (tt >= tail_tiles) return;
  const uint32_t e = idx & 16383u, row = e >> 6, c4 = e & 63u;
  const uint32_t S = p.sk_split;
  const float4* part = reinterpret_cast<const float4*>(p.sk_ws) + (size_t)tt * S * 16384 + e;
  float4 acc = part[0];
#pragma unroll 4
  for (uint32_t q = 1; q < S; ++q) {
    const float4 v = part[(size_t)q * 16384];
    acc.x = __fadd_rn(acc.x, v.x);
    acc.y = __fadd_rn(acc.y, v.y);
    acc.z = __fadd_rn(acc.z, v.z);
    acc.w = __fadd_rn(acc.w, v.w);
  }
  float alpha = __fmul_rn(*p.a_scale, *p.b_scale);
  if (alpha == 0.0f) alpha = 1.0f;
  const uint32_t tiles_m = p.M / 256, tiles_n = p.N / 256, mt = p.dp_tiles + tt;
  const uint32_t mb2 = p.raster_n ? mt / tiles_n : mt % tiles_m;
  const uint32_t nb2 = p.raster_n ? mt % tiles_n : mt / tiles_m;
  const size_t off = (size_t)(mb2 * 256 + row) * p.ldc + nb2 * 256 + c4 * 4;
  const float x = __fmul_rn(alpha, acc.x), y = __fmul_rn(alpha, acc.y), z = __fmul_rn(alpha, acc.z),
              w = __fmul_rn(alpha, acc.w);
  if (p.c_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.C) + off) = make_float4(x, y, z, w);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x, y), hi = __floats2bfloat162_rn(z, w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.C) + off) =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

// The branch fold on its own (the scale warps' in-kernel form, run before the GEMM):
// Pt = bf16(fl32(P * g)), g = fl32(beta / alpha), alpha = fl32(S_tA * S_tB) (1 when 0).
__global__ void __launch_bounds__(256) fold_branch_kernel(const uint32_t* P, uint32_t nwords,
                                                          const float* a_scale, const float* b_scale, float beta,
                                                          uint32_t* Pt) {
  pdl_trigger();
  pdl_wait();
  float alpha = __fmul_rn(*a_scale, *b_scale);
  if (alpha == 0.0f) alpha = 1.0f;
  const float g = __fdiv_rn(beta, alpha);
  for (uint32_t i = blockIdx.x * 256 + threadIdx.x; i < nwords; i += gridDim.x * 256) {
    const uint32_t v = P[i];
    __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(bf16_lo(v), g), __fmul_rn(bf16_hi(v), g));
    Pt[i] = *reinterpret_cast<uint32_t*>(&b2);
  }
}

cudaError_t launch_fold_branch(const void* P, int64_t M, int r, const float* a_scale, const float* b_scale,
                               float beta, void* Pt, cudaStream_t s) {
  const uint32_t nwords = static_cast<uint32_t>(M * r / 2);
  uint32_t blocks = (nwords + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  const cudaError_t e = launch_pdl(fold_branch_kernel, dim3(blocks), dim3(256), 0, s, static_cast<const uint32_t*>(P),
                                   nwords, a_scale, b_scale, beta, static_cast<uint32_t*>(Pt));
  count_launch();
  return e;
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
// row pitch `pitch_bytes`, box inner x outer, 128-byte swizzle by default.
// A tensor map is a pure function of these parameters, so encoded maps are kept
// in a small cache keyed on all of them (64 entries, replaced round-robin): a call
// on the same buffers and shapes as an earlier one skips the driver's encoder.
struct TmapKey {
  int dt, swizzle;
  const void* base;
  uint64_t inner, outer, pitch;
  uint32_t box_inner, box_outer;
};
static bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  constexpr int kCache = 64;
  static std::mutex mu;
  static TmapKey keys[kCache];
  static CUtensorMap maps[kCache];
  static int used = 0, next = 0;
  TmapKey k;
  std::memset(&k, 0, sizeof(k));  // padding included, for the byte-wise comparison
  k.dt = static_cast<int>(dt);
  k.swizzle = static_cast<int>(swizzle);
  k.base = base;
  k.inner = inner;
  k.outer = outer;
  k.pitch = pitch_bytes;
  k.box_inner = box_inner;
  k.box_outer = box_outer;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
      if (std::memcmp(&keys[i], &k, sizeof(k)) == 0) {
        *m = maps[i];
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  if (fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> g(mu);
  keys[next] = k;
  maps[next] = *m;
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  return true;
}

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  return make_tmap(m, dt, base, inner, outer, pitch_bytes, box_inner, box_outer, swizzle);
}

static cudaError_t launch_gemm_single(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tp,
                                      const CUtensorMap& tq, const GemmParams& p, int num_sms, cudaStream_t s) {
  using namespace g4;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // one CTA per SM (its shared memory allows no more), at most one per tile
  const uint32_t tiles = p.num_m * p.num_n;
  const uint32_t grid = tiles < (uint32_t)num_sms ? tiles : (uint32_t)num_sms;
  const cudaError_t e = launch_pdl(gemm_nvf4_kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, ta, tb, tp, tq, p);
  count_launch();
  return e;
}

static cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tp,
                                    const CUtensorMap& tq, const CUtensorMap& tc, const CUtensorMap& tsfb,
                                    const GemmParams& p, int num_sms,
                                    float* sk_ws, size_t sk_ws_bytes, cudaStream_t s) {
  using namespace g2;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(gemm_nvf4_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms / 2 * 2);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, gemm_nvf4_pair_kernel, &cfg) != cudaSuccess ||
        max_clusters <= 0)
      max_clusters = num_sms / 2;
    (void)cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  const uint32_t tiles = (p.M / 256) * (p.N / 256);
  const uint32_t clusters = tiles < (uint32_t)max_clusters ? tiles : (uint32_t)max_clusters;
  GemmParams q = p;
  q.sk_split = 0;
  q.dp_tiles = tiles;
  // Split tail: with W full waves and R < clusters tiles left over, the last wave would keep
  // clusters - R pairs idle for a whole tile.  Cutting each of the R tiles into S = clusters / R
  // K pieces (one per pair) ends the wave after about 1/S of a tile, plus the reduction.  Taken
  // when the pieces stay long enough (K of at least kSplitMinStages stages) to repay the partial
  // stores and the extra launch.
  const uint32_t num_k = (p.K + BK - 1) / BK, rem = tiles % clusters;
  if (sk_ws && tiles > clusters && rem > 0 && num_k >= kSplitMinStages) {
    uint32_t S = clusters / rem;
    if (S > num_k) S = num_k;
    if (S >= 2 && (size_t)rem * S * 65536 * sizeof(float) <= sk_ws_bytes) {
      q.sk_split = S;
      q.dp_tiles = tiles - rem;
      q.sk_ws = sk_ws;
    }
  }
  cudaError_t e =
      launch_pdl(gemm_nvf4_pair_kernel, dim3(clusters * 2), dim3(NUM_THREADS), SMEM_BYTES, s, ta, tb, tp, tq, tc, tsfb, q);
  count_launch();
  if (e == cudaSuccess && q.sk_split) {
    e = launch_pdl(gemm_splitk_reduce_kernel, dim3(rem * 64), dim3(256), 0, s, q, rem);
    count_launch();
  }
  return e;
}

size_t gemm_splitk_ws_bytes(int num_sms) { return (size_t)(num_sms / 2) * 65536 * sizeof(float); }

cudaError_t launch_gemm_nvf4(const GemmArgs& g, int num_sms, cudaStream_t s) {
  using namespace g4;
  if (g.M % 256 == 0 && g.N % 256 == 0) {
    // 2-SM path: each CTA TMA-loads 128 rows of A and of B
    CUtensorMap ta, tb, tp, tq;
    if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a_codes, g.K / 2, g.M, g.K / 2, BK / 2, 128) ||
        !make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b_codes, g.K / 2, g.N, g.K / 2, BK / 2, 128))
      return cudaErrorInvalidValue;
    if (g.r > 0) {
      if (!make_tmap(&tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.P, g.r, g.M, (uint64_t)g.r * 2, BR_K, 128) ||
          !make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.Q, g.r, g.N, (uint64_t)g.r * 2, BR_K, 128))
        return cudaErrorInvalidValue;
    } else {
      tp = ta;
      tq = tb;
    }
    GemmParams p{};
    p.a_scales = static_cast<const uint8_t*>(g.a_scales);
    p.b_scales = static_cast<const uint8_t*>(g.b_scales);
    p.a_scale = g.a_scale;
    p.b_scale = g.b_scale;
    p.M = (uint32_t)g.M;
    p.N = (uint32_t)g.N;
    p.K = (uint32_t)g.K;
    p.atoms_k = (uint32_t)(g.K / 64);
    p.num_m = (uint32_t)(g.M / 128);
    p.num_n = (uint32_t)(g.N / 128);
    p.r = g.r;
    p.beta = g.beta;
    p.C = g.C;
    p.c_f32 = g.c_f32;
    p.ldc = g.ldc;
    p.raster_n = g.M > g.N ? 1 : 0;  // A (M x K) is the larger operand: walk N fastest
    p.p_folded = g.p_folded && g.r > 0;
    // BF16 output leaves through TMA stores of 32 x 32 tiles (64-byte rows, 64-byte swizzle)
    CUtensorMap tc = ta;
    if (!g.c_f32 && !make_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.C, g.N, g.M, (uint64_t)g.ldc * 2, 32, 32,
                               CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    // B's scales as a 2-D tensor of 8-byte units: one row per 128-row block, K/64 atoms of 512 B each
    // (a stage's box of four atoms needs K >= 256)
    CUtensorMap tsfb = ta;
    p.sfb_tma = g.K >= 256;
    if (p.sfb_tma && !make_tmap(&tsfb, CU_TENSOR_MAP_DATA_TYPE_UINT64, g.b_scales, (uint64_t)(g.K / 64) * 64,
                                (uint64_t)(g.N / 128), (uint64_t)(g.K / 64) * 512, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    return launch_gemm_pair(ta, tb, tp, tq, tc, tsfb, p, num_sms, g.sk_ws, g.sk_ws_bytes, s);
  }
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
  GemmParams p{};
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
  p.raster_n = 0;
  p.p_folded = g.p_folded && g.r > 0;  // the scale warps skip their fold (one CTA: a local arrive)
  return launch_gemm_single(ta, tb, tp, tq, p, num_sms, s);
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
