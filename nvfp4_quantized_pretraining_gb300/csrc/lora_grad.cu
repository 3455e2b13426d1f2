// Gradients of the LoRA-SVD branch factors (sm_103a).
//
// "Full-Stack FP4" (gist.science explainer), section 2.1: the weight is
// W = W_res + beta * L2 L1 with the subspace L2 L1 in BF16, and the backward pass
// is restricted to that subspace.  With the branch factors P = bf16(X L1^T) of the
// forward and P' = bf16(dY L2) of the backward, the factors' gradients are
//   dL2 = beta * dY^T P      (N x r)        dL1 = beta * P'^T X      (r x K),
// both of the form C = beta * A^T B with A: T x M and B: T x r row-major and the
// sum over the T tokens.  (The Cholesky-QR constraint the pages mention is not
// specified there and is not applied.)
//
// One BF16 tcgen05 product per 128-row block of C (MMA M = 128, N = r, K = 16):
// both operands are read MN-major straight from their row-major storage (TMA boxes
// of 64 tokens x 64 columns, 128-byte swizzle), so neither A nor B is transposed in
// memory.  The token range is split over several CTAs when C has few row blocks;
// each writes its FP32 partial sum, and a second kernel adds the partials in split
// order (deterministic) and scales by beta.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace lg {
constexpr int BM = 128;                 // rows of C per CTA (two 64-column boxes of A)
constexpr int BT = 64;                  // tokens per stage
constexpr int STAGES = 6;
constexpr int BOX_BYTES = BT * 64 * 2;  // 8 KB: 64 tokens x 64 BF16 columns
constexpr int A_BYTES = 2 * BOX_BYTES;  // 16 KB
constexpr int B_BYTES = BOX_BYTES;      // 8 KB (r <= 64 columns; the rest of the box is zero fill)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 128;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
}  // namespace lg

// kind::f16 instruction descriptor with both operands MN-major (transpose bits 15 and 16).
__host__ __device__ constexpr uint32_t idesc_bf16_mn(uint32_t M, uint32_t N) {
  return idesc_bf16(M, N) | (1u << 15) | (1u << 16);
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait_x16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// partial[split][m][j] = sum over this split's tokens of A[t][m0 + m] * B[t][j]
__global__ void __launch_bounds__(lg::NUM_THREADS, 1)
    lora_grad_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     uint32_t T, uint32_t M, int r, uint32_t stages_per_split, float* __restrict__ partial) {
  using namespace lg;
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
  const uint32_t m0 = blockIdx.x * BM;
  const uint32_t total = (T + BT - 1) / BT;
  const uint32_t s_begin = blockIdx.y * stages_per_split;
  const uint32_t n_st = s_begin < total ? min(stages_per_split, total - s_begin) : 0;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (uint32_t it = 0; it < n_st; ++it) {
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        const int32_t t0 = (int32_t)((s_begin + it) * BT);
        mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        tma_load_2d(sA, &tmap_a, &full[stage], (int32_t)m0, t0);
        tma_load_2d(sA + BOX_BYTES, &tmap_a, &full[stage], (int32_t)(m0 + 64), t0);
        tma_load_2d(sA + A_BYTES, &tmap_b, &full[stage], 0, t0);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_mn(BM, (uint32_t)r);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (uint32_t it = 0; it < n_st; ++it) {
        if (*abort_flag || !mbar_wait(&full[stage], phase)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sB = sA + A_BYTES;
        // MN-major, 128-byte swizzle: 8-token groups 1024 bytes apart (SBO); A's two 64-column
        // halves one box apart (LBO).  B has a single 64-column block.
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          mma_bf16(tmem, smem_desc(sA + kk * 2048, BOX_BYTES, 1024, kSwizzle128B),
                   smem_desc(sB + kk * 2048, 1024, 1024, kSwizzle128B), idesc, (it | kk) != 0);
        tc_commit(&empty[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (!ok) *abort_flag = 1;
      tc_commit(acc_full);
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
  }
  __syncwarp();
  // epilogue, all four warps: TMEM lane quadrant = warp, row m0 + 32 warp + lane
  if (mbar_wait_warp(acc_full, 0) && !*abort_flag) {
    tc_fence_after();
    float* dst = partial + ((size_t)blockIdx.y * M + m0 + warp * 32 + lane) * r;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (16 * j >= r) break;
      uint32_t v[16];
      tmem_ld_x16(tmem + ((warp * 32) << 16) + 16 * j, v);
      tmem_ld_wait_x16(v);
      if (n_st == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0u;  // an empty token range contributes zeros
      }
      float4* d4 = reinterpret_cast<float4*>(dst + 16 * j);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        d4[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                            __uint_as_float(v[4 * q + 3]));
    }
    tc_fence_before();
  } else {
    *abort_flag = 1;
  }
  __syncthreads();
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

// C = beta * sum over splits (in split order) of partial[s]; C[m][j] at m * ldc + j, or
// C[j][m] at j * ldc + m when transposed.
__global__ void lora_grad_reduce_kernel(const float* __restrict__ partial, uint32_t splits, uint32_t M, int r,
                                        float beta, float* __restrict__ C, int64_t ldc, int transpose_c) {
  const uint32_t n = M * (uint32_t)r;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const uint32_t m = transpose_c ? i % M : i / r;
    const uint32_t j = transpose_c ? i / M : i % r;
    float s = 0.0f;
    for (uint32_t k = 0; k < splits; ++k) s = __fadd_rn(s, partial[(size_t)k * n + (size_t)m * r + j]);
    const float v = __fmul_rn(beta, s);
    if (transpose_c) C[(size_t)j * ldc + m] = v;
    else C[(size_t)m * ldc + j] = v;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// A BF16 row-major tensor of `rows` x `cols` (pitch in elements) as 64-column x 64-row boxes.
static bool lg_tmap(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, pitch * 2, 64, (uint32_t)lg::BT,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

uint32_t lora_grad_splits(int64_t T, int64_t M, int num_sms) {
  const int64_t blocks = M / lg::BM;
  const int64_t stages = (T + lg::BT - 1) / lg::BT;
  int64_t s = blocks > 0 ? num_sms / blocks : 1;
  if (s < 1) s = 1;
  if (s > stages / 4) s = stages / 4 > 0 ? stages / 4 : 1;  // at least four stages of tokens per split
  if (s > 32) s = 32;
  return (uint32_t)s;
}

cudaError_t launch_lora_grad(const void* A, int64_t T, int64_t M, int64_t lda, const void* B, int r, float beta,
                             float* C, int64_t ldc, int transpose_c, float* partial, uint32_t splits, cudaStream_t s) {
  using namespace lg;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(lora_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ta, tb;
  if (!lg_tmap(&ta, A, (uint64_t)M, (uint64_t)T, (uint64_t)lda) ||
      !lg_tmap(&tb, B, (uint64_t)r, (uint64_t)T, (uint64_t)r))
    return cudaErrorInvalidValue;
  const uint64_t stages = (uint64_t)((T + BT - 1) / BT);
  const uint32_t per_split = (uint32_t)((stages + splits - 1) / splits);
  dim3 grid((unsigned)(M / BM), splits);
  lora_grad_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, (uint32_t)T, (uint32_t)M, r, per_split, partial);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint32_t n = (uint32_t)(M * r);
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  lora_grad_reduce_kernel<<<blocks, 256, 0, s>>>(partial, splits, (uint32_t)M, r, beta, C, ldc, transpose_c);
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
