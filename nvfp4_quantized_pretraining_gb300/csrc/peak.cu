// Dense NVFP4 tensor-core rate probe (sm_103a): every SM issues back-to-back
// tcgen05.mma kind::mxf4nvf4 block-scaled MMAs on operands resident in shared
// memory, with no global-memory traffic, so the measured rate is the
// denominator for the block-scaled GEMM's fraction of peak.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int n, int iters) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;               // 128 rows x 128 B
  uint8_t* sB = smem + 16384;       // 256 rows x 128 B
  uint8_t* sSF = smem + 49152;      // 4 atoms of 512 B
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 51200);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int warp = threadIdx.x >> 5;
  // operands: E2M1 code 0x2 (1.0) everywhere, scales 0x38 (1.0)
  for (int i = threadIdx.x; i < 49152 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x22222222u;
  for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sSF)[i] = 0x38383838u;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) tmem_alloc(slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_nvf4(128, (uint32_t)n);
    const uint32_t tsf = tmem + 256;
    for (int a = 0; a < 4; ++a)
      tc_cp_32x128b_warpx4(tsf + a * 4, smem_desc(smem_u32(sSF + a * 512), 0, 128, kSwizzleNone));
    const uint32_t aS = smem_u32(sA), bS = smem_u32(sB);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_nvf4(tmem, smem_desc(aS + kk * 32, 16, 1024, kSwizzle128B), smem_desc(bS + kk * 32, 16, 1024, kSwizzle128B),
                 idesc, tsf, tsf + 4, (it | kk) != 0);
    }
    tc_commit(bar);
    mbar_wait(bar, 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_mma_peak(int n, int iters, int num_sms, cudaStream_t s) {
  const int smem = 51200 + 1024 + 64;
  cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_peak_kernel<<<num_sms, 128, smem, s>>>(n, iters);
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
