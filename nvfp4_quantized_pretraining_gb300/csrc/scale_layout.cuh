// Layout of the UE4M3 block scales of an NVFP4 tensor in HBM: the layout the
// block-scaled MMA reads, used for every stored NVFP4 tensor of the library.
#pragma once

#include <stdint.h>

namespace nvfp4 {

// Byte offset of scale (r, k) in the MMA layout of a tensor with kb scale
// columns: 128-row x 4-column atoms of 512 bytes, row-block-major.
__device__ __forceinline__ uint32_t sf_offset(uint32_t r, uint32_t k, uint32_t atoms_k) {
  return (((r >> 7) * atoms_k + (k >> 2)) << 9) + ((r & 31u) << 4) + (((r >> 5) & 3u) << 2) + (k & 3u);
}

}  // namespace nvfp4
