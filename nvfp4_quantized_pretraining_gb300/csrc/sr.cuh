// Stochastic rounding to the E2M1 grid: the Philox4x32-10 counter generator
// that supplies its random bits, and the rounding rule itself.  Used by the
// quantizer only.
#pragma once
#include <stdint.h>

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11)
// ---------------------------------------------------------------------------
// The ten round keys of a (seed lo, seed hi) key: round r uses
// (k0 + r * 0x9E3779B9, k1 + r * 0xBB67AE85).  Computed once on the host and
// passed in a kernel's parameters (constant memory, which the XOR instructions
// read as an operand: no registers held).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};
__host__ __device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys k;
  uint32_t a = static_cast<uint32_t>(seed), b = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = a;
    k.k1[r] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}
// One round: 64-bit products give hi and lo of c0*M0 and c2*M1 in one multiply each.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k.k0[r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k.k1[r], static_cast<uint32_t>(p0));
  }
  return c;
}

// The 128 random bits for element group j (elements 8j..8j+7) of a tensor:
// counter (j lo, j hi, stream, 0).  Element e of the group takes the 16-bit
// half e % 2 (low half for even e) of word e / 2.
__device__ __forceinline__ uint4 sr_random(const PhiloxKeys& k, uint32_t stream, uint64_t j) {
  return philox4x32_10(make_uint4(static_cast<uint32_t>(j), static_cast<uint32_t>(j >> 32), stream, 0u), k);
}
// The same for j < 2^32 (counter word 1 zero): with words 1 and 3 known zero and word 2 (the
// stream) the same for every call, part of the first two rounds no longer depends on j, and the
// compiler takes it out of the element loops.
__device__ __forceinline__ uint4 sr_random32(const PhiloxKeys& k, uint32_t stream, uint32_t j) {
  return philox4x32_10(make_uint4(j, 0u, stream, 0u), k);
}

// ---------------------------------------------------------------------------
// The rounding rule
// ---------------------------------------------------------------------------
// With a = |y|, lo the grid point <= a and sp the gap above it (0.5 below 2, 1 in
// [2, 4), 2 in [4, 8)), y rounds away from lo iff rnd16 < frac * 65536 with
// frac = (a - lo) / sp; a value above 6 ends on 6 or 8 and the saturating
// conversion that follows makes both 6, as the clamp min(a, 6) would.
//
// For a >= 1 the grid points of a binade are its floats with one mantissa bit
// (1, 1.5 | 2, 3 | 4, 6 | 8), so frac * 2^22 is the low 22 bits L of a's bit
// pattern and the rule reads: round up iff L > 64 rnd16.  Adding
// bias = 2^22 - 1 - 64 rnd16 to the pattern carries into bit 22 exactly then, and
// clearing the low 22 bits leaves lo or the next grid point (a carry out of the
// mantissa steps into the next binade, which is that point).
//
// For a < 1 the gap is 0.5 throughout, as it is in [1, 2).  Both cases are handled
// at once on z = a * 2^-126 rounded upward: for a >= 1 the product is exact (a
// normal float with a's mantissa), and for a < 1 it lands in FP32's subnormal
// range, whose spacing 2^-149 is uniform like E2M1's below 1: its pattern is the
// integer ceil(a * 2^23), and bit 22 of it is the half-step.  The carry rule on
// that pattern rounds a in units of 0.5 exactly as on [1, 2) (a grid point there,
// scaled back by 2^126, is 0, 0.5 or 1).  Rounding upward to that grid keeps the
// decision: lo and 64 rnd16 * 2^-23 are on it, and for such a point m,
// ceil(a) > m iff a > m.
//
// bias comes from the Philox word: sr_bias_lo for the low half-word (even
// element), sr_bias_hi for the high half-word (odd element).
__device__ __forceinline__ uint32_t sr_bias_lo(uint32_t w) { return ~(w << 6) & 0x3FFFFFu; }
__device__ __forceinline__ uint32_t sr_bias_hi(uint32_t w) { return (~(w >> 10) & 0x3FFFC0u) | 63u; }

// The rounded value (a grid point, or 8; sign of y kept), for the saturating
// E2M1 conversion that follows.  Exact for every finite y below 2^127 in
// magnitude, denormals included (no flush to zero in this code).
__device__ __forceinline__ float sr_round(float y, uint32_t bias) {
  const float z = __fmul_ru(fabsf(y), 0x1p-126f);  // (needs denormals kept: no -ftz in this build)
  const float w = __fmul_rn(__uint_as_float((__float_as_uint(z) + bias) & 0xFFC00000u), 0x1p126f);
  return __uint_as_float(__float_as_uint(w) | (__float_as_uint(y) & 0x80000000u));
}
// The same for two values, the multiply back by 2^126 done as one packed FP32x2 multiply (exact
// either way).  The upward-rounded multiply stays scalar: it takes |y| as a free operand modifier.
__device__ __forceinline__ float2 sr_round2(float2 y, uint32_t bias_x, uint32_t bias_y) {
  const float zx = __fmul_ru(fabsf(y.x), 0x1p-126f), zy = __fmul_ru(fabsf(y.y), 0x1p-126f);
  const float2 w = __fmul2_rn(make_float2(__uint_as_float((__float_as_uint(zx) + bias_x) & 0xFFC00000u),
                                          __uint_as_float((__float_as_uint(zy) + bias_y) & 0xFFC00000u)),
                              make_float2(0x1p126f, 0x1p126f));
  return make_float2(__uint_as_float(__float_as_uint(w.x) | (__float_as_uint(y.x) & 0x80000000u)),
                     __uint_as_float(__float_as_uint(w.y) | (__float_as_uint(y.y) & 0x80000000u)));
}

}  // namespace nvfp4
