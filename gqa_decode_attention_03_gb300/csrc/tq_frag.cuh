// tq_frag.cuh -- f16 fragment helpers shared by the TurboQuant tensor-core kernels (tq_mma.cu,
// tq_rows.cu): 2-bit centroid fields to f16 through byte permutes, hi / lo splits, and the
// power-of-two scales that keep the f16 parts clear of overflow and of the subnormal range.
#pragma once

#include <cuda_fp16.h>

#include "partial_mma.cuh"
#include "tq_common.cuh"

namespace gqa {

// A byte permute of the 8-byte table {hi4, lo4} by the low 16 bits of sel.  The PTX form takes
// each selector nibble as it is (bit 3 would ask for sign replication: every selector built here
// keeps it clear); __byte_perm would first mask the selector, one more integer instruction per
// permute on the kernel's busiest pipe.
__device__ __forceinline__ uint32_t prmt(uint32_t lo4, uint32_t hi4, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo4), "r"(hi4), "r"(sel));
  return d;
}

// Four 2-bit fields (bytes 0..3 of y, values 0..3) -> prmt selectors picking f16 numbers
// (y.b0, y.b1) and (y.b2, y.b3) of an 8-byte table: each byte k becomes 0x22 k + 0x10 (nibbles
// 2k, 2k + 1).  The high selector comes from a multiply-high on the FMA pipe, which leaves the
// integer ALU pipe (the kernel's busiest) to the field extraction and the permutes.
__device__ __forceinline__ void field_sel(uint32_t y, uint32_t& lo, uint32_t& hi) {
  lo = y * 0x22u + 0x10101010u;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(hi) : "r"(y), "r"(0x220000u), "r"(0x1010u));
}

// f16x2 of (a, b): the hi parts (part 0) or the lo parts a - hi, b - hi (part 1).
__device__ __forceinline__ uint32_t f16_part(float a, float b, int part) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  return h2_bits(part ? l : h);
}

// 2^(14 - e) for a = m 2^e, m in [0.5, 1): scales max |x| = a into [2^13, 2^14).
__device__ __forceinline__ float pow2_scale(float a) {
  if (!(a > 0.f) || !isfinite(a)) return 1.f;
  int e;
  frexpf(a, &e);
  return ldexpf(1.f, 14 - e);
}

}  // namespace gqa
