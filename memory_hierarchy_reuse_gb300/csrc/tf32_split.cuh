// The 3xTF32 split of one fp32 value into two tf32 parts, big + small, used
// by the split pre-pass (tc_prepass.cu) and by the CTA-pair kernel's in-kernel
// converter warps (tc_gemm_pair.cu).  big keeps the top 11 significant bits
// of x, rounded to nearest-even; small is the exact remainder x - big, itself
// rounded to tf32.  Products big*big + big*small + small*big then carry about
// 22 significant bits, against 11 for one tf32 product.
#pragma once

#include <cstdint>

namespace mhr {

// Round an fp32 value to tf32 (10 explicit mantissa bits) to nearest, ties to
// even: one cvt.rn.tf32.f32, whose result is the fp32 bit pattern with the low
// 13 bits cleared.  On GB300 it equals the integer rounding
// (u + 0xFFF + bit 13 of u) & ~0x1FFF for every non-NaN pattern -- checked
// over all 2^32 -- including subnormals and the overflow of values near
// FLT_MAX to infinity; NaNs stay NaNs.
__device__ __forceinline__ float tf32_rne(float x) {
  uint32_t r;
  asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// small is zero when big already equals x, which also covers infinities
// (where x - big would be NaN).
__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
  big = tf32_rne(x);
  const float rest = x - big;  // exact: the discarded low bits
  small = big == x ? 0.f : tf32_rne(rest);
}

__device__ __forceinline__ void split4(const float4 v, float4& b, float4& s) {
  split_tf32(v.x, b.x, s.x);
  split_tf32(v.y, b.y, s.y);
  split_tf32(v.z, b.z, s.z);
  split_tf32(v.w, b.w, s.w);
}

}  // namespace mhr
