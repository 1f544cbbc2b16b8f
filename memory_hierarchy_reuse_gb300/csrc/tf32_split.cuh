// The 3xTF32 split of one fp32 value into two tf32 parts, big + small, used
// by the split pre-pass (tc_prepass.cu) and by the CTA-pair kernel's in-kernel
// converter warps (tc_gemm_pair.cu).  big keeps the top 11 significant bits
// of x, truncated (below: that is what the tensor core reads from an fp32
// operand, so A and B themselves can serve as their big parts), and small is
// the exact remainder x - big, itself rounded to tf32.  Products
// big*big + big*small + small*big then carry about 22 significant bits,
// against 11 for one tf32 product.
#pragma once

#include <cstdint>

namespace mhr {

// Round an fp32 value to tf32 (10 explicit mantissa bits) to nearest, ties to
// even.  Two equivalent forms:
//   CVT = true:  one cvt.rn.tf32.f32 (the fp32 bit pattern with the low 13
//                bits cleared); fewest instructions, but a longer-latency
//                conversion;
//   CVT = false: integer arithmetic on the bit pattern, (u + 0xFFF + bit 13
//                of u) with the low 13 bits cleared, Inf and NaN passed
//                unchanged; more instructions, each short.
// On GB300 they agree on every non-NaN fp32 pattern -- checked over all 2^32,
// subnormals and the overflow of values near FLT_MAX to infinity included --
// and both keep NaNs NaN, so callers pick whichever is faster where they run:
// GB300 measurements favour the conversion where 16-byte loads keep the
// split memory-bound, and the integer form where 4-byte loads make it
// latency-bound (3000 x 2050 x 1000: 33.5 us with the conversion, 23.3 us
// without).
template <bool CVT>
__device__ __forceinline__ float tf32_rne(float x) {
  if constexpr (CVT) {
    uint32_t r;
    asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
  } else {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) == 0x7F800000u) return x;
    u += 0x0FFFu + ((u >> 13) & 1u);
    return __uint_as_float(u & 0xFFFFE000u);
  }
}

// The split: big = x with its low 13 bits cleared, which is what the tensor
// core itself reads from an fp32 operand under kind::tf32 (measured on GB300:
// u & ~0x1FFF for every value of a sweep), so A and B themselves can serve as
// their big parts; small = the exact remainder x - big, below 2^-10 |x|,
// rounded to tf32 to nearest.  small is zero when big already equals x, which
// also covers infinities (where x - big would be NaN).
template <bool CVT>
__device__ __forceinline__ void split_tf32_trunc(float x, float& big, float& small) {
  big = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  const float rest = x - big;  // exact
  small = big == x ? 0.f : tf32_rne<CVT>(rest);
}

// The small part alone for a truncated big part, small = tf32_rn(x - (x with
// its low 13 bits cleared)), for finite x (an infinite x gives NaN here, where
// split_tf32_trunc gives 0).  Used where the big part is x itself, read by the
// tensor core.
__device__ __forceinline__ float small_tf32_trunc(float x) {
  const float big = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  return tf32_rne<true>(x - big);  // x - big is exact
}

__device__ __forceinline__ float4 small4_tf32_trunc(const float4 v) {
  return make_float4(small_tf32_trunc(v.x), small_tf32_trunc(v.y), small_tf32_trunc(v.z),
                     small_tf32_trunc(v.w));
}

template <bool CVT>
__device__ __forceinline__ void split4_trunc(const float4 v, float4& b, float4& s) {
  split_tf32_trunc<CVT>(v.x, b.x, s.x);
  split_tf32_trunc<CVT>(v.y, b.y, s.y);
  split_tf32_trunc<CVT>(v.z, b.z, s.z);
  split_tf32_trunc<CVT>(v.w, b.w, s.w);
}

}  // namespace mhr
