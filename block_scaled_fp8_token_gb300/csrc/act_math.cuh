// act_math.cuh -- device arithmetic shared by the standalone 1x128 quantizers
// and the fused gate/up epilogue, so that both produce the same bytes:
//   h = bf16(silu(g) * u)            [dense-FFN gate/up/down arm]
//   q = RNE_sat_e4m3(x / s)          [Module w8a8_prefill: per-token 1x128
//                                     FP32 activation scales]
#pragma once

#include "bfp8_internal.h"

namespace bfp8 {
namespace dev {

// h = bf16(silu(g) * u). SiLU only feeds a BF16 rounding, so the fast
// exponential and division (a few FP32 ulps) change h only where the product
// sits within those ulps of a BF16 rounding boundary.
__device__ __forceinline__ float silu_mul_bf16_round(float g, float u) {
  const float s = __fdividef(g, 1.0f + __expf(-g));
  return __bfloat162float(__float2bfloat16_rn(s * u));
}

// The 1x128 scale of a group with maximum |x| = amax: the correctly rounded
// max(amax, 1e-10f) / 448, formed as div_by_scale below with the correctly
// rounded reciprocal of 448 (a constant), so no division is issued.
__device__ __forceinline__ float div_by_scale(float x, float s, float y);
__device__ __forceinline__ float group_scale(float amax) {
  return div_by_scale(fmaxf(amax, 1e-10f), 448.0f, 1.0f / 448.0f);
}

// RN(x / s) given y = RN(1 / s): one remainder correction. Markstein's
// theorem: with y within half an ulp of 1/s and q0 = RN(x*y) within one ulp
// of x/s, r = x - q0*s is exact under FMA and RN(q0 + r*y) = RN(x/s). The
// theorem assumes no underflow; a quotient in the FP32 subnormal range is
// below 2^-126, far under half the smallest E4M3 step (2^-10), so its code is
// 0 either way.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q0 = x * y;
  const float r = fmaf(-q0, s, x);
  return fmaf(r, y, q0);
}

// div_by_scale on two values at once (packed FP32 operations, the same
// roundings per lane): ns = (-s, -s), y = (RN(1/s), RN(1/s)).
__device__ __forceinline__ float2 div_by_scale2(float2 x, float2 ns, float2 y) {
  const float2 q0 = __fmul2_rn(x, y);
  const float2 r = __ffma2_rn(q0, ns, x);
  return __ffma2_rn(r, y, q0);
}

}  // namespace dev
}  // namespace bfp8
