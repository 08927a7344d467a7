// act_math.cuh -- device arithmetic shared by the standalone 1x128 quantizers
// and the fused gate/up epilogue, so that both produce the same bytes:
//   h = bf16(silu(g) * u)            [dense-FFN gate/up/down arm]
//   q = RNE_sat_e4m3(x / s)          [Module w8a8_prefill: per-token 1x128
//                                     FP32 activation scales]
#pragma once

#include "bfp8_internal.h"

namespace bfp8 {
namespace dev {

// h = bf16(silu(g) * u) for BF16 g and u, with silu(g) = g / (1 + exp(-g)):
// bit-identical to that expression evaluated in double and rounded once to
// BF16 (round to nearest even), which is how the definition reads.
//
// Fast path, FP32. With c = -log2(e) split as c_hi + c_lo, c_hi of 16
// significant bits, g * c_hi is exact for a BF16 g (8 significant bits), so
//   e = 2^(g c_hi) * (1 + g c_lo ln 2)       (ex2.approx of an exact argument,
//                                              first-order correction; the
//                                              dropped term is below 2^-25)
//   s = g * rcp(1 + e),  p = RN(s * u).
// Measured over every BF16 g with 2^-100 <= |g| < 64 against double,
// |s - silu(g)| <= 2^-22.2 |silu(g)|, so p is within 2^-22.2 + 2^-24 (relative)
// of silu(g) u: under 4.5 units in the last place of p. RN_bf16(p) is the
// correctly rounded result unless a BF16 rounding midpoint lies that close to
// p, i.e. unless p's low 16 bits lie within 4.5 of 0x8000; kSiluMidUlps = 5
// flags every p within 5 units. Those elements (11 in 65536 of them) and g
// outside the range are recomputed in double. The check works on FP32 subnormals too: there every
// rounding is at most half a unit of the fixed subnormal spacing.
constexpr float kNegLog2eHi = -1.44268798828125f;   // -23637 / 16384
constexpr float kNegLog2eLoLn2 = -0x1.480fb6p-18f;  // (-log2(e) - kNegLog2eHi) * ln 2
constexpr uint32_t kSiluMidUlps = 5;

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// silu(g) within 2^-22.2 relative, for a BF16 g with 2^-100 <= |g| < 64 (or 0).
__device__ __forceinline__ float silu_fast(float g) {
  const float e0 = ex2_approx(g * kNegLog2eHi);
  const float e = fmaf(e0, g * kNegLog2eLoLn2, e0);
  return g * rcp_approx(1.0f + e);
}

// The BF16 g values the fast path covers: 0, and 2^-100 <= |g| < 64.
__device__ __forceinline__ bool silu_fast_domain(float g) {
  const uint32_t a = __float_as_uint(g) & 0x7FFFFFFFu;
  return a == 0u || (a - 0x0D800000u) < (0x42800000u - 0x0D800000u);
}

// True if RN_bf16(p) may differ from the correct rounding of a value within
// kSiluMidUlps FP32 units of p: p's low 16 bits lie that close to 0x8000.
__device__ __forceinline__ bool near_bf16_midpoint(float p) {
  return ((__float_as_uint(p) - (0x8000u - kSiluMidUlps)) & 0xFFFFu) <= 2u * kSiluMidUlps;
}

// x rounded once to BF16 (nearest, ties to even), returned as the FP32 value
// of that BF16 number. Normal results keep 8 significant bits; below 2^-126 the
// spacing is the BF16 subnormal step 2^-133.
__device__ __forceinline__ float f64_to_bf16_value(double x) {
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
  const uint64_t sign = bits & 0x8000000000000000ull;
  const uint64_t mag = bits ^ sign;
  if (mag >= 0x7FF0000000000000ull) return static_cast<float>(x);  // inf, NaN
  const int e = static_cast<int>(mag >> 52) - 1023;                 // -1023: zero or subnormal
  const int qe = (e > -126 ? e : -126) - 7;                         // exponent of the BF16 step
  const double down = __longlong_as_double(static_cast<long long>(1023 - qe) << 52);  // 2^-qe
  const double up = __longlong_as_double(static_cast<long long>(1023 + qe) << 52);    // 2^qe
  double r = rint(__longlong_as_double(static_cast<long long>(mag)) * down) * up;
  if (r >= 0x1p128) r = __longlong_as_double(0x7FF0000000000000ll);
  const float f = static_cast<float>(r);  // exact: r has at most 8 significant bits
  return sign ? -f : f;
}

// The fallback: the definition evaluated in double, rounded once to BF16.
static __device__ __noinline__ float silu_mul_bf16_slow(float g, float u) {
  const double gd = g;
  return f64_to_bf16_value(gd / (1.0 + exp(-gd)) * static_cast<double>(u));
}

__device__ __forceinline__ float silu_mul_bf16_round(float g, float u) {
  const float p = silu_fast(g) * u;
  if (!silu_fast_domain(g) || near_bf16_midpoint(p)) return silu_mul_bf16_slow(g, u);
  return __bfloat162float(__float2bfloat16_rn(p));
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
// The remainder step turns a zero quotient into +0 whatever the sign of x
// (-0 + +0 is +0), while IEEE division keeps -0 / s = -0, which encodes as the
// E4M3 code 0x80: the sign of x is put back (a no-op for every nonzero x,
// whose quotient already has it).
__device__ __forceinline__ float with_sign_of(float q, float x) {
  return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q0 = x * y;
  const float r = fmaf(-q0, s, x);
  return with_sign_of(fmaf(r, y, q0), x);
}

// div_by_scale on two values at once (packed FP32 operations, the same
// roundings per lane): ns = (-s, -s), y = (RN(1/s), RN(1/s)).
__device__ __forceinline__ float2 div_by_scale2(float2 x, float2 ns, float2 y) {
  const float2 q0 = __fmul2_rn(x, y);
  const float2 r = __ffma2_rn(q0, ns, x);
  const float2 q = __ffma2_rn(r, y, q0);
  return make_float2(with_sign_of(q.x, x.x), with_sign_of(q.y, x.y));
}

}  // namespace dev
}  // namespace bfp8
