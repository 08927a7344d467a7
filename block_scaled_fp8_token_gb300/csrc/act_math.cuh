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

// ---- double-float arithmetic: a value hi + lo held as two FP32 numbers, used
// by the fallback below. The elementary steps are the error-free transforms
// (Knuth's TwoSum, Dekker's Fast2Sum, the FMA product error); every operation
// uses the round-to-nearest intrinsics so that none is fused or reordered.
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
__device__ __forceinline__ ff fast_two_sum(float a, float b) {  // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ ff two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const ff p = two_prod(a.hi, b.hi);
  return fast_two_sum(p.hi, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo)));
}

// e^x as hi + lo with relative error below 2^-46, for |x| < 64. x = k ln2 + r
// with k the integer nearest x / ln2 and |r| <= 0.35: ln2 is split in three
// parts, the first of 16 significant bits so that k times it is exact, and
// e^r is its Taylor series to degree 11 (the first dropped term is below
// 2^-47), degrees 7 to 11 in FP32 (their rounding reaches the sum below
// 2^-47) and the rest in double-float by Horner's rule. Then e^x = 2^k e^r.
__device__ __forceinline__ ff ff_exp(float x) {
  constexpr float kLn2Hi = 0x1.62e4p-1f, kLn2Lo = 0x1.7f7d1cp-20f, kLn2Lo2 = 0x1.ef357ap-45f;
  const float kf = rintf(x * 1.44269504f);
  const float t = __fsub_rn(x, __fmul_rn(kf, kLn2Hi));   // exact
  const ff kl = two_prod(kf, kLn2Lo);
  const ff r0 = two_sum(t, -kl.hi);
  const ff r = fast_two_sum(r0.hi, __fsub_rn(r0.lo, __fmaf_rn(kf, kLn2Lo2, kl.lo)));
  // 1/n! as hi + lo, n = 0 .. 11
  constexpr float c_hi[12] = {1.0f, 1.0f, 0.5f, 0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                              0x1.6c16c2p-10f, 0x1.a01a02p-13f, 0x1.a01a02p-16f, 0x1.71de3ap-19f,
                              0x1.27e4fcp-22f, 0x1.ae6456p-26f};
  constexpr float c_lo[7] = {0.0f, 0.0f, 0.0f, -0x1.555556p-28f, -0x1.555556p-30f,
                             -0x1.dddddep-32f, -0x1.27d27ep-35f};
  float tail = c_hi[11];
#pragma unroll
  for (int n = 10; n >= 7; --n) tail = __fmaf_rn(tail, r.hi, c_hi[n]);
  ff acc{tail, 0.0f};
#pragma unroll
  for (int n = 6; n >= 0; --n) acc = ff_add(ff{c_hi[n], c_lo[n]}, ff_mul(acc, r));
  const float scale = __int_as_float((static_cast<int>(kf) + 127) << 23);   // 2^k, exact
  return {__fmul_rn(acc.hi, scale), __fmul_rn(acc.lo, scale)};
}

// BF16 rounding of hi + lo (nearest, ties to even) for a finite hi + lo
// above 2^-90 in magnitude: their FP32 sum s rounds like the exact value
// unless s is itself a BF16 midpoint; then the sign of the remainder decides,
// by moving s one FP32 unit toward it.
__device__ __forceinline__ float ff_to_bf16_value(ff v) {
  const ff s = fast_two_sum(v.hi, v.lo);
  uint32_t b = __float_as_uint(s.hi);
  if ((b & 0xFFFFu) == 0x8000u && s.lo != 0.0f) b += ((s.lo > 0.0f) == (s.hi > 0.0f)) ? 1u : 0xFFFFFFFFu;
  return __bfloat162float(__float2bfloat16_rn(__uint_as_float(b)));
}

// The fallback for the elements the float32 path cannot round with
// certainty: h = bf16(g / (1 + exp(-g)) * u), the value of that double-
// precision expression rounded once.
//  - For BF16 g with -64 < g < 34 and |g| >= 2^-45, in double-float (about
//    2^-44 relative): e = exp(-g), d = 1 + e, q = g / d (FP32 quotient plus
//    the correction of its remainder), q u. There the exact value lies
//    either inside the open interval between two BF16 midpoints with room
//    far above double rounding, or next to a midpoint by a margin that both
//    evaluations resolve alike (a product g u on a midpoint moves off it by
//    at least |g|/2 or e^-34 relative, both far above 2^-52), so the two
//    roundings agree except within about 2^-44 of a midpoint.
//  - Elsewhere (|g| below 2^-45, where double arithmetic turns 1 + exp(-g)
//    into exactly 2; g >= 34, where it comes within a unit of exactly 1;
//    g <= -64; and results below 2^-90) it is evaluated in double precision,
//    the same expression in the same order.
static __device__ __noinline__ float silu_mul_bf16_slow(float g, float u) {
  const uint32_t ag = __float_as_uint(g) & 0x7FFFFFFFu;
  if (ag >= 0x29000000u && g < 34.0f && g > -64.0f) {
    const ff e = ff_exp(-g);
    const ff d = ff_add(ff{1.0f, 0.0f}, e);
    const float q1 = __fdiv_rn(g, d.hi);
    const float rem = __fsub_rn(__fmaf_rn(-q1, d.hi, g), __fmul_rn(q1, d.lo));
    const ff q = fast_two_sum(q1, __fdiv_rn(rem, d.hi));
    const ff p = two_prod(q.hi, u);
    const ff v{p.hi, __fmaf_rn(q.lo, u, p.lo)};
    const float av = fabsf(v.hi);
    if (av >= 0x1p-90f && av <= 0x1p127f) return ff_to_bf16_value(v);
  }
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
