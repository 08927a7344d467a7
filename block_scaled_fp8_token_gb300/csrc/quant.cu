// quant.cu -- the memory-bound quantizers:
//   * per-token 1x128 dynamic E4M3 activation quantization
//     [Module w8a8_prefill, arithmetic paragraph: per-token 1x128 FP32
//      activation scales];
//   * the same, fused behind SiLU(gate)*up (the dense-FFN gate/up/down arm);
//   * ahead-of-time 128x128 weight block quantization (a conversion endpoint
//     [th#1803 decoder PR: quantization is ahead of time, never at load]).
// Half a warp owns one (token, 128-column group). Each lane holds 8
// consecutive elements, the group maximum is a 4-step shuffle reduction, and
// the scale is max(amax, 1e-10f) / 448.0f with IEEE division. Codes come from
// cvt.rn.satfinite.e4m3x2.f32 applied to the correctly rounded quotient x / s,
// which makes the result bit-exact against the CPU definition. All 128
// elements of a group share the divisor, so the quotient is formed from one
// correctly rounded reciprocal per group and a remainder correction per
// element (act_math.cuh).
#include "bfp8_internal.h"
#include "ptx.cuh"
#include "act_math.cuh"

namespace bfp8 {
namespace {

using namespace dev;

constexpr int kThreads = 256;

// SILU == false: x is [M, K] with row stride ld; values are x[m, c].
// SILU == true : x is [M, 2K] with row stride ld; values are
//                bf16(silu(x[m, c]) * x[m, K + c]).
// A half-warp owns one (token, 128-column group): each lane holds 8 consecutive
// elements (one 16-byte load), the group maximum is a 4-step shuffle within the
// half-warp, and each half-warp keeps kUnroll groups in flight.
constexpr int kUnroll = 2;

template <bool SILU>
__device__ __forceinline__ void load8(const __nv_bfloat16* row, int64_t c, int64_t K, bool vec,
                                      float (&v)[8]) {
  if (vec && c + 8 <= K) {
    const uint4 raw = *reinterpret_cast<const uint4*>(row + c);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_bits_to_f32(static_cast<uint16_t>(w[i] & 0xFFFFu));
      v[2 * i + 1] = bf16_bits_to_f32(static_cast<uint16_t>(w[i] >> 16));
    }
    if (SILU) {
      const uint4 ru = *reinterpret_cast<const uint4*>(row + K + c);
      const uint32_t u[4] = {ru.x, ru.y, ru.z, ru.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = silu_mul_bf16_round(v[2 * i], bf16_bits_to_f32(static_cast<uint16_t>(u[i] & 0xFFFFu)));
        v[2 * i + 1] = silu_mul_bf16_round(v[2 * i + 1], bf16_bits_to_f32(static_cast<uint16_t>(u[i] >> 16)));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = 0.0f;
      if (c + i < K) {
        v[i] = __bfloat162float(row[c + i]);
        if (SILU) v[i] = silu_mul_bf16_round(v[i], __bfloat162float(row[K + c + i]));
      }
    }
  }
}

template <bool SILU>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K, int64_t ld,
    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s, int64_t ssm, int64_t sskb,
    int vec_in, int vec_out) {
  const int64_t Kb = (K + 127) / 128;
  const int64_t total = M * Kb;
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;                      // lane within the half-warp
  const int64_t hw0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int64_t nhw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 4;
  for (int64_t base = hw0; base < total; base += nhw * kUnroll) {
    float v[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t item = base + u * nhw;
      if (item < total) {
        const int64_t m = item / Kb, g = item - m * Kb;
        load8<SILU>(x + m * ld, g * 128 + hl * 8, K, vec_in, v[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[u][i] = 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t item = base + u * nhw;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[u][i]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (item >= total) continue;
      const float sc = group_scale(amax);
      const float rc = __frcp_rn(sc);
      const int64_t m = item / Kb, g = item - m * Kb;
      const int64_t c = g * 128 + hl * 8;
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint16_t lo = f32x2_to_e4m3x2(div_by_scale(v[u][4 * i], sc, rc),
                                            div_by_scale(v[u][4 * i + 1], sc, rc));
        const uint16_t hi = f32x2_to_e4m3x2(div_by_scale(v[u][4 * i + 2], sc, rc),
                                            div_by_scale(v[u][4 * i + 3], sc, rc));
        w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      uint8_t* qrow = q + m * ldq;
      if (vec_out && c + 8 <= K) {
        *reinterpret_cast<uint2*>(qrow + c) = make_uint2(w[0], w[1]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c + i < K) qrow[c + i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
      }
      if (hl == 0) s[m * ssm + g * sskb] = sc;
    }
  }
}

// One CTA per 128x128 weight block. Pass 1 finds the block maximum; pass 2
// writes the codes against the stored (BF16-rounded or F32) scale.
__global__ void __launch_bounds__(kThreads) weight_quant_kernel(
    const float* __restrict__ w, int64_t N, int64_t K, int64_t ldw, uint8_t* __restrict__ q,
    int64_t ldq, void* __restrict__ scale, int scale_f32, int64_t Kb) {
  const int64_t nb = blockIdx.y, kb = blockIdx.x;
  const int64_t r0 = nb * 128, c0 = kb * 128;
  const int tid = threadIdx.x;
  // each thread: column quad cq = tid & 31 (4 columns), rows (tid >> 5) + 8 i
  const int cq = tid & 31;
  const int rsub = tid >> 5;
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    const int64_t r = r0 + rsub + 8 * i;
    if (r >= N) break;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t c = c0 + cq * 4 + e;
      if (c < K) amax = fmaxf(amax, fabsf(w[r * ldw + c]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  __shared__ float red[kThreads / 32];
  __shared__ float s_stored;
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
    for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    const float s32 = fmaxf(m, 1e-10f) / 448.0f;
    if (scale_f32) {
      static_cast<float*>(scale)[nb * Kb + kb] = s32;
      s_stored = s32;
    } else {
      const __nv_bfloat16 sb = __float2bfloat16_rn(s32);
      static_cast<__nv_bfloat16*>(scale)[nb * Kb + kb] = sb;
      s_stored = __bfloat162float(sb);
    }
  }
  __syncthreads();
  const float sc = s_stored;
  for (int i = 0; i < 16; ++i) {
    const int64_t r = r0 + rsub + 8 * i;
    if (r >= N) break;
    const int64_t c = c0 + cq * 4;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = (c + e < K) ? w[r * ldw + c + e] : 0.0f;
    const uint16_t p01 = f32x2_to_e4m3x2(v[0] / sc, v[1] / sc);
    const uint16_t p23 = f32x2_to_e4m3x2(v[2] / sc, v[3] / sc);
    const uint8_t b[4] = {static_cast<uint8_t>(p01 & 0xFF), static_cast<uint8_t>(p01 >> 8),
                          static_cast<uint8_t>(p23 & 0xFF), static_cast<uint8_t>(p23 >> 8)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (c + e < K) q[r * ldq + c + e] = b[e];
  }
}

int act_quant_common(bool silu, const void* x, int64_t M, int64_t K, int64_t ld, void* q,
                     int64_t ldq, float* s, int64_t ssm, int64_t sskb, void* stream) {
  if (M < 0 || K < 0) return BFP8_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return BFP8_OK;
  if (!x || !q || !s) return BFP8_ERR_INVALID_ARG;
  const int64_t width = silu ? 2 * K : K;
  if (ld < width || ldq < K) return BFP8_ERR_INVALID_ARG;
  const int64_t Kb = (K + 127) / 128;
  if (ssm < 0 || sskb < 0 || (M > 1 && ssm == 0) || (Kb > 1 && sskb == 0))
    return BFP8_ERR_INVALID_ARG;
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const int vec_in = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld % 8 == 0) && (K % 8 == 0);
  const int vec_out = (reinterpret_cast<uintptr_t>(q) % 8 == 0) && (ldq % 8 == 0);
  const int64_t items = M * Kb;
  const int64_t per_block = (kThreads / 16) * kUnroll;   // groups one block covers per pass
  const int64_t want = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (silu)
    act_quant_kernel<true><<<blocks, kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), M, K, ld, static_cast<uint8_t*>(q), ldq, s, ssm,
        sskb, vec_in, vec_out);
  else
    act_quant_kernel<false><<<blocks, kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), M, K, ld, static_cast<uint8_t*>(q), ldq, s, ssm,
        sskb, vec_in, vec_out);
  return check_launch();
}

}  // namespace

int launch_act_quant(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                     float* s, int64_t ssm, int64_t sskb, void* stream) {
  return act_quant_common(false, x, M, K, ldx, q, ldq, s, ssm, sskb, stream);
}

int launch_silu_mul_act_quant(const void* gu, int64_t M, int64_t I, int64_t ld, void* q,
                              int64_t ldq, float* s, int64_t ssm, int64_t sskb, void* stream) {
  return act_quant_common(true, gu, M, I, ld, q, ldq, s, ssm, sskb, stream);
}

int launch_weight_quant(const float* w, int64_t N, int64_t K, int64_t ldw, void* q, int64_t ldq,
                        void* scale, int32_t scale_dtype, void* stream) {
  if (N < 0 || K < 0) return BFP8_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return BFP8_OK;
  if (!w || !q || !scale || ldw < K || ldq < K) return BFP8_ERR_INVALID_ARG;
  if (scale_dtype != BFP8_DT_BF16 && scale_dtype != BFP8_DT_F32) return BFP8_ERR_SCALE_DTYPE;
  const int64_t Nb = (N + 127) / 128, Kb = (K + 127) / 128;
  if (Nb > 65535 || Kb > 0x7FFFFFFF) return BFP8_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(Kb), static_cast<unsigned>(Nb));
  weight_quant_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      w, N, K, ldw, static_cast<uint8_t*>(q), ldq, scale, scale_dtype == BFP8_DT_F32, Kb);
  return check_launch();
}

}  // namespace bfp8
