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

// A quad of lanes owns one (token, 128-column group). Lane ql of the quad holds
// the 8-column chunks that start at 32 i + 8 ql (i = 0..3), so each 16-byte
// load of a quad covers 64 contiguous bytes and each 8-byte store 32. The
// per-group work (the maximum over the quad, the scale, its reciprocal, the
// scale store, the index update) is spread over 32 elements per lane. (Small
// inputs use 16 lanes a group: act_quant_kernel's GT.)
constexpr int kQuad = 4;

// row[c .. c+8) as four bf16x2 words, zero past K. FULL: the caller knows the
// chunk is in range and 16-byte aligned.
template <bool FULL>
__device__ __forceinline__ void load_chunk(const __nv_bfloat16* row, int64_t c, int64_t K,
                                           bool vec, uint32_t (&w)[4]) {
  if (FULL || (vec && c + 8 <= K)) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(row + c));
    w[0] = raw.x;
    w[1] = raw.y;
    w[2] = raw.z;
    w[3] = raw.w;
  } else {
    const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = c + 2 * j < K ? r16[c + 2 * j] : 0u;
      const uint32_t hi = c + 2 * j + 1 < K ? r16[c + 2 * j + 1] : 0u;
      w[j] = lo | (hi << 16);
    }
  }
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// SILU == false: x is [M, K] with row stride ld; values are x[m, c].
// SILU == true : x is [M, 2K] with row stride ld; values are
//                bf16(silu(x[m, c]) * x[m, K + c]).
// rows == nullptr: output row m quantizes input row m. Otherwise output row m
// quantizes input row rows[m] (a gather, e.g. routed MoE rows); an index
// outside [0, n_src) quantizes a zero row.
// For finite inputs the codes and scales equal the CPU definition bit for bit:
// the group maximum is exact (taken on the BF16 bit patterns of |x|, or on the
// BF16-rounded h), and every quotient is the correctly rounded x / s.
// FULL: K is a multiple of 128 and every row and pitch is aligned for 16-byte
// loads and 8-byte stores, so no chunk needs a bounds or alignment test.
// GT threads share a 128-value group, 128 / GT values each: 4 (32 values a
// thread) for large inputs; 16 (8 values) when the groups are too few to fill
// the GPU with 4 threads each (the decode step's SiLU*up quantization of 16
// tokens is ~40 instructions a value and ran latency-bound on 4).
template <bool SILU, bool FULL, int GT = kQuad>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K, int64_t ld,
    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s, int64_t ssm, int64_t sskb,
    int vec_in, int vec_out, const int32_t* __restrict__ rows, int64_t n_src,
    int32_t* __restrict__ clr, int32_t n_clr) {
  // a programmatic dependent of the previous kernel: wait before any access
  pdl_launch_dependents();
  pdl_wait();
  // zero a following kernel's counters (the decode step's GEMV tile counters),
  // which saves that kernel a launch of its own
  if (clr != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_clr; i += blockDim.x) clr[i] = 0;
  const int64_t Kb = (K + 127) / 128;
  constexpr int kCh = 16 / GT;  // 8-value chunks per thread
  const int ql = threadIdx.x & (GT - 1);
  const int64_t quad = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / GT;
  const int64_t nquad = static_cast<int64_t>(gridDim.x) * blockDim.x / GT;
  // (m, g) of this quad's group, advanced by nquad groups per pass without a division
  int64_t m = quad / Kb, g = quad - m * Kb;
  const int64_t dm = nquad / Kb, dg = nquad - dm * Kb;
  while (__any_sync(0xffffffffu, m < M)) {
    const bool live = m < M;
    const int64_t src = !live ? -1 : (rows ? static_cast<int64_t>(__ldg(rows + m)) : m);
    const bool ok = src >= 0 && src < n_src;
    const __nv_bfloat16* row = x + (ok ? src : 0) * ld;
    const int64_t c0 = g * 128 + ql * 8;   // chunk i at c0 + 8 * GT * i
    uint32_t a[kCh][4];
    float h[SILU ? kCh : 1][8];
    float amax;
    if constexpr (SILU) {
      amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        uint32_t u[4] = {0u, 0u, 0u, 0u};
        a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0u;
        if (ok) {
          load_chunk<FULL>(row, c0 + 8 * GT * i, K, vec_in, a[i]);
          load_chunk<FULL>(row + K, c0 + 8 * GT * i, K, vec_in, u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          h[i][2 * j] = silu_mul_bf16_round(lo_bf16(a[i][j]), lo_bf16(u[j]));
          h[i][2 * j + 1] = silu_mul_bf16_round(hi_bf16(a[i][j]), hi_bf16(u[j]));
          amax = fmaxf(amax, fmaxf(fabsf(h[i][2 * j]), fabsf(h[i][2 * j + 1])));
        }
      }
#pragma unroll
      for (int o = 1; o < GT; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    } else {
      uint32_t mx = 0u;
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0u;
        if (ok) load_chunk<FULL>(row, c0 + 8 * GT * i, K, vec_in, a[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max_u16x2(mx, a[i][j] & 0x7FFF7FFFu);
      }
      // |x| of a finite BF16 orders like its bit pattern with the sign cleared
      uint32_t am = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
      for (int o = 1; o < GT; o <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
      amax = __uint_as_float(am << 16);
    }
    const float sc = group_scale(amax);
    const float rc = __frcp_rn(sc);
    const float2 y2 = make_float2(rc, rc), ns2 = make_float2(-sc, -sc);
    uint8_t* qrow = q + (live ? m : 0) * ldq;
#pragma unroll
    for (int i = 0; i < kCh; ++i) {
      uint16_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = SILU ? make_float2(h[SILU ? i : 0][2 * j], h[SILU ? i : 0][2 * j + 1])
                              : make_float2(lo_bf16(a[i][j]), hi_bf16(a[i][j]));
        const float2 qv = div_by_scale2(v, ns2, y2);
        p[j] = f32x2_to_e4m3x2(qv.x, qv.y);
      }
      const uint32_t w0 = static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 16);
      const uint32_t w1 = static_cast<uint32_t>(p[2]) | (static_cast<uint32_t>(p[3]) << 16);
      const int64_t c = c0 + 8 * GT * i;
      if (!live) continue;
      if (FULL || (vec_out && c + 8 <= K)) {
        *reinterpret_cast<uint2*>(qrow + c) = make_uint2(w0, w1);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c + e < K) qrow[c + e] = static_cast<uint8_t>((e < 4 ? w0 : w1) >> (8 * (e & 3)));
      }
    }
    if (live && ql == 0) s[m * ssm + g * sskb] = sc;
    m += dm;
    g += dg;
    if (g >= Kb) {
      g -= Kb;
      ++m;
    }
  }
}

// h[m, c] = bf16(silu(gu[m, c]) * gu[m, I + c]) for the W8A16 arm (no
// quantization). Each thread owns 8 consecutive columns of one row; with
// `vec`, 16-byte loads and stores.
__global__ void __launch_bounds__(kThreads) silu_mul_kernel(
    const __nv_bfloat16* __restrict__ gu, int64_t M, int64_t I, int64_t ld,
    __nv_bfloat16* __restrict__ h, int64_t ldh, int vec) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t cpr = (I + 7) / 8;  // 8-column chunks per row
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < M * cpr;
       it += step) {
    const int64_t m = it / cpr;
    const int64_t c = (it - m * cpr) * 8;
    const __nv_bfloat16* row = gu + m * ld;
    uint32_t g[4], u[4];
    load_chunk<false>(row, c, I, vec, g);
    load_chunk<false>(row + I, c, I, vec, u);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float h0 = silu_mul_bf16_round(lo_bf16(g[j]), lo_bf16(u[j]));
      const float h1 = silu_mul_bf16_round(hi_bf16(g[j]), hi_bf16(u[j]));
      o[j] = (__float_as_uint(h0) >> 16) | (__float_as_uint(h1) & 0xFFFF0000u);
    }
    __nv_bfloat16* dst = h + m * ldh + c;
    if (vec && c + 8 <= I) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c + e < I) d16[e] = static_cast<uint16_t>(o[e >> 1] >> (16 * (e & 1)));
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

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// out[t, c] = bf16( sum_j w[t, j] * y[rows[t, j], c] ), FP32 fused multiply-adds
// in slot order j (deterministic). A row index outside [0, R) adds nothing.
// Each thread owns 8 consecutive columns of one token; the slots are fetched
// kSlotBatch at a time, all loads issued before the first multiply-add.
constexpr int kSlotBatch = 8;

__global__ void __launch_bounds__(kThreads) moe_combine_kernel(
    const __nv_bfloat16* __restrict__ y, int64_t R, int64_t H, int64_t ldy,
    const int32_t* __restrict__ rows, const float* __restrict__ w, int64_t T, int topk,
    __nv_bfloat16* __restrict__ out, int64_t ldo, int vec) {
  // a programmatic dependent of the previous kernel: wait before any access
  pdl_launch_dependents();
  pdl_wait();
  const int64_t hc = (H + 7) / 8;
  const int64_t it0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t t = it0 / hc, cc = it0 - t * hc;
  const int64_t dt = step / hc, dc = step - dt * hc;
  for (; t < T; t += dt, cc += dc) {
    if (cc >= hc) {
      cc -= hc;
      ++t;
      if (t >= T) break;
    }
    const int64_t c = cc * 8;
    const bool full = vec && c + 8 <= H;
    float2 acc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.0f, 0.0f);
    const int32_t* rt = rows + t * topk;
    const float* wt = w + t * topk;
    for (int j0 = 0; j0 < topk; j0 += kSlotBatch) {
      int64_t r[kSlotBatch];
      float wj[kSlotBatch];
      uint4 raw[kSlotBatch];
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u) {
        const bool in = j0 + u < topk;
        r[u] = in ? static_cast<int64_t>(__ldg(rt + j0 + u)) : -1;
        wj[u] = in ? __ldg(wt + j0 + u) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u) {
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r[u] < 0 || r[u] >= R) continue;
        const __nv_bfloat16* src = y + r[u] * ldy + c;
        if (full) {
          raw[u] = __ldg(reinterpret_cast<const uint4*>(src));
        } else {
          const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
          uint32_t wd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t lo = c + 2 * e < H ? s16[2 * e] : 0u;
            const uint32_t hi = c + 2 * e + 1 < H ? s16[2 * e + 1] : 0u;
            wd[e] = lo | (hi << 16);
          }
          raw[u] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
      }
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u) {
        if (r[u] < 0 || r[u] >= R) continue;
        const float2 w2 = make_float2(wj[u], wj[u]);
        const uint32_t wd[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc[e] = __ffma2_rn(w2, make_float2(lo_bf16(wd[e]), hi_bf16(wd[e])), acc[e]);
      }
    }
    __nv_bfloat16* dst = out + t * ldo + c;
    if (full) {
      uint4 o;
      o.x = pack_bf16x2(acc[0].x, acc[0].y);
      o.y = pack_bf16x2(acc[1].x, acc[1].y);
      o.z = pack_bf16x2(acc[2].x, acc[2].y);
      o.w = pack_bf16x2(acc[3].x, acc[3].y);
      *reinterpret_cast<uint4*>(dst) = o;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c + e < H) dst[e] = __float2bfloat16_rn(e & 1 ? acc[e >> 1].y : acc[e >> 1].x);
    }
  }
}

// Launch as a programmatic dependent of the previous work on the stream (the
// kernels wait for it before any memory access).
template <typename Kernel, typename... Args>
int launch_dependent(Kernel kernel, unsigned blocks, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? BFP8_OK : BFP8_ERR_CUDA;
}

// Blocks of kThreads that one SM keeps resident for `kernel` (at least 1):
// the grid-stride kernels launch exactly one wave of them.
template <typename Kernel>
int resident_blocks(Kernel kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 1;
  }
  return n;
}

int act_quant_common(bool silu, const void* x, int64_t M, int64_t K, int64_t ld, void* q,
                     int64_t ldq, float* s, int64_t ssm, int64_t sskb, void* stream,
                     const int32_t* rows = nullptr, int64_t n_src = 0, int32_t* clr = nullptr,
                     int32_t n_clr = 0) {
  if (M < 0 || K < 0 || n_clr < 0) return BFP8_ERR_INVALID_ARG;
  // an empty input launches nothing, so it cannot carry a counter clear
  if (M == 0 || K == 0) return clr ? BFP8_ERR_INVALID_ARG : BFP8_OK;
  if (!x || !q || !s) return BFP8_ERR_INVALID_ARG;
  const int64_t width = silu ? 2 * K : K;
  if (ld < width || ldq < K) return BFP8_ERR_INVALID_ARG;
  const int64_t Kb = (K + 127) / 128;
  if (ssm < 0 || sskb < 0 || (M > 1 && ssm == 0) || (Kb > 1 && sskb == 0))
    return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({x, q, s, rows, clr});
  if (rc != BFP8_OK) return rc;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const int vec_in = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld % 8 == 0) && (K % 8 == 0);
  const int vec_out = (reinterpret_cast<uintptr_t>(q) % 8 == 0) && (ldq % 8 == 0);
  const bool full = vec_in && vec_out && K % 128 == 0;
  static const int per_sm[4] = {
      resident_blocks(act_quant_kernel<false, false>), resident_blocks(act_quant_kernel<true, false>),
      resident_blocks(act_quant_kernel<false, true>), resident_blocks(act_quant_kernel<true, true>)};
  const int64_t items = M * Kb;
  // 16 lanes a group when 4 would not give every SM two blocks
  const bool wide = items * kQuad < static_cast<int64_t>(2 * sms) * kThreads;
  const int64_t per_block = kThreads / (wide ? 16 : kQuad);   // groups one block covers per pass
  const int64_t want = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm[(silu ? 1 : 0) + (full ? 2 : 0)];
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto go = [&](auto kernel) {
    return launch_dependent(kernel, blocks, st, static_cast<const __nv_bfloat16*>(x), M, K, ld,
                            static_cast<uint8_t*>(q), ldq, s, ssm, sskb, vec_in, vec_out, rows,
                            rows ? n_src : M, clr, clr ? n_clr : 0);
  };
  int lrc;
  if (wide)
    lrc = silu ? (full ? go(act_quant_kernel<true, true, 16>) : go(act_quant_kernel<true, false, 16>))
               : (full ? go(act_quant_kernel<false, true, 16>) : go(act_quant_kernel<false, false, 16>));
  else
    lrc = silu ? (full ? go(act_quant_kernel<true, true>) : go(act_quant_kernel<true, false>))
               : (full ? go(act_quant_kernel<false, true>) : go(act_quant_kernel<false, false>));
  if (lrc != BFP8_OK) return lrc;
  return check_launch();
}

}  // namespace

int launch_act_quant(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                     float* s, int64_t ssm, int64_t sskb, void* stream, int32_t* clear,
                     int32_t n_clear) {
  return act_quant_common(false, x, M, K, ldx, q, ldq, s, ssm, sskb, stream, nullptr, 0, clear,
                          n_clear);
}

int launch_silu_mul_act_quant(const void* gu, int64_t M, int64_t I, int64_t ld, void* q,
                              int64_t ldq, float* s, int64_t ssm, int64_t sskb, void* stream,
                              int32_t* clear, int32_t n_clear) {
  return act_quant_common(true, gu, M, I, ld, q, ldq, s, ssm, sskb, stream, nullptr, 0, clear,
                          n_clear);
}

int launch_silu_mul(const void* gu, int64_t M, int64_t I, int64_t ld, void* h, int64_t ldh,
                    void* stream) {
  if (M < 0 || I < 0) return BFP8_ERR_INVALID_ARG;
  if (M == 0 || I == 0) return BFP8_OK;
  if (!gu || !h || ld < 2 * I || ldh < I) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({gu, h});
  if (rc != BFP8_OK) return rc;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const int vec = (reinterpret_cast<uintptr_t>(gu) % 16 == 0) && (ld % 8 == 0) && (I % 8 == 0) &&
                  (reinterpret_cast<uintptr_t>(h) % 16 == 0) && (ldh % 8 == 0);
  static const int per_sm = resident_blocks(silu_mul_kernel);
  const int64_t items = M * ((I + 7) / 8);
  const int64_t want = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  rc = launch_dependent(silu_mul_kernel, blocks, static_cast<cudaStream_t>(stream),
                        static_cast<const __nv_bfloat16*>(gu), M, I, ld,
                        static_cast<__nv_bfloat16*>(h), ldh, vec);
  if (rc != BFP8_OK) return rc;
  return check_launch();
}

int launch_moe_gather_act_quant(const void* x, int64_t T, int64_t H, int64_t ldx,
                                const int32_t* row_token, int64_t R, void* q, int64_t ldq,
                                float* s, int64_t ssm, int64_t sskb, void* stream) {
  if (T < 0 || R < 0 || H < 0) return BFP8_ERR_INVALID_ARG;
  if (R == 0 || H == 0) return BFP8_OK;
  if (!row_token) return BFP8_ERR_INVALID_ARG;
  return act_quant_common(false, x, R, H, ldx, q, ldq, s, ssm, sskb, stream, row_token, T);
}

int launch_moe_combine(const void* y, int64_t R, int64_t H, int64_t ldy, const int32_t* token_rows,
                       const float* token_weights, int64_t T, int32_t topk, void* out, int64_t ldo,
                       void* stream) {
  if (R < 0 || H < 0 || T < 0 || topk < 1) return BFP8_ERR_INVALID_ARG;
  if (T == 0 || H == 0) return BFP8_OK;
  if (!y || !token_rows || !token_weights || !out || ldy < H || ldo < H) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({y, token_rows, token_weights, out});
  if (rc != BFP8_OK) return rc;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const int vec = (reinterpret_cast<uintptr_t>(y) % 16 == 0) && (ldy % 8 == 0) &&
                  (reinterpret_cast<uintptr_t>(out) % 16 == 0) && (ldo % 8 == 0);
  static const int per_sm = resident_blocks(moe_combine_kernel);
  const int64_t items = T * ((H + 7) / 8);
  const int64_t want = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  rc = launch_dependent(moe_combine_kernel, blocks, static_cast<cudaStream_t>(stream),
                        static_cast<const __nv_bfloat16*>(y), R, H, ldy, token_rows,
                        token_weights, T, static_cast<int>(topk),
                        static_cast<__nv_bfloat16*>(out), ldo, vec);
  if (rc != BFP8_OK) return rc;
  return check_launch();
}

int launch_weight_quant(const float* w, int64_t N, int64_t K, int64_t ldw, void* q, int64_t ldq,
                        void* scale, int32_t scale_dtype, void* stream) {
  if (N < 0 || K < 0) return BFP8_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return BFP8_OK;
  if (!w || !q || !scale || ldw < K || ldq < K) return BFP8_ERR_INVALID_ARG;
  if (scale_dtype != BFP8_DT_BF16 && scale_dtype != BFP8_DT_F32) return BFP8_ERR_SCALE_DTYPE;
  const int64_t Nb = (N + 127) / 128, Kb = (K + 127) / 128;
  if (Nb > 65535 || Kb > 0x7FFFFFFF) return BFP8_ERR_UNSUPPORTED;
  const int rc = check_device_ptrs({w, q, scale});
  if (rc != BFP8_OK) return rc;
  dim3 grid(static_cast<unsigned>(Kb), static_cast<unsigned>(Nb));
  weight_quant_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      w, N, K, ldw, static_cast<uint8_t*>(q), ldq, scale, scale_dtype == BFP8_DT_F32, Kb);
  return check_launch();
}

}  // namespace bfp8
