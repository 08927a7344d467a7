// gemv_decode.cu -- the memory-bound small-M (decode) block-FP8 projection.
//
//   y[m, n] = sum_kb s_w[r(n), kb] * sum_{k in kb} x[m, k] * e4m3(W[n, k]),  1 <= M <= 16
//
// W8A16 arithmetic: BF16 tokens, E4M3 weights decoded exactly, FP32
// accumulation, block multipliers applied inside the reduction [Qwen
// checkpoints with block FP8 weights, paragraph 2]. The GB10 design on the
// pages is an unfused per-projection GEMV [Module w8a8_prefill, "Reachability"].
//
// Design for GB300:
//   * Work unit = 128 weight rows x one 128-wide K-block (16 KB of E4M3).
//     There are ceil(N/128) * ceil(K/128) units. They are split into equal
//     contiguous ranges over one persistent CTA per SM (stream-K), so every
//     SM streams the same number of bytes whatever N and K are.
//   * Warp 0 streams units into an 8-deep ring with TMA (128-byte swizzle):
//     the weight tile plus the matching 128-column slice of x (up to 16
//     tokens). 160 KB stays in flight per SM, which covers HBM latency.
//   * Warps 1-8 work in four pairs. Unit i goes to pair i % 4, and each warp
//     of the pair owns 64 of the 128 rows. A warp reads 16-byte chunks of its
//     rows and runs the legacy m16n8k16 MMA with tokens as the n dimension,
//     on F16 operands:
//       - E4M3 -> F16 is one exact conversion per two weights.
//       - Each token's 128 BF16 values of the K-block are multiplied by a
//         power of two 2^e chosen so that their maximum lies in [2^14, 2^15),
//         then converted to F16. A BF16 significand (8 bits) fits F16's 11,
//         so every value within 28 binades of its row's maximum is carried
//         exactly, and every product x * w is formed exactly, as with BF16
//         operands.
//     The per-K-block FP32 partial is multiplied by 2^-e (exact) and by the
//     block's weight scale. The permutation of K inside a 64-wide half is the
//     same for both operands, so the sums are unchanged.
//   * At the end of a row tile's segment, the four pairs' accumulators are
//     summed through shared memory. A CTA that owns a whole row tile writes
//     BF16 directly. Partial tiles go to the workspace, and the last CTA to
//     arrive sums the partials in CTA order (deterministic) and writes y. No
//     CTA ever waits on another.
#include <mutex>

#include "bfp8_internal.h"
#include "ptx.cuh"

namespace bfp8 {

namespace {
using namespace dev;

__device__ int g_gemv_err;

constexpr int kRows = 128;          // weight rows per unit
constexpr int kStages = 8;          // must be a multiple of 4 (pairs own stages s, s+4)
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr uint32_t kWBytes = kRows * 128;
constexpr uint32_t kRedBytes = 4 * kRows * 16 * 4;
constexpr unsigned long long kDrainLimitNs = 100000000ull;

template <int NTB>
struct GCfg {
  static constexpr int kMB = 8 * NTB;                        // token rows per x half-tile
  static constexpr uint32_t kXHalf = kMB * 128;
  static constexpr uint32_t kStage = kWBytes + 2 * kXHalf;   // multiple of 1024
  static constexpr uint32_t kTmaBytes = kStage;
  static constexpr uint32_t kOffRed = kStages * kStage;
  static constexpr uint32_t kOffBar = kOffRed + kRedBytes;
  static constexpr uint32_t kOffMisc = kOffBar + 2 * kStages * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct GemvParams {
  int32_t M, N, K, Kb, RT;
  int64_t U;  // RT * Kb
  int32_t grid;
  const void* s_w;
  int32_t sw_f32;
  int32_t n_members;
  int32_t mem_n0[BFP8_MAX_MEMBERS], mem_rows[BFP8_MAX_MEMBERS], mem_sbase[BFP8_MAX_MEMBERS];
  __nv_bfloat16* y;
  int64_t ldy;
  int32_t* counters;  // [RT], zero at kernel start
  float* partials;    // [grid][2][128][16]
};

BFP8_DEV int64_t unit_begin(const GemvParams& p, int64_t c) { return (c * p.U) / p.grid; }
// The CTA whose range [unit_begin(c), unit_begin(c+1)) holds unit u.
BFP8_DEV int64_t cta_of_unit(const GemvParams& p, int64_t u) {
  return ((u + 1) * p.grid + p.U - 1) / p.U - 1;
}

BFP8_DEV int scale_row_of(const GemvParams& p, int n) {
  if (n >= p.N) return 0;
  int i = 0;
#pragma unroll 1
  while (i + 1 < p.n_members && n >= p.mem_n0[i + 1]) ++i;
  return p.mem_sbase[i] + (n - p.mem_n0[i]) / 128;
}

BFP8_DEV float load_scale(const GemvParams& p, int64_t idx) {
  return p.sw_f32 ? __ldg(static_cast<const float*>(p.s_w) + idx)
                  : bf16_bits_to_f32(__ldg(static_cast<const uint16_t*>(p.s_w) + idx));
}

BFP8_DEV bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && globaltimer() - t0 > limit_ns) return false;
  }
}

BFP8_DEV void raise_abort(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(&g_gemv_err, static_cast<int>(BFP8_ERR_TIMEOUT));
}

template <int NTB>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ GemvParams p) {
  using C = GCfg<NTB>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_u32);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kOffMisc);
  volatile int* last_flag = reinterpret_cast<volatile int*>(base_ptr + C::kOffMisc + 4);
  float* red = reinterpret_cast<float*>(base_ptr + C::kOffRed);

  const int64_t ub = unit_begin(p, blockIdx.x);
  const int64_t ue = unit_begin(p, blockIdx.x + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 2);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      for (int64_t i = 0; ub + i < ue; ++i) {
        const int s = static_cast<int>(i % kStages);
        const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
        if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) { ok = false; break; }
        const int64_t u = ub + i;
        const int rt = static_cast<int>(u / p.Kb);
        const int kb = static_cast<int>(u - static_cast<int64_t>(rt) * p.Kb);
        const uint32_t sW = base + s * C::kStage;
        const uint32_t sX = sW + kWBytes;
        mbar_arrive_expect_tx(full_bar(s), C::kTmaBytes);
        tma_load_2d(sW, &tmW, kb * 128, rt * kRows, full_bar(s));
        tma_load_2d(sX, &tmX, kb * 128, 0, full_bar(s));
        tma_load_2d(sX + C::kXHalf, &tmX, kb * 128 + 64, 0, full_bar(s));
        armed |= 1u << s;
        armed_phase = (armed_phase & ~(1u << s)) | (ph << s);
      }
      if (!ok) raise_abort(abort_flag);
      for (int s = 0; s < kStages; ++s)
        if ((armed >> s) & 1u) wait_bounded(full_bar(s), (armed_phase >> s) & 1u, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int pair = cw >> 1, hw = cw & 1;
    const int g = lane >> 2, t = lane & 3;
    const int ct = threadIdx.x - 32;  // 0..255
    bool ok = true;
    int64_t u = ub;
    while (u < ue) {
      const int rt = static_cast<int>(u / p.Kb);
      const int64_t tile_u0 = static_cast<int64_t>(rt) * p.Kb;
      const int64_t seg_end = min(ue, tile_u0 + p.Kb);
      const int64_t i0 = u - ub, i1 = seg_end - ub;
      int64_t srow_idx[4][2];
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          srow_idx[rg][hh] =
              static_cast<int64_t>(scale_row_of(p, rt * kRows + 64 * hw + 16 * rg + g + 8 * hh)) * p.Kb;
      float acc[4][NTB][4];
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int tb = 0; tb < NTB; ++tb)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[rg][tb][c] = 0.0f;

      if (ok) {
        for (int64_t i = i0 + ((pair - i0 % 4 + 4) % 4); i < i1; i += 4) {
          const int s = static_cast<int>(i % kStages);
          const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
          const int kb = static_cast<int>(ub + i - tile_u0);
          float sc[4][2];
#pragma unroll
          for (int rg = 0; rg < 4; ++rg)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) sc[rg][hh] = load_scale(p, srow_idx[rg][hh] + kb);
          const bool w_ok = mbar_wait(full_bar(s), ph, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
          const uint32_t sW = base + s * C::kStage;
          const uint32_t sX = sW + kWBytes;
          // x fragments: token row r = 8*tb + g, 16 values at K offset 16*t of each half
          uint32_t xf[2][NTB][8];
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int tb = 0; tb < NTB; ++tb) {
              const int r = 8 * tb + g;
              const uint32_t rowa = sX + half * C::kXHalf + r * 128;
              const uint4 v0 = lds128(rowa + (static_cast<uint32_t>((2 * t) ^ (r & 7)) << 4));
              const uint4 v1 = lds128(rowa + (static_cast<uint32_t>((2 * t + 1) ^ (r & 7)) << 4));
              xf[half][tb][0] = v0.x; xf[half][tb][1] = v0.y; xf[half][tb][2] = v0.z; xf[half][tb][3] = v0.w;
              xf[half][tb][4] = v1.x; xf[half][tb][5] = v1.y; xf[half][tb][6] = v1.z; xf[half][tb][7] = v1.w;
            }
          // BF16 -> F16 with a power of two per token: the quad of lanes
          // holding token row 8*tb + g finds the row's max |x| exponent E,
          // scales by 2^e, e = 141 - E (so the max lands in [2^14, 2^15)),
          // and hands 2^-e to the lanes whose accumulator columns are that
          // token. Non-negative BF16 patterns order like their values.
          float xinv[NTB][2];
#pragma unroll
          for (int tb = 0; tb < NTB; ++tb) {
            uint32_t m = 0;
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int j = 0; j < 8; ++j) m = __vmaxu2(m, xf[half][tb][j] & 0x7FFF7FFFu);
            m = max(m & 0xFFFFu, m >> 16);
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const int e = min(max(141 - static_cast<int>((m >> 7) & 0xFFu), -126), 126);
            const float up = __int_as_float((e + 127) << 23);
            const float dn = __int_as_float((127 - e) << 23);
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint32_t w = xf[half][tb][j];
                xf[half][tb][j] = f32x2_to_f16x2(__uint_as_float(w << 16) * up,
                                                 __uint_as_float(w & 0xFFFF0000u) * up);
              }
            xinv[tb][0] = __shfl_sync(0xffffffffu, dn, 8 * t);       // token 8*tb + 2t
            xinv[tb][1] = __shfl_sync(0xffffffffu, dn, 8 * t + 4);   // token 8*tb + 2t + 1
          }
#pragma unroll
          for (int rg = 0; rg < 4; ++rg) {
            float part[NTB][4];
#pragma unroll
            for (int tb = 0; tb < NTB; ++tb)
#pragma unroll
              for (int c = 0; c < 4; ++c) part[tb][c] = 0.0f;
            const int r_lo = 64 * hw + 16 * rg + g;
            const int r_hi = r_lo + 8;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint4 wl = lds128(sW + r_lo * 128 + (static_cast<uint32_t>((4 * half + t) ^ (r_lo & 7)) << 4));
              const uint4 wh = lds128(sW + r_hi * 128 + (static_cast<uint32_t>((4 * half + t) ^ (r_hi & 7)) << 4));
              const uint32_t wlw[4] = {wl.x, wl.y, wl.z, wl.w};
              const uint32_t whw[4] = {wh.x, wh.y, wh.z, wh.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(wlw[j] & 0xFFFFu));
                const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(wlw[j] >> 16));
                const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(whw[j] & 0xFFFFu));
                const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(whw[j] >> 16));
#pragma unroll
                for (int tb = 0; tb < NTB; ++tb)
                  mma_f16_16816(part[tb], a0, a1, a2, a3, xf[half][tb][2 * j], xf[half][tb][2 * j + 1]);
              }
            }
#pragma unroll
            for (int tb = 0; tb < NTB; ++tb) {
              // undo the token scale first (exact), then apply the block scale
              acc[rg][tb][0] = fmaf(part[tb][0] * xinv[tb][0], sc[rg][0], acc[rg][tb][0]);
              acc[rg][tb][1] = fmaf(part[tb][1] * xinv[tb][1], sc[rg][0], acc[rg][tb][1]);
              acc[rg][tb][2] = fmaf(part[tb][2] * xinv[tb][0], sc[rg][1], acc[rg][tb][2]);
              acc[rg][tb][3] = fmaf(part[tb][3] * xinv[tb][1], sc[rg][1], acc[rg][tb][3]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty_bar(s));
        }
      }
      // ---- segment reduction over the four pairs
#pragma unroll
      for (int rg = 0; rg < 4; ++rg)
#pragma unroll
        for (int tb = 0; tb < NTB; ++tb) {
          const int r_lo = 64 * hw + 16 * rg + g;
          const int tok = 8 * tb + 2 * t;
          float* lo = red + ((pair * kRows + r_lo) * 16 + tok);
          float* hi = red + ((pair * kRows + r_lo + 8) * 16 + tok);
          *reinterpret_cast<float2*>(lo) = make_float2(acc[rg][tb][0], acc[rg][tb][1]);
          *reinterpret_cast<float2*>(hi) = make_float2(acc[rg][tb][2], acc[rg][tb][3]);
        }
      named_bar_sync(1, 32 * kConsumerWarps);
      const int row = ct >> 1;
      const int tk0 = (ct & 1) * 8;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        const float4* src = reinterpret_cast<const float4*>(red + ((pr * kRows + row) * 16 + tk0));
        const float4 a = src[0], b = src[1];
        v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
        v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
      }
      const int n = rt * kRows + row;
      const bool whole = (u == tile_u0) && (seg_end == tile_u0 + p.Kb);
      if (whole) {
        if (n < p.N)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (tk0 + j < p.M) p.y[static_cast<int64_t>(tk0 + j) * p.ldy + n] = __float2bfloat16_rn(v[j]);
      } else {
        const int slot = (u == ub) ? 0 : 1;
        float* dst = p.partials + ((static_cast<int64_t>(blockIdx.x) * 2 + slot) * kRows + row) * 16 + tk0;
        reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
        __threadfence();
        named_bar_sync(1, 32 * kConsumerWarps);
        const int64_t c_first = cta_of_unit(p, tile_u0);
        const int64_t c_last = cta_of_unit(p, tile_u0 + p.Kb - 1);
        if (ct == 0) {
          const int old = atomicAdd(p.counters + rt, 1);
          *last_flag = (old == static_cast<int>(c_last - c_first)) ? 1 : 0;
        }
        named_bar_sync(1, 32 * kConsumerWarps);
        if (*last_flag) {
          __threadfence();
          float s[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = 0.0f;
          for (int64_t c = c_first; c <= c_last; ++c) {
            const int sl = (unit_begin(p, c) >= tile_u0) ? 0 : 1;
            const float4* srcp = reinterpret_cast<const float4*>(
                p.partials + ((c * 2 + sl) * kRows + row) * 16 + tk0);
            const float4 a = __ldcg(srcp), b = __ldcg(srcp + 1);
            s[0] += a.x; s[1] += a.y; s[2] += a.z; s[3] += a.w;
            s[4] += b.x; s[5] += b.y; s[6] += b.z; s[7] += b.w;
          }
          if (n < p.N)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (tk0 + j < p.M) p.y[static_cast<int64_t>(tk0 + j) * p.ldy + n] = __float2bfloat16_rn(s[j]);
          if (ct == 0) p.counters[rt] = 0;
        }
      }
      named_bar_sync(1, 32 * kConsumerWarps);
      u = seg_end;
    }
    if (!ok) raise_abort(abort_flag);
  }
  __syncthreads();
}

template <int NTB>
int launch_t(const CUtensorMap& tw, const CUtensorMap& tx, const GemvParams& p, void* stream) {
  using C = GCfg<NTB>;
  auto kernel = gemv_kernel<NTB>;
  int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), C::kSmemBytes);
  if (rc != BFP8_OK) return rc;
  kernel<<<p.grid, kThreads, C::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(tw, tx, p);
  return check_launch();
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K, int sms) {
  (void)M;
  (void)K;
  if (N <= 0 || sms <= 0) return 0;
  const int64_t RT = (N + kRows - 1) / kRows;
  return align256(static_cast<size_t>(RT) * 4) +
         static_cast<size_t>(sms) * 2 * kRows * 16 * sizeof(float);
}

int launch_gemv(const void* x, int64_t ldx, const void* w, const void* w_scale,
                int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y, int64_t ldy,
                const MemberTable& mt, void* workspace, size_t ws_bytes, void* stream) {
  if (K % 16 != 0 || ldx % 8 != 0) return BFP8_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(w) % 16 != 0)
    return BFP8_ERR_UNSUPPORTED;
  if (N > 0x7FFFFFFF || K > 0x7FFFFFFF) return BFP8_ERR_UNSUPPORTED;
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const size_t need = gemv_workspace_bytes(M, N, K, sms);
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return BFP8_ERR_INVALID_ARG;
  GemvParams p{};
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + 127) / 128);
  p.RT = static_cast<int32_t>((N + kRows - 1) / kRows);
  p.U = static_cast<int64_t>(p.RT) * p.Kb;
  p.grid = static_cast<int32_t>(p.U < sms ? p.U : sms);
  p.s_w = w_scale;
  p.sw_f32 = w_scale_dtype == BFP8_DT_F32;
  p.n_members = mt.count;
  for (int i = 0; i < mt.count; ++i) {
    p.mem_n0[i] = static_cast<int32_t>(mt.n0[i]);
    p.mem_rows[i] = static_cast<int32_t>(mt.rows[i]);
    p.mem_sbase[i] = static_cast<int32_t>(mt.sbase[i]);
  }
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  p.counters = static_cast<int32_t*>(workspace);
  p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        align256(static_cast<size_t>(p.RT) * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, static_cast<size_t>(p.RT) * 4, st) != cudaSuccess)
    return BFP8_ERR_CUDA;
  const int ntb = M <= 8 ? 1 : 2;
  const uint32_t mb = 8u * ntb;
  CUtensorMap tw, tx;
  rc = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, 128, kRows,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  rc = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, 64, mb,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  return ntb == 1 ? launch_t<1>(tw, tx, p, stream) : launch_t<2>(tw, tx, p, stream);
}

// ---------------------------------------------------------------------------
// bfp8_gemv_decode_noalloc: the decode GEMV for callers that cannot allocate
// device memory. Its split-K scratch (tile counters + partial tiles) lives in
// this fixed array instead of a caller-provided workspace. Every GPU that
// loads the library holds the array until the process exits. All calls on one
// device share it, so calls that overlap on the GPU race.
static __device__ __align__(256) unsigned char g_gemv_noalloc_scratch[BFP8_GEMV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
NoAllocSlot g_noalloc_slots[kNoAllocMaxDevices];

// The host-side name of a __device__ array is only a stand-in, not a device
// address, so look the real address up once per device, with that device
// current (the first call on each device does this).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BFP8_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return BFP8_ERR_UNSUPPORTED;
  NoAllocSlot& slot = g_noalloc_slots[dev];
  std::call_once(slot.once, [&slot] {
    slot.err = cudaGetSymbolAddress(&slot.ptr, g_gemv_noalloc_scratch);
  });
  if (slot.err != cudaSuccess || slot.ptr == nullptr) return BFP8_ERR_CUDA;
  *out = slot.ptr;
  return BFP8_OK;
}

}  // namespace

int gemv_read_clear_error() {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_err, sizeof(int)) != cudaSuccess) return BFP8_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_gemv_err, &zero, sizeof(int)) != cudaSuccess)
    return BFP8_ERR_CUDA;
  return v == 0 ? BFP8_OK : v;
}

}  // namespace bfp8

extern "C" int bfp8_gemv_decode_noalloc(const void* x_bf16, int64_t ldx, const void* w_e4m3,
                                        const void* w_scale, int32_t w_scale_dtype, int64_t M,
                                        int64_t N, int64_t K, void* y_bf16, int64_t ldy,
                                        const bfp8_members* members, void* stream) {
  using namespace bfp8;
  if (M < 1 || M > 16 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (!x_bf16 || !w_e4m3 || !w_scale || !y_bf16 || ldy < N || ldx < K)
    return BFP8_ERR_INVALID_ARG;
  if (w_scale_dtype != BFP8_DT_BF16 && w_scale_dtype != BFP8_DT_F32) return BFP8_ERR_SCALE_DTYPE;
  MemberTable mt;
  int rc = resolve_members(N, members, &mt);
  if (rc != BFP8_OK) return rc;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  if (gemv_workspace_bytes(M, N, K, sms) > BFP8_GEMV_NOALLOC_SCRATCH_BYTES)
    return BFP8_ERR_UNSUPPORTED;  // the problem needs more scratch than the fixed array holds
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != BFP8_OK) return rc;
  return launch_gemv(x_bf16, ldx, w_e4m3, w_scale, w_scale_dtype, M, N, K, y_bf16, ldy, mt,
                     scratch, BFP8_GEMV_NOALLOC_SCRATCH_BYTES, stream);
}
