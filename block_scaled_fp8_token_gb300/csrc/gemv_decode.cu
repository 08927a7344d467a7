// gemv_decode.cu -- the memory-bound small-M (decode) block-FP8 projection.
//
//   y[m, n] = sum_kb s_w[r(n), kb] * sum_{k in kb} x[m, k] * e4m3(W[n, k]),  1 <= M <= 16
//
// W8A16 arithmetic: BF16 tokens, E4M3 weights, FP32 accumulation, block
// multipliers applied inside the reduction [Qwen checkpoints with block FP8
// weights, paragraph 2]. The GB10 design on the pages is an unfused
// per-projection GEMV [Module w8a8_prefill, "Reachability"].
//
// Design for GB300: the weights go from HBM to the tensor cores untouched.
//   * Work unit = 128 weight rows x one 128-wide K-block (16 KB of E4M3).
//     There are ceil(N/128) * ceil(K/128) units. They are split into equal
//     contiguous ranges over one persistent CTA per SM (stream-K), so every
//     SM streams the same number of bytes whatever N and K are.
//   * A small kernel first turns the tokens into the MMA's B operand, once
//     per K-block. Token m's 128 values are multiplied by a power of two 2^e
//     that puts their maximum in [2^7, 2^8). Each scaled value v is written as
//     two E4M3 terms, hi = e4m3(v) and lo = e4m3(v - hi), in rows m and 16 + m
//     of a 32 x 128 byte tile; 2^-e goes to a small table. A BF16 significand
//     has 8 bits, hi keeps 4 and the remainder needs at most 4, so
//     hi + lo == v exactly for every value within 2^-10 of the maximum.
//     Smaller values are carried to within 2^-10 in the scaled units, that
//     is max|x| * 2^-18. The GEMV is launched behind it as a programmatic
//     dependent launch: it starts streaming weights at once and waits for
//     the token tiles (griddepcontrol.wait) only before it first needs them.
//   * Warp 4 streams units into an 8-slot ring with TMA: the weight tile and
//     the K-block's token tile, both with the 128-byte swizzle of the tcgen05
//     K-major layout. Slots are filled and released in groups of kGroup
//     consecutive units under one barrier: HBM delivers several 16 KB tiles
//     per barrier round trip much faster than one.
//   * Warp 5 issues four tcgen05.mma kind::f8f6f4 (M = 128 weight rows,
//     N = 32, K = 32) per unit into one of eight 32-column TMEM buffers:
//     exact E4M3 products, FP32 accumulation.
//   * Warps 0-3 (one TMEM lane quarter each, one weight row per thread) add
//     the hi and lo columns, undo 2^e (exact), apply the block's weight scale
//     and accumulate the 16 token sums in FP32 registers.
//   * A CTA that owns a whole row tile writes BF16 directly. Partial tiles
//     go to the workspace. Warp 6 publishes each partial with one
//     acquire-release atomic on the tile's counter while the epilogue goes
//     on; the CTA that arrives last on a tile sums its partials in CTA order
//     (deterministic) and writes y at the end. No CTA ever waits on another.
#include <mutex>

#include "bfp8_internal.h"
#include "ptx.cuh"
#include "act_math.cuh"

namespace bfp8 {

namespace {
using namespace dev;

__device__ int g_gemv_err;

constexpr int kRows = 128;           // weight rows per unit (the MMA's M)
#ifndef BFP8_GEMV_GROUP
#define BFP8_GEMV_GROUP 4
#endif
#ifndef BFP8_GEMV_SLOTS
#define BFP8_GEMV_SLOTS 8
#endif
constexpr int kStages = BFP8_GEMV_SLOTS;  // unit slots in shared memory
constexpr int kGroup = BFP8_GEMV_GROUP;  // consecutive units per fill / release
constexpr int kGroups = kStages / kGroup;
constexpr int kTBufs = 8;            // TMEM partial buffers, 32 columns each
constexpr int kThreads = 224;        // warps 0-3 epilogue, 4 producer, 5 MMA, 6 publisher
constexpr int kProducerWarp = 4, kMmaWarp = 5, kPublisherWarp = 6;
constexpr int kBarPartial = 2, kBarFinal = 3;  // named barriers: epilogue + publisher
constexpr uint32_t kTmemCols = kTBufs * 32;
constexpr uint32_t kWBytes = kRows * 128;            // E4M3 weight tile
constexpr uint32_t kXTile = 32 * 128;                // token tile: hi rows 0-15, lo rows 16-31
constexpr uint32_t kOffXTile = kWBytes;
constexpr uint32_t kStage = kWBytes + kXTile;
// bytes TMA brings per unit: the weight tile and the token tile (32 hi/lo
// rows for the W8A16 arm, 16 quantized token rows for the W8A8 arm)
template <bool W8A8>
constexpr uint32_t kTmaBytes = kWBytes + (W8A8 ? 16u * 128u : kXTile);
constexpr uint32_t kOffBar = kStages * kStage;
constexpr uint32_t kNumBars = 2 * kGroups + 2 * kTBufs + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // TMEM slot, abort flag, last flags [2]
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kThreads == 32 * (kPublisherWarp + 1), "one warp per role after the epilogue");
template <bool W8A8>
constexpr uint32_t kIdesc = idesc_e4m3(kRows, W8A8 ? 16 : 32);
constexpr unsigned long long kDrainLimitNs = 100000000ull;
static_assert(kStage % 1024 == 0 && kOffXTile % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kStages % kGroup == 0, "slot groups must tile the ring");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct GemvParams {
  int32_t M, N, K, Kb, RT;
  int64_t U;  // RT * Kb
  int32_t grid;
  const void* s_w;
  int32_t sw_f32;
  // scale (row block r, K-block kb) at s_w[r * sw_rs + kb * sw_ks]: (Kb, 1) for a
  // block grid, (0, 0) for a per-tensor multiplier
  int32_t sw_rs, sw_ks;
  int32_t n_members;
  int32_t mem_n0[BFP8_MAX_MEMBERS], mem_rows[BFP8_MAX_MEMBERS], mem_sbase[BFP8_MAX_MEMBERS];
  __nv_bfloat16* y;
  int64_t ldy;
  int32_t* counters;  // [RT], zero at kernel start
  float* partials;    // [grid][2][128][16]
  const float* xinv;  // [Kb][16]: 2^-e of each token's K-block (W8A16 arm)
  const float* s_a;   // token scales (W8A8 arm): (m, kb) at s_a[m*sa_sm + kb*sa_skb]
  int64_t sa_sm, sa_skb;
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

BFP8_DEV float2 f16x2_bits_to_f32x2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}


// Launches `kernel` as a programmatic dependent of the previous work on the
// stream: it may start before that work ends, so it must griddepcontrol.wait
// before touching anything the previous work reads or writes.
template <typename Kernel, typename... Args>
int launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
               Args... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? BFP8_OK : BFP8_ERR_CUDA;
}

// One CTA per K-block, 256 threads: thread t handles token t / 16 and the 8
// values [8*(t%16), +8) of the block (16 threads per token: the exact SiLU*up
// of the second split is ~40 instructions a value, and 64 threads a block
// left it latency-bound). Writes the hi/lo E4M3 rows of the block's 32 x 128
// token tile (row-major; TMA applies the swizzle on load) and 2^-e per token.
// Tokens past M get zero rows.
// It also clears the GEMV's split-tile counters; the GEMV touches them only
// after its griddepcontrol.wait.
// SILU == true: x is a gate/up output [M, 2K] (gate columns 0..K-1, up columns
// K..2K-1) and the tokens are h = bf16(silu(gate) * up), formed with the same
// arithmetic as the SiLU*up quantizer.
constexpr int kSplitThreads = 256;

BFP8_DEV void load_token_words8(const __nv_bfloat16* row, bool in_range, int c0, int K,
                                uint32_t (&xw)[4]) {
  if (in_range && c0 + 8 <= K) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + c0);   // 16-byte aligned: ldx % 8 == 0
    xw[0] = v.x; xw[1] = v.y; xw[2] = v.z; xw[3] = v.w;
  } else {
    const uint16_t* xr = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = (in_range && c0 + 2 * j < K) ? xr[c0 + 2 * j] : 0u;
      const uint32_t hi = (in_range && c0 + 2 * j + 1 < K) ? xr[c0 + 2 * j + 1] : 0u;
      xw[j] = lo | (hi << 16);
    }
  }
}

template <bool SILU>
__global__ void __launch_bounds__(kSplitThreads) gemv_split_tokens_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t ldx, int32_t M, int32_t K,
    uint8_t* __restrict__ xtile, float* __restrict__ xinv, int32_t* __restrict__ counters,
    int32_t n_counters) {
  pdl_launch_dependents();  // let the GEMV start streaming weights now
  // This kernel may start while the previous GEMV (which reads the same
  // workspace, or wrote x) is still running: wait for it before any access.
  pdl_wait();
  const int kb = blockIdx.x;
  for (int i = kb * kSplitThreads + threadIdx.x; i < n_counters; i += gridDim.x * kSplitThreads)
    counters[i] = 0;
  const int tok = threadIdx.x >> 4, s16 = threadIdx.x & 15;
  const int c0 = kb * 128 + 8 * s16;
  const bool live = tok < M;
  const __nv_bfloat16* row = x + static_cast<int64_t>(live ? tok : 0) * ldx;
  uint32_t xw[4];
  load_token_words8(row, live, c0, K, xw);
  if constexpr (SILU) {
    uint32_t uw[4];
    load_token_words8(row + K, live, c0, K, uw);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float h0 = silu_mul_bf16_round(__uint_as_float(xw[j] << 16), __uint_as_float(uw[j] << 16));
      const float h1 = silu_mul_bf16_round(__uint_as_float(xw[j] & 0xFFFF0000u),
                                           __uint_as_float(uw[j] & 0xFFFF0000u));
      xw[j] = (__float_as_uint(h0) >> 16) | (__float_as_uint(h1) & 0xFFFF0000u);
    }
  }
  // the token's max |x| over the block (non-negative BF16 patterns order like
  // their values), across its 16 threads
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = __vmaxu2(m, xw[j] & 0x7FFF7FFFu);
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int e = min(max(134 - static_cast<int>((m >> 7) & 0xFFu), -126), 126);
  const float up = __int_as_float((e + 127) << 23);
  uint32_t hw[2], lw[2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float v0 = __uint_as_float(xw[j] << 16) * up;
    const float v1 = __uint_as_float(xw[j] & 0xFFFF0000u) * up;
    const uint16_t hi = f32x2_to_e4m3x2(v0, v1);
    const float2 hf = f16x2_bits_to_f32x2(e4m3x2_to_f16x2(hi));
    const uint16_t lo = f32x2_to_e4m3x2(v0 - hf.x, v1 - hf.y);
    if (j & 1) {
      hw[j >> 1] |= static_cast<uint32_t>(hi) << 16;
      lw[j >> 1] |= static_cast<uint32_t>(lo) << 16;
    } else {
      hw[j >> 1] = hi;
      lw[j >> 1] = lo;
    }
  }
  *reinterpret_cast<uint2*>(xtile + (static_cast<int64_t>(kb) * 32 + tok) * 128 + 8 * s16) =
      make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2*>(xtile + (static_cast<int64_t>(kb) * 32 + 16 + tok) * 128 + 8 * s16) =
      make_uint2(lw[0], lw[1]);
  if (s16 == 0) xinv[kb * 16 + tok] = __int_as_float((127 - e) << 23);
}

// Clears the split-tile counters ahead of the W8A8 arm's GEMV, which runs as
// its programmatic dependent and touches them only after griddepcontrol.wait.
__global__ void __launch_bounds__(256) gemv_clear_counters_kernel(int32_t* __restrict__ counters,
                                                                 int32_t n) {
  pdl_launch_dependents();
  pdl_wait();   // the previous GEMV may still be using the counters
  for (int i = threadIdx.x; i < n; i += 256) counters[i] = 0;
}

// W8A8 == false: W8A16 arithmetic, tokens as split hi/lo tiles (tmX over
// the split kernel's output). W8A8 == true: tokens already quantized to E4M3
// with 1x128 scales (tmX over q_a [M, K], rows past M read as zeros).
template <bool W8A8>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_u32);
  // The next call's first kernel (token split or counter clear) may launch
  // now; it waits for this grid before touching the workspace, and the next
  // GEMV's CTAs take SMs as this grid's CTAs leave and stream their weights.
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + kOffBar;
  auto full_bar = [&](int g) { return bar0 + 8u * g; };
  auto empty_bar = [&](int g) { return bar0 + 8u * (kGroups + g); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kGroups + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kGroups + kTBufs + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kGroups + 2 * kTBufs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kOffMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(base_ptr + kOffMisc + 8);

  const int64_t ub = unit_begin(p, blockIdx.x);
  const int64_t ue = unit_begin(p, blockIdx.x + 1);
  const int64_t nu = ue - ub;

  // The producer thread sets up the barriers and starts the first group's
  // weight loads before the CTA-wide sync, so HBM is busy from the start.
  auto unit_rt_kb = [&](int64_t u, int& rt, int& kb) {
    rt = static_cast<int>(u / p.Kb);
    kb = static_cast<int>(u - static_cast<int64_t>(rt) * p.Kb);
  };
  const int64_t n_first = min(static_cast<int64_t>(kStages), nu);  // units of the ring's first pass
  if (warp == kProducerWarp && lane == 0) {
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(full_bar(g), 1);
      mbar_init(empty_bar(g), 1);
    }
    for (int b = 0; b < kTBufs; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    for (int64_t i0 = 0; i0 < n_first; i0 += kGroup) {
      const int g = static_cast<int>(i0 / kGroup);
      const int n_in = static_cast<int>(min(static_cast<int64_t>(kGroup), nu - i0));
      mbar_arrive_expect_tx(full_bar(g), kTmaBytes<W8A8> * n_in);
      for (int j = 0; j < n_in; ++j) {
        int rt, kb;
        unit_rt_kb(ub + i0 + j, rt, kb);
        tma_load_2d(base + (i0 + j) * kStage, &tmW, kb * 128, rt * kRows, full_bar(g));
      }
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      bool tokens_ready = false;
      for (int64_t i0 = 0; i0 < nu; i0 += kGroup) {
        const int g = static_cast<int>((i0 / kGroup) % kGroups);
        const uint32_t ph = static_cast<uint32_t>((i0 / kStages) & 1);
        const int n_in = static_cast<int>(min(static_cast<int64_t>(kGroup), nu - i0));
        if (i0 >= n_first) {  // the first pass's weight loads went out before the CTA sync
          if (!mbar_wait_sleep(empty_bar(g), ph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(g), kTmaBytes<W8A8> * n_in);
          for (int j = 0; j < n_in; ++j) {
            int rt, kb;
            unit_rt_kb(ub + i0 + j, rt, kb);
            tma_load_2d(base + (g * kGroup + j) * kStage, &tmW, kb * 128, rt * kRows, full_bar(g));
          }
        }
        // the token tiles (W8A16: from the split kernel this grid depends on;
        // W8A8: from the caller, ordered before the counter clear this grid
        // depends on) are read only after the dependency wait
        if (!tokens_ready) {
          pdl_wait();
          tokens_ready = true;
        }
        for (int j = 0; j < n_in; ++j) {
          const int64_t u = ub + i0 + j;
          const int kb = static_cast<int>(u % p.Kb);
          if (W8A8)
            tma_load_2d(base + (g * kGroup + j) * kStage + kOffXTile, &tmX, kb * 128, 0, full_bar(g));
          else
            tma_load_2d(base + (g * kGroup + j) * kStage + kOffXTile, &tmX, 0, kb * 32, full_bar(g));
        }
        armed |= 1u << g;
        armed_phase = (armed_phase & ~(1u << g)) | (ph << g);
      }
      if (!ok) raise_abort(abort_flag);
      // no copy may still be landing in shared memory when the CTA exits
      for (int g = 0; g < kGroups; ++g)
        if ((armed >> g) & 1u) wait_bounded(full_bar(g), (armed_phase >> g) & 1u, kDrainLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Converged warp; one elected lane issues the MMAs and their commits.
    bool ok = true;
    for (int64_t i = 0; i < nu; ++i) {
      const int s = static_cast<int>(i % kStages);
      const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
      const int b = static_cast<int>(i % kTBufs);
      const uint32_t bph = static_cast<uint32_t>((i / kTBufs) & 1);
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(tempty_bar(b), bph ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(full_bar(s / kGroup), ph, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sW = base + s * kStage;
      if (elect_one()) {
        const uint64_t da = smem_desc_sw128(sW);
        const uint64_t db = smem_desc_sw128(sW + kOffXTile);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 32 bytes per MMA: +2 in 16-byte units
          umma_e4m3(tmem_base + static_cast<uint32_t>(b * 32), da + 2u * k, db + 2u * k, kIdesc<W8A8>,
                    k > 0 ? 1u : 0u);
        umma_commit(tfull_bar(b));
        if (s % kGroup == kGroup - 1 || i == nu - 1)  // the group's last unit frees its slots
          umma_commit(empty_bar(s / kGroup));
      }
      __syncwarp();
    }
    if (!ok) raise_abort(abort_flag);
    if (elect_one()) umma_commit(drain_bar);
    __syncwarp();
    wait_bounded(drain_bar, 0, kDrainLimitNs);
  } else if (warp < kProducerWarp) {
    // ------------------------------------------------------------ promotion + output
    pdl_wait();  // the counters (and the W8A16 arm's token scales) come from the first kernel
    const int q = warp;                  // warps 0-3: TMEM lane quarter
    const int row = 32 * q + lane;       // weight row within the unit's tile
    const int et = threadIdx.x;          // 0..127
    bool ok = true;
    int64_t u = ub;
    while (u < ue) {
      const int rt = static_cast<int>(u / p.Kb);
      const int64_t tile_u0 = static_cast<int64_t>(rt) * p.Kb;
      const int64_t seg_end = min(ue, tile_u0 + p.Kb);
      const int n = rt * kRows + row;
      const int64_t srow_idx = static_cast<int64_t>(scale_row_of(p, n)) * p.sw_rs;
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
      if (ok) {
        // Units go in pairs whose TMEM buffers are adjacent (first buffer
        // even): one 64-column load and one wait serve both.
        int64_t uu = u;
        while (uu < seg_end) {
          const int64_t i = uu - ub;
          const int b = static_cast<int>(i % kTBufs);
          const bool pair = ((b & 1) == 0) && (uu + 1 < seg_end);
          const int kb = static_cast<int>(uu - tile_u0);
          const float sw0 = load_scale(p, srow_idx + static_cast<int64_t>(kb) * p.sw_ks);
          const float sw1 = pair ? load_scale(p, srow_idx + static_cast<int64_t>(kb + 1) * p.sw_ks)
                                 : 0.0f;
          // per-token factors of the two K-blocks: 2^-e of the split (W8A16)
          // or the 1x128 activation scale (W8A8)
          float xi0[16], xi1[16];
          if (W8A8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              xi0[j] = j < p.M ? __ldg(p.s_a + j * p.sa_sm + kb * p.sa_skb) : 0.0f;
              xi1[j] = (pair && j < p.M) ? __ldg(p.s_a + j * p.sa_sm + (kb + 1) * p.sa_skb) : 0.0f;
            }
          } else {
            const float4* xi4 = reinterpret_cast<const float4*>(p.xinv + kb * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 a4 = __ldg(xi4 + j);
              xi0[4 * j] = a4.x; xi0[4 * j + 1] = a4.y; xi0[4 * j + 2] = a4.z; xi0[4 * j + 3] = a4.w;
            }
            if (pair) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 a4 = __ldg(xi4 + 4 + j);
                xi1[4 * j] = a4.x; xi1[4 * j + 1] = a4.y; xi1[4 * j + 2] = a4.z; xi1[4 * j + 3] = a4.w;
              }
            }
          }
          bool w = mbar_wait(tfull_bar(b), static_cast<uint32_t>((i / kTBufs) & 1), abort_flag);
          if (pair && w)
            w = mbar_wait(tfull_bar(b + 1), static_cast<uint32_t>(((i + 1) / kTBufs) & 1), abort_flag);
          if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * 32);
          float v[64];
          if (pair) {
            tmem_ld64(taddr, v);
          } else {
            float v1[32];
            tmem_ld32(taddr, v1);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = v1[j];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(tempty_bar(b));
            if (pair) mbar_arrive(tempty_bar(b + 1));
          }
          // column j of a buffer is token j (W8A16: plus its lo term at 16 + j)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            acc[j] = fmaf((W8A8 ? v[j] : v[j] + v[16 + j]) * xi0[j], sw0, acc[j]);
          if (pair) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc[j] = fmaf((W8A8 ? v[32 + j] : v[32 + j] + v[48 + j]) * xi1[j], sw1, acc[j]);
          }
          uu += pair ? 2 : 1;
        }
      }
      // ---- output: whole tile, or a partial for the last CTA to sum
      const bool whole = (u == tile_u0) && (seg_end == tile_u0 + p.Kb);
      if (whole) {
        if (ok && n < p.N)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < p.M) p.y[static_cast<int64_t>(j) * p.ldy + n] = __float2bfloat16_rn(acc[j]);
      } else {
        const int slot = (u == ub) ? 0 : 1;
        float4* dst = reinterpret_cast<float4*>(
            p.partials + ((static_cast<int64_t>(blockIdx.x) * 2 + slot) * kRows + row) * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
        // hand the arrival to the publisher warp and go on with the next segment
        named_bar_sync(kBarPartial, 160);
      }
      u = seg_end;
    }
    // ---- fixups: tiles this CTA arrived at last, summed in CTA order
    named_bar_sync(kBarFinal, 160);
    for (int k = 0; k < 2; ++k) {
      const int last_tile = last_flag[k];  // tile index + 1, or 0
      if (last_tile == 0) continue;
      const int rt = last_tile - 1;
      const int64_t tile_u0 = static_cast<int64_t>(rt) * p.Kb;
      const int64_t c_first = cta_of_unit(p, tile_u0);
      const int64_t c_last = cta_of_unit(p, tile_u0 + p.Kb - 1);
      const int n = rt * kRows + row;
      float sum[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) sum[j] = 0.0f;
      // up to 4 contributors at a time so their loads overlap
      for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
        float4 part[4][4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int64_t c = c0 + cc;
          if (c <= c_last) {
            const int sl = (unit_begin(p, c) >= tile_u0) ? 0 : 1;
            const float4* srcp = reinterpret_cast<const float4*>(
                p.partials + ((c * 2 + sl) * kRows + row) * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) part[cc][j] = __ldcg(srcp + j);
          }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (c0 + cc <= c_last) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sum[4 * j] += part[cc][j].x; sum[4 * j + 1] += part[cc][j].y;
              sum[4 * j + 2] += part[cc][j].z; sum[4 * j + 3] += part[cc][j].w;
            }
          }
        }
      }
      if (n < p.N)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < p.M) p.y[static_cast<int64_t>(j) * p.ldy + n] = __float2bfloat16_rn(sum[j]);
      if (et == 0) p.counters[rt] = 0;  // leave the workspace clean
    }
    if (!ok) raise_abort(abort_flag);
  } else if (warp == kPublisherWarp) {
    // ------------------------------------------------------------ arrivals
    pdl_wait();  // the counters belong to the previous call until its grid ends
    // For each split tile of this CTA (at most two: the first and the last
    // segment), once the epilogue has written its partial: one acquire-release
    // atomic on the tile's counter publishes the partial (cumulative release
    // after the barrier) and tells whether this CTA arrived last; if so it
    // also makes the other CTAs' partials visible here (acquire).
    int k = 0;
    int64_t u = ub;
    while (u < ue) {
      const int rt = static_cast<int>(u / p.Kb);
      const int64_t tile_u0 = static_cast<int64_t>(rt) * p.Kb;
      const int64_t seg_end = min(ue, tile_u0 + p.Kb);
      const bool whole = (u == tile_u0) && (seg_end == tile_u0 + p.Kb);
      if (!whole) {
        named_bar_sync(kBarPartial, 160);
        if (lane == 0) {
          int last_arrival = 0;
          if (!*abort_flag) {
            const int64_t c_first = cta_of_unit(p, tile_u0);
            const int64_t c_last = cta_of_unit(p, tile_u0 + p.Kb - 1);
            const int old = atomic_add_acq_rel_gpu(p.counters + rt, 1);
            last_arrival = (old == static_cast<int>(c_last - c_first)) ? rt + 1 : 0;
          }
          last_flag[k] = last_arrival;
        }
        ++k;
      }
      u = seg_end;
    }
    if (lane == 0)
      for (; k < 2; ++k) last_flag[k] = 0;
    __syncwarp();
    named_bar_sync(kBarFinal, 160);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// The split kernel, then the GEMV as its programmatic dependent.
int launch_kernels(const void* x, int64_t ldx, uint8_t* xtile, float* xinv, const CUtensorMap& tw,
                   const CUtensorMap& tx, const GemvParams& p, void* stream, bool silu = false) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  int rc = silu ? launch_pdl(gemv_split_tokens_kernel<true>, dim3(p.Kb), dim3(kSplitThreads), 0, st, xb, ldx,
                             p.M, p.K, xtile, xinv, p.counters, p.RT)
                : launch_pdl(gemv_split_tokens_kernel<false>, dim3(p.Kb), dim3(kSplitThreads), 0, st, xb, ldx,
                             p.M, p.K, xtile, xinv, p.counters, p.RT);
  if (rc != BFP8_OK) return rc;
  rc = check_launch();
  if (rc != BFP8_OK) return rc;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_kernel<false>), kSmemBytes);
  if (rc != BFP8_OK) return rc;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemv_kernel<false>, tw, tx, p) != cudaSuccess) return BFP8_ERR_CUDA;
  return check_launch();
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Workspace: [RT] tile counters | [sms][2][128][16] FP32 partial tiles |
// [Kb][32][128] E4M3 token tiles | [Kb][16] token scales, each part 256-byte aligned.
struct WsLayout {
  size_t partials, xtile, xinv, total;
};
WsLayout ws_layout(int64_t N, int64_t K, int sms) {
  const int64_t RT = (N + kRows - 1) / kRows;
  const int64_t Kb = (K + 127) / 128;
  WsLayout l;
  l.partials = align256(static_cast<size_t>(RT) * 4);
  l.xtile = l.partials + align256(static_cast<size_t>(sms) * 2 * kRows * 16 * sizeof(float));
  l.xinv = l.xtile + align256(static_cast<size_t>(Kb) * kXTile);
  l.total = l.xinv + align256(static_cast<size_t>(Kb) * 16 * sizeof(float));
  return l;
}

}  // namespace

int32_t gemv_counter_count(int64_t N) { return static_cast<int32_t>((N + kRows - 1) / kRows); }

size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K, int sms) {
  (void)M;
  if (N <= 0 || K <= 0 || sms <= 0) return 0;
  return ws_layout(N, K, sms).total;
}

namespace {

// Parameters shared by both arms; checks the workspace and the geometry.
int init_params(GemvParams& p, const void* w, const void* w_scale, int32_t w_scale_dtype,
                int64_t M, int64_t N, int64_t K, void* y, int64_t ldy, const MemberTable& mt,
                void* workspace, size_t ws_bytes, int* sms_out) {
  if (K % 16 != 0 || reinterpret_cast<uintptr_t>(w) % 16 != 0) return BFP8_ERR_UNSUPPORTED;
  if (N > 0x7FFFFFFF || K > 0x7FFFFFFF) return BFP8_ERR_UNSUPPORTED;
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const size_t need = gemv_workspace_bytes(M, N, K, sms);
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return BFP8_ERR_INVALID_ARG;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + 127) / 128);
  p.RT = static_cast<int32_t>((N + kRows - 1) / kRows);
  p.U = static_cast<int64_t>(p.RT) * p.Kb;
  p.grid = static_cast<int32_t>(p.U < sms ? p.U : sms);
  p.s_w = w_scale;
  p.sw_f32 = weight_scale_f32(w_scale_dtype) ? 1 : 0;
  p.sw_rs = weight_scale_per_tensor(w_scale_dtype) ? 0 : p.Kb;
  p.sw_ks = weight_scale_per_tensor(w_scale_dtype) ? 0 : 1;
  p.n_members = mt.count;
  for (int i = 0; i < mt.count; ++i) {
    p.mem_n0[i] = static_cast<int32_t>(mt.n0[i]);
    p.mem_rows[i] = static_cast<int32_t>(mt.rows[i]);
    p.mem_sbase[i] = static_cast<int32_t>(mt.sbase[i]);
  }
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  const WsLayout l = ws_layout(N, K, sms);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<int32_t*>(ws);
  p.partials = reinterpret_cast<float*>(ws + l.partials);
  p.xinv = reinterpret_cast<float*>(ws + l.xinv);
  *sms_out = sms;
  return BFP8_OK;
}

}  // namespace

int launch_gemv(const void* x, int64_t ldx, const void* w, const void* w_scale,
                int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y, int64_t ldy,
                const MemberTable& mt, void* workspace, size_t ws_bytes, void* stream, bool silu) {
  if (ldx % 8 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0) return BFP8_ERR_UNSUPPORTED;
  if (silu && K % 8 != 0) return BFP8_ERR_UNSUPPORTED;
  int rc = check_device_ptrs({x, w, w_scale, y, workspace});
  if (rc != BFP8_OK) return rc;
  GemvParams p{};
  int sms = 0;
  rc = init_params(p, w, w_scale, w_scale_dtype, M, N, K, y, ldy, mt, workspace, ws_bytes, &sms);
  if (rc != BFP8_OK) return rc;
  uint8_t* xtile = static_cast<uint8_t*>(workspace) + ws_layout(N, K, sms).xtile;
  CUtensorMap tw, tx;
  rc = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, 128, kRows,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  // the split kernel's token tiles, one 32-row box per K-block
  rc = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xtile, 128, static_cast<uint64_t>(p.Kb) * 32,
                    128, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  return launch_kernels(x, ldx, xtile, const_cast<float*>(p.xinv), tw, tx, p, stream, silu);
}

int launch_gemv_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                     const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                     int64_t N, int64_t K, void* y, int64_t ldy, const MemberTable& mt,
                     void* workspace, size_t ws_bytes, void* stream, bool clear_counters) {
  if (reinterpret_cast<uintptr_t>(q_a) % 16 != 0) return BFP8_ERR_UNSUPPORTED;
  if (sa_sm < 0 || sa_skb < 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({q_a, s_a, w, w_scale, y, workspace});
  if (rc != BFP8_OK) return rc;
  GemvParams p{};
  int sms = 0;
  rc = init_params(p, w, w_scale, w_scale_dtype, M, N, K, y, ldy, mt, workspace, ws_bytes, &sms);
  if (rc != BFP8_OK) return rc;
  p.s_a = s_a;
  p.sa_sm = sa_sm;
  p.sa_skb = sa_skb;
  CUtensorMap tw, tx;
  rc = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, 128, kRows,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  // the quantized tokens themselves: one 16-row box per K-block, rows past M zero
  rc = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_a, K, M, K, 128, 16,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clear_counters) {   // else the kernel before this one on the stream zeroed them
    rc = launch_pdl(gemv_clear_counters_kernel, dim3(1), dim3(256), 0, st, p.counters, p.RT);
    if (rc != BFP8_OK) return rc;
    rc = check_launch();
    if (rc != BFP8_OK) return rc;
  }
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_kernel<true>), kSmemBytes);
  if (rc != BFP8_OK) return rc;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemv_kernel<true>, tw, tx, p) != cudaSuccess) return BFP8_ERR_CUDA;
  return check_launch();
}

// ---------------------------------------------------------------------------
// The dense-FFN decode step: gate/up GEMV (members {I, I}) -> h = bf16(silu(g)*u)
// -> down GEMV, every launch on one stream with no host synchronisation, so the
// step can be captured in a CUDA graph.
//   W8A16: split(x) -> GEMV(gate/up) -> split(SiLU*up of gu) -> GEMV(down), the
//          SiLU*up formed inside the down GEMV's token split.
//   W8A8:  1x128 quant(x) -> GEMV(gate/up) -> SiLU*up + 1x128 quant -> GEMV(down).
// Workspace: the intermediates, then one GEMV scratch region that the two GEMVs
// use in turn (the second GEMV's first kernel starts only after the first GEMV
// has finished, and each GEMV touches its counters and partials only after its
// programmatic-dependency wait).
namespace {

struct DecodeFfnLayout {
  size_t qx, sx, gu, qh, sh, scratch, total;
};

DecodeFfnLayout decode_ffn_layout(int64_t M, int64_t H, int64_t I, int32_t arith, int sms) {
  const int64_t Hb = (H + 127) / 128, Ib = (I + 127) / 128;
  const bool w8a8 = arith == BFP8_DECODE_W8A8;
  DecodeFfnLayout l{};
  size_t off = 0;
  l.qx = off;
  off += w8a8 ? align256(static_cast<size_t>(M * H)) : 0;
  l.sx = off;
  off += w8a8 ? align256(static_cast<size_t>(M * Hb) * sizeof(float)) : 0;
  l.gu = off;
  off += align256(static_cast<size_t>(M * 2 * I) * 2);
  l.qh = off;
  off += w8a8 ? align256(static_cast<size_t>(M * I)) : 0;
  l.sh = off;
  off += w8a8 ? align256(static_cast<size_t>(M * Ib) * sizeof(float)) : 0;
  l.scratch = off;
  const size_t g1 = ws_layout(2 * I, H, sms).total, g2 = ws_layout(H, I, sms).total;
  l.total = off + (g1 > g2 ? g1 : g2);
  return l;
}

}  // namespace

size_t decode_ffn_workspace_bytes(int64_t M, int64_t H, int64_t I, int32_t arith, int sms) {
  if (M < 1 || M > 16 || H <= 0 || I <= 0 || sms <= 0) return 0;
  if (arith != BFP8_DECODE_W8A16 && arith != BFP8_DECODE_W8A8) return 0;
  return decode_ffn_layout(M, H, I, arith, sms).total;
}

int launch_decode_ffn(int32_t arith, const void* x, int64_t ldx, const void* w_gu,
                      const void* s_gu, const void* w_dn, const void* s_dn, int32_t w_scale_dtype,
                      int64_t M, int64_t H, int64_t I, void* y, int64_t ldy, void* workspace,
                      size_t ws_bytes, void* stream) {
  if (arith != BFP8_DECODE_W8A16 && arith != BFP8_DECODE_W8A8) return BFP8_ERR_INVALID_ARG;
  if (!x || !w_gu || !s_gu || !w_dn || !s_dn || !y || !workspace) return BFP8_ERR_INVALID_ARG;
  if (M < 1 || M > 16 || H <= 0 || I <= 0 || ldx < H || ldy < H) return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  if (H % 16 != 0 || I % 16 != 0) return BFP8_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({x, w_gu, s_gu, w_dn, s_dn, y, workspace});
  if (rc != BFP8_OK) return rc;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const DecodeFfnLayout l = decode_ffn_layout(M, H, I, arith, sms);
  if (ws_bytes < l.total) return BFP8_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* gu = ws + l.gu;
  void* scratch = ws + l.scratch;
  const size_t scratch_bytes = ws_bytes - l.scratch;
  const int64_t Hb = (H + 127) / 128, Ib = (I + 127) / 128;
  MemberTable gu_mt, dn_mt;
  const int64_t gu_rows[2] = {I, I};
  bfp8_members gm;
  gm.n_members = 2;
  gm.member_rows = gu_rows;
  rc = resolve_members(2 * I, &gm, &gu_mt);
  if (rc != BFP8_OK) return rc;
  rc = resolve_members(H, nullptr, &dn_mt);
  if (rc != BFP8_OK) return rc;
  if (arith == BFP8_DECODE_W8A16) {
    rc = launch_gemv(x, ldx, w_gu, s_gu, w_scale_dtype, M, 2 * I, H, gu, 2 * I, gu_mt, scratch,
                     scratch_bytes, stream);
    if (rc != BFP8_OK) return rc;
    return launch_gemv(gu, 2 * I, w_dn, s_dn, w_scale_dtype, M, H, I, y, ldy, dn_mt, scratch,
                       scratch_bytes, stream, /*silu=*/true);
  }
  uint8_t* qx = ws + l.qx;
  float* sx = reinterpret_cast<float*>(ws + l.sx);
  uint8_t* qh = ws + l.qh;
  float* sh = reinterpret_cast<float*>(ws + l.sh);
  // each quantizer zeroes the tile counters of the GEMV that follows it (the
  // GEMV counters sit at the scratch region's start), once the kernel before
  // it, which may be the previous GEMV still counting there, has finished
  int32_t* counters = static_cast<int32_t*>(scratch);
  rc = launch_act_quant(x, M, H, ldx, qx, H, sx, Hb, 1, stream, counters,
                        gemv_counter_count(2 * I));
  if (rc != BFP8_OK) return rc;
  rc = launch_gemv_w8a8(qx, sx, Hb, 1, w_gu, s_gu, w_scale_dtype, M, 2 * I, H, gu, 2 * I, gu_mt,
                        scratch, scratch_bytes, stream, /*clear_counters=*/false);
  if (rc != BFP8_OK) return rc;
  rc = launch_silu_mul_act_quant(gu, M, I, 2 * I, qh, I, sh, Ib, 1, stream, counters,
                                 gemv_counter_count(H));
  if (rc != BFP8_OK) return rc;
  return launch_gemv_w8a8(qh, sh, Ib, 1, w_dn, s_dn, w_scale_dtype, M, H, I, y, ldy, dn_mt,
                          scratch, scratch_bytes, stream, /*clear_counters=*/false);
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

// The device address of the array on each device, once a lookup succeeded.
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
std::mutex g_noalloc_mutex;

// The host-side name of a __device__ array is only a stand-in, not a device
// address, so look the real address up per device, with that device current.
// Only a successful lookup is kept: a failed one (for instance a first call
// made under stream capture) returns BFP8_ERR_CUDA, clears its error and is
// tried again by the next call.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BFP8_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return BFP8_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gemv_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return BFP8_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
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
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
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
