// gemm_sm103.cu -- block-scaled FP8 projections on the sm_103a tensor cores.
//
// One persistent, warp-specialised kernel template serves three entry points:
//   W8A8    y = sum_kb (s_a[m,kb] * s_w[r(n),kb]) * (qa_kb . qw_kb^T)
//           [Module w8a8_prefill, arithmetic paragraph: per-token 1x128
//            activation scales times 128x128 weight scales in an FP32
//            epilogue per K-block]
//   W8A16   y = sum_kb s_w[r(n),kb] * (x_kb . e4m3(qw_kb)^T), with the E4M3
//           weight tile decoded to BF16 in shared memory just before a BF16
//           MMA [FP8 Native Serving, "Native FP8 vs dequant-to-BF16"]
//   grouped the W8A8 arithmetic per expert over an expert-sorted token table
//           [Module w8a8_prefill, "WHY": MoE expert projections on W8A8]
//
// Roles per CTA (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: one elected lane streams the A and B K-block
//               tiles (128 deep, 128-byte swizzle) into a STAGES-deep ring.
//   warp 1      allocates TMEM. One lane issues the tcgen05.mma of each
//               K-block into a fresh TMEM partial (two partial buffers, so
//               the tensor cores run one K-block ahead of the promotion).
//   epilogue    eight warps (4-11 for W8A8, 2-9 for W8A16): tcgen05.ld the
//               partial, acc += P * f in FP32 registers (f = s_a * s_w), then
//               BF16 stores of the tile. Warp w reads TMEM lanes 32*(w%4)..+31
//               (the rows it owns) and one half of the tile's columns. For
//               W8A8, setmaxnreg gives these warps 224 registers (the 128x256
//               FP32 accumulator is 128 registers per thread) and warpgroup 0
//               56.
//   warps 10-13 (W8A16 only) decode the raw E4M3 tile to BF16 in the
//               canonical 128-byte-swizzled K-major layout the MMA reads.
//
// The 128x128 scale blocks are not powers of two, so they cannot be folded
// into the hardware's block-scaled MMA kinds (those take UE8M0 scales per 32
// elements). The promotion therefore runs as an FP32 epilogue per K-block, on
// TMEM partials.
//
// Every mbarrier wait is bounded. On a timeout the kernel raises a CTA-wide
// abort flag and the device error word, drains its in-flight copies and MMAs,
// frees TMEM and returns.
#include <mutex>

#include "bfp8_internal.h"
#include "ptx.cuh"
#include "act_math.cuh"

namespace bfp8 {

namespace {
using namespace dev;

__device__ int g_gemm_err;

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int kMaxExperts = 1024;
constexpr unsigned long long kDrainLimitNs = 100000000ull;

struct GemmParams {
  int32_t M;   // rows of A (dense) or total expert-sorted rows (grouped)
  int32_t K, Kb;
  const float* s_a;
  int64_t sa_sm, sa_skb;
  const void* s_w;
  int32_t sw_f32;
  int64_t sw_expert_stride;  // scale elements between two experts' grids
  // scale (row block r, K-block kb) at s_w[r * sw_rs + kb * sw_ks]: (Kb, 1) for a
  // block grid, (0, 0) for a per-tensor multiplier
  int64_t sw_rs;
  int32_t sw_ks;
  __nv_bfloat16* y;
  int64_t ldy;
  int32_t vec_store;
  int32_t tma_store;  // the output tensor map is set (grouped BF16 output)
  // dense / member mode
  int32_t m_tiles, total_tiles, n_members;
  int32_t mem_n0[BFP8_MAX_MEMBERS], mem_rows[BFP8_MAX_MEMBERS], mem_sbase[BFP8_MAX_MEMBERS];
  int32_t mem_tile0[BFP8_MAX_MEMBERS + 1];
  // grouped mode
  const int32_t* offsets;
  int32_t G, N, n_tiles;
  // fused SiLU(gate)*up + 1x128 quant epilogue: W stacks the gate rows
  // [0, I) over the up rows [I, 2I); the output is h's E4M3 codes and scales
  uint8_t* q_h;
  int64_t ldq;
  float* s_h;
  int64_t sh_sm, sh_skb;
  int32_t up_row0;    // first up row of W (of each expert's W when grouped): I
  int32_t up_sbase;   // first scale row of the up member's grid: ceil(I / 128)
  // stream-K: split tiles exchange FP32 partials through a caller workspace
  int32_t stream_k;
  int32_t* ws_counters;   // one arrival counter per tile, zero on entry
  float* ws_partials;     // [CTAs][2] FP32 partial tiles, each [BN/4][BM] float4s
};

// Work partition over G CTAs. Whole tiles: CTA c takes tiles c, c + G, ...,
// so the CTAs running at the same time work on neighbouring tiles and share
// weight tiles through L2. With stream-K, all but the last one-to-two waves are
// still whole tiles in that order. The K-block units of the remaining tiles are
// cut into G equal contiguous ranges, one per contributor, so the last wave
// leaves no SM idle, and each of those tiles has only two or three
// contributors (see the lockstep grouping below when every tile is split).
// Work is walked as segments: runs of K-blocks inside one tile.
struct SegIter {
  int64_t u, ue;   // stream-K part: next unit, end of this CTA's range (units of the split part)
  int t, t_end, step;  // whole-tile part: next tile, end, stride
  int mu, r;       // stream-K tile of unit u: t_end + (u / Kb) * mu + r
};
// Stream-K geometry. Plain: G = CTAs contributors, one per CTA (mu = 1).
// Lockstep (dense tiles, numbered M-fastest): when the whole-tile prefix and
// the split part are both whole multiples of mu = m_tiles, the CTAs form
// G = CTAs / mu groups; a group's contributor range runs over the split
// part's (N tile, K-block) units and member r of the group computes M tile r
// of each, so the mu CTAs that share a weight tile read each of its K-blocks
// at the same time (through L2, once from DRAM) instead of at staggered
// offsets. CTAs past the last group get no stream-K work.
struct SkGeo {
  int dp_tiles;    // tiles handed out whole (the split part starts there)
  int64_t U;       // stream-K units per member (contributor unit space)
  int G, mu;
};
BFP8_DEV SkGeo sk_geo(bool sk, int total, int Kb, int ncl, int mu_lock) {
  SkGeo g;
  const int waves = total / ncl;
  g.dp_tiles = sk ? (waves > 1 ? (waves - 1) * ncl : 0) : total;
  g.mu = 1;
  g.G = ncl;
  if (sk && mu_lock > 1 && mu_lock <= ncl && g.dp_tiles % mu_lock == 0 &&
      (total - g.dp_tiles) % mu_lock == 0) {
    g.mu = mu_lock;
    g.G = ncl / mu_lock;
  }
  g.U = static_cast<int64_t>((total - g.dp_tiles) / g.mu) * Kb;
  return g;
}
BFP8_DEV int64_t sk_unit_begin(int64_t U, int G, int64_t c) { return (c * U) / G; }
// The contributor whose range holds unit u.
BFP8_DEV int64_t sk_cta_of_unit(int64_t U, int G, int64_t u) { return ((u + 1) * G + U - 1) / U - 1; }

BFP8_DEV SegIter seg_begin(bool sk, int total, int Kb, int cid, int ncl, int mu_lock) {
  const SkGeo g = sk_geo(sk, total, Kb, ncl, mu_lock);
  SegIter it;
  it.t = cid;
  it.t_end = g.dp_tiles;
  it.step = ncl;
  it.mu = g.mu;
  it.r = cid % g.mu;
  const int v = cid / g.mu;
  const bool has = sk && v < g.G;
  it.u = has ? sk_unit_begin(g.U, g.G, v) : 0;
  it.ue = has ? sk_unit_begin(g.U, g.G, v + 1) : 0;
  return it;
}
BFP8_DEV bool next_seg(bool sk, SegIter& it, int total, int Kb, int& t, int& kb0, int& kb1) {
  (void)sk;
  (void)total;
  if (it.t < it.t_end) {
    t = it.t;
    kb0 = 0;
    kb1 = Kb;
    it.t += it.step;
    return true;
  }
  if (it.u >= it.ue) return false;
  const int nt = static_cast<int>(it.u / Kb);
  t = it.t_end + nt * it.mu + it.r;
  kb0 = static_cast<int>(it.u - static_cast<int64_t>(nt) * Kb);
  const int64_t left = it.ue - it.u;
  kb1 = left < Kb - kb0 ? kb0 + static_cast<int>(left) : Kb;
  it.u += kb1 - kb0;
  return true;
}

struct Tile {
  int32_t a_row0, m_valid;   // first A / output row, rows valid from it
  int32_t b_row0, expert;    // first weight row (expert-local when grouped)
  int32_t n_out0, n_valid;   // first output column, columns valid from it
  int32_t srow0, srow_last;  // scale row of the first 128 columns; member's last row
  int32_t b_row0_up, srow_up;  // fused SiLU*up: first up row and its scale row
};

template <int BN, int STAGES, bool W8A16, bool GROUPED, bool SWIGLU = false>
struct Cfg {
  static_assert(!SWIGLU || (!W8A16 && BN == 256),
                "the fused SiLU*up epilogue pairs 128 gate with 128 up columns of a W8A8 tile");
  // output columns a tile covers: BN, or BN/2 when a tile holds gate and up halves
  static constexpr int kOutCols = SWIGLU ? BN / 2 : BN;
  static constexpr int kEpiWarps = 8;
  static constexpr int kConvWarps = W8A16 ? 4 : 0;
  // W8A8: warpgroup 0 = producer, MMA and two idle warps; warpgroups 1-2 =
  // promotion/epilogue. setmaxnreg moves registers from warpgroup 0 to the
  // epilogue, whose FP32 tile accumulator takes 128 registers per thread.
  static constexpr bool kSplitRegs = !W8A16;
  static constexpr int kEpiWarp0 = kSplitRegs ? 4 : 2;
  static constexpr int kWarps = kEpiWarp0 + kEpiWarps + kConvWarps;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kLaunchRegs = 168;      // 65536 / 384 rounded down to a multiple of 8
  // The fused SiLU*up epilogue keeps a second factor live in the promotion
  // loop (8 more registers per epilogue thread), and its grouped factor warp
  // needs 56; together they take the whole launch allocation.
  static constexpr int kCtrlRegs = SWIGLU ? 56 : 64;
  static constexpr int kEpiRegs = SWIGLU ? 224 : 216;
  static_assert(!kSplitRegs || kCtrlRegs * 128 + kEpiRegs * 256 <= kLaunchRegs * kThreads,
                "register split must add up to the launch allocation");
  static constexpr int kEpiCols = BN / 2;
  static constexpr uint32_t kABytes = W8A16 ? BM * BK * 2 : BM * BK;
  static constexpr uint32_t kBRawBytes = BN * BK;
  static constexpr uint32_t kBConvBytes = W8A16 ? BN * BK * 2 : 0;
  // W8A16 keeps three rings with their own barriers: A (BF16) in STAGES
  // stages, the raw E4M3 B tile in kRawStages stages (freed as soon as the
  // decode warps have read it) and the decoded BF16 B tile in kConvBufs
  // buffers (freed by the MMA), so TMA, decode and MMA overlap. W8A8 stages
  // hold A and B together.
  static constexpr int kRawStages = W8A16 ? 2 : 0;
  static constexpr int kConvBufs = W8A16 ? 2 : 0;
  static constexpr uint32_t kStage = W8A16 ? kABytes : kABytes + kBRawBytes;
  static constexpr uint32_t kTmaBytes = kStage;   // bytes one stage's TMA loads bring
  static constexpr uint32_t kOffRaw = STAGES * kStage;
  static constexpr uint32_t kOffConv = kOffRaw + kRawStages * kBRawBytes;
  static constexpr uint32_t kStgPitch = 80;  // 32 BF16 (64 B) + 16 B pad per row
  // Grouped BF16-output instances store full 32-row x 128-column warp tiles
  // by TMA: the warp writes its rows into two 32 x 64 boxes (128-byte
  // swizzle, 8 KB per warp) and one thread issues the two tensor stores, so
  // the warp goes on to the next tile while the copy engine writes. (MoE
  // tiles are short in K, so the tile-end store was up to 40% of their time.)
  // Dense shapes measured no faster this way: they keep the stores below.
  static constexpr bool kTmaStore = GROUPED && !W8A16 && !SWIGLU;
  static constexpr uint32_t kStgWarp = SWIGLU ? 0 : (kTmaStore ? 8192 : 32 * kStgPitch);
  // Fused SiLU*up: at the end of a tile the epilogue warps form h =
  // bf16(silu(g) * u) in float32 (the MUFU-heavy part, spread over 256
  // threads), stage it in shared memory and go straight on to the next tile.
  // The staging holds per row [64 h-or-gate pairs | 64 up pairs] (512 bytes
  // a row, 16-byte chunks swizzled by row): the finished h pair, or for a pair
  // the float32 path cannot round with certainty (an element next to a BF16
  // rounding midpoint, or a gate value outside the fast path's range) the
  // BF16 gate pair in its place, marked in a flag word per thread.
  // Warps 2 and 3 (the SiLU warps) then take the tile, alternate blocks of 32
  // rows each: they resolve the flagged pairs exactly, form each row's 1x128
  // scale and E4M3 codes and store them. (These instances have no factor
  // warp: their promotion factors come from the in-loop fetch.)
  static constexpr int kSiluWarp0 = 2, kSiluWarps = 2;
  static constexpr uint32_t kHStgBytes = SWIGLU ? BM * 512 : 0;
  // flag words [2][BM], then the largest |h| of each half row [2][BM] (BF16 bits)
  static constexpr uint32_t kFixBytes = SWIGLU ? 4 * BM * 4 : 0;
  // TMEM (512 columns) holds 512/BN partial buffers, so the tensor cores run
  // up to that many K-blocks minus one ahead of the promotion.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kNumBufs = 512 / BN;
  static constexpr uint32_t kOffStg = kOffConv + kConvBufs * kBConvBytes;
  // Grouped and fused W8A8 instances: warp 2 (otherwise idle, on its own
  // sub-partition) computes each K-block's promotion factors s_a[m,kb] *
  // s_w[r,kb] for the tile's 128 rows into a ring of kFacSlots slots, two
  // factors per row: the two 128-column halves' (or the gate and up members')
  // scale rows. The epilogue reads them from shared memory instead of loading
  // and multiplying on its critical path. (Measured: 3-5% faster MoE, 1%
  // faster fused dense gate/up, 1-2% slower plain dense shapes, which keep
  // the in-loop fetch.)
  static constexpr bool kFacWarp = kSplitRegs && GROUPED && !SWIGLU;
  static constexpr int kFacSlots = 4;
  static constexpr uint32_t kFacBytes = 2 * BM * 4;
  static constexpr uint32_t kOffFix = kOffStg + kEpiWarps * kStgWarp + kHStgBytes;
  static constexpr uint32_t kOffFac = kOffFix + kFixBytes;
  static constexpr uint32_t kOffBar = kOffFac + (kFacWarp ? kFacSlots * kFacBytes : 0);
  static constexpr uint32_t kNumBars =
      3 * STAGES + 2 * kNumBufs + 1 + 2 * kFacSlots + 2 * kRawStages + 2 * kConvBufs + 2;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  // misc: TMEM slot, abort flag, last-arriver flag, tile handed to the SiLU warp
  static constexpr uint32_t kOffOff = kOffMisc + 16;
  static constexpr uint32_t kOffPre = kOffOff + (kMaxExperts + 1) * 4;
  static constexpr uint32_t kSmemUsed = GROUPED ? kOffPre + (kMaxExperts + 1) * 4 : kOffOff;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // 1024-byte alignment slack
  static constexpr uint32_t kIdesc = W8A16 ? idesc_bf16(BM, BN) : idesc_e4m3(BM, BN);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kNumBufs >= 2 && kNumBufs * BN == 512, "TMEM partial buffers must tile 512 columns");
  static_assert(kEpiCols % 32 == 0, "epilogue columns come in 32-column TMEM loads");
};

// Work item t is one M tile of one N tile of TW output columns (M tiles
// fastest). The up-half fields serve the fused SiLU*up epilogue, whose tile of
// TW output columns reads TW gate rows and the TW matching up rows of W.
// The expert of grouped tile t: the last e >= e_hint with s_pre[e] <= t
// (t < s_pre[G]). Each caller walks its tiles in increasing order, so the
// search starts at the previous tile's expert. lane >= 0: the whole
// (converged) warp tests 32 expert boundaries at once and a ballot counts
// those at or before t (s_pre is non-decreasing, so they are lanes 0..n-1);
// lane < 0: one thread scans forward. (A binary search over all experts took
// ~900 clk of every grouped tile end; the forward scan ~600.)
BFP8_DEV int find_expert(const int* s_pre, int G, int t, int e_hint, int lane) {
  int e = e_hint;
  if (lane < 0) {
#pragma unroll 1
    while (s_pre[e + 1] <= t) ++e;
    return e;
  }
#pragma unroll 1
  for (;;) {
    const int i = e + 1 + lane;
    const uint32_t m = __ballot_sync(0xffffffffu, i <= G && s_pre[i] <= t);
    const int n = __popc(m);
    e += n;
    if (n < 32) return e;
  }
}

template <int TW, bool GROUPED>
__device__ __forceinline__ void decode_tile(const GemmParams& p, const int* s_off,
                                            const int* s_pre, int t, Tile& tl, int& e_hint,
                                            int lane) {
  if (!GROUPED) {
    const int nt = t / p.m_tiles;
    const int mt = t - nt * p.m_tiles;
    int i = 0;
#pragma unroll 1
    while (i + 1 < p.n_members && nt >= p.mem_tile0[i + 1]) ++i;
    const int nl0 = (nt - p.mem_tile0[i]) * TW;
    tl.a_row0 = mt * BM;
    tl.m_valid = min(BM, p.M - tl.a_row0);
    tl.b_row0 = p.mem_n0[i] + nl0;
    tl.expert = 0;
    tl.n_out0 = tl.b_row0;
    tl.n_valid = min(TW, p.mem_rows[i] - nl0);
    tl.srow0 = p.mem_sbase[i] + nl0 / 128;
    tl.srow_last = p.mem_sbase[i] + (p.mem_rows[i] + 127) / 128 - 1;
    tl.b_row0_up = p.up_row0 + nl0;
    tl.srow_up = p.up_sbase + nl0 / 128;
  } else {
    const int e = find_expert(s_pre, p.G, t, e_hint, lane);
    e_hint = e;
    const int row0 = s_off[e];
    const int rows = s_off[e + 1] - row0;
    const int units = (rows + BM - 1) / BM;
    const int local = t - s_pre[e];
    const int nt = local / units;
    const int mt = local - nt * units;
    tl.a_row0 = row0 + mt * BM;
    tl.m_valid = min(BM, rows - mt * BM);
    tl.b_row0 = nt * TW;
    tl.expert = e;
    tl.n_out0 = nt * TW;
    tl.n_valid = min(TW, p.N - nt * TW);
    tl.srow0 = (nt * TW) / 128;
    tl.srow_last = (p.N + 127) / 128 - 1;
    tl.b_row0_up = p.up_row0 + nt * TW;
    tl.srow_up = p.up_sbase + (nt * TW) / 128;
  }
}

// Grouped schedule, built by one warp: clamp the offsets into [0, M], make
// them non-decreasing, then prefix-sum the work items (one M tile x one N
// tile) of every expert.
__device__ void build_schedule(const GemmParams& p, int* s_off, int* s_pre, int lane) {
  const int n = p.G + 1;
  const int per = (n + 31) / 32;
  const int b = min(n, lane * per), e = min(n, b + per);
  int run = 0;
  for (int i = b; i < e; ++i) {
    int v = p.offsets[i];
    v = max(0, min(v, p.M));
    run = max(run, v);
    s_off[i] = run;
  }
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl = max(incl, o);
  }
  int excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0;
  for (int i = b; i < e; ++i) s_off[i] = max(s_off[i], excl);
  __syncwarp();
  const int per2 = (p.G + 31) / 32;
  const int b2 = min(p.G, lane * per2), e2 = min(p.G, b2 + per2);
  int sum = 0;
  for (int i = b2; i < e2; ++i)
    sum += ((s_off[i + 1] - s_off[i] + BM - 1) / BM) * p.n_tiles;
  int incl2 = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl2, off);
    if (lane >= off) incl2 += o;
  }
  int run2 = incl2 - sum;
  for (int i = b2; i < e2; ++i) {
    s_pre[i] = run2;
    run2 += ((s_off[i + 1] - s_off[i] + BM - 1) / BM) * p.n_tiles;
  }
  if (lane == 31) s_pre[p.G] = incl2;
  __syncwarp();
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
  atomicExch(&g_gemm_err, static_cast<int>(BFP8_ERR_TIMEOUT));
}


BFP8_DEV uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

BFP8_DEV float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
BFP8_DEV float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
BFP8_DEV uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
BFP8_DEV uint32_t min_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// h for a BF16 pair (gate pair gb, up pair ub) by the exact scalar path,
// packed like pack_bf16x2. Out of line: only flagged pairs take it.
static __device__ __noinline__ uint32_t silu_mul_pair_exact(uint32_t gb, uint32_t ub) {
  const float h0 = silu_mul_bf16_round(__uint_as_float(gb << 16), __uint_as_float(ub << 16));
  const float h1 = silu_mul_bf16_round(__uint_as_float(gb & 0xFFFF0000u),
                                       __uint_as_float(ub & 0xFFFF0000u));
  return (__float_as_uint(h0) >> 16) | (__float_as_uint(h1) & 0xFFFF0000u);
}

// The SiLU warp's work on one staged fused gate/up tile: per row, h over its
// 128 columns, the row's 1x128 scale and its E4M3 codes. Warp sw of nsw takes
// every nsw-th block of 32 rows, starting at block sw. Rows go in blocks of
// 32, one row per lane first: a row with flagged pairs gets their exact h
// (written back to the staging) and its maximum again; every row gets its
// scale and reciprocal, and one store writes the block's scales. Then 8
// lanes take a row, each 16 consecutive columns (two 16-byte chunks of h
// pairs), four rows per step, with the row's scale by shuffle and one 16-byte
// store of codes per lane. The warp issues few memory instructions: they
// share the pipe with the epilogue's tensor-memory loads.
__device__ __forceinline__ void silu_quant_tile(const GemmParams& p, const Tile& tl, uint32_t stg,
                                                const uint32_t* flags, int lane, int sw, int nsw) {
  const int rq = lane >> 3;         // row of the step this lane takes
  const int j = lane & 7;           // its 16-column slice
  const int col0 = 16 * j;
  const bool vec = p.vec_store && col0 + 16 <= tl.n_valid;
#pragma unroll 1
  for (int rb = 32 * sw; rb < tl.m_valid; rb += 32 * nsw) {
    const uint32_t ra = static_cast<uint32_t>(rb + lane) & (BM - 1);
    const uint32_t f0 = flags[ra], f1 = flags[BM + ra];
    uint32_t am = max(flags[2 * BM + ra], flags[3 * BM + ra]);
    if (__any_sync(0xffffffffu, (f0 | f1) != 0u)) {
      if (f0 | f1) {
        // this lane's row: exact h for its flagged pairs, then its maximum
        const uint32_t row = stg + ra * 512u, sw = ra & 7u;
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t f = hf ? f1 : f0;
          while (f) {
            const uint32_t pr = 32u * hf + static_cast<uint32_t>(__ffs(f) - 1);
            f &= f - 1u;
            const uint32_t ag = row + (((pr >> 2) ^ sw) << 4) + (pr & 3u) * 4u;
            const uint32_t au = row + (((16u + (pr >> 2)) ^ sw) << 4) + (pr & 3u) * 4u;
            uint32_t gb, ub;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(gb) : "r"(ag));
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(ub) : "r"(au));
            const uint32_t hb = silu_mul_pair_exact(gb, ub);
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(ag), "r"(hb) : "memory");
          }
        }
        uint32_t mx = 0u;
        for (int c = 0; c < 16; ++c) {
          const uint4 v = lds128(row + ((static_cast<uint32_t>(c) ^ sw) << 4));
          mx = max_u16x2(mx, v.x & 0x7FFF7FFFu);
          mx = max_u16x2(mx, v.y & 0x7FFF7FFFu);
          mx = max_u16x2(mx, v.z & 0x7FFF7FFFu);
          mx = max_u16x2(mx, v.w & 0x7FFF7FFFu);
        }
        am = max(mx & 0xFFFFu, mx >> 16);
      }
      __syncwarp();
    }
    const float sc_a = group_scale(__uint_as_float(am << 16));
    const float rc_a = __frcp_rn(sc_a);
    if (rb + lane < tl.m_valid)
      p.s_h[(static_cast<int64_t>(tl.a_row0) + rb + lane) * p.sh_sm + (tl.n_out0 / 128) * p.sh_skb] = sc_a;
    const int nrows = min(32, tl.m_valid - rb);
#pragma unroll 1
    for (int i = 0; i < nrows; i += 4) {
      const int ri = i + rq;
      const uint32_t r = static_cast<uint32_t>(rb + ri) & (BM - 1);
      const uint32_t row = stg + r * 512u;
      const uint4 h0 = lds128(row + ((static_cast<uint32_t>(2 * j) ^ (r & 7u)) << 4));
      const uint4 h1 = lds128(row + ((static_cast<uint32_t>(2 * j + 1) ^ (r & 7u)) << 4));
      const float sc = __shfl_sync(0xffffffffu, sc_a, ri & 31);
      const float rc = __shfl_sync(0xffffffffu, rc_a, ri & 31);
      const float2 y2 = make_float2(rc, rc), ns2 = make_float2(-sc, -sc);
      const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      uint32_t wq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 q0 = div_by_scale2(make_float2(lo_bf16(hw[2 * q]), hi_bf16(hw[2 * q])), ns2, y2);
        const float2 q1 =
            div_by_scale2(make_float2(lo_bf16(hw[2 * q + 1]), hi_bf16(hw[2 * q + 1])), ns2, y2);
        wq[q] = static_cast<uint32_t>(f32x2_to_e4m3x2(q0.x, q0.y)) |
                (static_cast<uint32_t>(f32x2_to_e4m3x2(q1.x, q1.y)) << 16);
      }
      if (ri < nrows) {
        uint8_t* dst = p.q_h + (static_cast<int64_t>(tl.a_row0) + rb + ri) * p.ldq + tl.n_out0 + col0;
        if (vec) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (col0 + e < tl.n_valid) dst[e] = static_cast<uint8_t>(wq[e >> 2] >> (8 * (e & 3)));
        }
      }
    }
  }
}

template <int BN, int STAGES, bool W8A16, bool GROUPED, bool SWIGLU>
__global__ void __launch_bounds__(Cfg<BN, STAGES, W8A16, GROUPED, SWIGLU>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const __grid_constant__ GemmParams p) {
  using C = Cfg<BN, STAGES, W8A16, GROUPED, SWIGLU>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_u32);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cid = blockIdx.x;
  const int ncl = gridDim.x;

  const uint32_t bar0 = base + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  // (barriers 2*STAGES .. 3*STAGES-1 are unused)
  auto tfull_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + C::kNumBufs + b); };
  const uint32_t drain_bar = bar0 + 8u * (3 * STAGES + 2 * C::kNumBufs);
  auto ffull_bar = [&](int f) { return bar0 + 8u * (3 * STAGES + 2 * C::kNumBufs + 1 + f); };
  auto fempty_bar = [&](int f) {
    return bar0 + 8u * (3 * STAGES + 2 * C::kNumBufs + 1 + C::kFacSlots + f);
  };
  float* fac = reinterpret_cast<float*>(base_ptr + C::kOffFac);   // [slot][2][BM]
  // W8A16 rings: raw E4M3 B stages and decoded BF16 B buffers
  constexpr int kW16Bar0 = 3 * STAGES + 2 * C::kNumBufs + 1 + 2 * C::kFacSlots;
  auto raw_full = [&](int r) { return bar0 + 8u * (kW16Bar0 + r); };
  auto raw_empty = [&](int r) { return bar0 + 8u * (kW16Bar0 + C::kRawStages + r); };
  auto cv_full = [&](int c) { return bar0 + 8u * (kW16Bar0 + 2 * C::kRawStages + c); };
  auto cv_empty = [&](int c) {
    return bar0 + 8u * (kW16Bar0 + 2 * C::kRawStages + C::kConvBufs + c);
  };
  // the fused SiLU*up hand-off: staging full (8 epilogue warps arrive) / empty (SiLU warp)
  const uint32_t stg_full = bar0 + 8u * (kW16Bar0 + 2 * C::kRawStages + 2 * C::kConvBufs);
  const uint32_t stg_empty = stg_full + 8u;
  const uint32_t hstg = base + C::kOffStg;  // [BM][128] BF16 h, swizzled 16-byte chunks
  uint32_t* pair_flags = reinterpret_cast<uint32_t*>(base_ptr + C::kOffFix);  // [2][BM]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kOffMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(base_ptr + C::kOffMisc + 8);
  volatile int* stg_tile = reinterpret_cast<volatile int*>(base_ptr + C::kOffMisc + 12);
  int* s_off = reinterpret_cast<int*>(base_ptr + C::kOffOff);
  int* s_pre = reinterpret_cast<int*>(base_ptr + C::kOffPre);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);   // released by the MMA's commit
    }
    for (int b = 0; b < C::kNumBufs; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int f = 0; f < C::kFacSlots; ++f) {
      mbar_init(ffull_bar(f), 32);              // every lane of the factor warp
      mbar_init(fempty_bar(f), C::kEpiWarps);
    }
    for (int r = 0; r < C::kRawStages; ++r) {
      mbar_init(raw_full(r), 1);
      mbar_init(raw_empty(r), C::kConvWarps);
    }
    for (int c = 0; c < C::kConvBufs; ++c) {
      mbar_init(cv_full(c), C::kConvWarps);
      mbar_init(cv_empty(c), 1);
    }
    mbar_init(stg_full, C::kEpiWarps);
    mbar_init(stg_empty, C::kSiluWarps);
    *abort_flag = 0;
    *stg_tile = -1;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  // This grid runs as a programmatic dependent of the previous kernel on the
  // stream: let the next one launch (it waits for this grid before touching
  // what this grid reads or writes), and read nothing the previous kernels
  // wrote (activations, their scales, the expert offsets) and write no output
  // before griddepcontrol.wait. Weights and on-chip setup come first.
  pdl_launch_dependents();
  if (GROUPED && warp == C::kEpiWarp0) {
    pdl_wait();
    build_schedule(p, s_off, s_pre, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = GROUPED ? s_pre[p.G] : p.total_tiles;
  // Stream-K only pays when whole-tile waves would leave the last wave mostly
  // empty (partial tiles cost an FP32 round trip through L2 and a fixup); it
  // also needs every CTA to own at least one K-block unit of the split part.
  const int waves = (total + ncl - 1) / ncl;
  // Dense: last-wave fill < 85% (O at M=4096, 84%, gains 4%; QKV at 93% loses
  // 2%; plain gate/up at 89% gains nothing). The fused SiLU*up instance splits
  // below 95%: its tile end is longer, and at 89% (the dense-FFN gate/up,
  // 1,088 tiles) the 24 CTAs with an eighth whole tile ran ~30 us past the
  // others (-4% with the split). Grouped tiles are short and their split
  // tiles cost more: < 80%.
  const int fill_pct = GROUPED ? 80 : (SWIGLU ? 95 : 85);
  const bool sparse_tail = waves > 0 && 100 * total < fill_pct * waves * ncl;
  const bool sk = p.stream_k && sparse_tail &&
                  sk_geo(true, total, p.Kb, ncl, 0).U >= static_cast<int64_t>(ncl);
  // lockstep stream-K groups (dense tiles are numbered M-fastest)
  const int mu_lock = GROUPED ? 0 : p.m_tiles;

  if (warp < C::kEpiWarp0) {
    // warpgroup 0: producer (warp 0) and MMA issuer (warp 1)
    if constexpr (C::kSplitRegs) warpgroup_reg_dealloc<C::kCtrlRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, armed = 0, armed_phase = 0;
        bool ok = true;
        bool a_ready = false;    // activations are read only after the dependency wait
        int e_hint = 0;        // grouped: expert of the previous tile
        SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
        int t, kb0, kb1;
        while (ok && next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
          Tile tl;
          decode_tile<C::kOutCols, GROUPED>(p, s_off, s_pre, t, tl, e_hint, -1);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_sleep(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
            const uint32_t sA = base + stage * C::kStage;
            const uint32_t sB = sA + C::kABytes;
            mbar_arrive_expect_tx(full_bar(stage), C::kTmaBytes);
            if (!a_ready) {
              pdl_wait();
              a_ready = true;
            }
            if (W8A16) {
              tma_load_2d(sA, &tmA, kb * BK, tl.a_row0, full_bar(stage));
              tma_load_2d(sA + BM * 128, &tmA, kb * BK + 64, tl.a_row0, full_bar(stage));
            } else {
              tma_load_2d(sA, &tmA, kb * BK, tl.a_row0, full_bar(stage));
            }
            if constexpr (SWIGLU) {
              // gate rows into B rows [0, BN/2), the matching up rows into [BN/2, BN)
              const uint32_t sBu = sB + (BN / 2) * 128u;
              if (GROUPED) {
                tma_load_3d(sB, &tmB, kb * BK, tl.b_row0, tl.expert, full_bar(stage));
                tma_load_3d(sBu, &tmB, kb * BK, tl.b_row0_up, tl.expert, full_bar(stage));
              } else {
                tma_load_2d(sB, &tmB, kb * BK, tl.b_row0, full_bar(stage));
                tma_load_2d(sBu, &tmB, kb * BK, tl.b_row0_up, full_bar(stage));
              }
            } else if (GROUPED) {
              tma_load_3d(sB, &tmB, kb * BK, tl.b_row0, tl.expert, full_bar(stage));
            } else if (!W8A16) {
              tma_load_2d(sB, &tmB, kb * BK, tl.b_row0, full_bar(stage));
            }
            armed |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) raise_abort(abort_flag);
        // No copy may still be landing in shared memory when the CTA exits.
        for (int s = 0; s < STAGES; ++s)
          if ((armed >> s) & 1u) wait_bounded(full_bar(s), (armed_phase >> s) & 1u, kDrainLimitNs);
      } else if (W8A16 && lane == 1) {
        // W8A16: the raw E4M3 B tiles, in their own ring
        int rs = 0;
        uint32_t rphase = 0, armed = 0, armed_phase = 0;
        bool ok = true;
        int e_hint = 0;
        SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
        int t, kb0, kb1;
        while (ok && next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
          Tile tl;
          decode_tile<C::kOutCols, GROUPED>(p, s_off, s_pre, t, tl, e_hint, -1);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_sleep(raw_empty(rs), rphase ^ 1u, abort_flag)) { ok = false; break; }
            const uint32_t sR = base + C::kOffRaw + rs * C::kBRawBytes;
            mbar_arrive_expect_tx(raw_full(rs), C::kBRawBytes);
            tma_load_2d(sR, &tmB, kb * BK, tl.b_row0, raw_full(rs));
            armed |= 1u << rs;
            armed_phase = (armed_phase & ~(1u << rs)) | (rphase << rs);
            if (++rs == C::kRawStages) { rs = 0; rphase ^= 1u; }
          }
        }
        if (!ok) raise_abort(abort_flag);
        for (int r = 0; r < C::kRawStages; ++r)
          if ((armed >> r) & 1u) wait_bounded(raw_full(r), (armed_phase >> r) & 1u, kDrainLimitNs);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop (barrier waits, addresses) converged and
      // one elected lane issues the tcgen05 instructions and their commits; a
      // lone-lane loop issues them several times slower.
      int stage = 0, buf = 0, cs = 0;
      uint32_t phase = 0, bphase = 0, cphase = 0;
      bool ok = true;
      SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
      int t, kb0, kb1;
      while (ok && next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          // one vote for all of this K-block's waits
          const bool w_ok = mbar_wait_sleep(tempty_bar(buf), bphase ^ 1u, abort_flag) &&
                            mbar_wait_sleep(full_bar(stage), phase, abort_flag) &&
                            (!W8A16 || mbar_wait_sleep(cv_full(cs), cphase, abort_flag));
          if (!__all_sync(0xffffffffu, w_ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
          const uint32_t sA = base + stage * C::kStage;
          if (elect_one()) {
            if (!W8A16) {
              const uint64_t da = smem_desc_sw128(sA);
              const uint64_t db = smem_desc_sw128(sA + C::kABytes);
#pragma unroll
              for (int k = 0; k < BK / 32; ++k)  // K = 32 bytes per MMA: +2 in 16-byte units
                umma_e4m3(d, da + 2u * k, db + 2u * k, C::kIdesc, k > 0 ? 1u : 0u);
            } else {
              const uint32_t sConv = base + C::kOffConv + cs * C::kBConvBytes;
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {  // K = 16 BF16 = 32 bytes per MMA
                const int j = k >> 2, kk = k & 3;
                const uint64_t da = smem_desc_sw128(sA + j * (BM * 128)) + 2u * kk;
                const uint64_t db = smem_desc_sw128(sConv + j * (BN * 128)) + 2u * kk;
                umma_bf16(d, da, db, C::kIdesc, k > 0 ? 1u : 0u);
              }
            }
            umma_commit(empty_bar(stage));
            if (W8A16) umma_commit(cv_empty(cs));   // the decoded B buffer is free again
            umma_commit(tfull_bar(buf));
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++buf == C::kNumBufs) { buf = 0; bphase ^= 1u; }
          if (W8A16 && ++cs == C::kConvBufs) { cs = 0; cphase ^= 1u; }
        }
      }
      if (!ok) raise_abort(abort_flag);
      // the elected lane is the same one every time (lane 0 of a converged
      // warp), so this commit tracks every MMA the warp issued
      if (elect_one()) umma_commit(drain_bar);
      __syncwarp();
      wait_bounded(drain_bar, 0, kDrainLimitNs);
    } else if (C::kFacWarp && warp == 2) {
      // ------------------------------------------------------------ factors
      pdl_wait();
      // Walks the epilogue's segments in the same order. Lane l fills rows
      // l, l+32, l+64, l+96 of each slot; rows past the tile get 0.
      const uint16_t* fsw16 = static_cast<const uint16_t*>(p.s_w);
      const float* fsw32 = static_cast<const float*>(p.s_w);
      auto fscale = [&](int64_t idx) -> float {
        return p.sw_f32 ? __ldg(fsw32 + idx) : bf16_bits_to_f32(__ldg(fsw16 + idx));
      };
      int slot = 0;
      uint32_t fphase = 0;
      bool ok = true;
      int e_hint = 0;
      SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
      int t, kb0, kb1;
      while (ok && next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
        Tile tl;
        decode_tile<C::kOutCols, GROUPED>(p, s_off, s_pre, t, tl, e_hint, lane);
        const int64_t sw_base = GROUPED ? tl.expert * p.sw_expert_stride : 0;
        const int srow0 = SWIGLU ? tl.srow0 : tl.srow0;
        const int srow1 = SWIGLU ? tl.srow_up : min(tl.srow0 + C::kEpiCols / 128, tl.srow_last);
        const int64_t i0 = sw_base + static_cast<int64_t>(srow0) * p.sw_rs;
        const int64_t i1 = sw_base + static_cast<int64_t>(srow1) * p.sw_rs;
        for (int kb = kb0; kb < kb1; ++kb) {
          // voted: the warp stays converged for the warp-wide tile decode
          if (!__all_sync(0xffffffffu, mbar_wait_sleep(fempty_bar(slot), fphase ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          const float w0 = fscale(i0 + static_cast<int64_t>(kb) * p.sw_ks);
          const float w1 = fscale(i1 + static_cast<int64_t>(kb) * p.sw_ks);
          float* f = fac + slot * (2 * BM);
#pragma unroll
          for (int r = 0; r < BM / 32; ++r) {
            const int row = lane + 32 * r;
            const float sa = row < tl.m_valid
                                 ? __ldg(p.s_a + (static_cast<int64_t>(tl.a_row0) + row) * p.sa_sm +
                                         static_cast<int64_t>(kb) * p.sa_skb)
                                 : 0.0f;
            f[row] = sa * w0;
            f[BM + row] = sa * w1;
          }
          mbar_arrive(ffull_bar(slot));
          if (++slot == C::kFacSlots) { slot = 0; fphase ^= 1u; }
        }
      }
      if (!ok) raise_abort(abort_flag);
    } else if (SWIGLU && warp >= C::kSiluWarp0 && warp < C::kSiluWarp0 + C::kSiluWarps) {
      // ------------------------------------------------------------ SiLU*up + quant
      // Takes each tile the epilogue hands over (tile index -1 ends the work),
      // writes h's codes and scales, and frees the staging for the next tile.
      pdl_wait();
      uint32_t ph = 0;
      bool ok = true;
      int e_hint = 0;        // tiles arrive in increasing order
      for (;;) {
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(stg_full, ph, abort_flag))) {
          ok = false;
          break;
        }
        const int t = *stg_tile;
        if (t < 0) break;
        Tile tl;
        decode_tile<C::kOutCols, GROUPED>(p, s_off, s_pre, t, tl, e_hint, lane);
        silu_quant_tile(p, tl, hstg, pair_flags, lane, warp - C::kSiluWarp0, C::kSiluWarps);
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_empty);
        ph ^= 1u;
      }
      if (!ok) raise_abort(abort_flag);
    }
  } else if (warp < C::kEpiWarp0 + C::kEpiWarps) {
    if constexpr (C::kSplitRegs) warpgroup_reg_alloc<C::kEpiRegs>();
    // ------------------------------------------------------------ promotion + epilogue
    pdl_wait();
    const int ew = warp - C::kEpiWarp0;
    const int q = warp & 3;
    const int h = ew >> 2;
    const int row_in_tile = q * 32 + lane;
    const uint32_t stg = base + C::kOffStg + ew * C::kStgWarp;
    const uint16_t* sw16 = static_cast<const uint16_t*>(p.s_w);
    const float* sw32 = static_cast<const float*>(p.s_w);
    int buf = 0;
    uint32_t bphase = 0;
    int fslot = 0;          // factor ring slot (W8A8)
    uint32_t fphase = 0;
    uint32_t handed = 0;    // tiles handed to the SiLU warp
    bool ok = true;
    // Every epilogue warp walks every segment, even after a failed wait, so
    // that all of them reach the same named barriers (those cannot time out).
    int e_hint = 0;
    SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
    int t, kb0, kb1;
    while (next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
      Tile tl;
      decode_tile<C::kOutCols, GROUPED>(p, s_off, s_pre, t, tl, e_hint, lane);
      const bool row_ok = row_in_tile < tl.m_valid;
      const int64_t arow = static_cast<int64_t>(tl.a_row0) + row_in_tile;
      // This warp's columns of the tile: 128 consecutive ones (one weight-scale
      // block), or with the fused SiLU*up epilogue 64 gate columns and the
      // 64 matching up columns, each half with its own member's scale row.
      const int srow = SWIGLU ? tl.srow0 : min(tl.srow0 + (h * C::kEpiCols) / 128, tl.srow_last);
      const int64_t sw_base = GROUPED ? tl.expert * p.sw_expert_stride : 0;
      const int64_t sw_idx = sw_base + static_cast<int64_t>(srow) * p.sw_rs;
      const int64_t sw_idx_up = sw_base + static_cast<int64_t>(tl.srow_up) * p.sw_rs;
      const float* sa_row = p.s_a + (row_ok ? arow * p.sa_sm : 0);
      // The promotion factor is s_a[m,kb] * s_w[row,kb] (s_w alone for W8A16).
      // No value loaded in this loop is used before the loop's barrier wait:
      // a warp that stalled on a load there would hold up the TMEM buffer for
      // every other warp. s_w is fetched 32 K-blocks at a time, one K-block
      // per lane, as raw bits (a window ahead), and each K-block takes its
      // value with a shuffle; s_a is loaded one K-block ahead (loaded at the
      // top of its own K-block, its latency held up the promotion of every
      // K-block: the fused gate/up launch took 11% longer).
      auto sw_raw = [&](int64_t idx, int k) -> uint32_t {
        uint32_t r = 0u;
        if (k < kb1) {
          const int64_t i = idx + static_cast<int64_t>(k) * p.sw_ks;
          if (p.sw_f32)
            r = __ldg(reinterpret_cast<const uint32_t*>(sw32) + i);
          else
            r = __ldg(sw16 + i);
        }
        return r;
      };
      auto sw_value = [&](uint32_t raw) -> float {
        return __uint_as_float(p.sw_f32 ? raw : raw << 16);
      };
      // FP32 accumulator pairs: the promotion runs as packed FP32x2 FMAs
      float2 acc[C::kEpiCols / 2];
#pragma unroll
      for (int i = 0; i < C::kEpiCols / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
      // the up half's factor exists only with the fused SiLU*up epilogue
      // (without the factor warp: W8A16, whose factor is s_w alone)
      uint32_t sw_cur = 0u, su_cur = 0u, sw_nxt = 0u, su_nxt = 0u;
      auto sa_load = [&](int k) -> float {
        return (W8A16 || !row_ok || k >= kb1) ? (W8A16 ? 1.0f : 0.0f) : __ldg(sa_row + k * p.sa_skb);
      };
      float sa_nxt = 0.0f;   // s_a of the next K-block
      if constexpr (!C::kFacWarp) {
        sa_nxt = sa_load(kb0);
        sw_cur = sw_raw(sw_idx, kb0 + lane);
        su_cur = SWIGLU ? sw_raw(sw_idx_up, kb0 + lane) : 0u;
        sw_nxt = sw_raw(sw_idx, kb0 + 32 + lane);
        su_nxt = SWIGLU ? sw_raw(sw_idx_up, kb0 + 32 + lane) : 0u;
      }
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        float f, fu;
        if constexpr (C::kFacWarp) {
          const bool w_ok = mbar_wait(tfull_bar(buf), bphase, abort_flag) &&
                            mbar_wait(ffull_bar(fslot), fphase, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
          const float* fr = fac + fslot * (2 * BM);
          f = fr[(SWIGLU ? 0 : h) * BM + row_in_tile];
          fu = SWIGLU ? fr[BM + row_in_tile] : 0.0f;
        } else {
          const int wl = (kb - kb0) & 31;
          if (wl == 0 && kb != kb0) {
            sw_cur = sw_nxt;
            su_cur = su_nxt;
            sw_nxt = sw_raw(sw_idx, kb + 32 + lane);
            if (SWIGLU) su_nxt = sw_raw(sw_idx_up, kb + 32 + lane);
          }
          const uint32_t sw_bits = __shfl_sync(0xffffffffu, sw_cur, wl);
          const uint32_t su_bits = SWIGLU ? __shfl_sync(0xffffffffu, su_cur, wl) : 0u;
          const float sa = sa_nxt;
          sa_nxt = sa_load(kb + 1);
          const bool w_ok = mbar_wait(tfull_bar(buf), bphase, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
          f = W8A16 ? sw_value(sw_bits) : sa * sw_value(sw_bits);
          fu = SWIGLU ? sa * sw_value(su_bits) : 0.0f;
        }
        const float2 f2 = make_float2(f, f);
        tc_fence_after();
        const uint32_t tcol0 = static_cast<uint32_t>(buf * BN + h * (SWIGLU ? 64 : C::kEpiCols));
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + tcol0;
        if constexpr (C::kSplitRegs) {
          // 64-column single-instruction loads (fewer tcgen05 instructions per
          // K-block than 32-column ones), then packed FP32x2 FMAs.
          constexpr uint32_t kStep = SWIGLU ? BN / 2 : 64;
#pragma unroll
          for (int c = 0; c < C::kEpiCols / 64; ++c) {
            float v[64];
            tmem_ld64(taddr + kStep * c, v);
            const float2 fc = (SWIGLU && c == 1) ? make_float2(fu, fu) : f2;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[32 * c + j] = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]), fc, acc[32 * c + j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(tempty_bar(buf));
            if (C::kFacWarp) mbar_arrive(fempty_bar(fslot));
          }
          if (++fslot == C::kFacSlots) { fslot = 0; fphase ^= 1u; }
        } else {
#pragma unroll
          for (int c = 0; c < C::kEpiCols / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + 32u * c, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc[16 * c + j] = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]), f2, acc[16 * c + j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
        if (++buf == C::kNumBufs) { buf = 0; bphase ^= 1u; }
      }
      if (kb0 != 0 || kb1 != p.Kb) {
        // Split tile: publish this CTA's FP32 partial. The last contributor to
        // arrive sums every contributor's partial in CTA order (deterministic)
        // and stores the tile; nobody waits for anybody.
        // contributors are indexed v = cid / mu (member r = cid % mu of each)
        const SkGeo sg = sk_geo(true, total, p.Kb, ncl, mu_lock);
        const int64_t U = sg.U;
        const int G = sg.G;
        const int mu = sg.mu, r = cid % sg.mu;
        const int64_t tile_u0 = static_cast<int64_t>((t - sg.dp_tiles - r) / mu) * p.Kb;
        const int slot = (tile_u0 + kb0 == sk_unit_begin(U, G, cid / mu)) ? 0 : 1;
        // A partial tile is stored column-chunk-major ([BN/4][BM] float4s),
        // so each warp store (and each fixup load) covers 32 consecutive rows
        // of one 4-column chunk: 512 contiguous bytes.
        float4* mine = reinterpret_cast<float4*>(
                           p.ws_partials + (static_cast<int64_t>(cid) * 2 + slot) * BM * BN) +
                       (h * (C::kEpiCols / 4)) * BM + row_in_tile;
        if (ok) {
#pragma unroll
          for (int i = 0; i < C::kEpiCols / 4; ++i)
            __stcg(mine + i * BM,
                   make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y));
        }
        __threadfence();
        named_bar_sync(1, 32 * C::kEpiWarps);
        const int64_t c_first = sk_cta_of_unit(U, G, tile_u0);
        const int64_t c_last = sk_cta_of_unit(U, G, tile_u0 + p.Kb - 1);
        if (ew == 0 && lane == 0) {
          int last_arrival = 0;
          if (ok && !*abort_flag) {
            const int old = atomicAdd(p.ws_counters + t, 1);
            last_arrival = (old == static_cast<int>(c_last - c_first)) ? 1 : 0;
          }
          *last_flag = last_arrival;
        }
        named_bar_sync(1, 32 * C::kEpiWarps);
        const bool last = *last_flag != 0;
        named_bar_sync(1, 32 * C::kEpiWarps);  // the flag is read before the next segment rewrites it
        if (!last) continue;
        __threadfence();
#pragma unroll
        for (int i = 0; i < C::kEpiCols / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
        for (int64_t c = c_first; c <= c_last; ++c) {
          const int sl = (sk_unit_begin(U, G, c) >= tile_u0) ? 0 : 1;
          const int64_t cta = c * mu + r;
          const float4* src =
              reinterpret_cast<const float4*>(p.ws_partials + (cta * 2 + sl) * BM * BN) +
              (h * (C::kEpiCols / 4)) * BM + row_in_tile;
#pragma unroll
          for (int i = 0; i < C::kEpiCols / 4; ++i) {
            const float4 v = __ldcg(src + i * BM);
            acc[2 * i].x += v.x;
            acc[2 * i].y += v.y;
            acc[2 * i + 1].x += v.z;
            acc[2 * i + 1].y += v.w;
          }
        }
        if (ew == 0 && lane == 0) p.ws_counters[t] = 0;  // leave the workspace clean
      }
      if constexpr (SWIGLU) {
        // Fused dense-FFN glue, this thread's share: its row's 64 h values,
        // h = bf16(silu(bf16(g)) * bf16(u)), the gate and up accumulators
        // rounded to BF16 exactly where the unfused GEMM would store them.
        // Float32 fast path (act_math.cuh); a pair that the fast path cannot
        // round with certainty is staged as its gate and up values and
        // flagged for the SiLU warp, which takes the tile from the staging.
        const bool w_ok = mbar_wait(stg_empty, (handed & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) ok = false;
        if (ok) {
          const float2 c_hi = make_float2(kNegLog2eHi, kNegLog2eHi);
          const float2 c_lo = make_float2(kNegLog2eLoLn2, kNegLog2eLoLn2);
          const float2 one = make_float2(1.0f, 1.0f);
          // BF16 gate and up pairs first: the FP32 accumulator dies here
          uint32_t gw[32], uw[32], hw[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            gw[jj] = pack_bf16x2(acc[jj].x, acc[jj].y);
            uw[jj] = pack_bf16x2(acc[32 + jj].x, acc[32 + jj].y);
          }
          uint32_t fmask = 0u, gmax = 0u, gmin = 0xFFFFFFFFu;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t gb = gw[jj], ub = uw[jj];
            const float2 g = make_float2(lo_bf16(gb), hi_bf16(gb));
            const float2 u = make_float2(lo_bf16(ub), hi_bf16(ub));
            const float2 ea = __fmul2_rn(g, c_hi);
            const float2 e0 = make_float2(ex2_approx(ea.x), ex2_approx(ea.y));
            const float2 ex = __ffma2_rn(e0, __fmul2_rn(g, c_lo), e0);
            const float2 d = __fadd2_rn(ex, one);
            const float2 sg = __fmul2_rn(g, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
            const float2 pr = __fmul2_rn(sg, u);
            hw[jj] = pack_bf16x2(pr.x, pr.y);
            // |g| range of the fast path over the pair (zero maps to the top
            // of the second range, so it never counts as tiny)
            const uint32_t a2 = gb & 0x7FFF7FFFu;
            gmax = max_u16x2(gmax, a2);
            gmin = min_u16x2(gmin, (a2 + 0x7FFF7FFFu) & 0x7FFF7FFFu);
            if (near_bf16_midpoint(pr.x) || near_bf16_midpoint(pr.y)) fmask |= 1u << jj;
          }
          // some |g| >= 64, or 0 < |g| < 2^-100: every pair goes the exact way
          if (max(gmax & 0xFFFFu, gmax >> 16) >= 0x4280u ||
              min(gmin & 0xFFFFu, gmin >> 16) < 0x0D80u - 1u)
            fmask = 0xFFFFFFFFu;
          // columns past the tile's valid width hold 0 (their gate rows belong
          // to the up member); then the largest |h| of this half row
          if (tl.n_valid < C::kOutCols) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int col = h * 64 + 2 * jj;
              hw[jj] &= (col < tl.n_valid ? 0x0000FFFFu : 0u) | (col + 1 < tl.n_valid ? 0xFFFF0000u : 0u);
              if (col >= tl.n_valid) fmask &= ~(1u << jj);
            }
          }
          uint32_t hmax = 0u;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) hmax = max_u16x2(hmax, hw[jj] & 0x7FFF7FFFu);
          // pair jj: h (or the gate pair when flagged) in the first half of
          // the row, the up pair in the second
          const uint32_t rowa = hstg + static_cast<uint32_t>(row_in_tile) * 512u;
          const uint32_t sw = static_cast<uint32_t>(row_in_tile & 7);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = ((fmask >> (4 * c + k)) & 1u) ? gw[4 * c + k] : hw[4 * c + k];
            sts128(rowa + ((static_cast<uint32_t>(8 * h + c) ^ sw) << 4), make_uint4(v[0], v[1], v[2], v[3]));
            sts128(rowa + ((static_cast<uint32_t>(16 + 8 * h + c) ^ sw) << 4),
                   make_uint4(uw[4 * c], uw[4 * c + 1], uw[4 * c + 2], uw[4 * c + 3]));
          }
          pair_flags[h * BM + row_in_tile] = fmask;
          pair_flags[(2 + h) * BM + row_in_tile] = max(hmax & 0xFFFFu, hmax >> 16);
          if (ew == 0 && lane == 0) *stg_tile = t;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full);
        ++handed;
        continue;
      }
      if (!ok) continue;
      if constexpr (C::kTmaStore) {
        // the previous tile's tensor stores must have read the staged boxes
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        // Rows past this expert's belong to the next one: only a warp whose
        // 32 rows are all valid stores by TMA. Columns past N are clipped by
        // the tensor map.
        if (p.tma_store && q * 32 + 32 <= tl.m_valid) {
          if (h * C::kEpiCols < tl.n_valid) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {  // lane = box row; chunk c at c ^ (row & 7)
                const int j = 32 * b + 4 * c;
                sts128(stg + b * 4096 + lane * 128 + ((static_cast<uint32_t>(c) ^ (lane & 7)) << 4),
                       make_uint4(pack_bf16x2(acc[j].x, acc[j].y), pack_bf16x2(acc[j + 1].x, acc[j + 1].y),
                                  pack_bf16x2(acc[j + 2].x, acc[j + 2].y),
                                  pack_bf16x2(acc[j + 3].x, acc[j + 3].y)));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int b = 0; b < 2; ++b)
                if (h * C::kEpiCols + 64 * b < tl.n_valid)
                  tma_store_2d(&tmY, stg + b * 4096, tl.n_out0 + h * C::kEpiCols + 64 * b,
                               tl.a_row0 + q * 32);
              bulk_commit();
            }
          }
          continue;
        }
      }
      // BF16 tile store: stage 32 rows x 32 columns through shared memory so
      // that global stores are row-contiguous 64-byte segments.
#pragma unroll
      for (int ps = 0; ps < C::kEpiCols / 32; ++ps) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v;
          v.x = pack_bf16x2(acc[16 * ps + 4 * i + 0].x, acc[16 * ps + 4 * i + 0].y);
          v.y = pack_bf16x2(acc[16 * ps + 4 * i + 1].x, acc[16 * ps + 4 * i + 1].y);
          v.z = pack_bf16x2(acc[16 * ps + 4 * i + 2].x, acc[16 * ps + 4 * i + 2].y);
          v.w = pack_bf16x2(acc[16 * ps + 4 * i + 3].x, acc[16 * ps + 4 * i + 3].y);
          sts128(stg + lane * C::kStgPitch + 16u * i, v);
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int chunk = it * 32 + lane;
          const int r = chunk >> 2, cq = chunk & 3;
          const uint4 v = lds128(stg + r * C::kStgPitch + 16u * cq);
          const int rt = q * 32 + r;
          const int ct = h * C::kEpiCols + ps * 32 + cq * 8;
          if (rt < tl.m_valid) {
            __nv_bfloat16* dst = p.y + (static_cast<int64_t>(tl.a_row0) + rt) * p.ldy + tl.n_out0 + ct;
            if (p.vec_store && ct + 8 <= tl.n_valid) {
              *reinterpret_cast<uint4*>(dst) = v;
            } else {
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (ct + e < tl.n_valid)
                  reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(wv[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
        __syncwarp();
      }
    }
    if constexpr (C::kTmaStore) {
      // the staged boxes stay in use until read, and the grid's writes are
      // complete only with the tensor stores
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
    if constexpr (SWIGLU) {
      // no more tiles: once the SiLU warp has taken the last one, tell it to stop
      mbar_wait(stg_empty, (handed & 1u) ^ 1u, abort_flag);
      if (ew == 0 && lane == 0) *stg_tile = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_full);
    }
    if (!ok) raise_abort(abort_flag);
  } else {
    // ------------------------------------------------------------ E4M3 -> BF16 decode (W8A16)
    const int cw = warp - C::kEpiWarp0 - C::kEpiWarps;
    int stage = 0, cs = 0;          // raw B stage, decoded B buffer
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    SegIter it = seg_begin(sk, total, p.Kb, cid, ncl, mu_lock);
    int t, kb0, kb1;
    while (ok && next_seg(sk, it, total, p.Kb, t, kb0, kb1)) {
      for (int kb = kb0; kb < kb1; ++kb) {
        const bool w_ok = mbar_wait(raw_full(stage), phase, abort_flag) &&
                          mbar_wait(cv_empty(cs), cphase ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        const uint32_t sRaw = base + C::kOffRaw + stage * C::kBRawBytes;
        const uint32_t sConv = base + C::kOffConv + cs * C::kBConvBytes;
        for (int idx = cw * 32 + lane; idx < BN * 8; idx += C::kConvWarps * 32) {
          const int r = idx >> 3, c = idx & 7;  // row, 16-byte chunk (16 K values)
          const uint4 raw = lds128(sRaw + r * 128 + c * 16);
          uint4 o0, o1;
          e4m3x4_to_bf16x4(raw.x, o0.x, o0.y);
          e4m3x4_to_bf16x4(raw.y, o0.z, o0.w);
          e4m3x4_to_bf16x4(raw.z, o1.x, o1.y);
          e4m3x4_to_bf16x4(raw.w, o1.z, o1.w);
          const int j = c >> 2, cc = (c & 3) * 2;
          const uint32_t row_addr = sConv + j * (BN * 128) + r * 128;
          sts128(row_addr + (static_cast<uint32_t>(cc ^ (r & 7)) << 4), o0);
          sts128(row_addr + (static_cast<uint32_t>((cc + 1) ^ (r & 7)) << 4), o1);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(cv_full(cs));
          mbar_arrive(raw_empty(stage));
        }
        if (++stage == C::kRawStages) { stage = 0; phase ^= 1u; }
        if (++cs == C::kConvBufs) { cs = 0; cphase ^= 1u; }
      }
    }
    if (!ok) raise_abort(abort_flag);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, int STAGES, bool W8A16, bool GROUPED, bool SWIGLU = false>
int launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmParams& p,
           int work_items, void* stream) {
  using C = Cfg<BN, STAGES, W8A16, GROUPED, SWIGLU>;
  auto kernel = gemm_kernel<BN, STAGES, W8A16, GROUPED, SWIGLU>;
  if constexpr (C::kSplitRegs) {
    // setmaxnreg.inc waits until the CTA's launch allocation can cover the
    // request, so the split is only safe if the kernel was built with exactly
    // kLaunchRegs registers per thread. Refuse to launch otherwise.
    static int regs = -1;
    static std::once_flag once;
    std::call_once(once, [&] {
      cudaFuncAttributes attr{};
      if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(kernel)) == cudaSuccess)
        regs = attr.numRegs;
    });
    if (regs != C::kLaunchRegs) return BFP8_ERR_UNSUPPORTED;
  }
  int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), C::kSmemBytes);
  if (rc != BFP8_OK) return rc;
  // persistent: at most as many CTAs as can be resident at once (one per SM)
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, C::kThreads, C::kSmemBytes) !=
          cudaSuccess ||
      per_sm < 1)
    return BFP8_ERR_CUDA;
  rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  const int64_t max_ctas = static_cast<int64_t>(per_sm) * sms;
  int64_t items = work_items;
  if (p.stream_k) items = static_cast<int64_t>(work_items) * p.Kb;  // stream-K splits by K-block units
  const int ctas = static_cast<int>(items < max_ctas ? items : max_ctas);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see the kernel's first wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, ty, p) != cudaSuccess) return BFP8_ERR_CUDA;
  return check_launch();
}

bool aligned16(const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; }

// The weight-scale fields of the parameters: a block grid ([r, kb] at
// r * Kb + kb, expert_stride elements per expert) or, with
// BFP8_SCALE_PER_TENSOR, one multiplier (one per expert).
void set_weight_scale(GemmParams& p, int32_t w_scale_dtype, int64_t expert_stride) {
  p.sw_f32 = weight_scale_f32(w_scale_dtype) ? 1 : 0;
  if (weight_scale_per_tensor(w_scale_dtype)) {
    p.sw_rs = 0;
    p.sw_ks = 0;
    p.sw_expert_stride = 1;
  } else {
    p.sw_rs = p.Kb;
    p.sw_ks = 1;
    p.sw_expert_stride = expert_stride;
  }
}

int fill_members(GemmParams& p, const MemberTable& mt, int bn, int64_t M, const void* y,
                 int64_t ldy) {
  p.n_members = mt.count;
  int tiles = 0;
  bool vec = aligned16(y) && (ldy % 8 == 0);
  for (int i = 0; i < mt.count; ++i) {
    p.mem_n0[i] = static_cast<int32_t>(mt.n0[i]);
    p.mem_rows[i] = static_cast<int32_t>(mt.rows[i]);
    p.mem_sbase[i] = static_cast<int32_t>(mt.sbase[i]);
    p.mem_tile0[i] = tiles;
    tiles += static_cast<int>((mt.rows[i] + bn - 1) / bn);
    if (mt.n0[i] % 8 != 0) vec = false;
  }
  p.mem_tile0[mt.count] = tiles;
  p.m_tiles = static_cast<int32_t>((M + BM - 1) / BM);
  const int64_t total = static_cast<int64_t>(p.m_tiles) * tiles;
  if (total > 0x7FFFFFFF) return BFP8_ERR_UNSUPPORTED;
  p.total_tiles = static_cast<int32_t>(total);
  p.vec_store = vec ? 1 : 0;
  return BFP8_OK;
}

bool fits_i32(int64_t v) { return v >= 0 && v <= 0x7FFFFFFF; }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Stream-K workspace: [tile counters][CTAs x 2 FP32 partial tiles].
size_t sk_workspace_bytes(int64_t tiles, int sms, int bn) {
  return align256(static_cast<size_t>(tiles) * 4) +
         static_cast<size_t>(sms) * 2 * BM * bn * sizeof(float);
}

// Enables stream-K when the caller's workspace is large enough; the tile
// counters are cleared on the stream first (the kernel also leaves them clear).
int sk_setup(GemmParams& p, int64_t tiles, int bn, void* ws, size_t ws_bytes, void* stream) {
  p.stream_k = 0;
  if (!ws) return BFP8_OK;
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc != BFP8_OK) return rc;
  if (ws_bytes < sk_workspace_bytes(tiles, sms, bn) || reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return BFP8_ERR_INVALID_ARG;
  p.stream_k = 1;
  p.ws_counters = static_cast<int32_t*>(ws);
  p.ws_partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                           align256(static_cast<size_t>(tiles) * 4));
  if (cudaMemsetAsync(ws, 0, static_cast<size_t>(tiles) * 4, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return BFP8_ERR_CUDA;
  return BFP8_OK;
}

int64_t member_tiles(const MemberTable& mt, int bn) {
  int64_t tiles = 0;
  for (int i = 0; i < mt.count; ++i) tiles += (mt.rows[i] + bn - 1) / bn;
  return tiles;
}

}  // namespace

// Pipeline stages. The dense fused SiLU*up instance runs 3 (measured 2.7%
// faster than 4 on the dense-FFN gate/up shape; the grouped one is no faster
// with 3), and the grouped BF16-output instance gives its fourth stage's
// shared memory to the TMA store staging.
constexpr int kBN8 = 256, kStages8 = 4, kStagesSwiglu = 3, kStagesGrouped = 3;
constexpr int kBN16 = 128, kStages16 = 3;   // A stages; raw and decoded B have their own rings

size_t gemm_w8a8_workspace_bytes(int64_t M, int64_t N, const MemberTable& mt, int sms) {
  (void)N;
  const int64_t m_tiles = (M + BM - 1) / BM;
  return sk_workspace_bytes(m_tiles * member_tiles(mt, kBN8), sms, kBN8);
}

size_t grouped_w8a8_workspace_bytes(int64_t total_M, int32_t G, int64_t N, int sms) {
  // an upper bound on the device-built tile count: sum_e ceil(M_e/128) <= total_M/128 + G
  const int64_t tiles = ((total_M + BM - 1) / BM + G) * ((N + kBN8 - 1) / kBN8);
  return sk_workspace_bytes(tiles, sms, kBN8);
}

int launch_gemm_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                     const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                     int64_t N, int64_t K, void* y, int64_t ldy, const MemberTable& mt,
                     void* workspace, size_t ws_bytes, void* stream) {
  if (K % 16 != 0 || !aligned16(q_a) || !aligned16(w)) return BFP8_ERR_UNSUPPORTED;
  if (!fits_i32(M) || !fits_i32(N) || !fits_i32(K)) return BFP8_ERR_UNSUPPORTED;
  if (sa_sm < 0 || sa_skb < 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({q_a, s_a, w, w_scale, y, workspace});
  if (rc != BFP8_OK) return rc;
  CUtensorMap ta, tb;
  rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_a, K, M, K, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  rc = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, BK, kBN8,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  GemmParams p{};
  p.M = static_cast<int32_t>(M);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + BK - 1) / BK);
  p.s_a = s_a;
  p.sa_sm = sa_sm;
  p.sa_skb = sa_skb;
  p.s_w = w_scale;
  set_weight_scale(p, w_scale_dtype, 0);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  rc = fill_members(p, mt, kBN8, M, y, ldy);
  if (rc != BFP8_OK) return rc;
  rc = sk_setup(p, p.total_tiles, kBN8, workspace, ws_bytes, stream);
  if (rc != BFP8_OK) return rc;
  const CUtensorMap ty{};  // unused: dense BF16 tiles are stored by the warps
  return launch<kBN8, kStages8, false, false>(ta, tb, ty, p, p.total_tiles, stream);
}

int launch_gemm_w8a16(const void* x, int64_t ldx, const void* w, const void* w_scale,
                      int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y,
                      int64_t ldy, const MemberTable& mt, void* stream) {
  if (K % 16 != 0 || ldx % 8 != 0 || !aligned16(x) || !aligned16(w)) return BFP8_ERR_UNSUPPORTED;
  if (!fits_i32(M) || !fits_i32(N) || !fits_i32(K)) return BFP8_ERR_UNSUPPORTED;
  int rc = check_device_ptrs({x, w, w_scale, y});
  if (rc != BFP8_OK) return rc;
  CUtensorMap ta, tb;
  rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, 64, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  rc = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, BK, kBN16,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != BFP8_OK) return rc;
  GemmParams p{};
  p.M = static_cast<int32_t>(M);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + BK - 1) / BK);
  p.s_a = nullptr;
  p.s_w = w_scale;
  set_weight_scale(p, w_scale_dtype, 0);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  rc = fill_members(p, mt, kBN16, M, y, ldy);
  if (rc != BFP8_OK) return rc;
  const CUtensorMap ty{};
  return launch<kBN16, kStages16, true, false>(ta, tb, ty, p, p.total_tiles, stream);
}

int launch_grouped_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                        const void* w, const void* w_scale, int32_t w_scale_dtype,
                        const int32_t* offsets, int32_t G, int64_t total_M, int64_t N,
                        int64_t K, void* y, int64_t ldy, void* workspace, size_t ws_bytes,
                        void* stream) {
  if (K % 16 != 0 || !aligned16(q_a) || !aligned16(w)) return BFP8_ERR_UNSUPPORTED;
  if (!fits_i32(total_M) || !fits_i32(N) || !fits_i32(K)) return BFP8_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return BFP8_ERR_INVALID_ARG;
  if (sa_sm < 0 || sa_skb < 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({q_a, s_a, w, w_scale, offsets, y, workspace});
  if (rc != BFP8_OK) return rc;
  CUtensorMap ta, tb;
  rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_a, K, total_M, K, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  rc = make_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, G, K, N * K, BK, kBN8, 1,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  GemmParams p{};
  p.M = static_cast<int32_t>(total_M);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + BK - 1) / BK);
  p.s_a = s_a;
  p.sa_sm = sa_sm;
  p.sa_skb = sa_skb;
  p.s_w = w_scale;
  set_weight_scale(p, w_scale_dtype, ((N + 127) / 128) * static_cast<int64_t>(p.Kb));
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  p.vec_store = (aligned16(y) && ldy % 8 == 0) ? 1 : 0;
  p.offsets = offsets;
  p.G = G;
  p.N = static_cast<int32_t>(N);
  p.n_tiles = static_cast<int32_t>((N + kBN8 - 1) / kBN8);
  p.n_members = 1;
  const int64_t tile_bound = ((total_M + BM - 1) / BM + G) * p.n_tiles;
  rc = sk_setup(p, tile_bound, kBN8, workspace, ws_bytes, stream);
  if (rc != BFP8_OK) return rc;
  // the work-item count is only known on the device: launch every resident CTA
  CUtensorMap ty{};
  if (p.vec_store && total_M > 0 && N > 0) {
    // 32-row x 64-column boxes (128 bytes, the swizzle span) of y [total_M, N]
    rc = make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, total_M, ldy * 2, 64, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != BFP8_OK) return rc;
    p.tma_store = 1;
  }
  return launch<kBN8, kStagesGrouped, false, true>(ta, tb, ty, p, 0x7FFFFFFF, stream);
}

size_t gemm_w8a8_swiglu_workspace_bytes(int64_t M, int64_t I, int sms) {
  const int64_t m_tiles = (M + BM - 1) / BM;
  return sk_workspace_bytes(m_tiles * ((I + 127) / 128), sms, kBN8);
}

size_t grouped_w8a8_swiglu_workspace_bytes(int64_t total_M, int32_t G, int64_t I, int sms) {
  const int64_t tiles = ((total_M + BM - 1) / BM + G) * ((I + 127) / 128);
  return sk_workspace_bytes(tiles, sms, kBN8);
}

namespace {

// Shared part of the fused gate/up + SiLU*up + 1x128 quant launches.
void fill_swiglu(GemmParams& p, int64_t I, void* q_h, int64_t ldq, float* s_h, int64_t sh_sm,
                 int64_t sh_skb) {
  p.q_h = static_cast<uint8_t*>(q_h);
  p.ldq = ldq;
  p.s_h = s_h;
  p.sh_sm = sh_sm;
  p.sh_skb = sh_skb;
  p.up_row0 = static_cast<int32_t>(I);
  p.up_sbase = static_cast<int32_t>((I + 127) / 128);
  p.vec_store = (aligned16(q_h) && ldq % 16 == 0) ? 1 : 0;
}

}  // namespace

int launch_gemm_w8a8_swiglu(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                            const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                            int64_t I, int64_t K, void* q_h, int64_t ldq, float* s_h,
                            int64_t sh_sm, int64_t sh_skb, void* workspace, size_t ws_bytes,
                            void* stream) {
  if (K % 16 != 0 || !aligned16(q_a) || !aligned16(w)) return BFP8_ERR_UNSUPPORTED;
  if (!fits_i32(M) || !fits_i32(2 * I) || !fits_i32(K)) return BFP8_ERR_UNSUPPORTED;
  if (sa_sm < 0 || sa_skb < 0 || sh_sm < 0 || sh_skb < 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({q_a, s_a, w, w_scale, q_h, s_h, workspace});
  if (rc != BFP8_OK) return rc;
  CUtensorMap ta, tb;
  rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_a, K, M, K, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  // gate and up halves of a B tile are separate 128-row boxes
  rc = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, 2 * I, K, BK, kBN8 / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  GemmParams p{};
  p.M = static_cast<int32_t>(M);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + BK - 1) / BK);
  p.s_a = s_a;
  p.sa_sm = sa_sm;
  p.sa_skb = sa_skb;
  p.s_w = w_scale;
  set_weight_scale(p, w_scale_dtype, 0);
  // tiles walk h's I columns 128 at a time: one member of I rows
  MemberTable mt;
  mt.count = 1;
  mt.n0[0] = 0;
  mt.rows[0] = I;
  mt.sbase[0] = 0;
  mt.scale_rows = (I + 127) / 128;
  rc = fill_members(p, mt, kBN8 / 2, M, nullptr, 0);
  if (rc != BFP8_OK) return rc;
  fill_swiglu(p, I, q_h, ldq, s_h, sh_sm, sh_skb);
  rc = sk_setup(p, p.total_tiles, kBN8, workspace, ws_bytes, stream);
  if (rc != BFP8_OK) return rc;
  const CUtensorMap ty{};
  return launch<kBN8, kStagesSwiglu, false, false, true>(ta, tb, ty, p, p.total_tiles, stream);
}

int launch_grouped_w8a8_swiglu(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                               const void* w, const void* w_scale, int32_t w_scale_dtype,
                               const int32_t* offsets, int32_t G, int64_t total_M, int64_t I,
                               int64_t K, void* q_h, int64_t ldq, float* s_h, int64_t sh_sm,
                               int64_t sh_skb, void* workspace, size_t ws_bytes, void* stream) {
  if (K % 16 != 0 || !aligned16(q_a) || !aligned16(w)) return BFP8_ERR_UNSUPPORTED;
  if (!fits_i32(total_M) || !fits_i32(2 * I) || !fits_i32(K)) return BFP8_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return BFP8_ERR_INVALID_ARG;
  if (sa_sm < 0 || sa_skb < 0 || sh_sm < 0 || sh_skb < 0) return BFP8_ERR_INVALID_ARG;
  int rc = check_device_ptrs({q_a, s_a, w, w_scale, offsets, q_h, s_h, workspace});
  if (rc != BFP8_OK) return rc;
  CUtensorMap ta, tb;
  rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_a, K, total_M, K, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  rc = make_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, 2 * I, G, K, 2 * I * K, BK,
                    kBN8 / 2, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BFP8_OK) return rc;
  GemmParams p{};
  p.M = static_cast<int32_t>(total_M);
  p.K = static_cast<int32_t>(K);
  p.Kb = static_cast<int32_t>((K + BK - 1) / BK);
  p.s_a = s_a;
  p.sa_sm = sa_sm;
  p.sa_skb = sa_skb;
  p.s_w = w_scale;
  // each expert's grid stacks the gate member's rows over the up member's
  set_weight_scale(p, w_scale_dtype, 2 * ((I + 127) / 128) * static_cast<int64_t>(p.Kb));
  p.offsets = offsets;
  p.G = G;
  p.N = static_cast<int32_t>(I);
  p.n_tiles = static_cast<int32_t>((I + 127) / 128);
  p.n_members = 1;
  fill_swiglu(p, I, q_h, ldq, s_h, sh_sm, sh_skb);
  const int64_t tile_bound = ((total_M + BM - 1) / BM + G) * p.n_tiles;
  rc = sk_setup(p, tile_bound, kBN8, workspace, ws_bytes, stream);
  if (rc != BFP8_OK) return rc;
  const CUtensorMap ty{};
  return launch<kBN8, kStagesSwiglu, false, true, true>(ta, tb, ty, p, 0x7FFFFFFF, stream);
}

// The bounded waits' self-test: a barrier that expects two arrivals gets one.
// Warp 0 waits on it the way the promotion warps wait, warp 1 the way the
// control warps wait (suspending); both give up after limit_ns, and the
// timeout is recorded in the device error word like any kernel's.
__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 2);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(b);   // the second arrival is withheld
  __syncthreads();
  const bool ok = (threadIdx.x >> 5) == 0
                      ? __all_sync(0xffffffffu, mbar_wait(b, 0, abort_flag, limit_ns))
                      : __all_sync(0xffffffffu, mbar_wait_sleep(b, 0, abort_flag, limit_ns));
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(abort_flag);
}

int launch_wait_selftest(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return BFP8_ERR_INVALID_ARG;
  wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  return check_launch();
}

int gemm_read_clear_error() {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(int)) != cudaSuccess) return BFP8_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_gemm_err, &zero, sizeof(int)) != cudaSuccess)
    return BFP8_ERR_CUDA;
  return v == 0 ? BFP8_OK : v;
}

}  // namespace bfp8
