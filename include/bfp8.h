/*
 * bfp8.h -- C ABI of libbfp8, the block-scaled FP8 linear projection for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation: y[M,N] = x[M,K] . W^T. W is E4M3 [N,K] row-major ([out,in],
 * K contiguous), with a "weight_scale_inv" grid of one MULTIPLIER (not a
 * reciprocal) per 128x128 block, stored as BF16 or F32. Scale grids are
 * ceil-divided for partial tails. A grouped tensor (fused QKV, gate/up) keeps
 * a block-row origin per member.
 *   [Qwen checkpoints with block FP8 weights, paragraphs 1-3]
 *   [th#1803 decoder PR, "What lands"]
 *   [FP8 Native Serving, "The two FP8 checkpoint shapes"]
 *
 * Conventions that hold for every entry point:
 *  - Returns an int status (bfp8_status). 0 means success. No exception,
 *    abort or exit crosses this boundary. bfp8_status_string() names each code.
 *  - Tensor pointers are DEVICE pointers owned by the caller. The library
 *    allocates nothing and keeps no per-tensor state; the only state it holds
 *    is a per-device cache of attributes and kernel settings.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Work is enqueued asynchronously on it. Launch failures are
 *    reported as BFP8_ERR_CUDA.
 *  - Sizes and leading dimensions are in ELEMENTS unless a name says bytes.
 *  - Geometry that the tensor-memory-accelerator (TMA) path cannot address
 *    (row strides that are not multiples of 16 bytes, base pointers not
 *    16-byte aligned) is refused with BFP8_ERR_UNSUPPORTED. There is no
 *    silent fallback and no CPU path.
 *  - Calls are thread-safe and re-entrant. Calls on different streams may
 *    overlap on the GPU unless an entry point says otherwise.
 *  - Kernel waits are bounded. If one runs out (which means a bug, not a
 *    data condition), the kernel records BFP8_ERR_TIMEOUT in a device word and
 *    returns early. bfp8_device_status() reads and clears that word.
 */
#ifndef BFP8_H_
#define BFP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
enum bfp8_status {
  BFP8_OK = 0,
  BFP8_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad stride   */
  BFP8_ERR_E5M2 = 2,            /* E5M2 weight encoding                       */
  BFP8_ERR_NO_SCALE = 3,        /* FP8 weight without weight_scale_inv        */
  BFP8_ERR_ROW_SCALE = 4,       /* rank-1 / per-row weight_scale tree         */
  BFP8_ERR_AMBIGUOUS_SCALE = 5, /* both row and block scales, or a per-row grid */
  BFP8_ERR_GRID_TRANSPOSED = 6, /* grid shaped [ceil(K/128), ceil(N/128)]     */
  BFP8_ERR_GRID_SHAPE = 7,      /* any other mis-blocked grid                 */
  BFP8_ERR_SCALE_DTYPE = 8,     /* scale neither BF16 nor F32                 */
  BFP8_ERR_BLOCK_SIZE = 9,      /* declared weight_block_size != [128,128]    */
  BFP8_ERR_QUANT_METHOD = 10,   /* declared quant_method != fp8               */
  BFP8_ERR_GROUP = 11,          /* member rows do not partition N / grid not member-local */
  BFP8_ERR_NOT_FP8 = 12,        /* dense (BF16/F16/F32) weight                */
  BFP8_ERR_UNSUPPORTED = 13,    /* geometry outside what the kernels address  */
  BFP8_ERR_CUDA = 14,           /* a CUDA runtime/driver call failed          */
  BFP8_ERR_TIMEOUT = 15         /* a bounded device wait ran out              */
};

/* ---- element / scale types --------------------------------------------- */
enum bfp8_dtype {
  BFP8_DT_NONE = 0,
  BFP8_DT_E4M3 = 1,
  BFP8_DT_E5M2 = 2,
  BFP8_DT_BF16 = 3,
  BFP8_DT_F16 = 4,
  BFP8_DT_F32 = 5
};

/* OR into any w_scale_dtype argument of a projection (BFP8_DT_BF16 or
 * BFP8_DT_F32): the weight is per-tensor scaled, and w_scale points at ONE
 * multiplier of that dtype (one per expert for the grouped entry points),
 * read as the degenerate block grid whose single block covers the tensor.
 *   [FP8 Native Serving, "The two FP8 checkpoint shapes": per-tensor scaled
 *    checkpoints read as a block case with block_size = infinity]
 * With members, the one multiplier covers every member. */
#define BFP8_SCALE_PER_TENSOR 0x100

/* Largest number of members a grouped (fused) weight may have. */
#define BFP8_MAX_MEMBERS 8

/* Name of a status code ("OK", "E5M2", ...). Never NULL. */
const char* bfp8_status_string(int status);

/* ---- a1: grid validation (host only, metadata only) --------------------- */
/*
 * Header-only view of one weight tensor, as read from a checkpoint's
 * safetensors header and quantization config before any weight byte is read.
 *   [th#1803 decoder PR, "What lands": verification from headers alone]
 */
typedef struct {
  int32_t weight_dtype;        /* bfp8_dtype of the weight bytes              */
  int32_t weight_rank;         /* must be 2                                   */
  int64_t weight_shape[2];     /* [N, K]                                      */
  int32_t scale_dtype;         /* dtype of weight_scale_inv, BFP8_DT_NONE if absent */
  int32_t scale_rank;          /* rank of weight_scale_inv (1 or 2)           */
  int64_t scale_shape[2];      /* its shape (scale_shape[1] unused if rank 1) */
  int32_t has_row_scale;       /* a per-row "weight_scale" leaf is present    */
  int32_t declared_quant_fp8;  /* config declares quant_method == "fp8"       */
  int32_t declared_block[2];   /* config's weight_block_size                  */
  int32_t n_members;           /* 0 = plain tensor; else rows per member below */
  const int64_t* member_rows;  /* host array [n_members], NULL if n_members==0 */
  int32_t tensor_scale_dtype;  /* dtype of a one-element "weight_scale" leaf (a
                                  per-tensor scaled weight), BFP8_DT_NONE if absent */
} bfp8_weight_desc;

/*
 * bfp8_validate_grid -- accept or refuse a block-FP8 weight before upload.
 *   [Qwen checkpoints with block FP8 weights, paragraph 3: E5M2, ambiguous
 *    row/block scales, malformed grids and incompatible declarations refuse
 *    before model upload]
 *   [th#1803 decoder PR, "Why the refusals matter more than the load": a
 *    row-wise tree, a transposed or mis-blocked grid, an FP8 weight with no
 *    scale, a rank-1 scale and a config that disagrees with the bytes are each
 *    refused by name]
 * A per-tensor scaled weight (one multiplier, tensor_scale_dtype set) is the
 * degenerate grid [FP8 Native Serving, "The two FP8 checkpoint shapes"]:
 * after QUANT_METHOD it is refused as AMBIGUOUS_SCALE next to another scale
 * leaf, BLOCK_SIZE if the config declares a weight_block_size, SCALE_DTYPE
 * unless BF16/F32, GROUP if members do not partition N; otherwise OK (pass
 * its dtype OR'd with BFP8_SCALE_PER_TENSOR to the projections).
 * Pure host code; needs no GPU. The first failing rule decides:
 *   INVALID_ARG, E5M2, NOT_FP8, QUANT_METHOD, BLOCK_SIZE, AMBIGUOUS_SCALE
 *   (row+block), ROW_SCALE (row leaf only), NO_SCALE, ROW_SCALE (rank 1),
 *   SCALE_DTYPE, GRID_SHAPE (rank != 2), GROUP (members), OK (grid equals
 *   [sum ceil(N_i/128), ceil(K/128)]), GRID_TRANSPOSED, AMBIGUOUS_SCALE
 *   (rows == N), GROUP (grid built on the stacked rows), GRID_SHAPE.
 * msg (optional, may be NULL): receives a NUL-terminated explanation,
 * truncated to msg_len bytes.
 */
int bfp8_validate_grid(const bfp8_weight_desc* desc, char* msg, size_t msg_len);

/* ---- a2: per-token 1x128 activation quantization ------------------------ */
/*
 * bfp8_act_quant_group -- dynamic E4M3 quantization of BF16 activations.
 *   [Module w8a8_prefill, arithmetic paragraph: per-token 1x128 FP32
 *    activation scales, as per_token_group_quant_fp8 computes them]
 * For token m and group g (columns [128g, min(128g+128, K))):
 *   amax = max|x|, s = max(amax, 1e-10f) / 448.0f, q = RNE_satfinite_e4m3(x / s)
 * where s and x / s are the correctly rounded float32 quotients (IEEE
 * division). This is bit-exact with the CPU oracle for finite inputs.
 *   x_bf16  [M, K] BF16, row stride ldx >= K (elements)
 *   q_e4m3  [M, K] E4M3 bytes, row stride ldq >= K (bytes)
 *   scales  float32, element (m, g) at scales[m*s_stride_m + g*s_stride_kb];
 *           row-major [M, ceil(K/128)] is (ceil(K/128), 1); the token-
 *           contiguous (MN-major) layout is (1, M).
 * M == 0 or K == 0 is a no-op. Errors: INVALID_ARG for null pointers,
 * negative sizes or ld < K.
 */
int bfp8_act_quant_group(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                         void* q_e4m3, int64_t ldq, float* scales,
                         int64_t s_stride_m, int64_t s_stride_kb, void* stream);

/* ---- a10: SiLU(gate)*up fused with the 1x128 quantization --------------- */
/*
 * bfp8_silu_mul_act_quant -- the glue between the gate/up and down
 * projections of the dense FFN [Module w8a8_prefill, first paragraph: the
 * gate/up/down GEMM arm].
 *   gu_bf16 [M, 2I] BF16 (gate columns 0..I-1, up columns I..2I-1), row stride ld
 *   h = bf16_rn( silu(g) * u ), silu(g) = g / (1 + exp(-g)), the value of the
 *   definition evaluated in double and rounded once to BF16 (see bfp8_silu_mul),
 *   then the same quantization as bfp8_act_quant_group over [M, I]. Codes and
 *   scales are bit-exact with the CPU oracle for finite inputs.
 * Output arguments as for bfp8_act_quant_group with K = I.
 */
int bfp8_silu_mul_act_quant(const void* gu_bf16, int64_t M, int64_t I, int64_t ld,
                            void* q_e4m3, int64_t ldq, float* scales,
                            int64_t s_stride_m, int64_t s_stride_kb, void* stream);

/*
 * bfp8_silu_mul -- the same glue for the W8A16 arm, whose down projection
 * takes BF16 activations: h = bf16_rn( silu(g) * u ) without quantization.
 *   [Module w8a8_prefill, first paragraph: the gate/up/down arm]
 *   [FP8 Native Serving, "Native FP8 vs dequant-to-BF16": BF16 activations]
 *   gu_bf16 [M, 2I] BF16, row stride ld >= 2I; h_bf16 [M, I], row stride ldh >= I
 * Each element is bit-identical to g / (1 + exp(-g)) * u evaluated in double
 * (g, u widened exactly from BF16) and rounded once to BF16, nearest-even.
 * The kernel computes it in float32 with an error bound and recomputes in
 * double the rare elements that lie too close to a BF16 rounding boundary.
 * M == 0 or I == 0 is a no-op. Errors: INVALID_ARG (null pointers, negative
 * sizes, ld < 2I, ldh < I, memory that is not on the current device).
 */
int bfp8_silu_mul(const void* gu_bf16, int64_t M, int64_t I, int64_t ld, void* h_bf16,
                  int64_t ldh, void* stream);

/* ---- ahead-of-time weight block quantization (conversion endpoint) ------ */
/*
 * bfp8_quantize_weight_block -- produce a block-FP8 weight from float32.
 * Quantization happens ahead of time through a conversion step, never at load
 * [th#1803 decoder PR, "Why the refusals matter more than the load"]. Per
 * 128x128 block: s = max(amax, 1e-10f)/448.0f, stored RNE to BF16 (or as F32);
 * q = RNE_satfinite_e4m3(w / s_stored).
 *   w      [N, K] float32, row stride ldw (elements)
 *   q      [N, K] E4M3 bytes, row stride ldq (bytes)
 *   scale  [ceil(N/128), ceil(K/128)] row-major, BFP8_DT_BF16 or BFP8_DT_F32
 */
int bfp8_quantize_weight_block(const float* w, int64_t N, int64_t K, int64_t ldw,
                               void* q, int64_t ldq, void* scale, int32_t scale_dtype,
                               void* stream);

/* Member table of a grouped weight: rows of each stacked member, in order.
 * Host memory; NULL (or n_members == 0) means a single member of N rows. */
typedef struct {
  int32_t n_members;
  const int64_t* member_rows;
} bfp8_members;

/* ---- a3-a5, a8: W8A8 block-scaled projection (tcgen05 / TMEM) ----------- */
/* Workspace bytes that let bfp8_linear_w8a8 split tiles along K (stream-K)
 * on the current device; 0 on bad arguments. */
size_t bfp8_linear_w8a8_workspace(int64_t M, int64_t N, int64_t K, const bfp8_members* members);

/*
 * bfp8_linear_w8a8 -- y = dequant(q_a) . dequant(W)^T.
 *   [Module w8a8_prefill, arithmetic paragraph: per-token 1x128 activation
 *    scales times 128x128 weight scales in an FP32 epilogue per K-block, FP32
 *    accumulation]
 *   [FP8 Native Serving, "Native FP8 vs dequant-to-BF16": FP8 through the
 *    tensor cores, BF16 only when the result is written]
 * For every 128-wide K-block kb the tensor cores form the exact FP8 product
 * sum P in FP32. The kernel then does acc += P * (s_a[m,kb] * s_w[r(n),kb]) in
 * FP32 and finally writes y = bf16_rn(acc). r(n) is the member-local scale row.
 *   q_a      [M, K] E4M3, row stride K bytes (densely packed)
 *   s_a      float32 activation scales, (m,kb) at s_a[m*s_stride_m + kb*s_stride_kb]
 *   w_e4m3   [N, K] E4M3 row-major (members stacked), row stride K bytes
 *   w_scale  [sum_i ceil(N_i/128), ceil(K/128)] row-major, w_scale_dtype BF16 or F32
 *   y_bf16   [M, N] BF16, row stride ldy >= N (elements)
 *   members  member table (host), NULL for one member
 *   workspace, ws_bytes  optional device scratch, caller-owned and 256-byte
 *            aligned. With at least bfp8_linear_w8a8_workspace() bytes, the
 *            kernel balances work by cutting the (tiles x K-blocks) work into
 *            equal ranges per SM (stream-K). Split tiles exchange FP32
 *            partials here, and the last CTA sums them in a fixed order, so
 *            the result is deterministic. NULL (or too small) means whole
 *            tiles per SM. The call clears the tile counters it uses; two
 *            calls that share a workspace must not overlap on the GPU.
 * Requirements: K % 16 == 0 (TMA row pitch); q_a, w_e4m3 16-byte aligned;
 * y_bf16 16-byte aligned and ldy % 8 == 0. M == 0 is a no-op.
 */
int bfp8_linear_w8a8(const void* q_a, const float* s_a, int64_t s_stride_m, int64_t s_stride_kb,
                     const void* w_e4m3, const void* w_scale, int32_t w_scale_dtype,
                     int64_t M, int64_t N, int64_t K, void* y_bf16, int64_t ldy,
                     const bfp8_members* members, void* workspace, size_t ws_bytes,
                     void* stream);

/* ---- a6: W8A16 block-scaled projection ---------------------------------- */
/*
 * bfp8_linear_w8a16 -- BF16 activations, FP8 weights decoded exactly to BF16
 * in shared memory right before a BF16 tensor-core MMA.
 *   [FP8 Native Serving, "Native FP8 vs dequant-to-BF16": convert to BF16 in
 *    the GEMM fragment, MMA in BF16]
 *   [Qwen checkpoints with block FP8 weights, paragraph 2: block multipliers
 *    applied inside the projection reduction, F32 accumulation]
 * y[m,n] = bf16_rn( sum_kb s_w[r(n),kb] * sum_{k in kb} x[m,k] * e4m3(W[n,k]) ), FP32.
 *   x_bf16 [M, K] BF16, row stride ldx (elements), ldx % 8 == 0, 16-byte aligned
 *   other arguments and requirements as bfp8_linear_w8a8.
 */
int bfp8_linear_w8a16(const void* x_bf16, int64_t ldx, const void* w_e4m3, const void* w_scale,
                      int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K,
                      void* y_bf16, int64_t ldy, const bfp8_members* members, void* stream);

/* ---- a7: decode GEMV, M <= 16 ------------------------------------------- */
/*
 * bfp8_gemv_decode -- the memory-bound small-M projection (W8A16 arithmetic).
 *   [Module w8a8_prefill, "Reachability": the GB10 decode path is an unfused
 *    per-projection GEMV]
 * W streams from HBM to the tensor cores untouched (TMA, tcgen05 E4M3 MMAs,
 * FP32 accumulation in tensor memory, the per-128-K block scale applied in
 * FP32 registers). A small kernel launched first writes each token's
 * 128-column blocks as two E4M3 terms hi + lo at a per-(token, block) power of
 * two; hi + lo equals the BF16 value exactly for every entry within 2^-10 of
 * the block's max |x|, and smaller entries are carried to within max|x| * 2^-18.
 * The GEMV runs behind it as a programmatic dependent launch. Split-K partial
 * sums are reduced in a fixed order through `workspace`, so results are
 * deterministic.
 *   x_bf16 [M, K] BF16, row stride ldx (ldx % 8 == 0, 16-byte aligned), 1 <= M <= 16
 *   w_e4m3 [N, K], w_scale grid as bfp8_linear_w8a8 (K % 16 == 0); E4M3 NaN
 *          codes (0x7F, 0xFF) give NaN outputs
 *   y_bf16 [M, N] BF16, row stride ldy (elements)
 *   workspace  device scratch of at least bfp8_gemv_decode_workspace(M,N,K)
 *              bytes, caller-owned, 256-byte aligned. Its contents need not be
 *              initialised. Two calls that share one workspace must not
 *              overlap on the GPU.
 * The call is two kernel launches on `stream` and can be captured in a CUDA
 * graph.
 */
int bfp8_gemv_decode(const void* x_bf16, int64_t ldx, const void* w_e4m3, const void* w_scale,
                     int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K,
                     void* y_bf16, int64_t ldy, const bfp8_members* members,
                     void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes bfp8_gemv_decode needs on the current device (0 if none). */
size_t bfp8_gemv_decode_workspace(int64_t M, int64_t N, int64_t K);

/*
 * bfp8_gemv_decode_w8a8 -- the same decode GEMV with E4M3 tokens: the W8A8
 * arithmetic of bfp8_linear_w8a8 for M <= 16.
 *   [Module w8a8_prefill, arithmetic paragraph: per-token 1x128 activation
 *    scales times 128x128 weight scales, FP32 per K-block]
 * y[m,n] = bf16_rn( sum_kb s_a[m,kb] * s_w[r(n),kb] * sum_{k in kb} e4m3(q_a[m,k]) * e4m3(W[n,k]) ).
 * The quantized tokens go to the FP8 tensor cores as they are (no split).
 *   q_a    [M, K] E4M3 from bfp8_act_quant_group, row stride K bytes, 16-byte aligned
 *   s_a    float32 activation scales as bfp8_linear_w8a8
 *   other arguments, the workspace (bfp8_gemv_decode_workspace bytes) and
 *   requirements as bfp8_gemv_decode. Two kernel launches: a one-CTA kernel
 *   that zeroes the workspace's tile counters, then the GEMV as its
 *   programmatic dependent.
 */
int bfp8_gemv_decode_w8a8(const void* q_a, const float* s_a, int64_t s_stride_m,
                          int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                          int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y_bf16,
                          int64_t ldy, const bfp8_members* members, void* workspace,
                          size_t ws_bytes, void* stream);

/* ---- the dense-FFN decode step (graph-capturable) ------------------------ */
/* Arithmetic of a decode step: the W8A16 GEMV of bfp8_gemv_decode, or the
 * W8A8 GEMV of bfp8_gemv_decode_w8a8 behind 1x128 activation quantization. */
enum bfp8_decode_arith { BFP8_DECODE_W8A16 = 0, BFP8_DECODE_W8A8 = 1 };

/*
 * bfp8_decode_ffn -- one dense-FFN decode step for M <= 16 tokens, as a
 * chain of GEMVs on one stream:
 *   gu = GEMV(x, W_gate_up) with members {I, I}        (BF16 [M, 2I])
 *   h  = bf16_rn( silu(gu[:, :I]) * gu[:, I:] )        (as bfp8_silu_mul_act_quant)
 *   y  = GEMV(h, W_down)                               (BF16 [M, H])
 *   [Module w8a8_prefill, "Reachability": decode on GB10 runs one unfused
 *    GEMV per projection; first paragraph: the gate/up/down arm]
 * arith = BFP8_DECODE_W8A16: both GEMVs are bfp8_gemv_decode's arithmetic on
 *   x and h (4 launches: each GEMV behind its token split; the SiLU*up is
 *   formed inside the down GEMV's token split).
 * arith = BFP8_DECODE_W8A8: x is quantized as bfp8_act_quant_group, the
 *   gate/up GEMV is bfp8_gemv_decode_w8a8, h is quantized as
 *   bfp8_silu_mul_act_quant, and the down GEMV is bfp8_gemv_decode_w8a8
 *   (4 launches: each quantizer also zeroes the tile counters of the GEMV
 *   that follows it, in place of that GEMV's clearing kernel).
 * The result equals that sequence of entry points byte for byte.
 *   x_bf16     [M, H] BF16, row stride ldx (ldx % 8 == 0, 16-byte aligned)
 *   w_gate_up  [2I, H] E4M3, gate rows over up rows; s_gate_up its
 *              member-local grid [2*ceil(I/128), ceil(H/128)]
 *   w_down     [H, I] E4M3; s_down its grid [ceil(H/128), ceil(I/128)]
 *   w_scale_dtype  BFP8_DT_BF16 or BFP8_DT_F32, for both grids
 *   y_bf16     [M, H] BF16, row stride ldy
 *   workspace  at least bfp8_decode_ffn_workspace(M, H, I, arith) bytes,
 *              256-byte aligned, caller-owned; holds the intermediates and
 *              the GEMVs' split-K scratch. Calls sharing it must not overlap.
 * Requirements: 1 <= M <= 16; H % 16 == 0 and I % 16 == 0.
 * Every launch goes to `stream` and nothing synchronises with the host, so a
 * step can be captured once in a CUDA graph and replayed.
 */
size_t bfp8_decode_ffn_workspace(int64_t M, int64_t H, int64_t I, int32_t arith);
int bfp8_decode_ffn(int32_t arith, const void* x_bf16, int64_t ldx, const void* w_gate_up,
                    const void* s_gate_up, const void* w_down, const void* s_down,
                    int32_t w_scale_dtype, int64_t M, int64_t H, int64_t I, void* y_bf16,
                    int64_t ldy, void* workspace, size_t ws_bytes, void* stream);

/* ---- decode GEMV for callers that cannot allocate ------------------------- */
/*
 * The pages have no counterpart for this entry point. It exists for callers
 * that cannot call cudaMalloc: code that runs under an allocator it must not
 * bypass (a framework's memory pool, a plugin inside another process), or
 * code that must keep device memory fixed once serving has started.
 *
 * bfp8_gemv_decode_noalloc computes exactly what bfp8_gemv_decode computes,
 * with the same arguments minus the workspace. Its split-K scratch is a fixed
 * device array of BFP8_GEMV_NOALLOC_SCRATCH_BYTES compiled into the library.
 * Every GPU that loads libbfp8.so holds that array until the process exits.
 *  - Limit: the problem must need at most BFP8_GEMV_NOALLOC_SCRATCH_BYTES of
 *    scratch; bfp8_gemv_decode_workspace(M, N, K) <= 4 MiB is the exact test.
 *    The scratch holds, each part rounded up to 256 bytes: 4 bytes per
 *    128-row tile of W (4 * ceil(N/128)), two 128 x 16 float32 partial tiles
 *    per SM (2.49 MB on a 152-SM GB300), and 4096 + 64 bytes of token tiles
 *    and factors per 128-column block of K (4160 * ceil(K/128)). On 152 SMs
 *    that allows K up to 52,352 at N = 5120, and N up to about 36 million
 *    rows at K = 17,408. Larger problems return BFP8_ERR_UNSUPPORTED before
 *    any GPU work.
 *  - The first successful call on each device does a one-time set-up: it
 *    looks up the array's device address with cudaGetSymbolAddress and keeps
 *    it. Make that first call before capturing any stream. A lookup that
 *    fails returns BFP8_ERR_CUDA and is tried again on the next call.
 *  - All calls on one device share the array, and each call clears the
 *    counters it needs on its stream before the kernel runs. Calls that
 *    overlap on the GPU (two streams, or two host threads without ordering)
 *    race on the array and give wrong results. Order them on one stream or
 *    with events.
 *  - It allocates no memory and calls no allocating routine.
 */
#define BFP8_GEMV_NOALLOC_SCRATCH_BYTES (4u << 20)
int bfp8_gemv_decode_noalloc(const void* x_bf16, int64_t ldx, const void* w_e4m3,
                             const void* w_scale, int32_t w_scale_dtype, int64_t M, int64_t N,
                             int64_t K, void* y_bf16, int64_t ldy, const bfp8_members* members,
                             void* stream);

/* ---- a9: grouped (per-expert) W8A8 projection ---------------------------- */
/*
 * bfp8_grouped_linear -- the MoE expert projections over a token-offset table.
 *   [Module w8a8_prefill, "WHY": the MoE expert path on the W8A8 block-scaled
 *    projection]
 * Rows offsets[e] .. offsets[e+1]-1 of the expert-sorted activations use
 * expert e's weight W[e] and scale grid s_w[e]. The arithmetic per row is that
 * of bfp8_linear_w8a8. The tile schedule is built on the device from
 * `offsets_dev`, so there is no host synchronisation. Empty experts cost
 * nothing.
 *   q_a        [total_M, K] E4M3 (expert-sorted), row stride K bytes
 *   s_a        float32 activation scales as bfp8_linear_w8a8
 *   w_e4m3     [G, N, K] E4M3; w_scale [G, ceil(N/128), ceil(K/128)]
 *   offsets_dev int32 [G+1] on the device. They should be non-decreasing with
 *              offsets[0] == 0 and offsets[G] == total_M. The kernel clamps
 *              values outside [0, total_M] and never reads or writes outside
 *              the tensors.
 *   y_bf16     [total_M, N] BF16, row stride ldy
 *   workspace, ws_bytes  optional stream-K scratch, as bfp8_linear_w8a8, sized
 *              by bfp8_grouped_linear_workspace() (an upper bound, because
 *              the tile count is only known on the device)
 * Requirements: 1 <= G <= 1024; K % 16 == 0; alignments as bfp8_linear_w8a8.
 */
size_t bfp8_grouped_linear_workspace(int64_t total_M, int32_t G, int64_t N, int64_t K);
int bfp8_grouped_linear(const void* q_a, const float* s_a, int64_t s_stride_m, int64_t s_stride_kb,
                        const void* w_e4m3, const void* w_scale, int32_t w_scale_dtype,
                        const int32_t* offsets_dev, int32_t G, int64_t total_M, int64_t N,
                        int64_t K, void* y_bf16, int64_t ldy, void* workspace, size_t ws_bytes,
                        void* stream);

/* ---- a10 fused into the gate/up projection --------------------------------- */
/*
 * bfp8_linear_w8a8_silu_quant -- the dense-FFN gate/up projection with
 * SiLU(gate)*up and the 1x128 quantization of h in its epilogue, so that the
 * BF16 [M, 2I] gate/up output never reaches memory.
 *   [Module w8a8_prefill, first paragraph: the gate/up/down GEMM arm]
 * The result equals bfp8_linear_w8a8 with members {I, I} writing gu [M, 2I]
 * in BF16, followed by bfp8_silu_mul_act_quant(gu):
 *   g = bf16_rn(acc_gate), u = bf16_rn(acc_up), h = bf16_rn(silu(g) * u),
 *   then per (token m, 128 columns of h): s = max(max|h|, 1e-10f) / 448,
 *   q_h = RNE_satfinite_e4m3(h / s).
 *   q_a, s_a, s_stride_*  as bfp8_linear_w8a8 (K columns)
 *   w_e4m3   [2I, K] E4M3: the gate rows 0..I-1 stacked over the up rows
 *            I..2I-1, row stride K bytes
 *   w_scale  [2*ceil(I/128), ceil(K/128)]: the gate member's grid stacked over
 *            the up member's (member-local origins), BF16 or F32
 *   q_h      [M, I] E4M3, row stride ldq >= I bytes
 *   s_h      float32 scales of h, (m, g) at s_h[m*sh_stride_m + g*sh_stride_kb]
 *   workspace, ws_bytes  optional stream-K scratch as bfp8_linear_w8a8, sized
 *            by bfp8_linear_w8a8_silu_quant_workspace()
 * Requirements: K % 16 == 0; q_a and w_e4m3 16-byte aligned. M == 0 is a no-op.
 */
size_t bfp8_linear_w8a8_silu_quant_workspace(int64_t M, int64_t I, int64_t K);
int bfp8_linear_w8a8_silu_quant(const void* q_a, const float* s_a, int64_t s_stride_m,
                                int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                                int32_t w_scale_dtype, int64_t M, int64_t I, int64_t K,
                                void* q_h, int64_t ldq, float* s_h, int64_t sh_stride_m,
                                int64_t sh_stride_kb, void* workspace, size_t ws_bytes,
                                void* stream);

/*
 * bfp8_grouped_linear_silu_quant -- the MoE expert gate/up projection with the
 * same fused epilogue, over the token-offset table of bfp8_grouped_linear.
 *   [Module w8a8_prefill, "WHY": the MoE expert path; first paragraph: the
 *    gate/up/down arm]
 *   w_e4m3   [G, 2I, K] E4M3 (each expert: gate rows over up rows)
 *   w_scale  [G, 2*ceil(I/128), ceil(K/128)] (each expert: gate grid over up grid)
 *   q_h      [total_M, I] E4M3, row stride ldq; s_h as above
 *   other arguments, the workspace (sized by
 *   bfp8_grouped_linear_silu_quant_workspace()) and requirements as
 *   bfp8_grouped_linear.
 */
size_t bfp8_grouped_linear_silu_quant_workspace(int64_t total_M, int32_t G, int64_t I, int64_t K);
int bfp8_grouped_linear_silu_quant(const void* q_a, const float* s_a, int64_t s_stride_m,
                                   int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                                   int32_t w_scale_dtype, const int32_t* offsets_dev, int32_t G,
                                   int64_t total_M, int64_t I, int64_t K, void* q_h, int64_t ldq,
                                   float* s_h, int64_t sh_stride_m, int64_t sh_stride_kb,
                                   void* workspace, size_t ws_bytes, void* stream);

/* ---- the steps on either side of the grouped MoE projection -------------- */
/*
 * bfp8_moe_gather_act_quant -- permutation by expert fused with the per-token
 * 1x128 activation quantization: routed row r of the expert-sorted buffer
 * quantizes token row_token[r] of x.
 *   [Module w8a8_prefill, "WHY": the MoE expert path on the block-scaled
 *    prefill arm; arithmetic paragraph: per-token 1x128 FP32 activation scales]
 * Each output row equals bfp8_act_quant_group of its source token row, so
 * the E4M3 codes and scales are bit-exact with quantizing first and
 * permuting after.
 *   x_bf16     [T, H] BF16 tokens, row stride ldx >= H (elements)
 *   row_token  device int32 [R]: the source token of each routed row; an
 *              index outside [0, T) yields a zero row (codes 0, scale 1e-10f/448)
 *   q_e4m3     [R, H] E4M3, row stride ldq >= H (bytes)
 *   scales     float32, (r, g) at scales[r*s_stride_m + g*s_stride_kb]
 * R == 0 or H == 0 is a no-op. Errors: INVALID_ARG for null pointers,
 * negative sizes or ld < H.
 */
int bfp8_moe_gather_act_quant(const void* x_bf16, int64_t T, int64_t H, int64_t ldx,
                              const int32_t* row_token, int64_t R, void* q_e4m3, int64_t ldq,
                              float* scales, int64_t s_stride_m, int64_t s_stride_kb,
                              void* stream);

/*
 * bfp8_moe_combine -- un-permute and weight the routed rows of the down
 * projection back onto their tokens:
 *   out[t, c] = bf16_rn( sum_{j=0}^{topk-1} w[t, j] * y[rows[t, j], c] )
 * as float32 fused multiply-adds in slot order j = 0, 1, ... from 0, so the
 * result is deterministic (no atomics).
 *   [Module w8a8_prefill, "WHY": the MoE expert path; the weights are the
 *    renormalized top-k router probabilities]
 *   y_bf16         [R, H] BF16 routed rows (expert-sorted), row stride ldy >= H
 *   token_rows     device int32 [T, topk]: the routed row of each (token, slot);
 *                  an index outside [0, R) contributes nothing
 *   token_weights  device float32 [T, topk]
 *   out_bf16       [T, H] BF16, row stride ldo >= H; must not overlap y
 * T == 0 or H == 0 is a no-op. Errors: INVALID_ARG for null pointers,
 * negative sizes, topk < 1 or ld < H.
 */
int bfp8_moe_combine(const void* y_bf16, int64_t R, int64_t H, int64_t ldy,
                     const int32_t* token_rows, const float* token_weights, int64_t T,
                     int32_t topk, void* out_bf16, int64_t ldo, void* stream);

/* ---- diagnostics ---------------------------------------------------------- */
/*
 * bfp8_device_status -- synchronise `stream`, then read and clear the library's
 * device error word on the current device. Returns BFP8_OK, BFP8_ERR_TIMEOUT
 * if a bounded wait ran out in a kernel since the last call, or BFP8_ERR_CUDA.
 */
int bfp8_device_status(void* stream);

/*
 * bfp8_selftest_wait_timeout -- exercise the bounded device waits: launch one
 * CTA on `stream` whose barrier gets one of the two arrivals it expects. Two
 * warps wait on it, one in the promotion warps' spinning form and one in the
 * control warps' suspending form; both give up after limit_ns nanoseconds and
 * record BFP8_ERR_TIMEOUT in the device error word, which the next
 * bfp8_device_status() returns (and clears). The kernel then exits normally:
 * the context stays usable. This is a library diagnostic, not part of the
 * projection. Errors: INVALID_ARG unless 0 < limit_ns <= 2e9 (the kernels'
 * own limit).
 */
int bfp8_selftest_wait_timeout(uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BFP8_H_ */
