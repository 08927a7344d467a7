// api.cpp -- the extern "C" boundary of libbfp8: argument checks, the
// metadata-only grid validation, TMA descriptor encoding and the per-device
// caches. No device memory is allocated anywhere in the library.
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "bfp8_internal.h"

namespace bfp8 {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCache {
  std::once_flag once;
  int sms = 0;
  int err = cudaSuccess;
};
DeviceCache g_dev[kMaxDevices];

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return BFP8_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return BFP8_ERR_UNSUPPORTED;
  return BFP8_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int encode(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, const void* base,
           const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
           CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return BFP8_ERR_CUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BFP8_OK : BFP8_ERR_UNSUPPORTED;
}

void write_msg(char* msg, size_t len, const char* fmt, ...) {
  if (!msg || len == 0) return;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, len, fmt, ap);
  va_end(ap);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int sm_count(int* out) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != BFP8_OK) return rc;
  DeviceCache& c = g_dev[dev];
  std::call_once(c.once, [&c, dev] {
    c.err = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
  });
  if (c.err != cudaSuccess || c.sms <= 0) return BFP8_ERR_CUDA;
  *out = c.sms;
  return BFP8_OK;
}

int check_launch() {
  return cudaPeekAtLastError() == cudaSuccess ? BFP8_OK : BFP8_ERR_CUDA;
}

int check_device_ptrs(std::initializer_list<const void*> ptrs) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != BFP8_OK) return rc;
  for (const void* p : ptrs) {
    if (!p) continue;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();  // not sticky; keep it out of the next launch check
      return BFP8_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return BFP8_ERR_INVALID_ARG;
  }
  return BFP8_OK;
}

int set_max_dynamic_smem(const void* kernel, int bytes) {
  // Cheap and idempotent; done on every launch so that every device is covered.
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return BFP8_ERR_CUDA;
  return BFP8_OK;
}

int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                 uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                 CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  return encode(map, dt, 2, base, dims, strides, box, swizzle);
}

int make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                 uint64_t dim1, uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                 uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, box2};
  return encode(map, dt, 3, base, dims, strides, box, swizzle);
}

int resolve_members(int64_t N, const bfp8_members* members, MemberTable* out) {
  memset(out, 0, sizeof(*out));
  if (!members || members->n_members == 0) {
    out->count = 1;
    out->n0[0] = 0;
    out->rows[0] = N;
    out->sbase[0] = 0;
    out->scale_rows = cdiv(N, 128);
    return BFP8_OK;
  }
  if (members->n_members < 0 || members->n_members > BFP8_MAX_MEMBERS || !members->member_rows)
    return BFP8_ERR_INVALID_ARG;
  int64_t row0 = 0, base = 0;
  for (int i = 0; i < members->n_members; ++i) {
    const int64_t r = members->member_rows[i];
    if (r <= 0) return BFP8_ERR_GROUP;
    out->n0[i] = row0;
    out->rows[i] = r;
    out->sbase[i] = base;
    row0 += r;
    base += cdiv(r, 128);
  }
  if (row0 != N) return BFP8_ERR_GROUP;
  out->count = members->n_members;
  out->scale_rows = base;
  return BFP8_OK;
}

}  // namespace bfp8

using namespace bfp8;

extern "C" {

const char* bfp8_status_string(int status) {
  switch (status) {
    case BFP8_OK: return "OK";
    case BFP8_ERR_INVALID_ARG: return "INVALID_ARG";
    case BFP8_ERR_E5M2: return "E5M2";
    case BFP8_ERR_NO_SCALE: return "NO_SCALE";
    case BFP8_ERR_ROW_SCALE: return "ROW_SCALE";
    case BFP8_ERR_AMBIGUOUS_SCALE: return "AMBIGUOUS_SCALE";
    case BFP8_ERR_GRID_TRANSPOSED: return "GRID_TRANSPOSED";
    case BFP8_ERR_GRID_SHAPE: return "GRID_SHAPE";
    case BFP8_ERR_SCALE_DTYPE: return "SCALE_DTYPE";
    case BFP8_ERR_BLOCK_SIZE: return "BLOCK_SIZE";
    case BFP8_ERR_QUANT_METHOD: return "QUANT_METHOD";
    case BFP8_ERR_GROUP: return "GROUP";
    case BFP8_ERR_NOT_FP8: return "NOT_FP8";
    case BFP8_ERR_UNSUPPORTED: return "UNSUPPORTED";
    case BFP8_ERR_CUDA: return "CUDA";
    case BFP8_ERR_TIMEOUT: return "TIMEOUT";
    default: return "UNKNOWN";
  }
}

int bfp8_validate_grid(const bfp8_weight_desc* d, char* msg, size_t msg_len) {
  write_msg(msg, msg_len, "ok");
  if (!d || d->weight_rank != 2 || d->weight_shape[0] <= 0 || d->weight_shape[1] <= 0) {
    write_msg(msg, msg_len, "weight must be a rank-2 [N, K] tensor with positive sizes");
    return BFP8_ERR_INVALID_ARG;
  }
  const int64_t N = d->weight_shape[0], K = d->weight_shape[1];
  if (d->weight_dtype == BFP8_DT_E5M2) {
    write_msg(msg, msg_len, "E5M2 weight encoding is not the block-FP8 (E4M3) format");
    return BFP8_ERR_E5M2;
  }
  if (d->weight_dtype != BFP8_DT_E4M3) {
    write_msg(msg, msg_len, "dense (non-FP8) weight: not a block-scaled FP8 tensor");
    return BFP8_ERR_NOT_FP8;
  }
  if (!d->declared_quant_fp8) {
    write_msg(msg, msg_len, "checkpoint does not declare quant_method fp8");
    return BFP8_ERR_QUANT_METHOD;
  }
  const bool has_block = d->scale_dtype != BFP8_DT_NONE;
  if (d->tensor_scale_dtype != BFP8_DT_NONE) {
    // per-tensor scaled: one multiplier, read as a grid with a single block
    if (has_block || d->has_row_scale) {
      write_msg(msg, msg_len, "a one-element weight_scale next to another scale leaf");
      return BFP8_ERR_AMBIGUOUS_SCALE;
    }
    if (d->declared_block[0] != 0 || d->declared_block[1] != 0) {
      write_msg(msg, msg_len, "per-tensor scaled weight but weight_block_size [%d,%d] declared",
                d->declared_block[0], d->declared_block[1]);
      return BFP8_ERR_BLOCK_SIZE;
    }
    if (d->tensor_scale_dtype != BFP8_DT_BF16 && d->tensor_scale_dtype != BFP8_DT_F32) {
      write_msg(msg, msg_len, "per-tensor weight_scale must be BF16 or F32");
      return BFP8_ERR_SCALE_DTYPE;
    }
    if (d->n_members > 0) {
      if (!d->member_rows || d->n_members > BFP8_MAX_MEMBERS) {
        write_msg(msg, msg_len, "member table missing or longer than %d", BFP8_MAX_MEMBERS);
        return BFP8_ERR_GROUP;
      }
      int64_t sum = 0;
      for (int i = 0; i < d->n_members; ++i) {
        if (d->member_rows[i] <= 0) {
          write_msg(msg, msg_len, "member %d has %lld rows", i, (long long)d->member_rows[i]);
          return BFP8_ERR_GROUP;
        }
        sum += d->member_rows[i];
      }
      if (sum != N) {
        write_msg(msg, msg_len, "member rows sum to %lld, weight has %lld", (long long)sum,
                  (long long)N);
        return BFP8_ERR_GROUP;
      }
    }
    write_msg(msg, msg_len, "OK: per-tensor scaled, one multiplier covers the tensor");
    return BFP8_OK;
  }
  if (d->declared_block[0] != 128 || d->declared_block[1] != 128) {
    write_msg(msg, msg_len, "declared weight_block_size [%d,%d] is not [128,128]",
              d->declared_block[0], d->declared_block[1]);
    return BFP8_ERR_BLOCK_SIZE;
  }
  if (d->has_row_scale) {
    if (has_block) {
      write_msg(msg, msg_len, "both a per-row weight_scale and a weight_scale_inv grid");
      return BFP8_ERR_AMBIGUOUS_SCALE;
    }
    write_msg(msg, msg_len, "row-scaled tree (weight_scale per row): use the row path");
    return BFP8_ERR_ROW_SCALE;
  }
  if (!has_block) {
    write_msg(msg, msg_len, "FP8 weight without weight_scale_inv");
    return BFP8_ERR_NO_SCALE;
  }
  if (d->scale_rank == 1) {
    write_msg(msg, msg_len, "rank-1 scale: a per-row multiplier, not a 128x128 grid");
    return BFP8_ERR_ROW_SCALE;
  }
  if (d->scale_dtype != BFP8_DT_BF16 && d->scale_dtype != BFP8_DT_F32) {
    write_msg(msg, msg_len, "weight_scale_inv must be BF16 or F32");
    return BFP8_ERR_SCALE_DTYPE;
  }
  if (d->scale_rank != 2) {
    write_msg(msg, msg_len, "weight_scale_inv must be rank 2");
    return BFP8_ERR_GRID_SHAPE;
  }
  int64_t Nb = 0;
  const bool grouped = d->n_members > 0;
  if (grouped) {
    if (!d->member_rows || d->n_members > BFP8_MAX_MEMBERS) {
      write_msg(msg, msg_len, "member table missing or longer than %d", BFP8_MAX_MEMBERS);
      return BFP8_ERR_GROUP;
    }
    int64_t sum = 0;
    for (int i = 0; i < d->n_members; ++i) {
      if (d->member_rows[i] <= 0) {
        write_msg(msg, msg_len, "member %d has %lld rows", i, (long long)d->member_rows[i]);
        return BFP8_ERR_GROUP;
      }
      sum += d->member_rows[i];
      Nb += cdiv(d->member_rows[i], 128);
    }
    if (sum != N) {
      write_msg(msg, msg_len, "member rows sum to %lld, weight has %lld", (long long)sum,
                (long long)N);
      return BFP8_ERR_GROUP;
    }
  } else if (d->n_members < 0) {
    write_msg(msg, msg_len, "negative member count");
    return BFP8_ERR_GROUP;
  } else {
    Nb = cdiv(N, 128);
  }
  const int64_t Kb = cdiv(K, 128);
  const int64_t s0 = d->scale_shape[0], s1 = d->scale_shape[1];
  if (s0 == Nb && s1 == Kb) return BFP8_OK;
  if (s0 == Kb && s1 == Nb && Nb != Kb) {
    write_msg(msg, msg_len, "scale grid [%lld,%lld] is transposed; expected [%lld,%lld]",
              (long long)s0, (long long)s1, (long long)Nb, (long long)Kb);
    return BFP8_ERR_GRID_TRANSPOSED;
  }
  if (s0 == N && N != Nb) {
    write_msg(msg, msg_len, "scale grid has one row per weight row: row/block ambiguous");
    return BFP8_ERR_AMBIGUOUS_SCALE;
  }
  if (grouped && s0 == cdiv(N, 128) && s1 == Kb) {
    write_msg(msg, msg_len, "grid built on the stacked rows, not member-local origins");
    return BFP8_ERR_GROUP;
  }
  write_msg(msg, msg_len, "scale grid [%lld,%lld] is mis-blocked; expected [%lld,%lld]",
            (long long)s0, (long long)s1, (long long)Nb, (long long)Kb);
  return BFP8_ERR_GRID_SHAPE;
}

int bfp8_act_quant_group(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q_e4m3,
                         int64_t ldq, float* scales, int64_t s_stride_m, int64_t s_stride_kb,
                         void* stream) {
  return launch_act_quant(x_bf16, M, K, ldx, q_e4m3, ldq, scales, s_stride_m, s_stride_kb,
                          stream);
}

int bfp8_silu_mul_act_quant(const void* gu_bf16, int64_t M, int64_t I, int64_t ld,
                            void* q_e4m3, int64_t ldq, float* scales, int64_t s_stride_m,
                            int64_t s_stride_kb, void* stream) {
  return launch_silu_mul_act_quant(gu_bf16, M, I, ld, q_e4m3, ldq, scales, s_stride_m,
                                   s_stride_kb, stream);
}

int bfp8_silu_mul(const void* gu_bf16, int64_t M, int64_t I, int64_t ld, void* h_bf16,
                  int64_t ldh, void* stream) {
  return launch_silu_mul(gu_bf16, M, I, ld, h_bf16, ldh, stream);
}

size_t bfp8_decode_ffn_workspace(int64_t M, int64_t H, int64_t I, int32_t arith) {
  int sms = 0;
  if (sm_count(&sms) != BFP8_OK) return 0;
  return decode_ffn_workspace_bytes(M, H, I, arith, sms);
}

int bfp8_decode_ffn(int32_t arith, const void* x_bf16, int64_t ldx, const void* w_gate_up,
                    const void* s_gate_up, const void* w_down, const void* s_down,
                    int32_t w_scale_dtype, int64_t M, int64_t H, int64_t I, void* y_bf16,
                    int64_t ldy, void* workspace, size_t ws_bytes, void* stream) {
  return launch_decode_ffn(arith, x_bf16, ldx, w_gate_up, s_gate_up, w_down, s_down,
                           w_scale_dtype, M, H, I, y_bf16, ldy, workspace, ws_bytes, stream);
}

int bfp8_moe_gather_act_quant(const void* x_bf16, int64_t T, int64_t H, int64_t ldx,
                              const int32_t* row_token, int64_t R, void* q_e4m3, int64_t ldq,
                              float* scales, int64_t s_stride_m, int64_t s_stride_kb,
                              void* stream) {
  return launch_moe_gather_act_quant(x_bf16, T, H, ldx, row_token, R, q_e4m3, ldq, scales,
                                     s_stride_m, s_stride_kb, stream);
}

int bfp8_moe_combine(const void* y_bf16, int64_t R, int64_t H, int64_t ldy,
                     const int32_t* token_rows, const float* token_weights, int64_t T,
                     int32_t topk, void* out_bf16, int64_t ldo, void* stream) {
  return launch_moe_combine(y_bf16, R, H, ldy, token_rows, token_weights, T, topk, out_bf16, ldo,
                            stream);
}

int bfp8_quantize_weight_block(const float* w, int64_t N, int64_t K, int64_t ldw, void* q,
                               int64_t ldq, void* scale, int32_t scale_dtype, void* stream) {
  return launch_weight_quant(w, N, K, ldw, q, ldq, scale, scale_dtype, stream);
}

size_t bfp8_linear_w8a8_workspace(int64_t M, int64_t N, int64_t K, const bfp8_members* members) {
  (void)K;
  if (M <= 0 || N <= 0) return 0;
  MemberTable mt;
  int sms = 0;
  if (resolve_members(N, members, &mt) != BFP8_OK || sm_count(&sms) != BFP8_OK) return 0;
  return gemm_w8a8_workspace_bytes(M, N, mt, sms);
}

int bfp8_linear_w8a8(const void* q_a, const float* s_a, int64_t s_stride_m, int64_t s_stride_kb,
                     const void* w_e4m3, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                     int64_t N, int64_t K, void* y_bf16, int64_t ldy,
                     const bfp8_members* members, void* workspace, size_t ws_bytes,
                     void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (M == 0) return BFP8_OK;
  if (!q_a || !s_a || !w_e4m3 || !w_scale || !y_bf16 || ldy < N) return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  MemberTable mt;
  int rc = resolve_members(N, members, &mt);
  if (rc != BFP8_OK) return rc;
  return launch_gemm_w8a8(q_a, s_a, s_stride_m, s_stride_kb, w_e4m3, w_scale, w_scale_dtype, M,
                          N, K, y_bf16, ldy, mt, workspace, ws_bytes, stream);
}

int bfp8_linear_w8a16(const void* x_bf16, int64_t ldx, const void* w_e4m3, const void* w_scale,
                      int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y_bf16,
                      int64_t ldy, const bfp8_members* members, void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (M == 0) return BFP8_OK;
  if (!x_bf16 || !w_e4m3 || !w_scale || !y_bf16 || ldy < N || ldx < K)
    return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  MemberTable mt;
  int rc = resolve_members(N, members, &mt);
  if (rc != BFP8_OK) return rc;
  return launch_gemm_w8a16(x_bf16, ldx, w_e4m3, w_scale, w_scale_dtype, M, N, K, y_bf16, ldy,
                           mt, stream);
}

size_t bfp8_gemv_decode_workspace(int64_t M, int64_t N, int64_t K) {
  int sms = 0;
  if (sm_count(&sms) != BFP8_OK) return 0;
  return gemv_workspace_bytes(M, N, K, sms);
}

int bfp8_gemv_decode(const void* x_bf16, int64_t ldx, const void* w_e4m3, const void* w_scale,
                     int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y_bf16,
                     int64_t ldy, const bfp8_members* members, void* workspace,
                     size_t ws_bytes, void* stream) {
  if (M < 1 || M > 16 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (!x_bf16 || !w_e4m3 || !w_scale || !y_bf16 || ldy < N || ldx < K)
    return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  MemberTable mt;
  int rc = resolve_members(N, members, &mt);
  if (rc != BFP8_OK) return rc;
  return launch_gemv(x_bf16, ldx, w_e4m3, w_scale, w_scale_dtype, M, N, K, y_bf16, ldy, mt,
                     workspace, ws_bytes, stream);
}

int bfp8_gemv_decode_w8a8(const void* q_a, const float* s_a, int64_t s_stride_m,
                          int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                          int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y_bf16,
                          int64_t ldy, const bfp8_members* members, void* workspace,
                          size_t ws_bytes, void* stream) {
  if (M < 1 || M > 16 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (!q_a || !s_a || !w_e4m3 || !w_scale || !y_bf16 || ldy < N) return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  MemberTable mt;
  int rc = resolve_members(N, members, &mt);
  if (rc != BFP8_OK) return rc;
  return launch_gemv_w8a8(q_a, s_a, s_stride_m, s_stride_kb, w_e4m3, w_scale, w_scale_dtype, M,
                          N, K, y_bf16, ldy, mt, workspace, ws_bytes, stream);
}

size_t bfp8_grouped_linear_workspace(int64_t total_M, int32_t G, int64_t N, int64_t K) {
  (void)K;
  int sms = 0;
  if (total_M <= 0 || G < 1 || N <= 0 || sm_count(&sms) != BFP8_OK) return 0;
  return grouped_w8a8_workspace_bytes(total_M, G, N, sms);
}

int bfp8_grouped_linear(const void* q_a, const float* s_a, int64_t s_stride_m,
                        int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                        int32_t w_scale_dtype, const int32_t* offsets_dev, int32_t G,
                        int64_t total_M, int64_t N, int64_t K, void* y_bf16, int64_t ldy,
                        void* workspace, size_t ws_bytes, void* stream) {
  if (G < 1 || G > 1024 || total_M < 0 || N <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (total_M == 0) return BFP8_OK;
  if (!q_a || !s_a || !w_e4m3 || !w_scale || !offsets_dev || !y_bf16 || ldy < N)
    return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  return launch_grouped_w8a8(q_a, s_a, s_stride_m, s_stride_kb, w_e4m3, w_scale, w_scale_dtype,
                             offsets_dev, G, total_M, N, K, y_bf16, ldy, workspace, ws_bytes,
                             stream);
}

size_t bfp8_linear_w8a8_silu_quant_workspace(int64_t M, int64_t I, int64_t K) {
  (void)K;
  int sms = 0;
  if (M <= 0 || I <= 0 || sm_count(&sms) != BFP8_OK) return 0;
  return gemm_w8a8_swiglu_workspace_bytes(M, I, sms);
}

int bfp8_linear_w8a8_silu_quant(const void* q_a, const float* s_a, int64_t s_stride_m,
                                int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                                int32_t w_scale_dtype, int64_t M, int64_t I, int64_t K,
                                void* q_h, int64_t ldq, float* s_h, int64_t sh_stride_m,
                                int64_t sh_stride_kb, void* workspace, size_t ws_bytes,
                                void* stream) {
  if (M < 0 || I <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (M == 0) return BFP8_OK;
  if (!q_a || !s_a || !w_e4m3 || !w_scale || !q_h || !s_h || ldq < I) return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  return launch_gemm_w8a8_swiglu(q_a, s_a, s_stride_m, s_stride_kb, w_e4m3, w_scale,
                                 w_scale_dtype, M, I, K, q_h, ldq, s_h, sh_stride_m,
                                 sh_stride_kb, workspace, ws_bytes, stream);
}

size_t bfp8_grouped_linear_silu_quant_workspace(int64_t total_M, int32_t G, int64_t I, int64_t K) {
  (void)K;
  int sms = 0;
  if (total_M <= 0 || G < 1 || I <= 0 || sm_count(&sms) != BFP8_OK) return 0;
  return grouped_w8a8_swiglu_workspace_bytes(total_M, G, I, sms);
}

int bfp8_grouped_linear_silu_quant(const void* q_a, const float* s_a, int64_t s_stride_m,
                                   int64_t s_stride_kb, const void* w_e4m3, const void* w_scale,
                                   int32_t w_scale_dtype, const int32_t* offsets_dev, int32_t G,
                                   int64_t total_M, int64_t I, int64_t K, void* q_h, int64_t ldq,
                                   float* s_h, int64_t sh_stride_m, int64_t sh_stride_kb,
                                   void* workspace, size_t ws_bytes, void* stream) {
  if (G < 1 || G > 1024 || total_M < 0 || I <= 0 || K <= 0) return BFP8_ERR_INVALID_ARG;
  if (total_M == 0) return BFP8_OK;
  if (!q_a || !s_a || !w_e4m3 || !w_scale || !offsets_dev || !q_h || !s_h || ldq < I)
    return BFP8_ERR_INVALID_ARG;
  if (!weight_scale_dtype_ok(w_scale_dtype)) return BFP8_ERR_SCALE_DTYPE;
  return launch_grouped_w8a8_swiglu(q_a, s_a, s_stride_m, s_stride_kb, w_e4m3, w_scale,
                                    w_scale_dtype, offsets_dev, G, total_M, I, K, q_h, ldq, s_h,
                                    sh_stride_m, sh_stride_kb, workspace, ws_bytes, stream);
}

int bfp8_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  return launch_wait_selftest(limit_ns, stream);
}

int bfp8_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BFP8_ERR_CUDA;
  const int a = gemm_read_clear_error();
  const int b = gemv_read_clear_error();
  if (a == BFP8_ERR_CUDA || b == BFP8_ERR_CUDA) return BFP8_ERR_CUDA;
  if (a != BFP8_OK) return a;
  return b;
}

}  // extern "C"
