// bfp8_internal.h -- host-side glue shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <initializer_list>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bfp8.h"

namespace bfp8 {

// Multiprocessor count of the current device (cached per device).
int sm_count(int* out);
// Map the last launch error (if any) to a status.
int check_launch();
// Every pointer a kernel or a tensor map will dereference must be device
// memory of the current device (cudaMalloc, a stream-ordered pool, or the
// library's own __device__ arrays). Host memory, pinned or not, managed
// memory and another GPU's memory are refused with BFP8_ERR_INVALID_ARG,
// before anything is launched. Null entries are skipped.
int check_device_ptrs(std::initializer_list<const void*> ptrs);
// Make `kernel` accept `bytes` of dynamic shared memory on the current device.
int set_max_dynamic_smem(const void* kernel, int bytes);

// Tiled tensor maps (TMA descriptors). dims/strides innermost first; strides
// are in bytes for dimensions 1.. (dimension 0 is contiguous).
int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                 uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                 CUtensorMapSwizzle swizzle);
int make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                 uint64_t dim1, uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                 uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle);

// Member table resolved on the host: member i covers output rows
// [n0[i], n0[i] + rows[i]) and its scale rows start at sbase[i].
struct MemberTable {
  int32_t count;
  int64_t n0[BFP8_MAX_MEMBERS];
  int64_t rows[BFP8_MAX_MEMBERS];
  int64_t sbase[BFP8_MAX_MEMBERS];
  int64_t scale_rows;  // sum_i ceil(rows_i / 128)
};
int resolve_members(int64_t N, const bfp8_members* members, MemberTable* out);

// A projection's w_scale_dtype: BF16 or F32, optionally OR'd with
// BFP8_SCALE_PER_TENSOR (one multiplier for the whole tensor).
inline bool weight_scale_dtype_ok(int32_t d) {
  const int32_t b = d & ~static_cast<int32_t>(BFP8_SCALE_PER_TENSOR);
  return b == BFP8_DT_BF16 || b == BFP8_DT_F32;
}
inline bool weight_scale_f32(int32_t d) {
  return (d & ~static_cast<int32_t>(BFP8_SCALE_PER_TENSOR)) == BFP8_DT_F32;
}
inline bool weight_scale_per_tensor(int32_t d) { return (d & BFP8_SCALE_PER_TENSOR) != 0; }

// Launchers (argument checks beyond the common ones happen inside).
// The two 1x128 quantizers can also zero n_clear int32 counters at `clear`
// once the previous kernel on the stream has finished (the decode step hands
// them the next GEMV's tile counters); M and K must then be nonzero.
int launch_act_quant(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                     float* s, int64_t ssm, int64_t sskb, void* stream, int32_t* clear = nullptr,
                     int32_t n_clear = 0);
int launch_silu_mul_act_quant(const void* gu, int64_t M, int64_t I, int64_t ld, void* q,
                              int64_t ldq, float* s, int64_t ssm, int64_t sskb, void* stream,
                              int32_t* clear = nullptr, int32_t n_clear = 0);
int launch_silu_mul(const void* gu, int64_t M, int64_t I, int64_t ld, void* h, int64_t ldh,
                    void* stream);
int launch_moe_gather_act_quant(const void* x, int64_t T, int64_t H, int64_t ldx,
                                const int32_t* row_token, int64_t R, void* q, int64_t ldq,
                                float* s, int64_t ssm, int64_t sskb, void* stream);
int launch_moe_combine(const void* y, int64_t R, int64_t H, int64_t ldy, const int32_t* token_rows,
                       const float* token_weights, int64_t T, int32_t topk, void* out, int64_t ldo,
                       void* stream);
int launch_weight_quant(const float* w, int64_t N, int64_t K, int64_t ldw, void* q, int64_t ldq,
                        void* scale, int32_t scale_dtype, void* stream);

size_t gemm_w8a8_workspace_bytes(int64_t M, int64_t N, const MemberTable& mt, int sms);
size_t grouped_w8a8_workspace_bytes(int64_t total_M, int32_t G, int64_t N, int sms);
int launch_gemm_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                     const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                     int64_t N, int64_t K, void* y, int64_t ldy, const MemberTable& mt,
                     void* workspace, size_t ws_bytes, void* stream);
size_t gemm_w8a8_swiglu_workspace_bytes(int64_t M, int64_t I, int sms);
size_t grouped_w8a8_swiglu_workspace_bytes(int64_t total_M, int32_t G, int64_t I, int sms);
int launch_gemm_w8a8_swiglu(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                            const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                            int64_t I, int64_t K, void* q_h, int64_t ldq, float* s_h,
                            int64_t sh_sm, int64_t sh_skb, void* workspace, size_t ws_bytes,
                            void* stream);
int launch_grouped_w8a8_swiglu(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                               const void* w, const void* w_scale, int32_t w_scale_dtype,
                               const int32_t* offsets, int32_t G, int64_t total_M, int64_t I,
                               int64_t K, void* q_h, int64_t ldq, float* s_h, int64_t sh_sm,
                               int64_t sh_skb, void* workspace, size_t ws_bytes, void* stream);
int launch_gemm_w8a16(const void* x, int64_t ldx, const void* w, const void* w_scale,
                      int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y,
                      int64_t ldy, const MemberTable& mt, void* stream);
int launch_grouped_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                        const void* w, const void* w_scale, int32_t w_scale_dtype,
                        const int32_t* offsets, int32_t G, int64_t total_M, int64_t N,
                        int64_t K, void* y, int64_t ldy, void* workspace, size_t ws_bytes,
                        void* stream);

size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K, int sms);
int launch_gemv(const void* x, int64_t ldx, const void* w, const void* w_scale,
                int32_t w_scale_dtype, int64_t M, int64_t N, int64_t K, void* y, int64_t ldy,
                const MemberTable& mt, void* workspace, size_t ws_bytes, void* stream,
                bool silu = false);
int launch_gemv_w8a8(const void* q_a, const float* s_a, int64_t sa_sm, int64_t sa_skb,
                     const void* w, const void* w_scale, int32_t w_scale_dtype, int64_t M,
                     int64_t N, int64_t K, void* y, int64_t ldy, const MemberTable& mt,
                     void* workspace, size_t ws_bytes, void* stream, bool clear_counters = true);
// The W8A8 GEMV's tile counters: at the workspace's start, one per 128 rows of N.
int32_t gemv_counter_count(int64_t N);

// The dense-FFN decode step (gate/up GEMV -> SiLU*up -> down GEMV).
size_t decode_ffn_workspace_bytes(int64_t M, int64_t H, int64_t I, int32_t arith, int sms);
int launch_decode_ffn(int32_t arith, const void* x, int64_t ldx, const void* w_gu,
                      const void* s_gu, const void* w_dn, const void* s_dn, int32_t w_scale_dtype,
                      int64_t M, int64_t H, int64_t I, void* y, int64_t ldy, void* workspace,
                      size_t ws_bytes, void* stream);

// Device error words, one per translation unit with bounded waits: read and
// clear. Return BFP8_OK, BFP8_ERR_TIMEOUT or BFP8_ERR_CUDA.
int gemm_read_clear_error();
// One bounded wait that runs out after limit_ns (0 < limit_ns <= 2 s).
int launch_wait_selftest(uint64_t limit_ns, void* stream);
int gemv_read_clear_error();

}  // namespace bfp8
