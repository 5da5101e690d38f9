// bi_internal.h -- host-side interface between the C ABI layer (abi.cu) and
// the translation units that hold the kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "bi.h"

namespace bi {

// ---- per-device state kept by abi.cu --------------------------------------
// Device address of the current device's error word (nullptr on failure).
int* device_error_word();
// SM count of the current device (0 on failure); cached per device.
int device_sm_count();
// Encode a 2-D bf16 tensor map (rows x cols, row stride = cols elements) with
// a box of box_rows x box_cols and 128-byte swizzling.  Returns false if the
// driver entry point is unavailable or the encoding is rejected.
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows, uint32_t box_cols);
// Encode a bf16 tensor map over the same matrix as a 3-D view (64 columns,
// rows, the rows' 128-byte column groups) whose box is box_rows rows times
// box_groups consecutive column groups: one copy reads box_groups * 128
// contiguous bytes of each row, and the groups land one after another in
// shared memory (group g of every row, then group g + 1), each with the
// 128-byte swizzle of a box_rows x 64 box.  cols must be a multiple of 64 and
// box_groups at most cols / 64; groups past the last read as zero.
bool make_tmap_groups_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_groups);

inline bi_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BI_OK : BI_ERR_CUDA; }

// ---- RMSNorm (rmsnorm.cu) ---------------------------------------------------
bi_status launch_rmsnorm_invariant(const void* x, const void* w, void* y, float* y_f32,
                                   int64_t M, int64_t H, float eps, int* err, cudaStream_t s);
bi_status launch_add_rmsnorm_invariant(const void* x, void* res, const void* w, void* y,
                                       float* y_f32, int64_t M, int64_t H, float eps,
                                       cudaStream_t s);
bi_status launch_add_bf16(const void* x, void* res, int64_t elems, cudaStream_t s);
bi_status launch_gather_rows(const void* src, int64_t rows, int64_t H, const int32_t* idx,
                             int64_t n, void* dst, int* err, cudaStream_t s);
bi_status launch_rope_qkv(const void* qkv, const int32_t* pos, int64_t T, int Hq, int Hkv, int D,
                          double theta, void* q, void* k, void* v, cudaStream_t s);
bi_status launch_silu_mul(const void* gu, int64_t T, int64_t F, int64_t block, void* out,
                          cudaStream_t s);
bi_status launch_sample(const void* logits, int64_t B, int64_t V, const float* temperature,
                        const uint64_t* seed, const uint64_t* step, int32_t* tokens,
                        cudaStream_t s);
int rmsnorm_variant_splits(int64_t M, int64_t H, int num_sms);
bi_status launch_rmsnorm_variant(const void* x, const void* w, void* y, float* y_f32, int64_t M,
                                 int64_t H, float eps, int splits, float* ws, int* err,
                                 cudaStream_t s);

// ---- GEMM (gemm.cu) ---------------------------------------------------------
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;
constexpr int kGemmSmallRows = 32;    // at most this many rows of A: a 32-row A ring
constexpr int kGemmNarrowRows = 64;   // at most this many rows of A: the narrow ring may run
constexpr int kGemmNarrowBN = 64;     // the narrow ring's output tile width
constexpr int kGemmNarrowKBlocks = 4; // k-blocks per stage of the narrow ring
// The narrow ring (64-column output tiles, four k-blocks per stage) runs for
// at most 64 rows of A when its tiles fit in one wave of the device's
// num_sms blocks, K is whole 64-column groups (at least four) and the
// epilogue is not SwiGLU (whose tile pairs 128 gate and 128 up rows); every
// other shape takes 256-column tiles.  The tile width never changes a
// row's arithmetic (tcgen05.mma gives each output element the same sum for
// every N), only how many blocks stream the weight.
inline bool gemm_narrow(int64_t M, int64_t N, int64_t K, int num_sms, bool swiglu) {
  return !swiglu && M <= kGemmNarrowRows && K % kGemmBK == 0 &&
         K / kGemmBK >= kGemmNarrowKBlocks &&
         (N + kGemmNarrowBN - 1) / kGemmNarrowBN <= num_sms;
}
// Above the small batches, a 128 x 192 tile where its tiles fill the SMs
// better than 128 x 256 ones: rounds of num_sms tiles times the tile width,
// the 192-column cost weighted by 10/9 (its tiles ran ~10% slower per flop
// on GB300: 8192 x 6144 x 4096 took 266 us against 252 with 256-column
// tiles, while at 256 and 1024 rows, one or two rounds, it took 28 and 47 us
// against 35 and 57); 256 always with SwiGLU.
constexpr int kGemmMidBN = 192;
inline int gemm_wide_tile(int64_t M, int64_t N, int num_sms, bool swiglu) {
  if (swiglu || M <= kGemmSmallRows || num_sms <= 0) return kGemmBN;
  const int64_t mt = (M + kGemmBM - 1) / kGemmBM;
  auto cost = [&](int64_t bn) {
    const int64_t tiles = mt * ((N + bn - 1) / bn);
    return ((tiles + num_sms - 1) / num_sms) * bn;
  };
  return cost(kGemmMidBN) * 10 < cost(kGemmBN) * 9 ? kGemmMidBN : kGemmBN;
}
inline int gemm_n_tile(int64_t M, int64_t N, int64_t K, int num_sms, bool swiglu) {
  return gemm_narrow(M, N, K, num_sms, swiglu) ? kGemmNarrowBN
                                                : gemm_wide_tile(M, N, num_sms, swiglu);
}
// swiglu: C is [M, N/2], the SwiGLU product of each tile's two column halves
bi_status launch_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K,
                      int splits, float* ws, int* err, cudaStream_t s, bool swiglu = false);

// ---- attention (attention.cu) -------------------------------------------------
struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* kv_lens;
  const int32_t* cu_q;        // prefill only
  const int32_t* q_start;     // prefill only
  void* out;
  float* out_f32;
  int B, Hq, Hkv, D, page_size;
  int64_t num_pages;
  int max_blocks;
  int max_kv_len;
  int64_t total_q;            // prefill only
  int max_q_len;              // prefill only
  int split_size;             // invariant: fixed split size
  int split_count;            // variant: fixed split count (decode)
  bool variant;
  float sm_scale;
  float* ws;                  // decode partials
  int max_splits;             // decode: partial slots per (b, q-head)
  int* err;
};
int attn_decode_max_splits(int max_kv_len, int split_size, bool variant, int split_count);
int attn_variant_split_count(int B, int Hkv, int max_kv_len, int num_sms);
size_t attn_decode_workspace_bytes(int B, int Hq, int D, int max_splits);
bi_status launch_attn_decode(const AttnArgs& a, cudaStream_t s);
bi_status launch_attn_prefill(const AttnArgs& a, cudaStream_t s);
bi_status launch_kv_write(const void* k_new, const void* v_new, const int32_t* seq,
                          const int32_t* pos, int64_t n_tokens, void* k_cache, void* v_cache,
                          const int32_t* block_table, int Hkv, int D, int page_size,
                          int64_t num_pages, int max_blocks, int* err, cudaStream_t s);

}  // namespace bi
