// abi.cu -- the C ABI of libbi (declared in include/bi.h): argument checks,
// workspace sizing, the per-device error word, TMA descriptor encoding, and
// dispatch to the kernels.  Every entry point validates before it launches
// and never allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bi.h"
#include "bi_internal.h"
#include "device_common.cuh"

namespace bi {

// One error word per device (a __device__ variable exists once per device
// that loads the module); kernels record the first device-side error here.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_addr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int* device_error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_addr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_addr[d] = static_cast<int*>(p);
  }
  return g_err_addr[d];
}

int device_sm_count() {
  const int d = current_device();
  if (d < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_sm_count[d] = n;
  }
  return g_sm_count[d];
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows, uint32_t box_cols) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool make_tmap_groups_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_groups) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode || cols % 64 != 0 || box_groups < 1 || box_groups > cols / 64) return false;
  // dimension 0: 64 columns of a 128-byte group, 1: rows, 2: the row's groups
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, box_groups};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace bi

using namespace bi;

extern "C" {

const char* bi_version(void) { return "0.1.0"; }

const char* bi_status_string(bi_status s) {
  switch (s) {
    case BI_OK: return "ok";
    case BI_ERR_INVALID_ARG: return "invalid argument (null, negative or misaligned)";
    case BI_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case BI_ERR_WORKSPACE: return "workspace missing or too small";
    case BI_ERR_CUDA: return "CUDA call failed";
    case BI_ERR_DEVICE_BOUNDS: return "device-side bounds check failed (bad page id or length)";
    case BI_ERR_TIMEOUT: return "device-side bounded wait ran out";
  }
  return "unknown status";
}

bi_status bi_check_device_errors(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BI_ERR_CUDA;
  int* addr = device_error_word();
  if (!addr) return BI_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, addr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(addr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return BI_ERR_CUDA;
  }
  return static_cast<bi_status>(v);
}

// --------------------------------------------------------------- self-test
// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after limit_ns, records BI_ERR_TIMEOUT and the kernel returns.
static __global__ void wait_timeout_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, err, nullptr, limit_ns);
}

bi_status bi_selftest_wait_timeout(uint32_t timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 2000000u) return BI_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (!err) return BI_ERR_CUDA;
  wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      err, static_cast<uint64_t>(timeout_us) * 1000u);
  return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------------------ RMSNorm
size_t bi_rmsnorm_workspace_size(int64_t M, int64_t H, bi_mode mode) {
  (void)H;
  if (mode != BI_MODE_VARIANT || M <= 0) return 0;
  return static_cast<size_t>(M) * 64u * sizeof(float);
}

bi_status bi_rmsnorm(const void* x, const void* w, void* y, float* y_f32, int64_t M, int64_t H,
                     float eps, bi_mode mode, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (M < 0 || H <= 0) return BI_ERR_INVALID_ARG;
  if (mode != BI_MODE_INVARIANT && mode != BI_MODE_VARIANT) return BI_ERR_INVALID_ARG;
  if (H % 8 != 0 || H < 8 || H > 65536) return BI_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return BI_ERR_UNSUPPORTED;
  if (M == 0) return BI_OK;
  if (!x || !w || !y) return BI_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return BI_ERR_INVALID_ARG;
  if (y_f32 && !aligned16(y_f32)) return BI_ERR_INVALID_ARG;
  if (!(eps >= 0.0f)) return BI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_word();
  if (mode == BI_MODE_INVARIANT)
    return launch_rmsnorm_invariant(x, w, y, y_f32, M, H, eps, err, s);
  const int sms = device_sm_count();
  if (sms <= 0) return BI_ERR_CUDA;
  const int splits = rmsnorm_variant_splits(M, H, sms);
  if (splits > 1) {
    const size_t need = static_cast<size_t>(M) * splits * sizeof(float);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BI_ERR_WORKSPACE;
  }
  return launch_rmsnorm_variant(x, w, y, y_f32, M, H, eps, splits,
                                static_cast<float*>(workspace), err, s);
}

bi_status bi_add_rmsnorm(const void* x, void* residual, const void* w, void* y, float* y_f32,
                         int64_t M, int64_t H, float eps, bi_mode mode, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (M < 0 || H <= 0) return BI_ERR_INVALID_ARG;
  if (mode != BI_MODE_INVARIANT && mode != BI_MODE_VARIANT) return BI_ERR_INVALID_ARG;
  if (H % 8 != 0 || H < 8 || H > 65536) return BI_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return BI_ERR_UNSUPPORTED;
  if (M == 0) return BI_OK;
  if (!x || !residual || !w || !y) return BI_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(w) || !aligned16(y))
    return BI_ERR_INVALID_ARG;
  if (y_f32 && !aligned16(y_f32)) return BI_ERR_INVALID_ARG;
  if (!(eps >= 0.0f)) return BI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mode == BI_MODE_INVARIANT)
    return launch_add_rmsnorm_invariant(x, residual, w, y, y_f32, M, H, eps, s);
  const bi_status st = launch_add_bf16(x, residual, M * H, s);
  if (st != BI_OK) return st;
  return bi_rmsnorm(residual, w, y, y_f32, M, H, eps, mode, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------------- GEMM
// The variant's split count, over the output tiles bi_gemm uses for this
// shape (gemm_n_tile: 64 columns where the narrow ring runs, else 256).
// bi_gemm_swiglu takes the same count for its [M, 2F] shape, so that in
// either mode it gives the bytes of bi_gemm followed by the SwiGLU kernel.
int bi_gemm_variant_splits(int64_t M, int64_t N, int64_t K, int num_sms) {
  if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return 1;
  const int64_t bn = gemm_n_tile(M, N, K, num_sms, false);
  const int64_t tiles = ((M + kGemmBM - 1) / kGemmBM) * ((N + bn - 1) / bn);
  const int64_t kblocks = (K + kGemmBK - 1) / kGemmBK;
  int64_t s = 1;
  // split K only when the tiles leave most SMs idle (at most a quarter busy:
  // measured on GB300, splitting 48 or 56 tiles of K = 4096 was 13-40% slower
  // than not splitting, 24 tiles 15-20% faster), then until the slices cover
  // the SMs, keeping at least 4 k-blocks per slice
  if (tiles * 4 > num_sms) return 1;
  while (tiles * s < num_sms && kblocks / (s * 2) >= 4 && s < 16) s *= 2;
  return static_cast<int>(s);
}

size_t bi_gemm_workspace_size(int64_t M, int64_t N, int64_t K, bi_mode mode,
                              int variant_splits) {
  if (mode != BI_MODE_VARIANT || M <= 0 || N <= 0 || K <= 0) return 0;
  int s = variant_splits;
  if (s <= 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return static_cast<size_t>(-1);
    s = bi_gemm_variant_splits(M, N, K, sms);
  }
  if (s <= 1) return 0;
  return static_cast<size_t>(s) * static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
}

bi_status bi_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K,
                  bi_mode mode, int variant_splits, void* workspace, size_t workspace_bytes,
                  void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
  if (mode != BI_MODE_INVARIANT && mode != BI_MODE_VARIANT) return BI_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 8 != 0) return BI_ERR_UNSUPPORTED;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return BI_ERR_UNSUPPORTED;
  if (M == 0) return BI_OK;
  if (!A || !W || !C) return BI_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C)) return BI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_word();
  int splits = 1;
  if (mode == BI_MODE_VARIANT) {
    splits = variant_splits;
    if (splits <= 0) {
      const int sms = device_sm_count();
      if (sms <= 0) return BI_ERR_CUDA;
      splits = bi_gemm_variant_splits(M, N, K, sms);
    }
    const int64_t kblocks = (K + kGemmBK - 1) / kGemmBK;
    if (splits > kblocks) splits = static_cast<int>(kblocks);
    if (splits > 1) {
      const size_t need = static_cast<size_t>(splits) * M * N * sizeof(float);
      if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BI_ERR_WORKSPACE;
    }
  }
  return launch_gemm(A, W, C, M, N, K, splits, static_cast<float*>(workspace), err, s);
}

bi_status bi_gemm_swiglu(const void* A, const void* W, void* out, int64_t M, int64_t F,
                         int64_t K, bi_mode mode, int variant_splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (M < 0 || F <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
  if (mode != BI_MODE_INVARIANT && mode != BI_MODE_VARIANT) return BI_ERR_INVALID_ARG;
  if (F % (kGemmBN / 2) != 0 || K % 8 != 0) return BI_ERR_UNSUPPORTED;
  const int64_t N = 2 * F;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return BI_ERR_UNSUPPORTED;
  if (M == 0) return BI_OK;
  if (!A || !W || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(out)) return BI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int splits = 1;
  if (mode == BI_MODE_VARIANT) {
    splits = variant_splits;
    if (splits <= 0) {
      const int sms = device_sm_count();
      if (sms <= 0) return BI_ERR_CUDA;
      splits = bi_gemm_variant_splits(M, N, K, sms);
    }
    const int64_t kblocks = (K + kGemmBK - 1) / kGemmBK;
    if (splits > kblocks) splits = static_cast<int>(kblocks);
    if (splits > 1) {
      const size_t need = static_cast<size_t>(splits) * M * N * sizeof(float);
      if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BI_ERR_WORKSPACE;
    }
  }
  return launch_gemm(A, W, out, M, N, K, splits, static_cast<float*>(workspace),
                     device_error_word(), s, /*swiglu=*/true);
}

// ---------------------------------------------------------------- attention
// The softmax scale must be positive and finite: the kernels take the
// reference maximum of the raw scores and scale it once, which equals the
// maximum of the scaled scores only for a positive scale.
static bool scale_ok(float s) { return s > 0.0f && s <= 3.4e38f; }

static bi_status attn_common_checks(const void* q, const void* k, const void* v,
                                    const int32_t* bt, const int32_t* kl, const void* out,
                                    const float* out_f32, int B, int Hq, int Hkv, int D,
                                    int page_size, int64_t num_pages, int max_blocks,
                                    int max_kv_len, int split_size, bi_mode mode) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 ||
      max_blocks <= 0 || max_kv_len < 0)
    return BI_ERR_INVALID_ARG;
  if (mode != BI_MODE_INVARIANT && mode != BI_MODE_VARIANT) return BI_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BI_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0 || Hq / Hkv > 16) return BI_ERR_UNSUPPORTED;
  if (page_size != 16) return BI_ERR_UNSUPPORTED;
  if (split_size <= 0 || split_size % 64 != 0) return BI_ERR_UNSUPPORTED;
  if (num_pages * Hkv * page_size >= (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535) return BI_ERR_UNSUPPORTED;
  if (B == 0) return BI_OK;
  if (!q || !k || !v || !bt || !kl || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return BI_ERR_INVALID_ARG;
  if (out_f32 && !aligned16(out_f32)) return BI_ERR_INVALID_ARG;
  return BI_OK;
}

size_t bi_attn_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_kv_len,
                                     int split_size, bi_mode mode, int variant_splits) {
  if (B <= 0 || Hq <= 0 || D <= 0 || max_kv_len <= 0 || split_size <= 0) return 0;
  int count = variant_splits;
  if (mode == BI_MODE_VARIANT && count <= 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return static_cast<size_t>(-1);
    count = attn_variant_split_count(B, Hkv, max_kv_len, sms);
  }
  const int ms = attn_decode_max_splits(max_kv_len, split_size, mode == BI_MODE_VARIANT, count);
  return attn_decode_workspace_bytes(B, Hq, D, ms);
}

bi_status bi_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, const int32_t* kv_lens, void* out,
                         float* out_f32, int B, int Hq, int Hkv, int D, int page_size,
                         int64_t num_pages, int max_blocks_per_seq, int max_kv_len,
                         int split_size, float sm_scale, bi_mode mode, int variant_splits,
                         void* workspace, size_t workspace_bytes, void* stream) {
  bi_status st = attn_common_checks(q, k_cache, v_cache, block_table, kv_lens, out, out_f32, B,
                                    Hq, Hkv, D, page_size, num_pages, max_blocks_per_seq,
                                    max_kv_len, split_size, mode);
  if (st != BI_OK || B == 0) return st;
  if (!scale_ok(sm_scale)) return BI_ERR_INVALID_ARG;
  AttnArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.block_table = block_table;
  a.kv_lens = kv_lens; a.out = out; a.out_f32 = out_f32;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.page_size = page_size; a.num_pages = num_pages;
  a.max_blocks = max_blocks_per_seq; a.max_kv_len = max_kv_len; a.split_size = split_size;
  a.variant = mode == BI_MODE_VARIANT; a.sm_scale = sm_scale;
  a.err = device_error_word();
  if (a.variant) {
    int c = variant_splits;
    if (c <= 0) {
      const int sms = device_sm_count();
      if (sms <= 0) return BI_ERR_CUDA;
      c = attn_variant_split_count(B, Hkv, max_kv_len, sms);
    }
    a.split_count = c;
  }
  a.max_splits = attn_decode_max_splits(max_kv_len, split_size, a.variant, a.split_count);
  if (a.max_splits > 0) {
    const size_t need = attn_decode_workspace_bytes(B, Hq, D, a.max_splits);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return BI_ERR_WORKSPACE;
  }
  a.ws = static_cast<float*>(workspace);
  return launch_attn_decode(a, static_cast<cudaStream_t>(stream));
}

bi_status bi_attn_prefill_chunk(const void* q, const int32_t* cu_q, const int32_t* q_start_pos,
                                const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* kv_lens, void* out,
                                float* out_f32, int B, int Hq, int Hkv, int D, int page_size,
                                int64_t num_pages, int max_blocks_per_seq, int64_t total_q,
                                int max_q_len, int max_kv_len, int split_size, float sm_scale,
                                bi_mode mode, int variant_splits, void* workspace,
                                size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  bi_status st = attn_common_checks(q, k_cache, v_cache, block_table, kv_lens, out, out_f32, B,
                                    Hq, Hkv, D, page_size, num_pages, max_blocks_per_seq,
                                    max_kv_len, split_size, mode);
  if (st != BI_OK || B == 0) return st;
  if (total_q < 0 || max_q_len < 0 || !scale_ok(sm_scale)) return BI_ERR_INVALID_ARG;
  if (total_q == 0 || max_q_len == 0) return BI_OK;
  if (!cu_q || !q_start_pos) return BI_ERR_INVALID_ARG;
  if (total_q * Hq >= (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
  AttnArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.block_table = block_table;
  a.kv_lens = kv_lens; a.cu_q = cu_q; a.q_start = q_start_pos; a.out = out; a.out_f32 = out_f32;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.page_size = page_size; a.num_pages = num_pages;
  a.max_blocks = max_blocks_per_seq; a.max_kv_len = max_kv_len; a.total_q = total_q;
  a.max_q_len = max_q_len; a.split_size = split_size; a.sm_scale = sm_scale;
  a.variant = mode == BI_MODE_VARIANT;
  a.err = device_error_word();
  if (a.variant) {
    int c = variant_splits;
    if (c <= 0) {
      const int sms = device_sm_count();
      if (sms <= 0) return BI_ERR_CUDA;
      c = attn_variant_split_count(B, Hkv, max_kv_len, sms);
    }
    // chunk-derived split size: the boundaries move with the chunk's length
    const int per = (max_kv_len + c - 1) / c;
    a.split_size = ((per + 63) / 64) * 64;
    if (a.split_size <= 0) a.split_size = 64;
    a.split_count = c;
  }
  return launch_attn_prefill(a, static_cast<cudaStream_t>(stream));
}

bi_status bi_kv_write(const void* k_new, const void* v_new, const int32_t* seq,
                      const int32_t* pos, int64_t n_tokens, void* k_cache, void* v_cache,
                      const int32_t* block_table, int Hkv, int D, int page_size,
                      int64_t num_pages, int max_blocks_per_seq, void* stream) {
  if (n_tokens < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 ||
      max_blocks_per_seq <= 0)
    return BI_ERR_INVALID_ARG;
  if (D % 8 != 0) return BI_ERR_UNSUPPORTED;
  if (n_tokens == 0) return BI_OK;
  if (n_tokens * Hkv >= (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !seq || !pos || !k_cache || !v_cache || !block_table)
    return BI_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return BI_ERR_INVALID_ARG;
  return launch_kv_write(k_new, v_new, seq, pos, n_tokens, k_cache, v_cache, block_table, Hkv, D,
                         page_size, num_pages, max_blocks_per_seq, device_error_word(),
                         static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- element-wise layer ops
bi_status bi_gather_rows(const void* src, int64_t rows, int64_t H, const int32_t* idx, int64_t n,
                         void* dst, void* stream) {
  if (rows < 0 || H <= 0 || n < 0) return BI_ERR_INVALID_ARG;
  if (H % 8 != 0) return BI_ERR_UNSUPPORTED;
  if (n == 0) return BI_OK;
  if (!src || !idx || !dst || !aligned16(src) || !aligned16(dst)) return BI_ERR_INVALID_ARG;
  return launch_gather_rows(src, rows, H, idx, n, dst, device_error_word(),
                            static_cast<cudaStream_t>(stream));
}

bi_status bi_rope_qkv(const void* qkv, const int32_t* pos, int64_t T, int Hq, int Hkv, int D,
                      double theta, void* q, void* k, void* v, void* stream) {
  if (T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return BI_ERR_INVALID_ARG;
  if (!(theta > 1.0) || !(theta < 1e300)) return BI_ERR_INVALID_ARG;
  if (D % 16 != 0 || D > 1024 || Hq + 2 * Hkv > 65535) return BI_ERR_UNSUPPORTED;
  if (T == 0) return BI_OK;
  if (!qkv || !pos || !q || !k || !v) return BI_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return BI_ERR_INVALID_ARG;
  return launch_rope_qkv(qkv, pos, T, Hq, Hkv, D, theta, q, k, v,
                         static_cast<cudaStream_t>(stream));
}

bi_status bi_silu_mul(const void* gate_up, int64_t T, int64_t F, int64_t block, void* out,
                      void* stream) {
  if (T < 0 || F <= 0 || block <= 0) return BI_ERR_INVALID_ARG;
  if (block % 8 != 0 || F % block != 0 || F >= (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
  if (T == 0) return BI_OK;
  if (!gate_up || !out || !aligned16(gate_up) || !aligned16(out)) return BI_ERR_INVALID_ARG;
  return launch_silu_mul(gate_up, T, F, block, out, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ sampling
bi_status bi_sample(const void* logits, int64_t B, int64_t V, const float* temperature,
                    const uint64_t* seed, const uint64_t* step, int32_t* tokens, void* stream) {
  if (B < 0 || V <= 0) return BI_ERR_INVALID_ARG;
  if (B > 65535 || V >= (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
  if (B == 0) return BI_OK;
  if (!logits || !temperature || !seed || !step || !tokens) return BI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 1u) || (reinterpret_cast<uintptr_t>(seed) & 7u) ||
      (reinterpret_cast<uintptr_t>(step) & 7u) || (reinterpret_cast<uintptr_t>(temperature) & 3u) ||
      (reinterpret_cast<uintptr_t>(tokens) & 3u))
    return BI_ERR_INVALID_ARG;
  return launch_sample(logits, B, V, temperature, seed, step, tokens,
                       static_cast<cudaStream_t>(stream));
}

}  // extern "C"
