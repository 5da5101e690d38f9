// attn_noalloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// bi_attn_decode needs a caller-provided workspace for its per-split partial
// results.  Some callers have no way to provide one: an engine that has
// already handed every byte of HBM to its KV-cache pool and forbids further
// cudaMalloc calls, a plugin running inside a host framework that owns the
// allocator, or code that must not risk the implicit synchronisation an
// allocation can cause.  bi_attn_decode_noalloc serves them: it runs the same
// batch-invariant decode with its scratch taken from one fixed array that
// lives in this file, so the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which this
// code is loaded keeps kNoallocScratchBytes reserved for it until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it names a stand-in object), so the device address is looked
// up with cudaGetSymbolAddress, once per device, the first time the entry
// point runs on that device, with that device current.  That first call
// should therefore happen before any stream capture begins.  The address is
// kept for the life of the process; a cudaDeviceReset of the device makes it
// stale, so the entry point must not be used on a device after a reset.
//
// All calls share the one array and it keeps whatever the last call left
// there.  Nothing in it needs to start at zero: every partial result the
// merge step reads is written earlier in the same call.  Two calls whose
// kernels overlap on the GPU (different streams, or different host threads)
// would race on the array; callers must order them, e.g. by issuing them on
// one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "bi.h"
#include "bi_internal.h"

namespace bi {
namespace {

constexpr size_t kNoallocScratchBytes = BI_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on
// first use), or nullptr if it cannot be obtained.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace bi

extern "C" bi_status bi_attn_decode_noalloc(const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_table,
                                            const int32_t* kv_lens, void* out, float* out_f32,
                                            int B, int Hq, int Hkv, int D, int page_size,
                                            int64_t num_pages, int max_blocks_per_seq,
                                            int max_kv_len, int split_size, float sm_scale,
                                            void* stream) {
  // The scratch this call would need must fit the fixed array.
  const size_t need = bi_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, split_size,
                                                    BI_MODE_INVARIANT, 0);
  if (need > bi::kNoallocScratchBytes) return BI_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = bi::scratch_address();
    if (!scratch) return BI_ERR_CUDA;
  }
  return bi_attn_decode(q, k_cache, v_cache, block_table, kv_lens, out, out_f32, B, Hq, Hkv, D,
                        page_size, num_pages, max_blocks_per_seq, max_kv_len, split_size,
                        sm_scale, BI_MODE_INVARIANT, 0, scratch, bi::kNoallocScratchBytes,
                        stream);
}
