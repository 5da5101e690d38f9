// attention.cu -- softmax attention over a paged KV cache: decode (one query
// token per sequence) and causal chunked prefill, both batch-invariant.
//
// What fixes the reduction order ("Reproducible LLM Inference", §5.5; "Your
// Answer Depends on Who Else Is in the Batch", "The attention detail that gets
// missed"):
//   * Fixed split SIZE: the keys 0..L-1 of a query are cut at multiples of S,
//     so every boundary is a function of the absolute key index only.
//   * Inside a split, key tiles of 64 aligned to absolute positions are
//     reduced in increasing order with an online softmax (FlashAttention,
//     cited by the pages): running max m, running sum l, unnormalised o.
//   * Splits are merged by a left fold in split order with the log-sum-exp
//     rule, then o/l is rounded once ("Reproducible LLM Inference", §4.3: a
//     fixed, non-parallel clean-up step).
//   * New tokens are written into the paged cache before attention runs, so
//     cached and fresh keys are read from one layout (§5.5).
// Decode runs one thread block per (sequence, kv head, split) and a separate
// merge kernel; prefill runs one block per (query block, kv head, sequence)
// and folds its splits in registers as it goes.  Both call the same tile step
// and the same fold, so a prefill row at position p is bit-identical to a
// decode with L = p + 1, whatever the chunking.
//
// Arithmetic of the tile step (identical in both kernels): scores by
// mma.sync m16n8k16 bf16 -> fp32 over D in increasing k; scaling by
// sm_scale*log2(e) and exp2f; P is split into a bf16 high part and a bf16
// low part (P - hi) and both are multiplied with V, so the probabilities keep
// ~16 significant bits; row max / row sum by a fixed shuffle tree.  Explicit
// __fmul_rn/__fadd_rn keep the compiler from contracting differently in the
// two kernels.
//
// K/V staging: each 16-token page of one kv head is a contiguous
// [16][D] bf16 block; a 2-D TMA tensor map over the cache viewed as
// [num_pages*Hkv*16][D] copies it into shared memory with 128-byte swizzling
// (one 16x64 box per 64 columns), completion counted on an mbarrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "bi_internal.h"
#include "device_common.cuh"

namespace bi {
namespace {

constexpr int kPage = 16;
constexpr int kTile = 64;              // keys per tile (4 pages)
constexpr int kPagesPerTile = kTile / kPage;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct TileGeom {
  static constexpr int kHalves = D / 64;                 // 128-byte column groups
  static constexpr int kPageBytes = kHalves * 2048;      // one page of K (or V)
  static constexpr int kKBytes = kPagesPerTile * kPageBytes;
  static constexpr int kBufBytes = 2 * kKBytes;          // K then V
  static constexpr int kQStride = D + 8;                 // padded Q row (elements)
};

// byte offset of (key n of the tile, column d) in a swizzled K or V tile
template <int D>
__device__ __forceinline__ uint32_t tile_off(int n, int d) {
  const int p = n >> 4, r = n & 15, hf = d >> 6, chunk = (d & 63) >> 3;
  return (uint32_t)((p * TileGeom<D>::kHalves + hf) * 2048 + r * 128 + ((chunk ^ (r & 7)) << 4));
}

// ----------------------------------------------------------- warp MMA helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D(16x8,f32) += A(16x16,bf16,row) * B(16x8,bf16,col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------- split state
// Per thread: rows g = lane/4 (index 0) and g + 8 (index 1) of the warp's 16
// rows; o[nd] holds columns 8*nd + 2*(lane%4) + {0,1} of both rows.
template <int D>
struct SplitState {
  float m[2], l[2];
  float o[D / 8][4];
  __device__ __forceinline__ void reset() {
    m[0] = m[1] = -CUDART_INF_F;
    l[0] = l[1] = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  }
};

// Shared address this lane hands to ldmatrix for the Q (A operand, row-major
// 16 x D, padded rows) fragment of k-step 0; k-step ks adds 32*ks bytes.
template <int D>
__device__ __forceinline__ uint32_t q_lane_addr(const __nv_bfloat16* qs) {
  const int lane = threadIdx.x & 31;
  const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int col = (lane >> 4) << 3;
  return smem_u32(qs + row * TileGeom<D>::kQStride + col);
}

// One tile of 64 keys (absolute indices key0 .. key0+63) for the warp's 16
// rows.  Row i sees key k iff lo <= k < hi[i].  A row that sees no key of the
// tile is left exactly as it was.
template <int D>
__device__ __forceinline__ void tile_step(SplitState<D>& st, uint32_t qaddr, uint32_t kbase,
                                          uint32_t vbase, int key0, int lo, const int (&hi)[2],
                                          float scale_log2) {
  const int lane = threadIdx.x & 31;
  const int t = lane & 3;
  // ---- scores S = Q K^T, 8 n-tiles of 8 keys; every score accumulates the
  // k-steps 0, 1, ..., D/16-1 in that order
  float s[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
  for (int kp = 0; kp < D / 32; ++kp) {
    uint32_t qa[4], qb[4];
    ldsm_x4(qaddr + kp * 64, qa[0], qa[1], qa[2], qa[3]);
    ldsm_x4(qaddr + kp * 64 + 32, qb[0], qb[1], qb[2], qb[3]);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      uint32_t b0, b1, b2, b3;
      const int key = nt * 8 + (lane & 7);
      const int col = kp * 32 + ((lane >> 3) << 3);
      ldsm_x4(kbase + tile_off<D>(key, col), b0, b1, b2, b3);
      mma_bf16(s[nt], qa, b0, b1);
      mma_bf16(s[nt], qb, b2, b3);
    }
  }
  // ---- scale, mask, row max
  float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int ri = c >> 1;
      const int k = key0 + nt * 8 + 2 * t + (c & 1);
      const bool ok = k >= lo && k < hi[ri];
      const float x = ok ? __fmul_rn(s[nt][c], scale_log2) : -CUDART_INF_F;
      s[nt][c] = x;
      mx[ri] = fmaxf(mx[ri], x);
    }
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(kFull, mx[ri], 1));
    mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(kFull, mx[ri], 2));
  }
  // ---- probabilities, rescale factors
  float alpha[2], mnew[2];
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    if (mx[ri] == -CUDART_INF_F) {  // no visible key: exact no-op for this row
      alpha[ri] = 1.0f;
      mnew[ri] = st.m[ri];
    } else {
      mnew[ri] = fmaxf(st.m[ri], mx[ri]);
      alpha[ri] = st.m[ri] == -CUDART_INF_F ? 0.0f : exp2f(__fsub_rn(st.m[ri], mnew[ri]));
    }
  }
  float rs[2] = {0.0f, 0.0f};
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int ri = c >> 1;
      const float x = s[nt][c];
      const float p = x == -CUDART_INF_F ? 0.0f : exp2f(__fsub_rn(x, mnew[ri]));
      s[nt][c] = p;
      rs[ri] = __fadd_rn(rs[ri], p);
    }
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    rs[ri] = __fadd_rn(rs[ri], __shfl_xor_sync(kFull, rs[ri], 1));
    rs[ri] = __fadd_rn(rs[ri], __shfl_xor_sync(kFull, rs[ri], 2));
    st.l[ri] = __fadd_rn(__fmul_rn(st.l[ri], alpha[ri]), rs[ri]);
    st.m[ri] = mnew[ri];
  }
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) {
    st.o[nd][0] = __fmul_rn(st.o[nd][0], alpha[0]);
    st.o[nd][1] = __fmul_rn(st.o[nd][1], alpha[0]);
    st.o[nd][2] = __fmul_rn(st.o[nd][2], alpha[1]);
    st.o[nd][3] = __fmul_rn(st.o[nd][3], alpha[1]);
  }
  // ---- O += P V with P = hi + lo (two bf16 parts), keys in order
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int nt = 2 * kk + (q >> 1);
      const int c = (q & 1) * 2;
      const float p0 = s[nt][c], p1 = s[nt][c + 1];
      const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
      const float l0 = __fsub_rn(p0, __bfloat162float(h0));
      const float l1 = __fsub_rn(p1, __bfloat162float(h1));
      __nv_bfloat162 hh;
      hh.x = h0;
      hh.y = h1;
      ph[q] = *reinterpret_cast<uint32_t*>(&hh);
      pl[q] = pack_bf16x2(l0, l1);
    }
#pragma unroll
    for (int np = 0; np < D / 16; ++np) {
      uint32_t b0, b1, b2, b3;
      const int mi = lane >> 3;
      const int key = kk * 16 + (lane & 7) + ((mi & 1) << 3);
      const int col = np * 16 + ((mi >> 1) << 3);
      ldsm_x4_t(vbase + tile_off<D>(key, col), b0, b1, b2, b3);
      mma_bf16(st.o[2 * np], ph, b0, b1);
      mma_bf16(st.o[2 * np], pl, b0, b1);
      mma_bf16(st.o[2 * np + 1], ph, b2, b3);
      mma_bf16(st.o[2 * np + 1], pl, b2, b3);
    }
  }
}

// Log-sum-exp merge of partial (mb, lb, ob) into (m, l, o), in that order.
__device__ __forceinline__ void lse_coeffs(float m, float mb, float& mn, float& ca, float& cb) {
  mn = fmaxf(m, mb);
  ca = exp2f(__fsub_rn(m, mn));
  cb = exp2f(__fsub_rn(mb, mn));
}
__device__ __forceinline__ float lse_mix(float a, float ca, float b, float cb) {
  return __fadd_rn(__fmul_rn(a, ca), __fmul_rn(b, cb));
}

__device__ __forceinline__ void store_out(void* out, float* out_f32, int64_t idx, float v0,
                                          float v1) {
  *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(out) + idx) = pack_bf16x2(v0, v1);
  if (out_f32) *reinterpret_cast<float2*>(out_f32 + idx) = make_float2(v0, v1);
}

// ---------------------------------------------------------------- staging
// Issue the TMA copies of tile `key0` (pages below `limit` only) into buf.
template <int D>
__device__ __forceinline__ void issue_tile(uint8_t* buf, uint64_t* bar, const CUtensorMap* km,
                                           const CUtensorMap* vm, const int32_t* bt_row,
                                           int key0, int limit, int Hkv, int h) {
  int np = 0;
  for (int p = 0; p < kPagesPerTile; ++p)
    if (key0 + p * kPage < limit) ++np;
  mbar_arrive_expect_tx(bar, np * 2 * TileGeom<D>::kPageBytes);
  for (int p = 0; p < np; ++p) {
    const int page = bt_row[(key0 >> 4) + p];
    const int y = (page * Hkv + h) * kPage;
#pragma unroll
    for (int hf = 0; hf < TileGeom<D>::kHalves; ++hf) {
      const int off = (p * TileGeom<D>::kHalves + hf) * 2048;
      tma_load_2d(buf + off, km, hf * 64, y, bar);
      tma_load_2d(buf + TileGeom<D>::kKBytes + off, vm, hf * 64, y, bar);
    }
  }
}

// Zero the V rows of keys >= limit in a landed tile (unwritten cache slots may
// hold any bits; their probability is exactly 0 but 0 * NaN is not 0).
template <int D>
__device__ __forceinline__ void clear_v_tail(uint8_t* buf, int key0, int limit, int tid,
                                             int nthreads) {
  const int first = limit - key0;  // first tile row to clear
  if (first >= kTile) return;
  const int start = first < 0 ? 0 : first;
  const int chunks = (kTile - start) * (D / 8);  // 16-byte chunks
  for (int i = tid; i < chunks; i += nthreads) {
    const int n = start + i / (D / 8);
    const int d = (i % (D / 8)) * 8;
    *reinterpret_cast<uint4*>(buf + TileGeom<D>::kKBytes + tile_off<D>(n, d)) =
        make_uint4(0, 0, 0, 0);
  }
}

// Check that the pages covering keys [key_lo, key_hi) of a sequence exist.
__device__ __forceinline__ bool pages_ok(const int32_t* bt_row, int key_lo, int key_hi,
                                         int64_t num_pages, int lane, int nlanes) {
  bool ok = true;
  for (int pg = (key_lo >> 4) + lane; pg * kPage < key_hi; pg += nlanes) {
    const int v = bt_row[pg];
    if (v < 0 || v >= num_pages) ok = false;
  }
  return ok;
}

struct KernelParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* kv_lens;
  const int32_t* cu_q;
  const int32_t* q_start;
  void* out;
  float* out_f32;
  float* ws;
  int* err;
  int B, Hq, Hkv, G, max_blocks, max_kv_len, split_size, split_count, max_splits;
  int64_t num_pages;
  float scale_log2;
  bool variant;
};

__device__ __forceinline__ bool len_ok(int L, const KernelParams& p) {
  return L >= 0 && L <= p.max_kv_len && L <= p.max_blocks * kPage;
}

// ------------------------------------------------------------ decode split
// Block (j, h, b): split j of sequence b, kv head h, all G query heads of the
// group as rows 0..G-1 of one m16 tile.  One warp.
template <int D>
__global__ void __launch_bounds__(32) attn_decode_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const KernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* bufs = smem;                                           // 2 tile buffers
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + 2 * TileGeom<D>::kBufBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + 16 * TileGeom<D>::kQStride);

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x;
  const int L = p.kv_lens[b];
  if (!len_ok(L, p)) {
    if (j == 0 && h == 0 && lane == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
    return;
  }
  int lo, hi;
  if (p.variant) {
    if (j >= p.split_count) return;
    lo = (int)(((int64_t)j * L) / p.split_count);
    hi = (int)(((int64_t)(j + 1) * L) / p.split_count);
  } else {
    lo = j * p.split_size;
    if (lo >= L) return;
    hi = min(lo + p.split_size, L);
  }
  const int G = p.G;
  const int64_t slot0 = ((int64_t)b * p.Hq + (int64_t)h * G) * p.max_splits + j;
  float* ws_ml = p.ws;
  float* ws_o = p.ws + (int64_t)p.B * p.Hq * p.max_splits * 2;
  const int32_t* bt_row = p.block_table + (int64_t)b * p.max_blocks;
  const int first_tile = lo & ~(kTile - 1);
  bool ok = lo < hi && pages_ok(bt_row, first_tile, hi, p.num_pages, lane, 32);
  ok = __all_sync(kFull, ok);
  if (!ok) {
    if (lo < hi && lane == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
    if (lane < G) {
      const int64_t slot = slot0 + (int64_t)lane * p.max_splits;
      ws_ml[2 * slot] = -CUDART_INF_F;
      ws_ml[2 * slot + 1] = 0.0f;
    }
    return;
  }
  const int ntiles = (hi - first_tile + kTile - 1) / kTile;

  if (lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0) {
    issue_tile<D>(bufs, &bars[0], &kmap, &vmap, bt_row, first_tile, hi, p.Hkv, h);
    if (ntiles > 1)
      issue_tile<D>(bufs + TileGeom<D>::kBufBytes, &bars[1], &kmap, &vmap, bt_row,
                    first_tile + kTile, hi, p.Hkv, h);
  }
  // Q rows of the group -> padded shared tile (rows >= G are zero)
  for (int i = lane; i < 16 * (D / 8); i += 32) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G)
      v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + h * G + r) * D + c);
    *reinterpret_cast<uint4*>(qs + r * TileGeom<D>::kQStride + c) = v;
  }
  __syncwarp();
  const uint32_t qaddr = q_lane_addr<D>(qs);

  SplitState<D> st;
  st.reset();
  const int g = lane >> 2;
  const int hi_r[2] = {g < G ? hi : lo, g + 8 < G ? hi : lo};
  bool alive = true;
  int stuck = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int bi_ = i & 1;
    uint8_t* buf = bufs + bi_ * TileGeom<D>::kBufBytes;
    const bool landed = mbar_wait(&bars[bi_], (i >> 1) & 1, p.err);
    if (!__all_sync(kFull, landed)) {
      alive = false;
      stuck = i;
      break;
    }
    const int key0 = first_tile + i * kTile;
    if (key0 + kTile > hi) {
      clear_v_tail<D>(buf, key0, hi, lane, 32);
      __syncwarp();
    }
    tile_step<D>(st, qaddr, smem_u32(buf), smem_u32(buf + TileGeom<D>::kKBytes), key0, lo, hi_r,
                 p.scale_log2);
    fence_proxy_async_smem();
    __syncwarp();
    if (i + 2 < ntiles && lane == 0) {
      issue_tile<D>(buf, &bars[bi_], &kmap, &vmap, bt_row, key0 + 2 * kTile, hi, p.Hkv, h);
    }
  }
  if (!alive) {
    // a copy never landed: give the copies still in flight a bounded wait,
    // mark this split empty and leave
    if (lane == 0) {
      mbar_wait(&bars[stuck & 1], (stuck >> 1) & 1, nullptr);
      if (stuck + 1 < ntiles) mbar_wait(&bars[(stuck + 1) & 1], ((stuck + 1) >> 1) & 1, nullptr);
    }
    __syncwarp();
    if (lane < G) {
      const int64_t slot = slot0 + (int64_t)lane * p.max_splits;
      ws_ml[2 * slot] = -CUDART_INF_F;
      ws_ml[2 * slot + 1] = 0.0f;
    }
    return;
  }
  // ---- write the partial state of rows < G
  const int t = lane & 3;
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int r = g + 8 * ri;
    if (r >= G) continue;
    const int64_t slot = slot0 + (int64_t)r * p.max_splits;
    if (t == 0) {
      ws_ml[2 * slot] = st.m[ri];
      ws_ml[2 * slot + 1] = st.l[ri];
    }
    float* orow = ws_o + slot * D;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(orow + nd * 8 + 2 * t) =
          make_float2(st.o[nd][2 * ri], st.o[nd][2 * ri + 1]);
  }
}

// ------------------------------------------------------------ decode merge
// Block (qh, b), D/2 threads: left fold over the splits in index order, then
// o / l.  Empty splits (variant plan at L < count) are skipped.
template <int D>
__global__ void __launch_bounds__(64) attn_decode_merge_kernel(const KernelParams p) {
  const int qh = blockIdx.x, b = blockIdx.y;
  const int d = threadIdx.x * 2;
  const int64_t row = (int64_t)b * p.Hq + qh;
  const int L = p.kv_lens[b];
  if (!len_ok(L, p) || L == 0) {
    store_out(p.out, p.out_f32, row * D + d, 0.0f, 0.0f);
    return;
  }
  const int ns = p.variant ? p.split_count : (L + p.split_size - 1) / p.split_size;
  const float* ml = p.ws + row * p.max_splits * 2;
  const float* ob = p.ws + (int64_t)p.B * p.Hq * p.max_splits * 2 + row * p.max_splits * D;
  float m = -CUDART_INF_F, l = 0.0f, o0 = 0.0f, o1 = 0.0f;
  bool have = false;
  for (int j = 0; j < ns; ++j) {
    const float mj = ml[2 * j], lj = ml[2 * j + 1];
    if (mj == -CUDART_INF_F) continue;  // empty split
    const float2 oj = *reinterpret_cast<const float2*>(ob + (int64_t)j * D + d);
    if (!have) {
      m = mj; l = lj; o0 = oj.x; o1 = oj.y;
      have = true;
    } else {
      float mn, ca, cb;
      lse_coeffs(m, mj, mn, ca, cb);
      l = lse_mix(l, ca, lj, cb);
      o0 = lse_mix(o0, ca, oj.x, cb);
      o1 = lse_mix(o1, ca, oj.y, cb);
      m = mn;
    }
  }
  if (!have) {
    store_out(p.out, p.out_f32, row * D + d, 0.0f, 0.0f);
    return;
  }
  store_out(p.out, p.out_f32, row * D + d, __fdiv_rn(o0, l), __fdiv_rn(o1, l));
}

// ------------------------------------------------------------- prefill
// Block (qb, h, b): kNW warps; each warp owns 16 rows = TPW tokens x G heads
// of query block qb of sequence b, kv head h.  Tiles of 64 keys are staged
// once per block and shared by the warps; splits are folded in registers.
constexpr int kPrefillWarps = 8;

template <int D>
__global__ void __launch_bounds__(kPrefillWarps * 32, 1) attn_prefill_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const KernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* bufs = smem;
  __nv_bfloat16* qs_all = reinterpret_cast<__nv_bfloat16*>(smem + 2 * TileGeom<D>::kBufBytes);
  // merged state of each warp's rows, thread-private: value i of lane l at
  // [i * 32 + l] (i = 4 * nd + c, as in SplitState::o)
  float* mg_all = reinterpret_cast<float*>(qs_all + kPrefillWarps * 16 * TileGeom<D>::kQStride);
  uint64_t* bars = reinterpret_cast<uint64_t*>(mg_all + kPrefillWarps * (D / 2) * 32);
  __shared__ int s_abort;

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, TPW = 16 / G;
  const int QB = kPrefillWarps * TPW;
  const int q_begin = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - q_begin;
  const int tok0 = qb * QB;
  if (tok0 >= q_len) return;
  const int start = p.q_start[b];
  const int kvl = p.kv_lens[b];
  if (!len_ok(kvl, p) || start < 0 || q_len < 0 || start + q_len > kvl) {
    if (tid == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
    return;
  }
  const int ntok = min(QB, q_len - tok0);
  const int p_last = start + tok0 + ntok - 1;  // last position in this block
  const int32_t* bt_row = p.block_table + (int64_t)b * p.max_blocks;
  const int ntiles = (p_last + kTile) / kTile;  // tiles 0 .. covering key p_last
  {
    const int loaded_hi = min(kvl, ntiles * kTile);  // keys a tile copy may read
    bool ok = pages_ok(bt_row, 0, loaded_hi, p.num_pages, tid, blockDim.x);
    ok = __syncthreads_and(ok);
    if (!ok) {
      if (tid == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
      return;
    }
  }
  if (tid == 0) {
    s_abort = 0;
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    issue_tile<D>(bufs, &bars[0], &kmap, &vmap, bt_row, 0, kvl, p.Hkv, h);
    if (ntiles > 1)
      issue_tile<D>(bufs + TileGeom<D>::kBufBytes, &bars[1], &kmap, &vmap, bt_row, kTile, kvl,
                    p.Hkv, h);
  }
  // this warp's rows: row r -> token r / G, head r % G of the group
  __nv_bfloat16* qs = qs_all + warp * 16 * TileGeom<D>::kQStride;
  for (int i = lane; i < 16 * (D / 8); i += 32) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    const int tk = warp * TPW + r / G;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < TPW * G && tk < ntok)
      v = *reinterpret_cast<const uint4*>(
          p.q + ((int64_t)(q_begin + tok0 + tk) * p.Hq + h * G + r % G) * D + c);
    *reinterpret_cast<uint4*>(qs + r * TileGeom<D>::kQStride + c) = v;
  }
  __syncwarp();
  const uint32_t qaddr = q_lane_addr<D>(qs);

  const int g = lane >> 2, t = lane & 3;
  int pos[2];  // absolute position of the two rows, -1 for padding rows
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int r = g + 8 * ri;
    const int tk = warp * TPW + r / G;
    pos[ri] = (r < TPW * G && tk < ntok) ? start + tok0 + tk : -1;
  }
  float* mgo = mg_all + warp * (D / 2) * 32 + lane;
  SplitState<D> st;  // current split
  float mg_m[2] = {-CUDART_INF_F, -CUDART_INF_F}, mg_l[2] = {0.0f, 0.0f};
  bool have[2] = {false, false};
  const int S = p.split_size;
  for (int i = 0; i < ntiles; ++i) {
    const int bi_ = i & 1;
    uint8_t* buf = bufs + bi_ * TileGeom<D>::kBufBytes;
    const int key0 = i * kTile;
    const int lo = (key0 / S) * S;  // split start
    if (key0 == lo) st.reset();
    bool landed = mbar_wait(&bars[bi_], (i >> 1) & 1, p.err, &s_abort);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) {
        s_abort = 1;
        mbar_wait(&bars[bi_], (i >> 1) & 1, nullptr);
        if (i + 1 < ntiles) mbar_wait(&bars[(i + 1) & 1], ((i + 1) >> 1) & 1, nullptr);
      }
      __syncthreads();
      break;
    }
    if (key0 + kTile > kvl) {
      clear_v_tail<D>(buf, key0, kvl, tid, blockDim.x);
      __syncthreads();
    }
    int hi_r[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) hi_r[ri] = pos[ri] >= lo ? min(lo + S, pos[ri] + 1) : lo;
    tile_step<D>(st, qaddr, smem_u32(buf), smem_u32(buf + TileGeom<D>::kKBytes), key0, lo, hi_r,
                 p.scale_log2);
    fence_proxy_async_smem();
    __syncthreads();
    if (i + 2 < ntiles && tid == 0) {
      issue_tile<D>(buf, &bars[bi_], &kmap, &vmap, bt_row, key0 + 2 * kTile, kvl, p.Hkv, h);
    }
    // end of split: fold it into the merged state (rows that reach it)
    if (key0 + kTile == lo + S || i + 1 == ntiles) {
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        if (pos[ri] < lo) continue;
        if (!have[ri]) {
          mg_m[ri] = st.m[ri];
          mg_l[ri] = st.l[ri];
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd) {
            mgo[(4 * nd + 2 * ri) * 32] = st.o[nd][2 * ri];
            mgo[(4 * nd + 2 * ri + 1) * 32] = st.o[nd][2 * ri + 1];
          }
          have[ri] = true;
        } else {
          float mn, ca, cb;
          lse_coeffs(mg_m[ri], st.m[ri], mn, ca, cb);
          mg_l[ri] = lse_mix(mg_l[ri], ca, st.l[ri], cb);
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd) {
            float* a0 = &mgo[(4 * nd + 2 * ri) * 32];
            float* a1 = &mgo[(4 * nd + 2 * ri + 1) * 32];
            *a0 = lse_mix(*a0, ca, st.o[nd][2 * ri], cb);
            *a1 = lse_mix(*a1, ca, st.o[nd][2 * ri + 1], cb);
          }
          mg_m[ri] = mn;
        }
      }
    }
  }
  if (s_abort) return;
  // ---- out = o / l for the real rows
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    if (pos[ri] < 0) continue;
    const int r = g + 8 * ri;
    const int tk = warp * TPW + r / G;
    const int64_t orow = ((int64_t)(q_begin + tok0 + tk) * p.Hq + h * G + r % G) * D;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      store_out(p.out, p.out_f32, orow + nd * 8 + 2 * t,
                __fdiv_rn(mgo[(4 * nd + 2 * ri) * 32], mg_l[ri]),
                __fdiv_rn(mgo[(4 * nd + 2 * ri + 1) * 32], mg_l[ri]));
  }
}

// --------------------------------------------------------------- KV write
__global__ void kv_write_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                const int32_t* __restrict__ seq, const int32_t* __restrict__ pos,
                                int64_t n_tokens, uint4* __restrict__ k_cache,
                                uint4* __restrict__ v_cache, const int32_t* __restrict__ bt,
                                int Hkv, int dvec, int page_size, int64_t num_pages,
                                int max_blocks, int* err) {
  const int64_t tok = blockIdx.x;
  const int h = blockIdx.y;
  const int s = seq[tok], ps = pos[tok];
  if (s < 0 || ps < 0 || ps >= max_blocks * page_size) {
    if (threadIdx.x == 0 && h == 0) record_error(err, BI_ERR_DEVICE_BOUNDS);
    return;
  }
  const int page = bt[(int64_t)s * max_blocks + ps / page_size];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0 && h == 0) record_error(err, BI_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t dst = (((int64_t)page * Hkv + h) * page_size + ps % page_size) * dvec;
  const int64_t src = (tok * Hkv + h) * dvec;
  for (int i = threadIdx.x; i < dvec; i += blockDim.x) {
    k_cache[dst + i] = k_new[src + i];
    v_cache[dst + i] = v_new[src + i];
  }
}

template <int D>
size_t decode_smem() {
  return 1024 + 2 * TileGeom<D>::kBufBytes + 16 * TileGeom<D>::kQStride * 2 + 64;
}
template <int D>
size_t prefill_smem() {
  return 1024 + 2 * TileGeom<D>::kBufBytes + kPrefillWarps * 16 * TileGeom<D>::kQStride * 2 +
         kPrefillWarps * (D / 2) * 32 * 4 + 64;
}

KernelParams make_params(const AttnArgs& a) {
  KernelParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_table = a.block_table;
  p.kv_lens = a.kv_lens;
  p.cu_q = a.cu_q;
  p.q_start = a.q_start;
  p.out = a.out;
  p.out_f32 = a.out_f32;
  p.ws = a.ws;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.max_blocks = a.max_blocks;
  p.max_kv_len = a.max_kv_len;
  p.split_size = a.split_size;
  p.split_count = a.split_count;
  p.max_splits = a.max_splits;
  p.num_pages = a.num_pages;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.variant = a.variant;
  return p;
}

bool make_kv_maps(const AttnArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.Hkv * kPage;
  return make_tmap_2d_bf16(km, a.k_cache, rows, a.D, kPage, 64) &&
         make_tmap_2d_bf16(vm, a.v_cache, rows, a.D, kPage, 64);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

template <int D>
bi_status decode_impl(const AttnArgs& a, cudaStream_t s) {
  CUtensorMap km, vm;
  if (!make_kv_maps(a, &km, &vm)) return BI_ERR_CUDA;
  const KernelParams p = make_params(a);
  if (a.max_splits > 0) {
    const size_t sm = decode_smem<D>();
    if (set_smem(attn_decode_split_kernel<D>, sm) != cudaSuccess) return BI_ERR_CUDA;
    const dim3 grid(a.max_splits, a.Hkv, a.B);
    attn_decode_split_kernel<D><<<grid, 32, sm, s>>>(km, vm, p);
  }
  attn_decode_merge_kernel<D><<<dim3(a.Hq, a.B), D / 2, 0, s>>>(p);
  return cuda_status(cudaGetLastError());
}

template <int D>
bi_status prefill_impl(const AttnArgs& a, cudaStream_t s) {
  CUtensorMap km, vm;
  if (!make_kv_maps(a, &km, &vm)) return BI_ERR_CUDA;
  KernelParams p = make_params(a);
  const int G = a.Hq / a.Hkv;
  const int QB = kPrefillWarps * (16 / G);
  const int nqb = (a.max_q_len + QB - 1) / QB;
  const size_t sm = prefill_smem<D>();
  if (set_smem(attn_prefill_kernel<D>, sm) != cudaSuccess) return BI_ERR_CUDA;
  attn_prefill_kernel<D><<<dim3(nqb, a.Hkv, a.B), kPrefillWarps * 32, sm, s>>>(km, vm, p);
  return cuda_status(cudaGetLastError());
}

}  // namespace

int attn_variant_split_count(int B, int Hkv, int num_sms) {
  // FlashDecoding-style: enough splits that B * Hkv * c blocks cover the SMs twice
  const int64_t units = static_cast<int64_t>(B) * Hkv;
  int64_t c = (2 * static_cast<int64_t>(num_sms) + units - 1) / (units > 0 ? units : 1);
  if (c < 1) c = 1;
  if (c > 64) c = 64;
  return static_cast<int>(c);
}

int attn_decode_max_splits(int max_kv_len, int split_size, bool variant, int split_count) {
  if (max_kv_len <= 0) return 0;
  if (variant) return split_count > 0 ? split_count : 1;
  return (max_kv_len + split_size - 1) / split_size;
}

bi_status launch_attn_decode(const AttnArgs& a, cudaStream_t s) {
  if (a.D == 64) return decode_impl<64>(a, s);
  if (a.D == 128) return decode_impl<128>(a, s);
  return BI_ERR_UNSUPPORTED;
}

bi_status launch_attn_prefill(const AttnArgs& a, cudaStream_t s) {
  if (a.D == 64) return prefill_impl<64>(a, s);
  if (a.D == 128) return prefill_impl<128>(a, s);
  return BI_ERR_UNSUPPORTED;
}

bi_status launch_kv_write(const void* k_new, const void* v_new, const int32_t* seq,
                          const int32_t* pos, int64_t n_tokens, void* k_cache, void* v_cache,
                          const int32_t* block_table, int Hkv, int D, int page_size,
                          int64_t num_pages, int max_blocks, int* err, cudaStream_t s) {
  if (n_tokens > 0x7fffffff || Hkv > 65535) return BI_ERR_UNSUPPORTED;
  const int dvec = D / 8;
  const int threads = dvec < 32 ? 32 : (dvec > 256 ? 256 : dvec);
  kv_write_kernel<<<dim3(static_cast<unsigned>(n_tokens), Hkv), threads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), seq, pos, n_tokens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_table, Hkv, dvec,
      page_size, num_pages, max_blocks, err);
  return cuda_status(cudaGetLastError());
}

}  // namespace bi
