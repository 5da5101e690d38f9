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
//     rule, then o times the rounded 1/l is rounded once ("Reproducible LLM
//     Inference", §4.3: a fixed, non-parallel clean-up step).
//   * New tokens are written into the paged cache before attention runs, so
//     cached and fresh keys are read from one layout (§5.5).
// Decode runs a small plan kernel (the list of (sequence, split) units), a
// persistent split kernel whose blocks walk that list, and a merge kernel;
// prefill runs one block per (query block, kv head, sequence) and folds its
// splits as it goes.  Decode (mma.sync) and prefill (tcgen05) perform the
// same per-element arithmetic in the same order, and the two instructions
// give bit-identical fp32 results for the same operands and k order, so a
// prefill row at position p is bit-identical to a decode with L = p + 1,
// whatever the chunking.
//
// The tile step works on transposed scores: S^T = K Q^T (keys are the MMA's
// M dimension, query rows its N dimension, 8 per n-tile) and O^T = V^T P^T,
// with mma.sync m16n8k16 bf16 -> fp32, every sum over k in increasing order.
// P^T comes from the S^T accumulators by an in-register 8x8 transpose
// (movmatrix).  A decode row group (the G query heads of one kv head) fills
// one 8-wide n-tile, so padding costs at most half of an n-tile.  With
// c = sm_scale*log2(e) a probability is 2^(s c - m), one fused multiply-add
// before ex2.approx, and the reference maximum is the raw scores' maximum
// scaled once (rounding is monotone, c > 0); P is split into a
// bf16 high part and a bf16 low part (P - hi), both taken by truncation and
// both multiplied with V, so the probabilities keep 16 significant bits.
// Column max / sum use a fixed shuffle tree.  Explicit __fmul_rn/__fadd_rn/__fmaf_rn keep the compiler from
// contracting differently in the two kernels.
//
// K/V staging: each 16-token page of one kv head is a contiguous [16][D]
// bf16 block; a 2-D TMA tensor map over the cache viewed as
// [num_pages*Hkv*16][D] copies it into shared memory with 128-byte swizzling
// (one 16x64 box per 64 columns), completion counted on an mbarrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <algorithm>
#include <queue>
#include <type_traits>
#include <utility>
#include <vector>

#include "bi_internal.h"
#include "device_common.cuh"
#include "tcgen05.cuh"

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
};

// byte offset of (key n of the tile, column d) in a swizzled K or V tile
template <int D>
__device__ __forceinline__ uint32_t tile_off(int n, int d) {
  const int p = n >> 4, r = n & 15, hf = d >> 6, chunk = (d & 63) >> 3;
  return (uint32_t)((p * TileGeom<D>::kHalves + hf) * 2048 + r * 128 + ((chunk ^ (r & 7)) << 4));
}

// 2^x on the special function unit (ex2.approx.ftz: relative error about
// 2^-22, results below 2^-126 flushed to zero).  Decode and prefill use it
// for the probabilities and the rescale factors.
__device__ __forceinline__ float exp2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------- warp MMA helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// C(16x8,f32) += A(16x16,bf16,row) * B(16x8,bf16,col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------- split state
// NQ n-tiles of 8 query columns.  Per thread, column index cc in {0,1} is
// query 8*nq + 2*(lane%4) + cc; o[md][nq] holds O^T rows d = 16*md + lane/4
// (c = 0,1) and d + 8 (c = 2,3), columns 2*(lane%4) + (c & 1).
template <int D, int NQ>
struct SplitState {
  float m[NQ][2], l[NQ][2];
  float o[D / 16][NQ][4];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
      m[nq][0] = m[nq][1] = -CUDART_INF_F;
      l[nq][0] = l[nq][1] = 0.0f;
#pragma unroll
      for (int md = 0; md < D / 16; ++md)
        o[md][nq][0] = o[md][nq][1] = o[md][nq][2] = o[md][nq][3] = 0.0f;
    }
  }
};

// Q^T fragments (B operand: k = d, n = query) for every k-step from a
// row-major [8*NQ][stride] bf16 shared tile.
template <int D, int NQ>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[NQ][D / 16][2],
                                             const __nv_bfloat16* qs, int stride) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
    for (int kp = 0; kp < D / 32; ++kp) {
      uint32_t r[4];
      ldsm_x4(smem_u32(qs + (8 * nq + (lane & 7)) * stride + 32 * kp + 8 * (lane >> 3)), r);
      qf[nq][2 * kp][0] = r[0];
      qf[nq][2 * kp][1] = r[1];
      qf[nq][2 * kp + 1][0] = r[2];
      qf[nq][2 * kp + 1][1] = r[3];
    }
}

// P = hi + lo: the probabilities of keys k, k+1 as two bf16 pairs (key k in
// the low half).  hi is p with its low 16 bits cleared (bf16 by truncation),
// lo the exact remainder p - hi truncated the same way, so hi + lo keeps 16
// significant bits of p (|p - hi - lo| < 2^-14 p) with no conversion
// instruction; decode and prefill split every probability with this function.
__device__ __forceinline__ void split_p_bf16(float p0, float p1, uint32_t& hp, uint32_t& lp) {
  const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
  hp = __byte_perm(b0, b1, 0x7632);
  const float r0 = __fsub_rn(p0, __uint_as_float(b0 & 0xffff0000u));
  const float r1 = __fsub_rn(p1, __uint_as_float(b1 & 0xffff0000u));
  lp = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}

// Two fp32 operations in one instruction (the packed f32x2 forms of sm_100
// and later): each lane is the IEEE operation, rounded to nearest, that the
// scalar form computes, so the results are bit-identical to __fadd_rn /
// __fmaf_rn; the prefill softmax uses them to issue fewer instructions.
__device__ __forceinline__ void add2_rn(float& r0, float& r1, float a0, float a1, float b0,
                                        float b1) {
  asm("{\n\t.reg .b64 a, b, r;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 r, a, b;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma2_rn(float& r0, float& r1, float a0, float a1, float b,
                                        float c) {
  asm("{\n\t.reg .b64 a, b, c, r;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\t"
      "mov.b64 c, {%5, %5};\n\tfma.rn.f32x2 r, a, b, c;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// The largest of three values (exact, as any fmaxf order).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The running reference maximum of a row moves only when a tile's maximum
// exceeds it by more than this many powers of two (and on the first tile
// with a visible key); otherwise the tile's probabilities are taken against
// the old reference (so they are at most 2^8) and the accumulated sum and o
// are left as they are.  The split's m is this reference; the merge rule is
// exact for any reference.  Decode and prefill apply the same rule to the
// same values, so they stay bit-identical.
constexpr float kRescaleLog2 = 8.0f;

// One tile of 64 keys (absolute indices key0 .. key0+63).  Query column
// (nq, cc) sees key k iff lo <= k < hi[nq][cc].  A column that sees no key
// of the tile is left exactly as it was.
template <int D, int NQ>
__device__ __forceinline__ void tile_step(SplitState<D, NQ>& st,
                                          const uint32_t (&qf)[NQ][D / 16][2], uint32_t kbase,
                                          uint32_t vbase, int key0, int lo,
                                          const int (&hi)[NQ][2], float scale_log2) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, mi = lane >> 3, r8 = lane & 7;
  // ---- S^T = K Q^T: 4 m-tiles of 16 keys; each score sums k-steps in order
  float s[4][NQ][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) s[mt][nq][0] = s[mt][nq][1] = s[mt][nq][2] = s[mt][nq][3] = 0.0f;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(kbase + tile_off<D>(16 * mt + r8 + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1)), a);
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq) mma_bf16(s[mt][nq], a, qf[nq][ks][0], qf[nq][ks][1]);
    }
  // ---- mask, column max of the raw scores, scaled once: rounding is
  // monotone, so RN(max s * c) = max RN(s * c) for the positive scale c
  float mx[NQ][2];
#pragma unroll
  for (int nq = 0; nq < NQ; ++nq) {
    mx[nq][0] = mx[nq][1] = -CUDART_INF_F;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = c & 1;
        const int k = key0 + 16 * mt + g + 8 * (c >> 1);
        const bool ok = k >= lo && k < hi[nq][cc];
        const float x = ok ? s[mt][nq][c] : -CUDART_INF_F;
        s[mt][nq][c] = x;
        mx[nq][cc] = fmaxf(mx[nq][cc], x);
      }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      mx[nq][cc] = fmaxf(mx[nq][cc], __shfl_xor_sync(kFull, mx[nq][cc], 4));
      mx[nq][cc] = fmaxf(mx[nq][cc], __shfl_xor_sync(kFull, mx[nq][cc], 8));
      mx[nq][cc] = fmaxf(mx[nq][cc], __shfl_xor_sync(kFull, mx[nq][cc], 16));
      mx[nq][cc] = __fmul_rn(mx[nq][cc], scale_log2);
    }
  }
  // ---- probabilities, rescale factors, column sums
  float alpha[NQ][2];
#pragma unroll
  for (int nq = 0; nq < NQ; ++nq) {
    float mnew[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const float m_in = st.m[nq][cc], t = mx[nq][cc];
      alpha[nq][cc] = 1.0f;
      mnew[cc] = m_in;
      if (t == -CUDART_INF_F) {
        // no visible key: exact no-op for this column
      } else if (m_in == -CUDART_INF_F) {
        mnew[cc] = t;
        alpha[nq][cc] = 0.0f;
      } else if (__fsub_rn(t, m_in) > kRescaleLog2) {
        mnew[cc] = t;
        alpha[nq][cc] = exp2_sfu(__fsub_rn(m_in, t));
      }
    }
    // masked keys hold -inf, and 2^(-inf - base) = +0 for any finite base
    const float mb[2] = {mnew[0] == -CUDART_INF_F ? 0.0f : mnew[0],
                         mnew[1] == -CUDART_INF_F ? 0.0f : mnew[1]};
    float cs[2] = {0.0f, 0.0f};
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = c & 1;
        const float pv = exp2_sfu(__fmaf_rn(s[mt][nq][c], scale_log2, -mb[cc]));
        s[mt][nq][c] = pv;
        cs[cc] = __fadd_rn(cs[cc], pv);
      }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      cs[cc] = __fadd_rn(cs[cc], __shfl_xor_sync(kFull, cs[cc], 4));
      cs[cc] = __fadd_rn(cs[cc], __shfl_xor_sync(kFull, cs[cc], 8));
      cs[cc] = __fadd_rn(cs[cc], __shfl_xor_sync(kFull, cs[cc], 16));
      st.l[nq][cc] = __fadd_rn(__fmul_rn(st.l[nq][cc], alpha[nq][cc]), cs[cc]);
      st.m[nq][cc] = mnew[cc];
    }
#pragma unroll
    for (int md = 0; md < D / 16; ++md)
#pragma unroll
      for (int c = 0; c < 4; ++c) st.o[md][nq][c] = __fmul_rn(st.o[md][nq][c], alpha[nq][c & 1]);
  }
  // ---- O^T += V^T P^T with P = hi + lo (two bf16 parts), keys in order
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t bh[NQ][2], bl[NQ][2];
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t hp, lp;
        split_p_bf16(s[kk][nq][2 * half], s[kk][nq][2 * half + 1], hp, lp);
        bh[nq][half] = transpose8x8(hp);
        bl[nq][half] = transpose8x8(lp);
      }
#pragma unroll
    for (int md = 0; md < D / 16; ++md) {
      uint32_t a[4];
      ldsm_x4_t(vbase + tile_off<D>(16 * kk + r8 + 8 * (mi >> 1), 16 * md + 8 * (mi & 1)), a);
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq) {
        mma_bf16(st.o[md][nq], a, bh[nq][0], bh[nq][1]);
        mma_bf16(st.o[md][nq], a, bl[nq][0], bl[nq][1]);
      }
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
// The output's normalisation: o times the correctly rounded reciprocal of l
// (one reciprocal per row, then one product per element; an IEEE division
// per element cost the prefill's output phase 2.7 us a block).  Decode, its
// merge and prefill all normalise with this, so they stay bit-identical.
__device__ __forceinline__ float inv_l(float l) { return __frcp_rn(l); }
__device__ __forceinline__ float normalize(float o, float rl) { return __fmul_rn(o, rl); }

// ---------------------------------------------------------------- staging
// Issue the TMA copies of the first np pages of a tile; page ids in pid.
template <int D>
__device__ __forceinline__ void issue_pages(uint8_t* buf, uint64_t* bar, const CUtensorMap* km,
                                            const CUtensorMap* vm, const int (&pid)[4], int np,
                                            int Hkv, int h) {
  // each cached K/V byte is read once per call: evict it first, so that the
  // split partials written meanwhile are still in L2 for the merge
  // One copy per page and tensor: the page's 16 rows of this head, both
  // 128-byte column groups (the maps' boxes are whole rows).
  const uint64_t pol = l2_policy_evict_first();
  for (int p = 0; p < np; ++p) {
    const int y = (pid[p] * Hkv + h) * kPage;
    const int off = p * TileGeom<D>::kPageBytes;
    tma_load_3d_hint(buf + off, km, 0, y, 0, bar, pol);
    tma_load_3d_hint(buf + TileGeom<D>::kKBytes + off, vm, 0, y, 0, bar, pol);
  }
}

__device__ __forceinline__ int pages_below(int key0, int limit) {
  int np = 0;
#pragma unroll
  for (int p = 0; p < kPagesPerTile; ++p) np += (key0 + p * kPage < limit) ? 1 : 0;
  return np;
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
  int* unit_count;   // decode plan: number of (sequence, split) units
  int4* units;       // decode plan: {b, j, lo, hi} per unit
  float* ml;         // decode partials: {m, l} per (b, q-head, split)
  float* o;          // decode partials: o[D] per (b, q-head, split)
  int* err;
  int B, Hq, Hkv, G, max_blocks, max_kv_len, split_size, split_count, max_splits;
  int ml_stride;     // decode partials: {m, l} pairs per (b, q-head) row, even
  int local_plan;    // decode: the split kernel works out its units itself
  int2* order;       // decode, in-kernel plan: {sequence, split count}, most splits first
  int target_units;  // decode variant: work units the batch is cut into (about)
  int64_t num_pages;
  float scale_log2;
  bool variant;
};

__device__ __forceinline__ bool len_ok(int L, const KernelParams& p) {
  return L >= 0 && L <= p.max_kv_len && L <= p.max_blocks * kPage;
}

// --------------------------------------------------------------- decode plan
// The fixed split size gives ceil(L/S) splits with boundaries at multiples of
// S.  The batch-variant plan (as a throughput-tuned engine plans decode)
// picks one chunk size C for the whole call from the batch itself: enough
// chunks over all sequences and kv heads to give every SM several work units
// (about target_units), and few enough that no sequence has more than
// split_count (the workspace's capacity); sequence b then gets ceil(L_b / C)
// chunks with boundaries at multiples of C.  C, and with it every boundary,
// moves with the batch's lengths: the plan is not batch-invariant.
__device__ __forceinline__ int variant_chunk_tiles(int64_t total_tiles, int max_tiles,
                                                   const KernelParams& p) {
  const int64_t units = total_tiles * p.Hkv;
  const int64_t by_work = (units + p.target_units - 1) / p.target_units;
  const int64_t by_cap = (max_tiles + p.split_count - 1) / p.split_count;
  const int64_t c = by_work > by_cap ? by_work : by_cap;
  return c < 1 ? 1 : static_cast<int>(c);
}
__device__ __forceinline__ int plan_splits(int L, int chunk, const KernelParams& p) {
  const int c = p.variant ? chunk : p.split_size;
  return (L + c - 1) / c;
}

// One block: the list of (sequence, split) units, in sequence order.
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(const KernelParams p) {
  __shared__ int warp_tot[32];
  __shared__ long long warp_tiles[32];
  __shared__ int warp_max[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (p.B + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(p.B, tid * chunk), b1 = min(p.B, b0 + chunk);
  int csize = 0;  // variant: the call's chunk size in keys
  if (p.variant) {
    long long tiles = 0;
    int tmax = 0;
    for (int b = b0; b < b1; ++b) {
      const int L = p.kv_lens[b];
      if (!len_ok(L, p)) continue;
      tiles += (L + kTile - 1) / kTile;
      tmax = max(tmax, (L + kTile - 1) / kTile);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      tiles += __shfl_xor_sync(kFull, tiles, o);
      tmax = max(tmax, __shfl_xor_sync(kFull, tmax, o));
    }
    if (lane == 0) {
      warp_tiles[warp] = tiles;
      warp_max[warp] = tmax;
    }
    __syncthreads();
    tiles = warp_tiles[lane];
    tmax = warp_max[lane];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      tiles += __shfl_xor_sync(kFull, tiles, o);
      tmax = max(tmax, __shfl_xor_sync(kFull, tmax, o));
    }
    csize = kTile * variant_chunk_tiles(tiles, tmax, p);
    if (tid == 0) p.unit_count[1] = csize;
  }
  int n = 0;
  for (int b = b0; b < b1; ++b) {
    const int L = p.kv_lens[b];
    if (!len_ok(L, p)) {
      record_error(p.err, BI_ERR_DEVICE_BOUNDS);
      continue;
    }
    if (L > 0) n += plan_splits(L, csize, p);
  }
  // block exclusive scan of n
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += v;
    }
    warp_tot[lane] = wi - w;  // exclusive
    if (lane == 31) *p.unit_count = wi;
  }
  __syncthreads();
  int base = warp_tot[warp] + incl - n;
  for (int b = b0; b < b1; ++b) {
    const int L = p.kv_lens[b];
    if (!len_ok(L, p) || L == 0) continue;
    const int ns = plan_splits(L, csize, p);
    const int c = p.variant ? csize : p.split_size;
    for (int j = 0; j < ns; ++j) p.units[base++] = make_int4(b, j, j * c, min((j + 1) * c, L));
  }
}

// ------------------------------------------------------------ decode split
// Persistent: block x takes units u = x, x + gridDim.x, ... (unit u = split
// u / Hkv of the plan, kv head u % Hkv).  Two warps per block:
//   warp 1 (producer) works out the plan, opens the units in order (page ids
//     fetched one unit ahead, checked and staged in shared memory, the unit's
//     descriptor put in a queue of kQueue slots) and issues the TMA copies of
//     every tile into a ring of two tile buffers, each as soon as the compute
//     warp has freed its buffer; the q rows of a unit ride with its first
//     tile;
//   warp 0 (compute) takes the descriptors in order, runs the tile steps (the
//     G query heads of the kv head are the columns of NQ 8-wide n-tiles) and
//     writes the unit's partial state, or the output when the sequence has a
//     single split.
// Measured on one block with a single warp doing everything: issuing a
// tile's copies (one lane, 9 copies) took ~1,400 cycles against ~1,800 for
// the tile's arithmetic, and opening a unit ~870; both are off the compute
// warp's path here.  Barriers: full / empty per ring
// buffer, ready / free per descriptor slot; every wait is bounded, a wait
// that runs out raises a flag that makes the other warp's waits return, and
// the producer lets its copies in flight land before it exits.  A unit whose
// pages are not all in the pool is recorded as BI_ERR_DEVICE_BOUNDS and
// marked with l = -1.
constexpr int kQueue = 4;
constexpr int kUnitPages = 64;                     // page ids staged per unit
constexpr int kLocalSlabs = 4;                     // 32 sequences per slab
constexpr int kLocalPlanMax = 32 * kLocalSlabs;    // largest batch planned in-kernel
constexpr int kSplitThreads = 64;                  // compute warp, producer warp

__device__ __forceinline__ int unit_tiles(int4 d) {  // {b, j, lo, hi}
  return d.z < d.w ? (d.w - (d.z & ~(kTile - 1)) + kTile - 1) / kTile : 0;
}

// At most three blocks per SM (shared memory), so registers are not what
// limits residency: the bound lets ptxas keep the whole tile step in
// registers instead of its default for this block size, which measurably
// starved the G <= 8 instantiation.
template <int D, int NQ>
__global__ void __maxnreg__(NQ == 1 ? 192 : 255) attn_decode_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const KernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* bufs = smem;  // 2 tile buffers
  __nv_bfloat16* qbuf = reinterpret_cast<__nv_bfloat16*>(smem + 2 * TileGeom<D>::kBufBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(qbuf + 2 * 8 * NQ * D);  // [2]
  uint64_t* empty = full + 2;                                            // [2]
  uint64_t* ready = empty + 2;                                           // [kQueue]
  uint64_t* freed = ready + kQueue;                                      // [kQueue]
  __shared__ int4 q_unit[kQueue];            // b, j, lo, hi of opened units (b < 0: no more)
  __shared__ int q_head[kQueue];             // kv head h, or -(h+1) if its pages are bad
  __shared__ int q_single[kQueue];           // the sequence has this one split
  __shared__ int q_pid[kQueue][kUnitPages];  // page ids of the unit's first pages
  __shared__ int s_incl[kLocalPlanMax], s_len[kLocalPlanMax];
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, Hkv = p.Hkv;
  if (threadIdx.x == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&ready[i], 1);
      mbar_init(&freed[i], 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  // padding query rows G .. 8*NQ-1 stay zero in both buffers
  {
    const int pad = (8 * NQ - G) * (D / 8);  // 16-byte chunks per buffer
    for (int i = threadIdx.x; i < 2 * pad; i += kSplitThreads) {
      const int bsel = i / pad, rem = i % pad;
      const int r = G + rem / (D / 8), c = (rem % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(qbuf + (bsel * 8 * NQ + r) * D + c) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();  // the zeroed rows before any copy into the buffers
  __syncthreads();
  // No early trigger for the merge kernel (launched behind this grid with
  // programmatic stream serialisation): it launches as these blocks exit.
  // Triggered at the start, its blocks queued up beside the split blocks and
  // the call took ~5 us longer whenever a kernel holding tensor memory and
  // ~200 KB of shared memory had run before it (64-request case on GB300:
  // 92.2 against 86.8 us; without the trigger 86.6 us either way).
  grid_dependency_wait();  // inputs and the plan kernel's unit list are complete from here

  if (warp == 1) {
    // ============================================================ producer
    // Units in sequence order.  For small batches the running split count
    // (inclusive) and the length of every sequence are kept in shared
    // memory; the sequence of split s is the number of sequences whose
    // running count is <= s, found with one ballot per 32 sequences.
    int total = 0;
    int csize = 0;  // variant: the call's chunk size in keys
    if (p.local_plan) {
      if (p.variant) {
        long long tiles = 0;
        int tmax = 0;
#pragma unroll
        for (int k = 0; k < kLocalSlabs; ++k) {
          const int b = lane + 32 * k;
          const int L = b < p.B ? p.kv_lens[b] : 0;
          if (b < p.B && len_ok(L, p)) {
            tiles += (L + kTile - 1) / kTile;
            tmax = max(tmax, (L + kTile - 1) / kTile);
          }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          tiles += __shfl_xor_sync(kFull, tiles, o);
          tmax = max(tmax, __shfl_xor_sync(kFull, tmax, o));
        }
        csize = kTile * variant_chunk_tiles(tiles, tmax, p);
        if (blockIdx.x == 0 && lane == 0) p.unit_count[1] = csize;  // for the merge
      }
#pragma unroll
      for (int k = 0; k < kLocalSlabs; ++k) {
        const int b = lane + 32 * k;
        int L = 0, n = 0;
        if (b < p.B) {
          L = p.kv_lens[b];
          if (!len_ok(L, p)) {
            record_error(p.err, BI_ERR_DEVICE_BOUNDS);
            L = 0;
          }
          if (L > 0) n = plan_splits(L, csize, p);
        }
        int v = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kFull, v, o);
          if (lane >= o) v += t;
        }
        s_incl[b] = total + v;
        s_len[b] = L;
        total += __shfl_sync(kFull, v, 31);
      }
      __syncwarp();
      // the merge takes sequences longest first: rank of sequence x among all
      // (more splits first, then lower index)
      for (int x = blockIdx.x; x < p.B; x += gridDim.x) {
        auto splits = [&](int b) { return s_incl[b] - (b > 0 ? s_incl[b - 1] : 0); };
        const int nx = splits(x);
        int ahead = 0;
#pragma unroll
        for (int k = 0; k < kLocalSlabs; ++k) {
          const int b = lane + 32 * k;
          if (b < p.B) {
            const int nb = splits(b);
            ahead += (nb > nx || (nb == nx && b < x)) ? 1 : 0;
          }
        }
        ahead = __reduce_add_sync(kFull, ahead);
        if (lane == 0) p.order[ahead] = make_int2(x, nx);
      }
    } else {
      total = *p.unit_count;
      if (p.variant) csize = p.unit_count[1];
    }
    const int U = total * Hkv;
    // A sequence with a single split has no merge: its unit writes the
    // output itself (o * (1/l), the merge's arithmetic for one split).  Split 0
    // is the only one iff it ends below the chunk size or the sequence is
    // exactly one chunk long.
    auto single_split = [&](int b, int j, int hi) -> bool {
      if (j != 0) return false;
      const int c = p.variant ? csize : p.split_size;
      if (hi < c) return true;
      return (p.local_plan ? s_len[b] : p.kv_lens[b]) == c;
    };
    auto unit_at = [&](int s) -> int4 {  // {b, j, lo, hi} of split s; warp-uniform s
      if (!p.local_plan) return p.units[s];
      int b = 0;
#pragma unroll
      for (int k = 0; k < kLocalSlabs; ++k)
        b += __popc(__ballot_sync(kFull, s_incl[lane + 32 * k] <= s));
      const int L = s_len[b];
      const int j = s - (b > 0 ? s_incl[b - 1] : 0);
      const int c = p.variant ? csize : p.split_size;
      return make_int4(b, j, j * c, min((j + 1) * c, L));
    };

    // the pending unit: its descriptor and page ids (in flight in registers)
    int lu = blockIdx.x;  // next unit to fetch
    bool pend = false;
    int4 pd = make_int4(0, 0, 0, 0);
    int ph = 0;
    int ppg[kUnitPages / 32];
    auto fetch = [&]() {
      pend = lu < U;
      if (!pend) return;
      ph = lu % Hkv;
      pd = unit_at(lu / Hkv);
      lu += gridDim.x;
      const int first = pd.z & ~(kTile - 1);
      const int npg = pd.z < pd.w ? (pd.w - first + kPage - 1) / kPage : 0;
      const int32_t* bt = p.block_table + (int64_t)pd.x * p.max_blocks + (first >> 4);
#pragma unroll
      for (int k = 0; k < kUnitPages / 32; ++k) {
        const int idx = lane + 32 * k;
        ppg[k] = idx < npg ? bt[idx] : 0;
      }
    };

    int n_units = 0, n_issued = 0, q_issued = 0;
    bool ok = true;
    fetch();
    while (ok) {
      const int slot = n_units % kQueue;
      if (n_units >= kQueue)
        ok = __all_sync(kFull, mbar_wait(&freed[slot], ((n_units / kQueue) - 1) & 1, p.err,
                                         &s_abort));
      if (!ok) break;
      if (!pend) {  // no more units: the end marker
        if (lane == 0) {
          q_unit[slot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&ready[slot]);
        }
        break;
      }
      // check the pending unit's pages, stage them, queue its descriptor
      const int4 d = pd;
      const int h = ph;
      const int first = d.z & ~(kTile - 1);
      const int npg = d.z < d.w ? (d.w - first + kPage - 1) / kPage : 0;
      bool good = true;
#pragma unroll
      for (int k = 0; k < kUnitPages / 32; ++k) {
        const int idx = lane + 32 * k;
        if (idx < npg) {
          if (ppg[k] < 0 || ppg[k] >= p.num_pages) good = false;
          q_pid[slot][idx] = ppg[k];
        }
      }
      if (npg > kUnitPages) {
        const int32_t* bt_row = p.block_table + (int64_t)d.x * p.max_blocks;
        if (!pages_ok(bt_row, first + kUnitPages * kPage, d.w, p.num_pages, lane, 32))
          good = false;
      }
      good = __all_sync(kFull, good);
      const bool single = single_split(d.x, d.y, d.w);
      if (lane == 0) {
        q_unit[slot] = d;
        q_head[slot] = good ? h : -(h + 1);
        q_single[slot] = single ? 1 : 0;
        if (!good) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[slot]);
      ++n_units;
      fetch();  // the next unit's page ids load while this unit's tiles are issued
      if (!good || d.z >= d.w) continue;
      const int ntiles = unit_tiles(d);
      for (int lt = 0; lt < ntiles; ++lt) {
        const int rs = n_issued & 1;
        if (n_issued >= 2)
          ok = __all_sync(kFull, mbar_wait(&empty[rs], ((n_issued >> 1) - 1) & 1, p.err,
                                           &s_abort));
        if (!ok) break;
        const int key0 = first + lt * kTile;
        const int np = pages_below(key0, d.w);
        int pid[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int idx = 4 * lt + pp;  // page index within the unit
          pid[pp] = pp >= np            ? 0
                    : idx < kUnitPages  ? q_pid[slot][idx]
                                        : p.block_table[(int64_t)d.x * p.max_blocks +
                                                        (first >> 4) + idx];
        }
        if (lane == 0) {
          uint8_t* buf = bufs + rs * TileGeom<D>::kBufBytes;
          const uint32_t qbytes = lt == 0 ? (uint32_t)(G * D * 2) : 0u;
          mbar_arrive_expect_tx(&full[rs], np * 2 * TileGeom<D>::kPageBytes + qbytes);
          if (lt == 0)
            bulk_load(qbuf + (q_issued & 1) * 8 * NQ * D,
                      p.q + ((int64_t)d.x * p.Hq + (int64_t)h * G) * D, qbytes, &full[rs]);
          issue_pages<D>(buf, &full[rs], &kmap, &vmap, pid, np, Hkv, h);
        }
        if (lt == 0) ++q_issued;
        ++n_issued;
      }
    }
    if (!ok) s_abort = 1;
    // the copies in flight land before the block exits
    if (lane == 0)
      for (int i = n_issued > 2 ? n_issued - 2 : 0; i < n_issued; ++i)
        mbar_wait(&full[i & 1], (i >> 1) & 1, nullptr);
    return;
  }
  // ============================================================== compute
  SplitState<D, NQ> st;
  uint32_t qf[NQ][D / 16][2];
  const int g = lane >> 2, t = lane & 3;
  int n = 0, n_done = 0, q_used = 0;
  bool alive = true;
  for (;;) {
    const int slot = n % kQueue;
    if (!__all_sync(kFull, mbar_wait(&ready[slot], (n / kQueue) & 1, p.err, &s_abort))) {
      alive = false;
      break;
    }
    const int4 d = q_unit[slot];
    const int hv = q_head[slot];
    const bool single = q_single[slot] != 0;
    __syncwarp();
    if (lane == 0) mbar_arrive(&freed[slot]);
    ++n;
    if (d.x < 0) break;  // no more units
    const bool pages_good = hv >= 0;
    const int h = pages_good ? hv : -hv - 1;
    const int b = d.x, j = d.y, lo = d.z, hi = d.w;
    const int64_t row0 = (int64_t)b * p.Hq + (int64_t)h * G;  // first q-head row
    if (!pages_good || lo >= hi) {
      // bad pages (l = -1 makes the merge emit zeros) or an empty split
      if (!pages_good && single) {
        for (int i = lane; i < G * D; i += 32) {
          static_cast<__nv_bfloat16*>(p.out)[row0 * D + i] = __float2bfloat16_rn(0.0f);
          if (p.out_f32) p.out_f32[row0 * D + i] = 0.0f;
        }
      } else if (lane < G) {
        const int64_t s = (row0 + lane) * p.ml_stride + j;
        p.ml[2 * s] = -CUDART_INF_F;
        p.ml[2 * s + 1] = pages_good ? 0.0f : -1.0f;
      }
      continue;
    }
    const int first = lo & ~(kTile - 1);
    const int ntiles = (hi - first + kTile - 1) / kTile;
    int hcol[NQ][2];
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) hcol[nq][cc] = (8 * nq + 2 * t + cc) < G ? hi : lo;
    for (int ti = 0; ti < ntiles; ++ti) {
      const int rs = n_done & 1;
      if (!__all_sync(kFull, mbar_wait(&full[rs], (n_done >> 1) & 1, p.err, &s_abort))) {
        alive = false;
        break;
      }
      uint8_t* buf = bufs + rs * TileGeom<D>::kBufBytes;
      if (ti == 0) {
        load_q_frags<D, NQ>(qf, qbuf + (q_used & 1) * 8 * NQ * D, D);
        ++q_used;
        st.reset();
      }
      const int key0 = first + ti * kTile;
      const bool tail = key0 + kTile > hi;
      if (tail) {
        clear_v_tail<D>(buf, key0, hi, lane, 32);
        __syncwarp();
      }
      tile_step<D, NQ>(st, qf, smem_u32(buf), smem_u32(buf + TileGeom<D>::kKBytes), key0, lo,
                       hcol, p.scale_log2);
      ++n_done;
      // the buffer goes back to the producer; the rows this warp zeroed are
      // ordered before the copy that will overwrite them
      if (tail) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[rs]);
    }
    if (!alive) break;
    if (single) {
      // ---- the output of the valid columns
      if (NQ == 1 && G <= 4) {
        // lanes with t >= 2 hold padding columns: each takes the odd column
        // of lane t - 2 (one exchange), so every lane divides 16 values
        const bool helper = t >= 2;
        const int col = 2 * (t & 1) + (helper ? 1 : 0);
        const float l_odd = __shfl_xor_sync(kFull, st.l[0][1], 2);
        const float lv = helper ? l_odd : st.l[0][0];
        const int64_t orow = (row0 + col) * D;
#pragma unroll
        for (int md = 0; md < D / 16; ++md)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float o_odd = __shfl_xor_sync(kFull, st.o[md][0][2 * hh + 1], 2);
            const float ov = helper ? o_odd : st.o[md][0][2 * hh];
            if (col < G) {
              const float v = lv > 0.0f ? normalize(ov, inv_l(lv)) : 0.0f;
              const int64_t idx = orow + 16 * md + g + 8 * hh;
              static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
              if (p.out_f32) p.out_f32[idx] = v;
            }
          }
        continue;
      }
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = 8 * nq + 2 * t + cc;
          if (col >= G) continue;
          const float lv = st.l[nq][cc];
          const int64_t orow = (row0 + col) * D;
#pragma unroll
          for (int md = 0; md < D / 16; ++md)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float v = lv > 0.0f ? normalize(st.o[md][nq][2 * hh + cc], inv_l(lv)) : 0.0f;
              const int64_t idx = orow + 16 * md + g + 8 * hh;
              static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
              if (p.out_f32) p.out_f32[idx] = v;
            }
        }
      continue;
    }
    // ---- partial state of the valid columns
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col = 8 * nq + 2 * t + cc;
        if (col >= G) continue;
        const int64_t sm = (row0 + col) * p.ml_stride + j;
        if (g == 0) {
          p.ml[2 * sm] = st.m[nq][cc];
          p.ml[2 * sm + 1] = st.l[nq][cc];
        }
        float* orow = p.o + ((row0 + col) * p.max_splits + j) * D;
#pragma unroll
        for (int md = 0; md < D / 16; ++md) {
          orow[16 * md + g] = st.o[md][nq][cc];
          orow[16 * md + g + 8] = st.o[md][nq][2 + cc];
        }
      }
  }
  if (!alive) s_abort = 1;
}

// ------------------------------------------------------------ decode merge
// Block (qh, rank): one q-head row of the rank-th longest sequence (longest
// first), D threads, one output column each.  Each warp folds its 32
// columns over the splits in index order, 32 splits per chunk.  Lane j of a
// warp loads split j's {m, l} and derives that split's coefficients: the
// running maximum before a split is a prefix maximum, exact in any order,
// so the whole chunk's coefficients come from one scan; the fold proper is
// then a chain of products and sums with one select per split and no
// branch, bit-identical to folding one split at a time.  Empty splits are
// skipped; a split marked l = -1 (bad pages) makes the whole row zero.  The
// o values of a chunk are loaded at once (one coalesced 128-byte row per
// split and warp), and the next chunk's loads are issued before the current
// chunk is folded.  No shared memory and no waits: the row's latency is a
// load round trip per chunk plus the fold chain.  A row of a sequence with a
// single split was written by the split kernel and is skipped here.
constexpr int kMergeChunk = 32;

template <int D>
__global__ void __launch_bounds__(D) attn_decode_merge_kernel(const KernelParams p) {
  // each warp's coefficients of the chunk being folded: {ca, cb, l, kind}
  __shared__ float4 coef[D / 32][kMergeChunk];
  const int qh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dependency_wait();  // every split kernel block has finished
  int b, ns;
  if (p.order) {
    const int2 e = p.order[blockIdx.y];
    b = e.x;
    ns = e.y;
  } else {
    b = blockIdx.y;
    const int L = p.kv_lens[b];
    ns = (len_ok(L, p) && L > 0) ? plan_splits(L, p.variant ? p.unit_count[1] : 0, p) : 0;
  }
  if (ns == 1) return;  // the split kernel wrote this row
  const int64_t row = (int64_t)b * p.Hq + qh;
  const float2* mlrow = reinterpret_cast<const float2*>(p.ml) + row * p.ml_stride;
  const float* ocol = p.o + row * p.max_splits * D + tid;
  // chunk starting at split c0: {m, l} of split c0 + lane, o of every split
  auto load = [&](int c0, float2& ml, float (&ov)[kMergeChunk]) {
    const int cnt = min(kMergeChunk, ns - c0);
    ml = lane < cnt ? mlrow[c0 + lane] : make_float2(-CUDART_INF_F, 0.0f);
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j)
      ov[j] = j < cnt ? ocol[static_cast<int64_t>(c0 + j) * D] : 0.0f;
  };
  float run_m = -CUDART_INF_F;  // max over the splits folded so far
  bool have = false;            // a non-empty split was folded
  bool bad = false;             // a split with bad pages
  float o = 0.0f, l = 0.0f;
  // two chunk buffers: the chunk being folded and the next one in flight
  float2 ml0, ml1;
  float ov0[kMergeChunk], ov1[kMergeChunk];
  auto fold = [&](const float2 ml, const float (&ov)[kMergeChunk]) {
    // coefficients of the chunk's split lane
    const float m = ml.x, lj = ml.y;
    const bool nonempty = m != -CUDART_INF_F;
    float pm = m;  // inclusive prefix max over the chunk
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const float t = __shfl_up_sync(kFull, pm, s);
      if (lane >= s) pm = fmaxf(pm, t);
    }
    float before = __shfl_up_sync(kFull, pm, 1);
    before = fmaxf(run_m, lane == 0 ? -CUDART_INF_F : before);
    const unsigned ne = __ballot_sync(kFull, nonempty);
    const bool had = have || (ne & ((1u << lane) - 1u)) != 0;
    bad = bad || __any_sync(kFull, lj < 0.0f);
    float ca = 0.0f, cb = 0.0f;
    if (nonempty && had) {
      float mn;
      lse_coeffs(before, m, mn, ca, cb);
    }
    const int kind = nonempty ? (had ? 2 : 1) : 0;  // 0 empty, 1 first non-empty, 2 fold in
    run_m = fmaxf(run_m, __shfl_sync(kFull, pm, 31));
    have = have || ne != 0;
    // the fold reads split j's coefficients as one broadcast load, which
    // can be issued ahead of the chain (shuffles issued in place stalled
    // every step of it)
    coef[warp][lane] = make_float4(ca, cb, lj, __int_as_float(kind));
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
      const float4 cf = coef[warp][j];
      const int kj = __float_as_int(cf.w);
      const float nl = lse_mix(l, cf.x, cf.z, cf.y);
      const float no = lse_mix(o, cf.x, ov[j], cf.y);
      l = kj == 2 ? nl : (kj == 1 ? cf.z : l);
      o = kj == 2 ? no : (kj == 1 ? ov[j] : o);
    }
    __syncwarp();  // every lane is done with the chunk's coefficients
  };
  if (ns > 0) load(0, ml0, ov0);
  for (int c0 = 0; c0 < ns; c0 += 2 * kMergeChunk) {
    if (c0 + kMergeChunk < ns) load(c0 + kMergeChunk, ml1, ov1);
    fold(ml0, ov0);
    if (c0 + kMergeChunk >= ns) break;
    if (c0 + 2 * kMergeChunk < ns) load(c0 + 2 * kMergeChunk, ml0, ov0);
    fold(ml1, ov1);
  }
  const float r = (ns > 0 && !bad && l > 0.0f) ? normalize(o, inv_l(l)) : 0.0f;
  const int64_t oidx = row * D + tid;
  const float r_next = __shfl_down_sync(kFull, r, 1);
  if ((tid & 1) == 0)
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + oidx) =
        pack_bf16x2(r, r_next);
  if (p.out_f32) p.out_f32[oidx] = r;
}

// ---------------------------------------------------- prefill (tcgen05)
// Block: 128 query rows -- up to 128 / G tokens times the G heads of one kv
// head (row r is token r / G, head r % G).  Keys come in tiles of 64; the
// scores are computed for pairs of tiles:
//   S = Q K^T   tcgen05.mma M=128 N=128 over a pair of key tiles, k = d in
//               steps of 16, A = Q from tensor memory, into pair buffer
//               q % 2 (the next pair's S is computed while this pair's
//               softmax runs);
//   softmax     per 64-key tile, the decode tile step's per-element
//               arithmetic, key summation tree and P = hi + lo split, one
//               row per thread; P (bf16 pairs) is stored back over the
//               tile's own score columns;
//   O += P V    tcgen05.mma M=128 N=D with A = P read from tensor memory,
//               per 16-key chunk the hi part then the lo part, V read as an
//               MN-major operand, into the accumulator (started afresh at
//               each split's first tile, once the fold has read the
//               previous split's).
// An MMA instruction costs the tensor core about the same time at N = 64
// as at N = 128, so pairs of tiles take 12 MMAs per 64 keys instead of 16.
// tcgen05.mma and mma.sync give bit-identical fp32 results for the same
// operands and k order, so every output row equals the decode of its
// position bit for bit.
// Roles: warps 0-3 run the softmax (warp w owns rows 32w..32w+31, the TMEM
// lanes of quadrant w), keeping each row's split state (reference maximum m,
// sum l) in registers; warps 4-7 fold every finished split into the merged
// state (in shared memory) and write out = o * (1/l) at the end; one lane of
// warp 13 issues the S MMAs and one of warp 8 the PV MMAs (two schedulers:
// a single issuing lane shares its scheduler with a softmax warp and falls
// behind); warps 9-12 the TMA copies, one column half of K or of V each
// (page ids cached in shared memory).  A single lane issuing all of a tile's
// copies was the bottleneck: it shares its scheduler with a softmax warp and
// took ~130 cycles per 2 KB page box.  The fold and copy warps sleep in
// their barrier waits instead of polling, so that they leave the issue slots
// of their scheduler to the softmax warp beside them.  Blocks start longest
// first, or, for one sequence whose blocks leave the last wave part full, in
// a host-planned order (plan_prefill_order).
constexpr int kPfRows = 128;
constexpr int kPfThreads = 14 * 32;
constexpr int kPfSoftWarp0 = 0, kPfFoldWarp0 = 4, kPfMmaWarp = 8, kPfTmaWarp0 = 9, kPfSWarp = 13;
constexpr int kPfPageCache = 1024;  // page ids held in shared memory (16384 keys)
constexpr int kPfPair = 2 * kTile;  // keys per S computation
constexpr int kPfKStages = 2;       // K stages, a pair of tiles each
constexpr int kPfVStages = 4;       // V stages, one tile each
constexpr int kPfPready = 4;        // P-ready barriers (tiles in flight)

template <int D>
struct PfGeom {
  static constexpr int kHalves = D / 64;
  static constexpr int kKBytes = kHalves * kPfPair * 128;  // K pair: [half][128 keys][128 B]
  static constexpr int kVBytes = kHalves * kTile * 128;    // V tile: [half][64 keys][128 B]
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kPfKStages * kKBytes;
  // merged o, fp32 [D / 4][128 rows][4]: a row's four consecutive columns
  // are one 16-byte vector, and a warp's 32 rows a contiguous 512 bytes
  static constexpr int kMOff = kVOff + kPfVStages * kVBytes;
  static constexpr int kXOff = kMOff + D * kPfRows * 4;  // split m, l: [parity][2][128]
  static constexpr int kPidOff = kXOff + 4 * kPfRows * 4;
  static constexpr int kBarOff = kPidOff + kPfPageCache * 4;
  // kfull, kfree [KS]; vfull, vfree [VS]; sfull, pfree [2]; pready [4];
  // odone, ofree; sdone, folded [2]
  static constexpr int kNumBars = 2 * kPfKStages + 2 * kPfVStages + 4 + kPfPready + 2 + 4;
  static constexpr int kSmem = 1024 + kBarOff + kNumBars * 8;
  static constexpr uint32_t kTmemCols = 512;
  // two S / P pair buffers of 128 columns, the accumulator (D columns), Q
  // (bf16 pairs, D / 2 columns)
  static constexpr uint32_t kColS = 0, kColO = 2 * kPfPair, kColQ = kColO + 128;
};
static_assert(PfGeom<128>::kSmem <= 232448, "prefill shared memory");

// mbarrier wait for the roles with slack (the fold and TMA warps): the thread
// suspends in the wait (a hint of 20 us, then it tries again), leaving the
// issue slots of its scheduler to the softmax warp beside it; bounded in time
// like mbar_wait.  The MMA and softmax warps, whose waits are on the
// critical path, use mbar_wait itself.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool pf_wait_lazy(uint64_t* bar, uint32_t parity, int* err,
                                             volatile int* abort) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (abort && *abort) return false;
    if (global_ns() - t0 > kWaitNs) break;
  }
  record_error(err, BI_ERR_TIMEOUT);
  if (abort) *abort = 1;
  return false;
}

// Wait for up to three barriers: their first tests go out back to back (the
// common case is that all are complete), then each missing one is waited for.
__device__ __forceinline__ bool mbar_wait3(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                           uint64_t* c, uint32_t pc, int* err,
                                           volatile int* abort) {
  const bool ra = mbar_try_wait(a, pa);
  const bool rb = b == nullptr || mbar_try_wait(b, pb);
  const bool rc = c == nullptr || mbar_try_wait(c, pc);
  if (ra && rb && rc) return true;
  return (ra || mbar_wait(a, pa, err, abort)) && (rb || mbar_wait(b, pb, err, abort)) &&
         (rc || mbar_wait(c, pc, err, abort));
}

// D (tmem) += A (tmem) * B (smem descriptor), one CTA, kind::f16.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Which query block and kv head a block of the launch computes.  LpOrder:
// the longest query blocks (of every kv head) first.  TableOrder: a
// host-planned order of one sequence's blocks (see plan_prefill_order), one
// index qb * Hkv + h per block, carried in the kernel's parameters.
struct LpOrder {
  __device__ __forceinline__ void map(int x, int nqb, int Hkv, int& qb, int& h) const {
    qb = nqb - 1 - x / Hkv;
    h = x % Hkv;
  }
};
constexpr int kPfOrderMax = 4096;
struct TableOrder {
  uint16_t blk[kPfOrderMax];
  __device__ __forceinline__ void map(int x, int nqb, int Hkv, int& qb, int& h) const {
    (void)nqb;
    const int v = blk[x];
    qb = v / Hkv;
    h = v % Hkv;
  }
};

template <int D, class Order>
__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const KernelParams p, const __grid_constant__ Order order) {
  using Gm = PfGeom<D>;
  constexpr uint32_t kIdescS = umma_idesc_bf16(kPfRows, kPfPair, false, false);
  constexpr uint32_t kIdescPV = umma_idesc_bf16(kPfRows, D, false, true);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kst = smem + Gm::kKOff;
  uint8_t* vst = smem + Gm::kVOff;
  float* xsplit = reinterpret_cast<float*>(smem + Gm::kXOff);  // [parity][m, l][128]
  float4* omg = reinterpret_cast<float4*>(smem + Gm::kMOff);   // merged o [D/4][128]
  int* pid_s = reinterpret_cast<int*>(smem + Gm::kPidOff);      // page ids of this sequence
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Gm::kBarOff);  // K pair landed
  uint64_t* kfree = kfull + kPfKStages;  // the S that read the K stage is done
  uint64_t* vfull = kfree + kPfKStages;  // V tile landed
  uint64_t* vfree = vfull + kPfVStages;  // the PV that read the V stage is done
  uint64_t* sfull = vfree + kPfVStages;  // S of the pair computed [2]
  uint64_t* pfree = sfull + 2;           // both PVs of the pair done: its buffer is free [2]
  uint64_t* pready = pfree + 2;          // P of the tile written over its scores [4]
  uint64_t* odone = pready + kPfPready;  // the last PV of a split done
  uint64_t* ofree = odone + 1;           // the fold has read the accumulator
  uint64_t* sdone = ofree + 1;           // a split's m, l written [2]
  uint64_t* folded = sdone + 2;          // a split folded, its m, l slot free [2]
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  __shared__ int s_out[2];  // for the output: first row's (token * Hq + head), tokens

  const int nqb = static_cast<int>(gridDim.x) / p.Hkv;
  int qb, h;
  order.map(static_cast<int>(blockIdx.x), nqb, p.Hkv, qb, h);
  const int b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G, TPB = kPfRows / G;
  const int q_begin = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - q_begin;
  const int tok0 = qb * TPB;
  if (tok0 >= q_len) return;
  const int start = p.q_start[b];
  const int kvl = p.kv_lens[b];
  if (!len_ok(kvl, p) || start < 0 || q_len < 0 || start + q_len > kvl) {
    if (tid == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
    return;
  }
  const int ntok = min(TPB, q_len - tok0);
  const int p_last = start + tok0 + ntok - 1;  // last position in this block
  const int32_t* bt_row = p.block_table + (int64_t)b * p.max_blocks;
  const int ntiles = (p_last + kTile) / kTile;  // tiles 0 .. covering key p_last
  const int npairs = (ntiles + 1) / 2;
  const int key_hi = min(kvl, ntiles * kTile);  // keys the copies read: 0 .. key_hi - 1
  const int S = p.split_size;
  const int tps = S / kTile;                    // tiles per split
  const int nsplits = (ntiles + tps - 1) / tps;
  {
    // check every page a copy may read, and keep the first ids at hand
    bool ok = true;
    for (int pg = tid; pg * kPage < key_hi; pg += 2 * kPfThreads) {  // two loads in flight
      const int pg1 = pg + kPfThreads;
      const bool has1 = pg1 * kPage < key_hi;
      const int v = bt_row[pg];
      const int v1 = has1 ? bt_row[pg1] : 0;
      if (v < 0 || v >= p.num_pages || v1 < 0 || v1 >= p.num_pages) ok = false;
      if (pg < kPfPageCache) pid_s[pg] = v;
      if (has1 && pg1 < kPfPageCache) pid_s[pg1] = v1;
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
      if (tid == 0) record_error(p.err, BI_ERR_DEVICE_BOUNDS);
      return;
    }
  }
  if (tid == 0) {
    s_abort = 0;
    // kept here rather than in registers through the main loops
    s_out[0] = (q_begin + tok0) * p.Hq + h * G;
    s_out[1] = ntok;
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    for (int i = 0; i < kPfKStages; ++i) {
      mbar_init(&kfull[i], Gm::kHalves);  // one arrival per copying warp
      mbar_init(&kfree[i], 1);
    }
    for (int i = 0; i < kPfVStages; ++i) {
      mbar_init(&vfull[i], Gm::kHalves);
      mbar_init(&vfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfree[i], 1);
      mbar_init(&sdone[i], 4);   // the four softmax warps
      mbar_init(&folded[i], 4);  // the four fold warps
    }
    for (int i = 0; i < kPfPready; ++i) mbar_init(&pready[i], 4);
    mbar_init(odone, 1);
    mbar_init(ofree, 4);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, Gm::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp < 4) {
    // Q row r into tensor memory lane r, the A operand of the S MMA: column
    // c holds elements 2c, 2c + 1; padding rows are zero
    const int r = warp * 32 + lane;
    const int tk = r / G;
    const bool valid = r < TPB * G && tk < ntok;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + ((int64_t)(q_begin + tok0 + (valid ? tk : 0)) * p.Hq + h * G + r % G) * D);
    uint32_t v[D / 2];  // the row's D bf16 values: every load goes out before the stores
#pragma unroll
    for (int u = 0; u < D / 8; ++u) {
      const uint4 w = valid ? src[u] : make_uint4(0, 0, 0, 0);
      v[4 * u] = w.x;
      v[4 * u + 1] = w.y;
      v[4 * u + 2] = w.z;
      v[4 * u + 3] = w.w;
    }
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + Gm::kColQ + 32 * c,
                *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp >= kPfTmaWarp0 && warp < kPfSWarp) {
    // ================================================================ copies
    // Warps 9, 10: column halves 0, 1 of K; warps 11, 12: those of V (one
    // lane each; with D = 64 only warps 9 and 11 copy).  K goes by pairs of
    // tiles: pair q into stage q % KS once the S of pair q - KS is done
    // (kfree); V by tiles: tile i into stage i % VS once the PV of tile
    // i - VS is (vfree).  Each copying warp arrives on the stage's full
    // barrier with the bytes of its half.
    const int role = warp - kPfTmaWarp0;
    const bool is_v = role >= 2;
    const int hf = role & 1;
    if (lane == 0 && hf < Gm::kHalves) {
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      // the pages of keys k0 .. k0 + nkeys - 1 below key_hi, 2 KB apart
      auto issue = [&](uint8_t* dst, uint64_t* bar, int k0, int nkeys) {
        const int np = max(0, min(nkeys / kPage, (key_hi - k0 + kPage - 1) / kPage));
        mbar_arrive_expect_tx(bar, np * 2048);
        for (int pp = 0; pp < np; ++pp) {
          const int pg = (k0 >> 4) + pp;
          const int y = ((pg < kPfPageCache ? pid_s[pg] : bt_row[pg]) * p.Hkv + h) * kPage;
          tma_load_2d(dst + pp * 2048, map, hf * 64, y, bar);
        }
      };
      bool ok = true;
      int n = 0;
      if (!is_v) {
        for (int q = 0; q < npairs && ok; ++q) {
          if (q >= kPfKStages)
            ok = pf_wait_lazy(&kfree[q % kPfKStages], ((q / kPfKStages) - 1) & 1, p.err,
                              &s_abort);
          if (!ok) break;
          issue(kst + (q % kPfKStages) * Gm::kKBytes + hf * (kPfPair * 128),
                &kfull[q % kPfKStages], q * kPfPair, kPfPair);
          ++n;
        }
        // every copy lands before the block exits (bounded waits)
        for (int k = max(0, n - kPfKStages); k < n; ++k)
          pf_wait_lazy(&kfull[k % kPfKStages], (k / kPfKStages) & 1, ok ? p.err : nullptr,
                       ok ? &s_abort : nullptr);
      } else {
        for (int i = 0; i < ntiles && ok; ++i) {
          if (i >= kPfVStages)
            ok = pf_wait_lazy(&vfree[i % kPfVStages], ((i / kPfVStages) - 1) & 1, p.err,
                              &s_abort);
          if (!ok) break;
          issue(vst + (i % kPfVStages) * Gm::kVBytes + hf * (kTile * 128),
                &vfull[i % kPfVStages], i * kTile, kTile);
          ++n;
        }
        for (int k = max(0, n - kPfVStages); k < n; ++k)
          pf_wait_lazy(&vfull[k % kPfVStages], (k / kPfVStages) & 1, ok ? p.err : nullptr,
                       ok ? &s_abort : nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kPfMmaWarp || warp == kPfSWarp) {
    // ================================================================ MMA
    // Warp 13 issues the S of every pair as soon as its K has landed and its
    // buffer is free; warp 8 the PVs.  One lane each, no warp collective
    // between two MMA batches.  The two lanes' MMAs meet only through the
    // barriers: sfull (S done) before the softmax, pready (P written) before
    // the PV, pfree (both PVs of a pair done) before the next S into that
    // buffer.
    if (lane == 0) {
      const uint64_t kd = umma_desc_sw128(smem_u32(kst), 16, 1024);
      const uint64_t vd = umma_desc_sw128(smem_u32(vst), kTile * 128, 1024);
      uint64_t* last_bar = nullptr;  // the latest MMA commit
      uint32_t last_par = 0;
      // S of pair q once its K landed and both PVs of pair q - 2 (the last
      // readers of its buffer) are done
      auto issue_s = [&](int q) -> bool {
        const int ks_ = q % kPfKStages, sb = q & 1;
        if (!mbar_wait3(&kfull[ks_], (q / kPfKStages) & 1, q >= 2 ? &pfree[sb] : nullptr,
                        ((q >> 1) - 1) & 1, nullptr, 0, p.err, &s_abort))
          return false;
        tc_fence_after();
        const uint64_t kb = kd + static_cast<uint64_t>(ks_ * (Gm::kKBytes >> 4));
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_ts(tmem + Gm::kColS + kPfPair * sb, tmem + Gm::kColQ + 8 * ks,
                    kb + static_cast<uint64_t>((ks >> 2) * (kPfPair * 8) + (ks & 3) * 2),
                    kIdescS, ks > 0 ? 1u : 0u);
        tc_commit(&sfull[sb]);
        tc_commit(&kfree[ks_]);
        last_bar = &sfull[sb];
        last_par = (q >> 1) & 1;
        return true;
      };
      if (warp == kPfSWarp) {  // every pair's S, in order
        bool sok = true;
        for (int q = 0; q < npairs && sok; ++q) sok = issue_s(q);
        if (!sok && last_bar) mbar_wait(last_bar, last_par, nullptr);  // MMAs in flight
      }
      bool ok = warp == kPfMmaWarp;  // warp 8: every tile's PV, in order
      // split of tile i and the tile's place in it, kept by counters: a
      // division by the runtime tiles-per-split costs the single issuing
      // thread a few hundred cycles per tile
      int j = 0, t_in = 0;
      for (int i = 0; i < ntiles && ok; ++i, (++t_in == tps ? (t_in = 0, ++j) : 0)) {
        const int q = i >> 1, u = i & 1;
        const int stg = i % kPfVStages;
        uint8_t* vt = vst + stg * Gm::kVBytes;
        const int key0 = i * kTile;
        const bool split_first = t_in == 0;
        const bool split_last = t_in == tps - 1 || i + 1 == ntiles;
        // the next pair's S goes to the tensor core as this pair's first
        // tile comes up, so that it is ready when this pair's softmax ends
        // V landed, P written, and (at a split's first tile) the fold has
        // read the previous split's accumulator
        ok = mbar_wait3(&vfull[stg], (i / kPfVStages) & 1, &pready[i % kPfPready],
                        (i / kPfPready) & 1, split_first && j >= 1 ? ofree : nullptr,
                        (j - 1) & 1, p.err, &s_abort);
        if (!ok) break;
        if (key0 + kTile > kvl) {  // keys past the end: zero their V rows before PV
          const int first = kvl - key0;
          for (int idx = 0; idx < (kTile - first) * Gm::kHalves * 8; ++idx) {
            const int n = first + idx / (Gm::kHalves * 8);
            const int rem = idx % (Gm::kHalves * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kTile * 128) + n * 128 +
                                      (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_after();
        // ---- O += P V, per 16-key chunk the hi part then the lo part
        const uint64_t vb = vd + static_cast<uint64_t>(stg * (Gm::kVBytes >> 4));
        // P of tile i: hi in columns 0-31 of its 64, lo in 32-63
        const uint32_t pa = tmem + Gm::kColS + kPfPair * (q & 1) + kTile * u;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bd = vb + static_cast<uint64_t>(kk * 128);
          tc_mma_ts(tmem + Gm::kColO, pa + 8 * kk, bd, kIdescPV,
                    (split_first && kk == 0) ? 0u : 1u);
          tc_mma_ts(tmem + Gm::kColO, pa + 32 + 8 * kk, bd, kIdescPV, 1u);
        }
        tc_commit(&vfree[stg]);
        if (u == 1 || i + 1 == ntiles) tc_commit(&pfree[q & 1]);
        if (split_last) tc_commit(odone);
        last_bar = &vfree[stg];
        last_par = (i / kPfVStages) & 1;
      }
      if (warp == kPfMmaWarp && !ok && last_bar) mbar_wait(last_bar, last_par, nullptr);
    }
    __syncwarp();
  } else if (warp < kPfFoldWarp0) {
    // ================================================================= softmax
    const int r = (warp - kPfSoftWarp0) * 32 + lane;
    const int tk = r / G;
    const int pos = (r < TPB * G && tk < ntok) ? start + tok0 + tk : -1;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float m = -CUDART_INF_F, l = 0.0f;  // the split's reference maximum and sum
    bool live = true;                   // no wait has run out
    int j = 0, t_in = 0;                // split of tile i and the tile's place in it
    for (int i = 0; i < ntiles && live; ++i, (++t_in == tps ? (t_in = 0, ++j) : 0)) {
      const int q = i >> 1, u = i & 1;
      const int key0 = i * kTile;
      const bool split_first = t_in == 0;
      const bool split_last = t_in == tps - 1 || i + 1 == ntiles;
      const uint32_t sa = tl + Gm::kColS + kPfPair * (q & 1) + kTile * u;
      // ---- scores of the tile: all 64 in registers
      live = __all_sync(kFull, mbar_wait(&sfull[q & 1], (q >> 1) & 1, p.err, &s_abort));
      if (!live) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t sv[64];
        tmem_ld32_nowait(sa, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32_nowait(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(sv[e]);
      }
      // keys key0 .. key0 + nvis - 1 are visible to this row (the tile lies
      // inside one split, which starts at or before key0)
      const int nvis = pos >= key0 ? min(kTile, pos + 1 - key0) : 0;
      if (key0 + kTile - 1 > start + tok0) {  // some row of the block sees part of the tile
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = e < nvis ? x[e] : -CUDART_INF_F;
      }
      float mx;
      {
        // the row maximum of the raw scores is exact in any order (a tree of
        // 3-way maxima), and scaled once it is the maximum of the scaled
        // scores (rounding is monotone, the scale positive): the decode's
        float t[22];
#pragma unroll
        for (int e = 0; e < 21; ++e) t[e] = max3(x[3 * e], x[3 * e + 1], x[3 * e + 2]);
        t[21] = x[63];
        float u[8];
#pragma unroll
        for (int e = 0; e < 7; ++e) u[e] = max3(t[3 * e], t[3 * e + 1], t[3 * e + 2]);
        u[7] = t[21];
        mx = __fmul_rn(max3(max3(u[0], u[1], u[2]), max3(u[3], u[4], u[5]), fmaxf(u[6], u[7])),
                       p.scale_log2);
      }
      const float m_in = split_first ? -CUDART_INF_F : m;
      float mnew = m_in, alpha = 1.0f;  // the decode's reference rule (kRescaleLog2)
      if (mx == -CUDART_INF_F) {
        // no visible key: exact no-op for this row
      } else if (m_in == -CUDART_INF_F) {
        mnew = mx;
        alpha = 0.0f;
      } else if (__fsub_rn(mx, m_in) > kRescaleLog2) {
        mnew = mx;
        alpha = exp2_sfu(__fsub_rn(m_in, mx));
      }
      // ---- probabilities: P = hi + lo as bf16 pairs (column c holds keys
      // 2c, 2c+1), written over the scores; key e adds to partial sum e % 8
      // in increasing key order, then the tree ((0+1)+(2+3))+((4+5)+(6+7))
      // p = 2^(s * scale - base), one rounding (the decode's fma); masked keys
      // hold -inf, and 2^(-inf) = +0 for any finite base
      const float mb = mnew == -CUDART_INF_F ? 0.0f : mnew;
      float cs[8];
#pragma unroll
      for (int g8 = 0; g8 < 8; ++g8) cs[g8] = 0.0f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // keys 32hf .. 32hf+31: columns 16hf .. 16hf+15
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // keys 32hf+8c .. 32hf+8c+7
          const int k0 = 32 * hf + 8 * c;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            fma2_rn(x[k0 + e], x[k0 + e + 1], x[k0 + e], x[k0 + e + 1], p.scale_log2, -mb);
            x[k0 + e] = exp2_sfu(x[k0 + e]);
            x[k0 + e + 1] = exp2_sfu(x[k0 + e + 1]);
            add2_rn(cs[e], cs[e + 1], cs[e], cs[e + 1], x[k0 + e], x[k0 + e + 1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // split_p_bf16, both remainders in one instruction
            const float p0 = x[k0 + 2 * e], p1 = x[k0 + 2 * e + 1];
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            ph[4 * c + e] = __byte_perm(b0, b1, 0x7632);
            float r0, r1;
            add2_rn(r0, r1, p0, p1, -__uint_as_float(b0 & 0xffff0000u),
                    -__uint_as_float(b1 & 0xffff0000u));
            pl[4 * c + e] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
          }
        }
        tmem_st16(sa + 16 * hf, ph);
        tmem_st16(sa + 32 + 16 * hf, pl);
      }
      const float csum = __fadd_rn(__fadd_rn(__fadd_rn(cs[0], cs[1]), __fadd_rn(cs[2], cs[3])),
                                   __fadd_rn(__fadd_rn(cs[4], cs[5]), __fadd_rn(cs[6], cs[7])));
      l = __fadd_rn(__fmul_rn(split_first ? 0.0f : l, alpha), csum);
      m = mnew;
      // ---- o *= alpha where a reference moved: after the previous tile's PV,
      // before this one's (the tensor core accumulates in issue order)
      if (!split_first && __any_sync(kFull, alpha != 1.0f)) {
        const int ip = i - 1;
        live = __all_sync(kFull, mbar_wait(&vfree[ip % kPfVStages], (ip / kPfVStages) & 1,
                                         p.err, &s_abort));
        if (!live) break;
        tc_fence_after();
        const uint32_t oc = tl + Gm::kColO;
#pragma unroll 1  // a rare path: kept compact, out of the way of the hot loop's code
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v0[32];
          tmem_ld32(oc + 32 * c, v0);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v0[e] = __float_as_uint(__fmul_rn(__uint_as_float(v0[e]), alpha));
          tmem_st32(oc + 32 * c, v0);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[i % kPfPready]);
      if (split_last) {
        // hand the split's m, l to the fold warps (their slot was read when
        // the fold of split j - 2 finished)
        if (j >= 2)
          live = __all_sync(kFull, mbar_wait(&folded[j & 1], ((j - 2) >> 1) & 1, p.err,
                                           &s_abort));
        if (!live) break;
        xsplit[(j & 1) * 2 * kPfRows + r] = m;
        xsplit[(j & 1) * 2 * kPfRows + kPfRows + r] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sdone[j & 1]);
      }
    }
  } else {
    // ================================================================ fold
    // Split j's accumulator (m_s, l_s, o_s) into the merged state, in split
    // order: the decode merge's left fold, one row per thread.  The
    // accumulator is released (ofree) as soon as its last columns are read.
    const int r = (warp - kPfFoldWarp0) * 32 + lane;
    const int tk = r / G;
    const int pos = (r < TPB * G && tk < ntok) ? start + tok0 + tk : -1;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float mg_m = -CUDART_INF_F, mg_l = 0.0f;  // merged state
    bool have = false;
    bool live = true;
    for (int j = 0; j < nsplits && live; ++j) {
      live = __all_sync(kFull, pf_wait_lazy(&sdone[j & 1], (j >> 1) & 1, p.err, &s_abort) &&
                                   pf_wait_lazy(odone, j & 1, p.err, &s_abort));
      if (!live) break;
      tc_fence_after();
      const float m_s = xsplit[(j & 1) * 2 * kPfRows + r];
      const float l_s = xsplit[(j & 1) * 2 * kPfRows + kPfRows + r];
      const bool part = pos >= j * S;  // the split holds keys this row sees
      float mn = 0.0f, ca = 0.0f, cb = 0.0f;
      if (part && have) lse_coeffs(mg_m, m_s, mn, ca, cb);
      const bool any = __any_sync(kFull, part);
#pragma unroll 1  // once per split: compact code
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vo[32];
        if (any) tmem_ld32(Gm::kColO + tl + 32 * c, vo);
        if (c == D / 32 - 1) {  // the accumulator is read: the next split may start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ofree);
        }
        if (part) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4* slot = omg + (8 * c + v) * kPfRows + r;
            const float4 add = make_float4(__uint_as_float(vo[4 * v]),
                                           __uint_as_float(vo[4 * v + 1]),
                                           __uint_as_float(vo[4 * v + 2]),
                                           __uint_as_float(vo[4 * v + 3]));
            if (have) {
              const float4 m4 = *slot;
              *slot = make_float4(lse_mix(m4.x, ca, add.x, cb), lse_mix(m4.y, ca, add.y, cb),
                                  lse_mix(m4.z, ca, add.z, cb), lse_mix(m4.w, ca, add.w, cb));
            } else {
              *slot = add;
            }
          }
        }
      }
      if (part) {
        if (have) {
          mg_l = lse_mix(mg_l, ca, l_s, cb);
          mg_m = mn;
        } else {
          mg_m = m_s;
          mg_l = l_s;
          have = true;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&folded[j & 1]);
    }
    // the row's 1/l for the output below (the split m, l slots are free now)
    if (live && pos >= 0) xsplit[r] = inv_l(mg_l);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, Gm::kTmemCols);
  // ---- out = o * (1/l), rounded once, by every warp: a warp takes 8 rows x
  // 16 columns at a time (lane: row 8 rg + lane / 4, columns 4 c4 .. 4 c4 + 3
  // with c4 = 4 cg + lane % 4), so its reads of the merged state are 128-byte
  // runs and its writes 32-byte runs of each row
  if (s_abort) return;
  const int64_t row0 = s_out[0];
  const int otok = s_out[1], oG = p.G;
  for (int u = warp; u < (kPfRows / 8) * (D / 16); u += kPfThreads / 32) {
    const int r = 8 * (u % (kPfRows / 8)) + (lane >> 2);
    const int c4 = 4 * (u / (kPfRows / 8)) + (lane & 3);
    const int tk = r / oG;
    if (r >= (kPfRows / oG) * oG || tk >= otok) continue;
    const float rl = xsplit[r];
    const float4 a = omg[c4 * kPfRows + r];
    const float o0 = normalize(a.x, rl), o1 = normalize(a.y, rl);
    const float o2 = normalize(a.z, rl), o3 = normalize(a.w, rl);
    const int64_t idx = (row0 + (int64_t)tk * p.Hq + r % oG) * D + 4 * c4;
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + idx) =
        make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
    if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + idx) = make_float4(o0, o1, o2, o3);
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

template <int D, int NQ>
size_t decode_smem() {  // ring, q buffers, barriers (full, empty: 2 each; ready, free)
  return 1024 + 2 * TileGeom<D>::kBufBytes + 2 * 8 * NQ * D * 2 + (4 + 2 * kQueue) * 8;
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
// Decode: one box per (page, kv head), both column groups of its 16 rows.
bool make_kv_page_maps(const AttnArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.Hkv * kPage;
  return make_tmap_groups_bf16(km, a.k_cache, rows, a.D, kPage, a.D / 64) &&
         make_tmap_groups_bf16(vm, a.v_cache, rows, a.D, kPage, a.D / 64);
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous one in the stream drains, and waits for it in-kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// Workspace carve-up for decode: [unit count | units | {m,l} | o].  The
// {m, l} rows hold an even number of pairs so that every row starts on a
// 16-byte boundary.
struct DecodeWs {
  size_t units_off, ml_off, o_off, total;
  int ml_stride;
};
DecodeWs decode_ws_layout(int B, int Hq, int D, int max_splits) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  DecodeWs w;
  w.ml_stride = (max_splits + 1) & ~1;
  const size_t rows = static_cast<size_t>(B) * Hq;
  w.units_off = 256;
  w.ml_off = w.units_off + up(static_cast<size_t>(B) * max_splits * sizeof(int4));
  w.o_off = w.ml_off + up(rows * w.ml_stride * 2 * sizeof(float));
  w.total = w.o_off + rows * max_splits * D * sizeof(float);
  return w;
}

template <int D, int NQ>
bi_status decode_impl(const AttnArgs& a, cudaStream_t s) {
  KernelParams p = make_params(a);
  if (a.max_splits > 0) {
    CUtensorMap km, vm;
    if (!make_kv_page_maps(a, &km, &vm)) return BI_ERR_CUDA;
    const DecodeWs w = decode_ws_layout(a.B, a.Hq, a.D, a.max_splits);
    char* base = reinterpret_cast<char*>(a.ws);
    p.unit_count = reinterpret_cast<int*>(base);
    p.units = reinterpret_cast<int4*>(base + w.units_off);
    p.ml = reinterpret_cast<float*>(base + w.ml_off);
    p.o = reinterpret_cast<float*>(base + w.o_off);
    p.ml_stride = w.ml_stride;
    p.local_plan = a.B <= kLocalPlanMax;
    if (p.local_plan) p.order = reinterpret_cast<int2*>(base + w.units_off);  // units unused
    const size_t sm = decode_smem<D, NQ>();
    if (set_smem(attn_decode_split_kernel<D, NQ>, sm) != cudaSuccess) return BI_ERR_CUDA;
    static int per_sm[2][3] = {};
    int& occ = per_sm[D == 128][NQ];
    if (occ == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &occ, attn_decode_split_kernel<D, NQ>, kSplitThreads, sm) !=
                        cudaSuccess)
      return BI_ERR_CUDA;
    const int sms = device_sm_count();
    if (sms <= 0 || occ <= 0) return BI_ERR_CUDA;
    const int64_t max_units = static_cast<int64_t>(a.B) * a.Hkv * a.max_splits;
    const int64_t cap = static_cast<int64_t>(occ) * sms;
    // variant: 4 units per resident block (measured on GB300, 64 requests of
    // 1..32768 keys, mean of 40 calls: 2 -> 94.2 us, 4 -> 86.5, 8 -> 90.1,
    // 16 -> 92.1 us)
    p.target_units = static_cast<int>(4 * cap);
    if (!p.local_plan) attn_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
    const int grid = static_cast<int>(max_units < cap ? max_units : cap);
    if (launch_pdl(attn_decode_split_kernel<D, NQ>, dim3(grid), dim3(kSplitThreads), sm, s, km,
                   vm, p) !=
        cudaSuccess)
      return BI_ERR_CUDA;
  }
  if (launch_pdl(attn_decode_merge_kernel<D>, dim3(a.Hq, a.B), dim3(D), 0, s, p) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

// Launch order of one sequence's prefill blocks.  The hardware gives each
// block, in launch order, to the SM that frees first; with n similar blocks
// on m SMs (n = a m + r) longest-first leaves the last r blocks running
// alone after every SM has run a.  A block's time is modelled as a fixed
// start-up (as long as ~640 keys) plus its key count (the chunk assumed to
// end at max_kv_len).  The plan gives the r SMs that must run a + 1 blocks
// the shortest blocks and the others the longest a each (longest first
// within each group), then orders all blocks by their planned start times,
// so that the hardware's own dispatch reproduces it.  Both orders are
// simulated with the model; the plan is used only where it predicts a
// shorter run (1% or more).  The order changes no block's work or result.
bool plan_prefill_order(int nqb, int Hkv, int TPB, int max_q_len, int max_kv_len, int sms,
                        TableOrder* out) {
  const int n = nqb * Hkv;
  if (sms <= 0 || n <= sms || n > kPfOrderMax) return false;
  const int a = n / sms, r = n % sms;
  if (r == 0) return false;
  const int64_t start = std::max<int64_t>(0, int64_t(max_kv_len) - max_q_len);
  std::vector<double> d(n);  // modelled time of block b = qb * Hkv + h
  for (int qb = 0; qb < nqb; ++qb) {
    const int64_t keys = std::min<int64_t>(max_kv_len, start + int64_t(TPB) * (qb + 1));
    for (int h = 0; h < Hkv; ++h) d[qb * Hkv + h] = 640.0 + static_cast<double>(keys);
  }
  using Ev = std::pair<double, int>;  // (time the SM frees, SM)
  auto simulate = [&](const std::vector<int>& ord) {
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> q;
    for (int i = 0; i < sms; ++i) q.push({0.0, i});
    double end = 0.0;
    for (int b : ord) {
      Ev e = q.top();
      q.pop();
      e.first += d[b];
      end = std::max(end, e.first);
      q.push(e);
    }
    return end;
  };
  std::vector<int> lp(n);
  for (int x = 0; x < n; ++x) lp[x] = (nqb - 1 - x / Hkv) * Hkv + x % Hkv;
  std::vector<int> by_len(lp);  // longest first (ties: as the default order)
  std::stable_sort(by_len.begin(), by_len.end(), [&](int u, int v) { return d[u] > d[v]; });
  // the two groups, each by longest-first onto its SMs with a fixed count each
  std::vector<std::pair<double, int>> starts;  // (planned start, block)
  starts.reserve(n);
  auto place = [&](int first, int count, int nsm, int per) {
    // longest first onto the SM that frees first (the lowest index among
    // equals), exactly `per` blocks each
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> q;
    for (int i = 0; i < nsm; ++i) q.push({0.0, i});
    std::vector<int> cnt(nsm, 0);
    for (int k = first; k < first + count; ++k) {
      Ev e = q.top();
      q.pop();
      const int b = by_len[k];
      starts.push_back({e.first, b});
      e.first += d[b];
      if (++cnt[e.second] < per) q.push(e);
    }
  };
  place(0, (sms - r) * a, sms - r, a);
  place((sms - r) * a, r * (a + 1), r, a + 1);
  std::stable_sort(starts.begin(), starts.end(),
                   [](const std::pair<double, int>& u, const std::pair<double, int>& v) {
                     return u.first < v.first;
                   });
  std::vector<int> planned(n);
  for (int k = 0; k < n; ++k) planned[k] = starts[k].second;
  if (simulate(planned) > 0.99 * simulate(lp)) return false;
  for (int k = 0; k < n; ++k) out->blk[k] = static_cast<uint16_t>(planned[k]);
  return true;
}

template <int D>
bi_status prefill_impl(const AttnArgs& a, cudaStream_t s) {
  CUtensorMap km, vm;
  if (!make_kv_maps(a, &km, &vm)) return BI_ERR_CUDA;
  KernelParams p = make_params(a);
  const int G = a.Hq / a.Hkv;
  const int TPB = kPfRows / G;  // tokens per block
  const int nqb = (a.max_q_len + TPB - 1) / TPB;
  const size_t sm = PfGeom<D>::kSmem;
  const dim3 grid(nqb * a.Hkv, 1, a.B);
  // one sequence: a planned order, kept for the next call of the same shape
  thread_local TableOrder plan;
  thread_local int plan_key[6] = {-1, -1, -1, -1, -1, -1};
  thread_local bool plan_ok = false;
  if (a.B == 1) {
    const int key[6] = {nqb, a.Hkv, TPB, a.max_q_len, a.max_kv_len, device_sm_count()};
    if (!std::equal(key, key + 6, plan_key)) {
      plan_ok = plan_prefill_order(nqb, a.Hkv, TPB, a.max_q_len, a.max_kv_len, key[5], &plan);
      std::copy(key, key + 6, plan_key);
    }
    if (plan_ok) {
      if (set_smem(attn_prefill_kernel<D, TableOrder>, sm) != cudaSuccess) return BI_ERR_CUDA;
      attn_prefill_kernel<D, TableOrder><<<grid, kPfThreads, sm, s>>>(km, vm, p, plan);
      return cuda_status(cudaGetLastError());
    }
  }
  if (set_smem(attn_prefill_kernel<D, LpOrder>, sm) != cudaSuccess) return BI_ERR_CUDA;
  attn_prefill_kernel<D, LpOrder><<<grid, kPfThreads, sm, s>>>(km, vm, p, LpOrder{});
  return cuda_status(cudaGetLastError());
}

}  // namespace

int attn_variant_split_count(int B, int Hkv, int max_kv_len, int num_sms) {
  // the largest number of chunks the batch-variant plan may give one
  // sequence (it sizes the workspace): one per 256 keys of the longest
  // sequence, at most 128
  (void)B;
  (void)Hkv;
  (void)num_sms;
  int64_t c = (static_cast<int64_t>(max_kv_len) + 255) / 256;
  if (c < 1) c = 1;
  if (c > 128) c = 128;
  return static_cast<int>(c);
}

int attn_decode_max_splits(int max_kv_len, int split_size, bool variant, int split_count) {
  if (max_kv_len <= 0) return 0;
  if (variant) return split_count > 0 ? split_count : 1;
  return (max_kv_len + split_size - 1) / split_size;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int D, int max_splits) {
  if (B <= 0 || max_splits <= 0) return 0;
  return decode_ws_layout(B, Hq, D, max_splits).total;
}

bi_status launch_attn_decode(const AttnArgs& a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if (a.D == 64) return G <= 8 ? decode_impl<64, 1>(a, s) : decode_impl<64, 2>(a, s);
  if (a.D == 128) return G <= 8 ? decode_impl<128, 1>(a, s) : decode_impl<128, 2>(a, s);
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
