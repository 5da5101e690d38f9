// gemm.cu -- C = A * W^T in bf16 with fp32 accumulation, on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), operands staged
// by TMA.
//
// Batch invariance ("Reproducible LLM Inference", §5.4): a matmul loses it in
// two ways -- splitting K when M and N are small, and switching to a
// different tensor-core instruction or tile at small batch, since each
// instruction has its own internal order.  Every shape here runs the
// instruction tcgen05.mma.cta_group::1.kind::f16 (M=128, K=16) and
// accumulates the k-blocks of 64 in increasing k into one fp32 accumulator,
// rounded to bf16 once.  The output tile is 128 x 256, or 128 x 64 (N=64)
// for at most 64 rows of A where those narrow tiles fit in one wave: the
// instruction's N only sets how many output columns it computes, and every
// output element gets the same sum for N = 64 and N = 256 (checked bit for
// bit on GB300 against the 256-column tiles of large M for every M up to
// 256).  A row of C therefore depends only on its row of A, W and K: rows
// beyond M in a partial tile are zero-filled by TMA and never mix with real
// rows.  The work distribution (which block takes which tile, how wide the
// tiles are) may vary with M; the arithmetic of an output element does not.
//
// The batch-variant mode (split-K, §5.4) runs the same tile over s slices of
// the k-blocks, writes fp32 partial tiles, and sums them in slice order in a
// second kernel.
//
// SwiGLU epilogue: for a gate/up weight whose rows come in blocks of 128
// features (the gate rows of the block, then its up rows), each 256-column
// tile holds the gate and up values of the same 128 features, so the
// epilogue rounds both to bf16 (as a stored projection would be), applies
// silu(g) * u and writes 128 columns of the product: the bytes of the GEMM
// followed by the standalone SwiGLU kernel, without the round trip of the
// [M, 2F] projection through memory.
//
// Structure: persistent blocks (one per SM), 6 warps:
//   warp 0    : TMA producer, fills a ring of (A, W) stages, 128-byte
//               swizzled, completion on mbarriers (the ring geometries are
//               listed at struct Ring): 4 stages of A 128x64 and W 256x64;
//               with at most 32 rows of A, 6 stages whose A holds 32 rows
//               (the weight, which is what a block streams at small M, then
//               has 192 KB in flight instead of 128 KB); in the narrow ring,
//               stages of four k-blocks of A (32 or 64 rows) and W (64 rows),
//               one 3-D copy per operand;
//   warp 1    : allocates tensor memory for two accumulators of the tile's
//               width (512 or 128 columns); one thread issues the MMAs into
//               one of them and commits them to the ring's "empty" barriers;
//   warps 2-5 : epilogue; each reads its 32 accumulator lanes (rows) with
//               tcgen05.ld, converts and stores, then frees the accumulator,
//               so the epilogue of one tile overlaps the MMAs of the next.
// Every wait is bounded; a wait that runs out records BI_ERR_TIMEOUT, tells
// the other roles to stop, waits (bounded) for its copies and MMAs in flight,
// frees tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bi_internal.h"
#include "device_common.cuh"
#include "tcgen05.cuh"

namespace bi {
namespace {

constexpr int BM = kGemmBM, BK = kGemmBK;
constexpr int kThreads = 192;
constexpr int kSmallRows = kGemmSmallRows;

// Ring geometry for an output tile of 128 x kBN, kARows rows of A per stage
// (128, or 32 / 64 when A has at most that many rows: the MMA still reads a
// 128-row window, whose rows past M reach accumulator rows that are never
// stored) and kKG k-blocks per stage:
//   128-row A, 256-column tile : 4 stages;
//   32-row A, 256-column tile  : 6 stages (the weight is what a block
//                                streams at small M);
//   narrow ring, 32- or 64-row A, 64-column tile, four k-blocks a stage:
//                                4 or 3 stages, one 3-D copy per operand that
//                                reads 512 contiguous bytes of each row.
// A stage holds kKG sub-tiles per operand, k-block after k-block, each laid
// out as a single k-block stage would be.
template <int kARows, int kBN, int kKG>
struct Ring {
  static constexpr int kStages =
      kBN == 256 ? (kARows == BM ? 4 : 6) : kBN == 192 ? 5 : (kARows == 64 ? 3 : 4);
  static constexpr int kASub = kARows * BK * 2;  // one k-block of A
  static constexpr int kBSub = kBN * BK * 2;     // one k-block of W
  static constexpr int kABytes = kKG * kASub;
  static constexpr int kBBytes = kKG * kBSub;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 256;
  // two kBN-column fp32 accumulators, allocated as a power of two of at
  // least 32 columns
  static constexpr uint32_t kTmemCols = 2 * kBN <= 32 ? 32u : 2 * kBN <= 128 ? 128u
                                        : 2 * kBN <= 256 ? 256u : 512u;
  // the MMA reads a 128-row A window from each A sub-tile: it must stay
  // inside the block's shared memory (the W ring follows the A ring)
  static_assert((kStages * kKG - 1) * kASub + BM * BK * 2 <= kStages * kStageBytes,
                "small-batch A window leaves shared memory");
  static_assert(kSmemBytes <= 227 * 1024, "ring exceeds shared memory");
  static_assert(((kBN == 256 || kBN == kGemmMidBN) && kKG == 1) ||
                    (kBN == kGemmNarrowBN && kKG == kGemmNarrowKBlocks),
                "wide tiles take one k-block a stage, narrow tiles four");
};

// K-major tiles written by TMA with 128-byte swizzling: rows of 64 bf16
// (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return umma_desc_sw128(saddr, 16, 1024);
}

struct GemmParams {
  __nv_bfloat16* C;
  float* ws;      // split-K partials [splits][M][N] (variant only)
  int* err;
  int M, N, K;
  int m_tiles, n_tiles, splits, kb_total, kb_per_split;
  int group;      // tiles of the L2-resident operand per raster group
  int m_fast;     // 1: A rows stay resident, W streams; 0: the other way round
};

struct Unit {
  int m_tile, n_tile, split, kb0, kb1;
};

// Tile order (it never changes a tile's arithmetic, only which block runs
// it and when): the smaller operand is kept resident in L2 in groups of
// `group` tiles while the other one streams past it once per group.
__device__ __forceinline__ Unit unit_of(int u, const GemmParams& p) {
  const int tiles = p.m_tiles * p.n_tiles;
  Unit w;
  w.split = u / tiles;
  const int r = u - w.split * tiles;
  if (p.m_fast) {
    const int per = p.group * p.n_tiles;
    const int g = r / per, rr = r - g * per;
    const int gs = min(p.group, p.m_tiles - g * p.group);
    w.n_tile = rr / gs;
    w.m_tile = g * p.group + rr % gs;
  } else {
    const int per = p.group * p.m_tiles;
    const int g = r / per, rr = r - g * per;
    const int gs = min(p.group, p.n_tiles - g * p.group);
    w.m_tile = rr / gs;
    w.n_tile = g * p.group + rr % gs;
  }
  w.kb0 = w.split * p.kb_per_split;
  w.kb1 = min(w.kb0 + p.kb_per_split, p.kb_total);
  return w;
}

enum Epilogue : int {
  kEpiBf16 = 0,    // C [M, N] bf16
  kEpiF32 = 1,     // fp32 split-K partials ws [split][M][N]
  kEpiSwiglu = 2,  // C [M, N/2] bf16 = silu(gate) * up of the interleaved tile halves
};

template <int kEpi, int kARows, int kBN, int kKG>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(
    const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
    const GemmParams p) {
  using R = Ring<kARows, kBN, kKG>;
  constexpr int kStages = R::kStages;
  constexpr int kABytes = R::kABytes;
  constexpr int kBBytes = R::kBBytes;
  constexpr int kASub = R::kASub;
  constexpr int kBSub = R::kBSub;
  constexpr int kStageBytes = R::kStageBytes;
  constexpr uint32_t kTmemCols = R::kTmemCols;
  constexpr uint32_t kIdesc = umma_idesc_bf16(BM, kBN, false, false);
  static_assert(kEpi != kEpiSwiglu || kBN == 256, "the SwiGLU tile pairs 128 gate and 128 up rows");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.m_tiles * p.n_tiles * p.splits;

  if (threadIdx.x == 0) {
    prefetch_tmap(&ta);
    prefetch_tmap(&tb);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(u, p);
        for (int kb = w.kb0; kb < w.kb1; kb += kKG) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          if constexpr (kKG == 1) {
            tma_load_2d(sA + stage * kABytes, &ta, kb * BK, w.m_tile * BM, &full[stage]);
            tma_load_2d(sB + stage * kBBytes, &tb, kb * BK, w.n_tile * kBN, &full[stage]);
          } else {
            // k-blocks kb .. kb + kKG - 1 (those past the slice are loaded
            // and not used; those past K read as zero)
            tma_load_3d(sA + stage * kABytes, &ta, 0, w.m_tile * BM, kb, &full[stage]);
            tma_load_3d(sB + stage * kBBytes, &tb, 0, w.n_tile * kBN, kb, &full[stage]);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the block goes away
        const int first = issued > kStages ? issued - kStages : 0;
        for (int i = first; i < issued; ++i)
          mbar_wait(&full[i % kStages], (i / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(u, p);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb0 = w.kb0; kb0 < w.kb1; kb0 += kKG) {
          if (!mbar_wait(&full[stage], phase, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < kKG; ++g) {
            const int kb = kb0 + g;
            if (kb >= w.kb1) break;
            const uint64_t ad = smem_desc(smem_u32(sA + stage * kABytes + g * kASub));
            const uint64_t bd = smem_desc(smem_u32(sB + stage * kBBytes + g * kBSub));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // +32 bytes along K per step
              tc_mma(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        tc_commit(drain);  // all issued MMAs done before tensor memory is freed
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int wq = warp & 3;  // this warp may access accumulator lanes 32*wq ..
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = unit_of(u, p);
      if (!mbar_wait(&tfull[acc], acc_phase, p.err, abort_flag)) break;
      __syncwarp();
      tc_fence_after();
      const int row = w.m_tile * BM + wq * 32 + lane;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      if constexpr (kEpi == kEpiSwiglu) {
        // gate in accumulator columns 0 .. kBN/2-1, up in kBN/2 .. kBN-1
#pragma unroll 1
        for (int c = 0; c < kBN / 64; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32_nowait(tbase + c * 32, g);
          tmem_ld32_nowait(tbase + kBN / 2 + c * 32, u);
          tmem_wait_ld();
          if (row < p.M) {
            __nv_bfloat16* dst = p.C + static_cast<int64_t>(row) * (p.N / 2) +
                                 w.n_tile * (kBN / 2) + c * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float y[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                y[e] = silu_mul_f32(bf16_round(__uint_as_float(g[8 * q + e])),
                                    bf16_round(__uint_as_float(u[8 * q + e])));
              *reinterpret_cast<uint4*>(dst + 8 * q) =
                  make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                             pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          const int col0 = w.n_tile * kBN + c * 32;
          if (row < p.M) {
            if constexpr (kEpi == kEpiF32) {
              float* dst = p.ws + (static_cast<int64_t>(w.split) * p.M + row) * p.N + col0;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (col0 + 4 * q < p.N)
                  *reinterpret_cast<uint4*>(dst + 4 * q) =
                      make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              __nv_bfloat16* dst = p.C + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (col0 + 8 * q < p.N) {
                  uint4 o;
                  o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
                  o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                  o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                  o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                  *reinterpret_cast<uint4*>(dst + 8 * q) = o;
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// C = bf16(sum_s ws[s]) in slice order, 4 columns per thread.
__global__ void splitk_reduce_kernel(const float4* __restrict__ ws, uint2* __restrict__ C,
                                     int64_t mn4, int splits) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < mn4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = ws[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = ws[s * mn4 + i];
      a.x = __fadd_rn(a.x, b.x);
      a.y = __fadd_rn(a.y, b.y);
      a.z = __fadd_rn(a.z, b.z);
      a.w = __fadd_rn(a.w, b.w);
    }
    C[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  }
}

// out[i, j] = bf16(silu(g) * u), g and u the slice-ordered sums of the gate
// and up partials of output feature j (columns 256 (j / 128) + j % 128 and
// 128 more of ws), each rounded to bf16 first: the bytes of
// splitk_reduce_kernel followed by the standalone SwiGLU kernel.  Four
// features per thread.
__global__ void splitk_reduce_swiglu_kernel(const float* __restrict__ ws, uint2* __restrict__ out,
                                            int64_t M, int64_t F, int splits) {
  const int64_t f4 = F / 4, n4 = M * f4, N = 2 * F, slice = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / f4, j = (i - row * f4) * 4;
    const float* gp = ws + row * N + (j / 128) * 256 + j % 128;
    float4 g = *reinterpret_cast<const float4*>(gp);
    float4 u = *reinterpret_cast<const float4*>(gp + 128);
    for (int s = 1; s < splits; ++s) {
      const float4 b = *reinterpret_cast<const float4*>(gp + s * slice);
      const float4 c = *reinterpret_cast<const float4*>(gp + s * slice + 128);
      g.x = __fadd_rn(g.x, b.x);
      g.y = __fadd_rn(g.y, b.y);
      g.z = __fadd_rn(g.z, b.z);
      g.w = __fadd_rn(g.w, b.w);
      u.x = __fadd_rn(u.x, c.x);
      u.y = __fadd_rn(u.y, c.y);
      u.z = __fadd_rn(u.z, c.z);
      u.w = __fadd_rn(u.w, c.w);
    }
    out[i] = make_uint2(pack_bf16x2(silu_mul_f32(bf16_round(g.x), bf16_round(u.x)),
                                    silu_mul_f32(bf16_round(g.y), bf16_round(u.y))),
                        pack_bf16x2(silu_mul_f32(bf16_round(g.z), bf16_round(u.z)),
                                    silu_mul_f32(bf16_round(g.w), bf16_round(u.w))));
  }
}

template <int kEpi, int kARows, int kBN, int kKG>
bi_status launch_tc_ring(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                         int grid, cudaStream_t s) {
  constexpr size_t smem = Ring<kARows, kBN, kKG>::kSmemBytes;
  if (cudaFuncSetAttribute(gemm_tc_kernel<kEpi, kARows, kBN, kKG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return BI_ERR_CUDA;
  gemm_tc_kernel<kEpi, kARows, kBN, kKG><<<grid, kThreads, smem, s>>>(ta, tb, p);
  return cuda_status(cudaGetLastError());
}
// narrow: the narrow ring runs (gemm_narrow); a_rows: rows of A per stage;
// bn: the tile width (gemm_n_tile)
template <int kEpi>
bi_status launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int grid,
                    bool narrow, uint32_t a_rows, int bn, cudaStream_t s) {
  if constexpr (kEpi != kEpiSwiglu) {
    if (narrow)
      return a_rows == kSmallRows
                 ? launch_tc_ring<kEpi, kSmallRows, kGemmNarrowBN, kGemmNarrowKBlocks>(ta, tb, p,
                                                                                       grid, s)
                 : launch_tc_ring<kEpi, kGemmNarrowRows, kGemmNarrowBN, kGemmNarrowKBlocks>(
                       ta, tb, p, grid, s);
  }
  if (a_rows == kSmallRows) return launch_tc_ring<kEpi, kSmallRows, 256, 1>(ta, tb, p, grid, s);
  if constexpr (kEpi != kEpiSwiglu) {
    if (bn == kGemmMidBN) return launch_tc_ring<kEpi, BM, kGemmMidBN, 1>(ta, tb, p, grid, s);
  }
  return launch_tc_ring<kEpi, BM, 256, 1>(ta, tb, p, grid, s);
}

}  // namespace

bi_status launch_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K,
                      int splits, float* ws, int* err, cudaStream_t s, bool swiglu) {
  const int sms = device_sm_count();
  if (sms <= 0) return BI_ERR_CUDA;
  CUtensorMap ta, tb;
  const bool narrow = gemm_narrow(M, N, K, sms, swiglu);
  const int bn = gemm_n_tile(M, N, K, sms, swiglu);
  // rows of A per stage (the A box)
  const uint32_t a_rows = M <= kSmallRows ? kSmallRows : (narrow ? kGemmNarrowRows : BM);
  const bool ok =
      narrow ? make_tmap_groups_bf16(&ta, A, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                                     a_rows, kGemmNarrowKBlocks) &&
                   make_tmap_groups_bf16(&tb, W, static_cast<uint64_t>(N),
                                         static_cast<uint64_t>(K), bn, kGemmNarrowKBlocks)
             : make_tmap_2d_bf16(&ta, A, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                                 a_rows, BK) &&
                   make_tmap_2d_bf16(&tb, W, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                                     bn, BK);
  if (!ok) return BI_ERR_CUDA;
  GemmParams p{};
  p.C = static_cast<__nv_bfloat16*>(C);
  p.ws = ws;
  p.err = err;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  p.n_tiles = static_cast<int>((N + bn - 1) / bn);
  p.kb_total = static_cast<int>((K + BK - 1) / BK);
  if (splits < 1) splits = 1;
  if (splits > p.kb_total) splits = p.kb_total;
  p.kb_per_split = (p.kb_total + splits - 1) / splits;
  p.splits = (p.kb_total + p.kb_per_split - 1) / p.kb_per_split;  // no empty slice
  // raster: keep the smaller operand in L2 (about 40 MB of it per group)
  const int64_t resident_budget = int64_t(40) << 20;
  p.m_fast = M <= N ? 1 : 0;
  const int64_t tile_bytes = static_cast<int64_t>(p.m_fast ? BM : bn) * K * 2;
  int64_t grp = resident_budget / (tile_bytes > 0 ? tile_bytes : 1);
  if (grp < 1) grp = 1;
  const int span = p.m_fast ? p.m_tiles : p.n_tiles;
  p.group = static_cast<int>(grp < span ? grp : span);
  const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.splits;
  if (units > 0x7fffffff) return BI_ERR_UNSUPPORTED;
  const int grid = static_cast<int>(units < sms ? units : sms);
  if (p.splits == 1)
    return swiglu ? launch_tc<kEpiSwiglu>(ta, tb, p, grid, narrow, a_rows, bn, s)
                  : launch_tc<kEpiBf16>(ta, tb, p, grid, narrow, a_rows, bn, s);
  const bi_status st = launch_tc<kEpiF32>(ta, tb, p, grid, narrow, a_rows, bn, s);
  if (st != BI_OK) return st;
  const int64_t n4 = swiglu ? M * N / 8 : M * N / 4;  // threads of the reduction
  const int rb = static_cast<int>((n4 + 255) / 256 < 4 * sms ? (n4 + 255) / 256 : 4 * sms);
  if (swiglu)
    splitk_reduce_swiglu_kernel<<<rb, 256, 0, s>>>(ws, static_cast<uint2*>(C), M, N / 2, p.splits);
  else
    splitk_reduce_kernel<<<rb, 256, 0, s>>>(reinterpret_cast<const float4*>(ws),
                                            static_cast<uint2*>(C), n4, p.splits);
  return cuda_status(cudaGetLastError());
}

}  // namespace bi
