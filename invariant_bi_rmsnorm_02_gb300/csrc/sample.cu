// sample.cu -- next-token selection from a row of bf16 logits per request:
// the plain argmax at temperature 0, seeded Gumbel-max sampling above it
// ("Reproducible LLM Inference - Batch Invariance, the Cost of Determinism,
// and Where Bitwise Identity Is Actually Required", §9.2 and §9.3).
//
// Gumbel-max: argmax_v (z_v / T + G_v), G_v = -log(-log(u_v)) standard
// Gumbel, is a draw from softmax(z / T).  The uniforms come from a
// counter-based generator, Philox4x64-10 (Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011), keyed by the
// request's seed and counted by its step and the vocabulary index, so u_v of
// a request depends on (seed, step, v) alone: never on the batch around it.
//
// The reduction is an argmax under a total order (score, then lowest
// index), which gives the same token in any reduction order; a row is split
// over a thread-block cluster of kCluster CTAs whose winners are combined
// through distributed shared memory.  One launch, no workspace, no atomics.
#include <cooperative_groups.h>
#include <math_constants.h>
#include <cuda_runtime.h>

#include "bi_internal.h"
#include "device_common.cuh"

namespace bi {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

// Philox4x64-10: ten rounds of two 64 x 64 -> 128-bit products; the key is
// advanced by the two Weyl constants (golden ratio, sqrt(3) - 1) between
// rounds.
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                              uint64_t k0, uint64_t k1, uint64_t (&out)[4]) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t hi0 = __umul64hi(kM0, c0), lo0 = kM0 * c0;
    const uint64_t hi1 = __umul64hi(kM1, c2), lo1 = kM1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// Orderable 64-bit key of (score, index): larger key = larger score, and on
// equal scores the lower index.  -0 counts as +0; a NaN score counts as -inf.
__device__ __forceinline__ uint64_t argmax_key(float s, uint32_t v) {
  uint32_t b = __float_as_uint(s);
  if (s == 0.0f) b = 0u;
  if (s != s) b = 0xff800000u;
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(b) << 32) | static_cast<uint32_t>(~v);
}

__device__ __forceinline__ uint64_t max_u64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = max_u64(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Grid (C, B); the C CTAs of one row form a cluster (C = 8 for small batches,
// so that one row keeps several SMs busy; C = 1 once the rows alone fill the
// GPU).  Each CTA scans a fixed slice of groups of 8 vocabulary entries (one
// Philox block per group); rank 0 combines the slice winners and writes the
// token.  The token does not depend on C: the argmax is order-free.
template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(kThreads)
    sample_kernel(const uint16_t* __restrict__ logits, int64_t V, bool vec_ok,
                  const float* __restrict__ temperature, const uint64_t* __restrict__ seed,
                  const uint64_t* __restrict__ step, int32_t* __restrict__ tokens) {
  constexpr int kCluster = C;
  __shared__ uint64_t s_warp[kThreads / 32];
  __shared__ uint64_t s_best;
  const int rank = static_cast<int>(blockIdx.x);  // the rank within the row's cluster
  const int64_t b = blockIdx.y;
  const float T = temperature[b];
  const bool greedy = !(T > 0.0f);
  const float inv_t = greedy ? 0.0f : __frcp_rn(T);
  const uint64_t key = seed[b], ctr1 = step[b];
  const int64_t groups = (V + 7) >> 3;
  const int64_t g_begin = groups * rank / kCluster, g_end = groups * (rank + 1) / kCluster;
  const uint16_t* row = logits + b * V;

  // This thread's best (score, index): it visits its entries in increasing
  // index order, so a strict > keeps the lowest index among equal scores;
  // scores are canonical (-0 -> +0, NaN -> -inf) so that == is the order's
  // equality.  bv < 0: no entry yet.
  float bs = -CUDART_INF_F;
  int64_t bv = -1;
  // one group of 8 entries (entries past the end of the row hold NaN, so
  // every real entry of the group has a lower index)
  auto group = [&](int64_t g, const float (&x)[8]) {
    if (greedy) {
      // the group's maximum (fmaxf passes over NaN), then its lowest index
      float m = x[0];
#pragma unroll
      for (int j = 1; j < 8; ++j) m = fmaxf(m, x[j]);
      if (m != m) m = -CUDART_INF_F;
      if (m > bs || bv < 0) {
        // the lowest index scoring m; a NaN scores -inf
        const bool low = m == -CUDART_INF_F;
        int jj = 0;
#pragma unroll
        for (int j = 7; j >= 0; --j)
          if (x[j] == m || (low && x[j] != x[j])) jj = j;
        bs = m == 0.0f ? 0.0f : m;
        bv = g * 8 + jj;
      }
      return;
    }
    uint64_t r[4];
    philox4x64_10(static_cast<uint64_t>(g), ctr1, 0, 0, key, 0, r);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t v = g * 8 + j;
      if (v >= V) break;
      const uint64_t word = r[j >> 1];
      const uint32_t half = (j & 1) ? static_cast<uint32_t>(word >> 32)
                                    : static_cast<uint32_t>(word);
      // u = (k + 1/2) 2^-23 for the top 23 bits k: exact in fp32, in (0, 1)
      const float u = __fmul_rn(static_cast<float>(half >> 9) + 0.5f, 0x1p-23f);
      const float gumbel = -logf(-logf(u));
      float s = __fadd_rn(__fmul_rn(x[j], inv_t), gumbel);
      if (s != s) s = -CUDART_INF_F;
      if (s == 0.0f) s = 0.0f;
      if (s > bs || bv < 0) {
        bs = s;
        bv = v;
      }
    }
  };
  if (vec_ok) {
    // kUnroll 16-byte loads in flight per thread before any is used
    constexpr int kUnroll = 4;
    for (int64_t g0 = g_begin + threadIdx.x; g0 < g_end; g0 += kUnroll * kThreads) {
      uint4 q[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t g = g0 + u * kThreads;
        q[u] = g < g_end ? __ldcs(reinterpret_cast<const uint4*>(row) + g) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t g = g0 + u * kThreads;
        if (g >= g_end) break;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[2 * i] = bf16_lo(w[i]);
          x[2 * i + 1] = bf16_hi(w[i]);
        }
        group(g, x);
      }
    }
  } else {
    for (int64_t g = g_begin + threadIdx.x; g < g_end; g += kThreads) {
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t v = g * 8 + j;
        x[j] = v < V ? __uint_as_float(static_cast<uint32_t>(row[v]) << 16) : CUDART_NAN_F;
      }
      group(g, x);
    }
  }
  uint64_t best = bv < 0 ? 0 : argmax_key(bs, static_cast<uint32_t>(bv));  // 0: below any key
  best = warp_max_u64(best);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s_warp[warp] = best;
  __syncthreads();
  if (warp == 0) {
    uint64_t t = lane < kThreads / 32 ? s_warp[lane] : 0;
    t = warp_max_u64(t);
    if (lane == 0) s_best = t;
  }
  if constexpr (kCluster == 1) {
    __syncthreads();
    if (threadIdx.x == 0) tokens[b] = static_cast<int32_t>(~static_cast<uint32_t>(s_best));
  } else {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
      uint64_t m = s_best;
#pragma unroll
      for (int q = 1; q < kCluster; ++q) m = max_u64(m, *cluster.map_shared_rank(&s_best, q));
      tokens[b] = static_cast<int32_t>(~static_cast<uint32_t>(m));
    }
    cluster.sync();  // the other CTAs' shared memory lives until rank 0 has read it
  }
}

}  // namespace

bi_status launch_sample(const void* logits, int64_t B, int64_t V, const float* temperature,
                        const uint64_t* seed, const uint64_t* step, int32_t* tokens,
                        cudaStream_t s) {
  if (B == 0) return BI_OK;
  const bool vec_ok = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  const auto* z = static_cast<const uint16_t*>(logits);
  // CTAs per row: 8 for fewer than 128 rows (one row then keeps several SMs
  // busy), 1 from 128 rows on (measured at 256 rows: 25 us against 33 us for
  // clusters of 4)
  const unsigned by = static_cast<unsigned>(B);
  if (B >= 128) {
    sample_kernel<1><<<dim3(1, by), kThreads, 0, s>>>(z, V, vec_ok, temperature, seed, step,
                                                      tokens);
  } else {
    sample_kernel<8><<<dim3(8, by), kThreads, 0, s>>>(z, V, vec_ok, temperature, seed, step,
                                                      tokens);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace bi
