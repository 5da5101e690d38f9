// layer_ops.cu -- the element-wise steps of a Llama-style decoder layer
// around the reductions: a row gather (token embedding, selecting the rows
// that need logits), rotary position embedding fused with the split of the
// QKV projection into q / k / v, and the SwiGLU product silu(gate) * up.
// None of them reduces across a row of the batch, so each output element is
// a function of its own inputs only ("Reproducible LLM Inference - Batch
// Invariance, the Cost of Determinism, and Where Bitwise Identity Is Actually
// Required", §5.4: element-wise operations are batch-invariant by nature).
#include <cuda_runtime.h>

#include "bi_internal.h"
#include "device_common.cuh"

namespace bi {
namespace {

constexpr int kThreads = 256;

unsigned blocks_for(int64_t work, int64_t cap = 152 * 32) {
  int64_t b = (work + kThreads - 1) / kThreads;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

// ------------------------------------------------------------ gather rows
// dst[i, :] = src[idx[i], :], 16-byte vectors, one block per row (rows taken
// in a grid-stride loop); an index outside [0, rows) is recorded and its row
// is written as zeros.
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(
    const uint4* __restrict__ src, int64_t rows, int vec_per_row,
    const int32_t* __restrict__ idx, int64_t n, uint4* __restrict__ dst, int* err) {
  for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int64_t r = idx[i];
    const bool ok = r >= 0 && r < rows;
    if (!ok && threadIdx.x == 0) record_error(err, BI_ERR_DEVICE_BOUNDS);
    const uint4* s = src + (ok ? r : 0) * vec_per_row;
    uint4* d = dst + i * vec_per_row;
#pragma unroll 4
    for (int c = threadIdx.x; c < vec_per_row; c += kThreads)
      __stcs(d + c, ok ? __ldg(s + c) : make_uint4(0, 0, 0, 0));
  }
}

// --------------------------------------------------------------- rotary
// One thread per (token, group of 8 frequency pairs).  Pair i (0 <= i < D/2)
// of a head rotates elements i and i + D/2 (the rotate-half arrangement) by
// the angle pos * theta^(-2i/D).  The angle is formed in fp64 and reduced
// modulo 2 pi before the fp32 sine and cosine, so it is accurate at any
// position; the rotation itself is fp32 with one rounding to bf16.
__global__ void __launch_bounds__(kThreads) rope_qkv_kernel(
    const uint4* __restrict__ qkv, const int32_t* __restrict__ pos, int64_t T, int Hq, int Hkv,
    int D, double log2_theta, uint4* __restrict__ q, uint4* __restrict__ k,
    uint4* __restrict__ v) {
  const int groups = D / 16;               // groups of 8 pairs per head
  const int vec_head = D / 8;              // 16-byte vectors per head
  const int64_t vec_row = static_cast<int64_t>(Hq + 2 * Hkv) * vec_head;
  const int64_t total = T * groups;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = e / groups;
    const int g = static_cast<int>(e - t * groups);
    const double p = static_cast<double>(pos[t]);
    float cs[8], sn[8];
    // theta^(-2i/D) for i = 8g .. 8g+7: the first power directly, the rest
    // by the constant ratio theta^(-2/D)
    const double ratio = exp2(-2.0 / D * log2_theta);
    double f = exp2(-2.0 * (8 * g) / D * log2_theta);
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const double a = p * f;
      const double r = fma(-kTwoPi, rint(a * kInvTwoPi), a);  // |r| <= pi (+ a few ulps)
      sincosf(static_cast<float>(r), &sn[j], &cs[j]);
      f *= ratio;
    }
    const uint4* row = qkv + t * vec_row;
    // heads in groups of kHeadBatch: all loads of a group before its stores,
    // so that many loads are in flight per thread
    constexpr int kHeadBatch = 4;
    for (int h0 = 0; h0 < Hq + Hkv; h0 += kHeadBatch) {
      uint4 lo[kHeadBatch], hi[kHeadBatch];
#pragma unroll
      for (int u = 0; u < kHeadBatch; ++u) {
        const int h = h0 + u;
        if (h < Hq + Hkv) {
          lo[u] = __ldg(row + h * vec_head + g);
          hi[u] = __ldg(row + h * vec_head + groups + g);
        }
      }
#pragma unroll
      for (int u = 0; u < kHeadBatch; ++u) {
        const int h = h0 + u;
        if (h >= Hq + Hkv) break;
        const uint32_t a[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
        const uint32_t b[4] = {hi[u].x, hi[u].y, hi[u].z, hi[u].w};
        uint32_t ol[4], oh[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          float x1[2] = {bf16_lo(a[w]), bf16_hi(a[w])}, x2[2] = {bf16_lo(b[w]), bf16_hi(b[w])};
          float y1[2], y2[2];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const float c = cs[2 * w + s], si = sn[2 * w + s];
            y1[s] = __fsub_rn(__fmul_rn(x1[s], c), __fmul_rn(x2[s], si));
            y2[s] = __fadd_rn(__fmul_rn(x2[s], c), __fmul_rn(x1[s], si));
          }
          ol[w] = pack_bf16x2(y1[0], y1[1]);
          oh[w] = pack_bf16x2(y2[0], y2[1]);
        }
        uint4* dst =
            h < Hq ? q + (t * Hq + h) * vec_head : k + (t * Hkv + (h - Hq)) * vec_head;
        __stcs(dst + g, make_uint4(ol[0], ol[1], ol[2], ol[3]));
        __stcs(dst + groups + g, make_uint4(oh[0], oh[1], oh[2], oh[3]));
      }
    }
    for (int h0 = 0; h0 < Hkv; h0 += kHeadBatch) {
      uint4 lo[kHeadBatch], hi[kHeadBatch];
#pragma unroll
      for (int u = 0; u < kHeadBatch; ++u) {
        const uint4* src = row + (Hq + Hkv + h0 + u) * vec_head;
        if (h0 + u < Hkv) {
          lo[u] = __ldg(src + g);
          hi[u] = __ldg(src + groups + g);
        }
      }
#pragma unroll
      for (int u = 0; u < kHeadBatch; ++u) {
        if (h0 + u >= Hkv) break;
        uint4* dst = v + (t * Hkv + h0 + u) * vec_head;
        __stcs(dst + g, lo[u]);
        __stcs(dst + groups + g, hi[u]);
      }
    }
  }
}

// ---------------------------------------------------------------- SwiGLU
// out[t, j] = bf16(silu(gate) * up), silu(x) = x / (1 + exp(-x)) in fp32
// (silu_mul_f32); gate and up come in blocks of vb 16-byte vectors (8 features
// each): gate vector c at 2 vb (c / vb) + c % vb of the row, up vb after it.

__global__ void __launch_bounds__(kThreads) silu_mul_kernel(const uint4* __restrict__ gu,
                                                            int64_t T, int64_t vec_f,
                                                            int64_t vb,
                                                            uint4* __restrict__ out) {
  const int64_t total = T * vec_f;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = e / vec_f;
    // c, vb < vec_f < 2^31 (16-byte vectors of one row): 32-bit arithmetic;
    // one block (vb == vec_f) is the stacked-halves layout
    const int c = static_cast<int>(e - t * vec_f), v = static_cast<int>(vb);
    const int cb = v == static_cast<int>(vec_f) ? 0 : c / v;
    const uint4* src = gu + t * 2 * vec_f + static_cast<int64_t>(cb) * 2 * v + (c - cb * v);
    const uint4 gv = __ldcs(src);
    const uint4 uv = __ldcs(src + vb);
    const uint32_t g[4] = {gv.x, gv.y, gv.z, gv.w}, u[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      o[w] = pack_bf16x2(silu_mul_f32(bf16_lo(g[w]), bf16_lo(u[w])),
                         silu_mul_f32(bf16_hi(g[w]), bf16_hi(u[w])));
    out[e] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

bi_status launch_gather_rows(const void* src, int64_t rows, int64_t H, const int32_t* idx,
                             int64_t n, void* dst, int* err, cudaStream_t s) {
  const int vpr = static_cast<int>(H / 8);
  const unsigned grid = static_cast<unsigned>(n < 152 * 16 ? n : 152 * 16);
  gather_rows_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint4*>(src), rows, vpr, idx, n,
                                               static_cast<uint4*>(dst), err);
  return cuda_status(cudaGetLastError());
}

bi_status launch_rope_qkv(const void* qkv, const int32_t* pos, int64_t T, int Hq, int Hkv, int D,
                          double theta, void* q, void* k, void* v, cudaStream_t s) {
  rope_qkv_kernel<<<blocks_for(T * (D / 16)), kThreads, 0, s>>>(
      static_cast<const uint4*>(qkv), pos, T, Hq, Hkv, D, log2(theta), static_cast<uint4*>(q),
      static_cast<uint4*>(k), static_cast<uint4*>(v));
  return cuda_status(cudaGetLastError());
}

bi_status launch_silu_mul(const void* gu, int64_t T, int64_t F, int64_t block, void* out,
                          cudaStream_t s) {
  const int64_t vf = F / 8;
  silu_mul_kernel<<<blocks_for(T * vf), kThreads, 0, s>>>(static_cast<const uint4*>(gu), T, vf,
                                                          block / 8, static_cast<uint4*>(out));
  return cuda_status(cudaGetLastError());
}

}  // namespace bi
