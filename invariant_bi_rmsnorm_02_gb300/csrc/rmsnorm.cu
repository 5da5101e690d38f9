// rmsnorm.cu -- RMSNorm, batch-invariant and batch-variant.
//
//   y[i,:] = x[i,:] * (mean_j x[i,j]^2 + eps)^(-1/2) * w
//
// Invariant kernel ("Reproducible LLM Inference", §5.3): one row per thread
// block.  The block shape and every step of the in-row reduction are fixed by
// H alone: thread t owns the 16-byte vectors t, t+T, t+2T, ... of the row
// (loaded up front, so each thread has several 16-byte loads in flight) and
// accumulates their squares in that order (fp32 fused multiply-add); the 32
// lanes of a warp are combined by a fixed xor-butterfly of shuffles; the
// warps' sums are combined by the same butterfly over warp indices.  A larger
// batch only means more blocks, never a different order for a row.
//
// Variant kernels ("Reproducible LLM Inference", §5.3; "Your Answer Depends on
// Who Else Is in the Batch", "A Concrete Example" step 3): at small M the row
// is cut into s chunks reduced by separate blocks, and the partial sums are
// combined by a pairwise tree in a second kernel that also writes y.  s grows
// as M shrinks, so a row's reduction order depends on the batch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bi_internal.h"
#include "device_common.cuh"

namespace bi {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float sum_squares8(const uint4& v, float acc) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
    acc = __fmaf_rn(a, a, acc);
    acc = __fmaf_rn(b, b, acc);
  }
  return acc;
}

// Fixed xor-butterfly over the 32 lanes; every lane ends with the same sum
// (fp32 addition is commutative, so lane i and lane i^o add the same pair).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Sum of one value per thread over the block, in a fixed order: warp
// butterflies, then the same butterfly over the warp sums (missing warps
// contribute +0, which leaves a sum of squares unchanged).
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = (blockDim.x + 31) >> 5;
  float t = lane < nw ? red[lane] : 0.0f;
  return warp_sum(t);
}

// y = (x * r) * w for 8 elements; the bf16 result is returned, the fp32
// values are also stored to yf (8 floats) when it is not null.
__device__ __forceinline__ uint4 scale_row8(const uint4& xv, const uint4& wv, float r,
                                            float* yf) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
  uint32_t o[4];
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __fmul_rn(__fmul_rn(bf16_lo(xs[i]), r), bf16_lo(ws[i]));
    f[2 * i + 1] = __fmul_rn(__fmul_rn(bf16_hi(xs[i]), r), bf16_hi(ws[i]));
    o[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
  }
  if (yf) {
    reinterpret_cast<float4*>(yf)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(yf)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float inv_rms(float sum_sq, float inv_h, float eps) {
  return rsqrtf(__fadd_rn(__fmul_rn(sum_sq, inv_h), eps));
}

// ---------------------------------------------------------------- invariant
template <int VPT>
__global__ void __launch_bounds__(1024) rmsnorm_row_kernel(const uint4* __restrict__ x,
                                                           const uint4* __restrict__ w,
                                                           uint4* __restrict__ y,
                                                           float* __restrict__ yf, int nvec,
                                                           float inv_h, float eps) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const uint4* xr = x + row * nvec;
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nvec ? __ldcs(xr + v) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) ss = sum_squares8(xv[k], ss);
  const float r = inv_rms(block_sum(ss, red), inv_h, eps);
  uint4* yr = y + row * nvec;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec)
      __stcs(yr + v, scale_row8(xv[k], __ldg(w + v), r, yf ? yf + (row * nvec + v) * 8 : nullptr));
  }
}

// Residual add fused in front: h = bf16(x + res) (an fp32 add, rounded once)
// overwrites res, and y = RMSNorm(h) * w with exactly the row reduction of
// rmsnorm_row_kernel, so the result equals a bf16 add followed by RMSNorm.
__device__ __forceinline__ uint4 add_bf16x8(const uint4& a, const uint4& b) {
  const uint32_t as[4] = {a.x, a.y, a.z, a.w}, bs[4] = {b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = pack_bf16x2(__fadd_rn(bf16_lo(as[i]), bf16_lo(bs[i])),
                       __fadd_rn(bf16_hi(as[i]), bf16_hi(bs[i])));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int VPT>
__global__ void __launch_bounds__(1024) add_rmsnorm_row_kernel(
    const uint4* __restrict__ x, uint4* __restrict__ res, const uint4* __restrict__ w,
    uint4* __restrict__ y, float* __restrict__ yf, int nvec, float inv_h, float eps) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const uint4* xr = x + row * nvec;
  uint4* rr = res + row * nvec;
  uint4 hv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    hv[k] = v < nvec ? add_bf16x8(__ldcs(xr + v), __ldcs(rr + v)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) __stcs(rr + v, hv[k]);
  }
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) ss = sum_squares8(hv[k], ss);
  const float r = inv_rms(block_sum(ss, red), inv_h, eps);
  uint4* yr = y + row * nvec;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec)
      __stcs(yr + v, scale_row8(hv[k], __ldg(w + v), r, yf ? yf + (row * nvec + v) * 8 : nullptr));
  }
}

// The add alone, for the batch-variant path (which then runs the split
// RMSNorm over h).
__global__ void add_bf16_kernel(const uint4* __restrict__ x, uint4* __restrict__ res,
                                int64_t nvec_total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec_total;
       i += (int64_t)gridDim.x * blockDim.x)
    res[i] = add_bf16x8(x[i], res[i]);
}

// Block shape as a function of H only: VPT vectors of 8 elements per thread,
// T threads (a multiple of 32, at most 1024).
struct RowShape {
  int vpt, threads;
};
RowShape row_shape(int64_t H) {
  const int nvec = static_cast<int>(H / 8);
  int vpt = nvec >= 256 ? 4 : (nvec >= 64 ? 2 : 1);
  while ((nvec + vpt - 1) / vpt > 1024) vpt *= 2;
  int t = (nvec + vpt - 1) / vpt;
  t = (t + 31) / 32 * 32;
  return {vpt, t};
}

// ------------------------------------------------------------------ variant
// Pass 1: block (c, i) sums the squares of chunk c of row i.
__global__ void __launch_bounds__(256) rmsnorm_split_partial(const uint4* __restrict__ x,
                                                             float* __restrict__ part, int nvec,
                                                             int chunk_vec) {
  __shared__ float red[32];
  const int c = blockIdx.x, s = gridDim.x;
  const int64_t row = blockIdx.y;
  const uint4* xc = x + row * nvec + (int64_t)c * chunk_vec;
  float ss = 0.0f;
  for (int v = threadIdx.x; v < chunk_vec; v += blockDim.x) ss = sum_squares8(__ldg(xc + v), ss);
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) part[row * s + c] = ss;
}

// Pass 2: every block combines the row's s partials by a pairwise tree, then
// normalises its own chunk.
__global__ void __launch_bounds__(256) rmsnorm_split_finish(const uint4* __restrict__ x,
                                                            const uint4* __restrict__ w,
                                                            const float* __restrict__ part,
                                                            uint4* __restrict__ y,
                                                            float* __restrict__ yf, int nvec,
                                                            int chunk_vec, float inv_h,
                                                            float eps) {
  const int c = blockIdx.x, s = gridDim.x;
  const int64_t row = blockIdx.y;
  float p[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) p[i] = i < s ? part[row * s + i] : 0.0f;
#pragma unroll
  for (int width = 32; width >= 1; width >>= 1)
#pragma unroll
    for (int i = 0; i < width; ++i) p[i] = __fadd_rn(p[2 * i], p[2 * i + 1]);
  const float r = inv_rms(p[0], inv_h, eps);
  const int64_t base = row * nvec + (int64_t)c * chunk_vec;
  for (int v = threadIdx.x; v < chunk_vec; v += blockDim.x)
    y[base + v] = scale_row8(__ldg(x + base + v), __ldg(w + c * chunk_vec + v), r,
                             yf ? yf + (base + v) * 8 : nullptr);
}

}  // namespace

bi_status launch_rmsnorm_invariant(const void* x, const void* w, void* y, float* y_f32,
                                   int64_t M, int64_t H, float eps, int* err, cudaStream_t s) {
  (void)err;
  if (M == 0) return BI_OK;
  const RowShape sh = row_shape(H);
  const int nvec = static_cast<int>(H / 8);
  const float inv_h = 1.0f / static_cast<float>(H);
  const dim3 grid(static_cast<unsigned>(M));
  const auto* xp = static_cast<const uint4*>(x);
  const auto* wp = static_cast<const uint4*>(w);
  auto* yp = static_cast<uint4*>(y);
  switch (sh.vpt) {
    case 1: rmsnorm_row_kernel<1><<<grid, sh.threads, 0, s>>>(xp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 2: rmsnorm_row_kernel<2><<<grid, sh.threads, 0, s>>>(xp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 4: rmsnorm_row_kernel<4><<<grid, sh.threads, 0, s>>>(xp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 8: rmsnorm_row_kernel<8><<<grid, sh.threads, 0, s>>>(xp, wp, yp, y_f32, nvec, inv_h, eps); break;
    default: return BI_ERR_UNSUPPORTED;
  }
  return cuda_status(cudaGetLastError());
}

bi_status launch_add_rmsnorm_invariant(const void* x, void* res, const void* w, void* y,
                                       float* y_f32, int64_t M, int64_t H, float eps,
                                       cudaStream_t s) {
  if (M == 0) return BI_OK;
  const RowShape sh = row_shape(H);
  const int nvec = static_cast<int>(H / 8);
  const float inv_h = 1.0f / static_cast<float>(H);
  const dim3 grid(static_cast<unsigned>(M));
  const auto* xp = static_cast<const uint4*>(x);
  auto* rp = static_cast<uint4*>(res);
  const auto* wp = static_cast<const uint4*>(w);
  auto* yp = static_cast<uint4*>(y);
  switch (sh.vpt) {
    case 1: add_rmsnorm_row_kernel<1><<<grid, sh.threads, 0, s>>>(xp, rp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 2: add_rmsnorm_row_kernel<2><<<grid, sh.threads, 0, s>>>(xp, rp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 4: add_rmsnorm_row_kernel<4><<<grid, sh.threads, 0, s>>>(xp, rp, wp, yp, y_f32, nvec, inv_h, eps); break;
    case 8: add_rmsnorm_row_kernel<8><<<grid, sh.threads, 0, s>>>(xp, rp, wp, yp, y_f32, nvec, inv_h, eps); break;
    default: return BI_ERR_UNSUPPORTED;
  }
  return cuda_status(cudaGetLastError());
}

bi_status launch_add_bf16(const void* x, void* res, int64_t elems, cudaStream_t s) {
  const int64_t nvec = elems / 8;
  if (nvec == 0) return BI_OK;
  int64_t blocks = (nvec + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  add_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint4*>(x),
                                                               static_cast<uint4*>(res), nvec);
  return cuda_status(cudaGetLastError());
}

int rmsnorm_variant_splits(int64_t M, int64_t H, int num_sms) {
  const int64_t nvec = H / 8;
  int s = 1;
  while (s * 2 <= 64 && nvec % (s * 2) == 0 && H / (s * 2) >= 128 &&
         M * s < 2 * static_cast<int64_t>(num_sms))
    s *= 2;
  return s;
}

bi_status launch_rmsnorm_variant(const void* x, const void* w, void* y, float* y_f32, int64_t M,
                                 int64_t H, float eps, int splits, float* ws, int* err,
                                 cudaStream_t s) {
  if (M == 0) return BI_OK;
  if (splits <= 1) return launch_rmsnorm_invariant(x, w, y, y_f32, M, H, eps, err, s);
  if (M > 65535) return BI_ERR_UNSUPPORTED;
  const int nvec = static_cast<int>(H / 8);
  const int chunk_vec = nvec / splits;
  int threads = chunk_vec < 256 ? (chunk_vec + 31) / 32 * 32 : 256;
  const dim3 grid(splits, static_cast<unsigned>(M));
  rmsnorm_split_partial<<<grid, threads, 0, s>>>(static_cast<const uint4*>(x), ws, nvec,
                                                 chunk_vec);
  rmsnorm_split_finish<<<grid, threads, 0, s>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(w), ws, static_cast<uint4*>(y),
      y_f32, nvec, chunk_vec, 1.0f / static_cast<float>(H), eps);
  return cuda_status(cudaGetLastError());
}

}  // namespace bi
