// Next-layer prefetch predictor ("Speculating Experts Accelerates Inference for
// MoE" §2.A): the default vector d_l plus the residual r_l, layer-normalised,
// stands in for the next router's input LN(r_l + y_l). This file holds the fused
// LayerNorm of both rows and the hit count; routing reuses the gate/top-K kernels.
#include <algorithm>

#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPer = 32;  // d <= 8192

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

// Row t: q = LN(d_l + r_t) -> qs[t], s = LN(r_t + y_t) -> qs[T + t]; biased variance,
// eps 1e-5, two passes over values held in registers, output rounded to TE.
template <typename TE>
__global__ void __launch_bounds__(kThreads)
ln_pair_kernel(const float* __restrict__ r, const float* __restrict__ d_l,
               const TE* __restrict__ y, const float* __restrict__ gamma,
               const float* __restrict__ beta, TE* __restrict__ qs, int T, int d) {
  __shared__ float red[kThreads / 32];
  const int t = blockIdx.x;
  const float* rr = r + (size_t)t * d;
  const TE* yy = y + (size_t)t * d;
  float a[kMaxPer], b[kMaxPer];
  float sa = 0.0f, sb = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int j = threadIdx.x + i * kThreads;
    a[i] = b[i] = 0.0f;
    if (j < d) {
      const float rv = rr[j];
      a[i] = d_l[j] + rv;
      b[i] = rv + Elem<TE>::to_f32(yy[j]);
      sa += a[i];
      sb += b[i];
    }
  }
  const float ma = block_sum(sa, red) / d;
  const float mb = block_sum(sb, red) / d;
  float va = 0.0f, vb = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int j = threadIdx.x + i * kThreads;
    if (j < d) {
      va += (a[i] - ma) * (a[i] - ma);
      vb += (b[i] - mb) * (b[i] - mb);
    }
  }
  const float ia = rsqrtf(block_sum(va, red) / d + 1e-5f);
  const float ib = rsqrtf(block_sum(vb, red) / d + 1e-5f);
  TE* q = qs + (size_t)t * d;
  TE* s = qs + ((size_t)T + t) * d;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int j = threadIdx.x + i * kThreads;
    if (j < d) {
      q[j] = Elem<TE>::from_f32((a[i] - ma) * ia * gamma[j] + beta[j]);
      s[j] = Elem<TE>::from_f32((b[i] - mb) * ib * gamma[j] + beta[j]);
    }
  }
}

__global__ void __launch_bounds__(kThreads)
hits_kernel(const int32_t* __restrict__ pred, const int32_t* __restrict__ truth, int T, int K,
            unsigned long long* __restrict__ hits) {
  __shared__ unsigned long long red[kThreads / 32];
  unsigned long long c = 0;
  for (int t = blockIdx.x * kThreads + threadIdx.x; t < T; t += gridDim.x * kThreads) {
    const int32_t* p = pred + (size_t)t * K;
    const int32_t* q = truth + (size_t)t * K;
    for (int k = 0; k < K; ++k) {
      const int e = p[k];
      for (int k2 = 0; k2 < K; ++k2) c += (q[k2] == e);
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long s = 0;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    atomicAdd(hits, s);
  }
}

}  // namespace

cudaError_t launch_prefetch_ln(const smoe_desc& d, const float* r, const float* d_l,
                               const void* y, const float* gamma, const float* beta, void* qs,
                               cudaStream_t s) {
  SMOE_COUNT_LAUNCH(1);
  if (d.dtype == SMOE_F32)
    ln_pair_kernel<float><<<d.T, kThreads, 0, s>>>(r, d_l, static_cast<const float*>(y), gamma,
                                                   beta, static_cast<float*>(qs), d.T, d.d);
  else
    ln_pair_kernel<__nv_bfloat16><<<d.T, kThreads, 0, s>>>(
        r, d_l, static_cast<const __nv_bfloat16*>(y), gamma, beta,
        static_cast<__nv_bfloat16*>(qs), d.T, d.d);
  return cudaGetLastError();
}

cudaError_t launch_hits(const smoe_desc& d, const int32_t* pred_idx, const int32_t* true_idx,
                        unsigned long long* hits, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(hits, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(ceil_div(d.T, kThreads), 1024));
  SMOE_COUNT_LAUNCH(1);
  hits_kernel<<<grid, kThreads, 0, s>>>(pred_idx, true_idx, d.T, d.K, hits);
  return cudaGetLastError();
}

}  // namespace smoe
