// Next-layer prefetch predictor ("Speculating Experts Accelerates Inference for
// MoE" §2.A): the default vector d_l plus the residual r_l, layer-normalised,
// stands in for the next router's input LN(r_l + y_l). This file holds the fused
// LayerNorm of both rows and the hit count; routing reuses the gate/top-K kernels.
#include <algorithm>

#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    s.x += red[w].x;
    s.y += red[w].y;
  }
  return s;
}

__device__ __forceinline__ void load4(const float* p, float* v) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* v) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void store4(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float* v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) =
      make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// Row t: q = LN(d_l + r_t) -> qs[t], s = LN(r_t + y_t) -> qs[T + t]; biased variance,
// eps 1e-5, two passes over values held in registers (4-element chunks), output
// rounded to TE.
template <typename TE, int kMaxChunks>
__global__ void __launch_bounds__(kThreads)
ln_pair_kernel(const float* __restrict__ r, const float* __restrict__ d_l,
               const TE* __restrict__ y, const float* __restrict__ gamma,
               const float* __restrict__ beta, TE* __restrict__ qs, int T, int d) {
  pdl_wait_and_trigger();
  __shared__ float2 red[kThreads / 32];
  const int t = blockIdx.x;
  const float* rr = r + (size_t)t * d;
  const TE* yy = y + (size_t)t * d;
  float a[kMaxChunks][4], b[kMaxChunks][4];
  float2 sum = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int j = 4 * (threadIdx.x + i * kThreads);
    if (j < d) {
      float rv[4], dv[4], yv[4];
      load4(rr + j, rv);
      load4(d_l + j, dv);
      load4(yy + j, yv);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        a[i][c] = dv[c] + rv[c];
        b[i][c] = rv[c] + yv[c];
        sum.x += a[i][c];
        sum.y += b[i][c];
      }
    }
  }
  const float2 tot = block_sum2(sum, red);
  const float ma = tot.x / d, mb = tot.y / d;
  float2 sq = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int j = 4 * (threadIdx.x + i * kThreads);
    if (j < d) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sq.x += (a[i][c] - ma) * (a[i][c] - ma);
        sq.y += (b[i][c] - mb) * (b[i][c] - mb);
      }
    }
  }
  const float2 var = block_sum2(sq, red);
  const float ia = rsqrtf(var.x / d + 1e-5f), ib = rsqrtf(var.y / d + 1e-5f);
  TE* q = qs + (size_t)t * d;
  TE* s = qs + ((size_t)T + t) * d;
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int j = 4 * (threadIdx.x + i * kThreads);
    if (j < d) {
      float g[4], bt[4], oq[4], os[4];
      load4(gamma + j, g);
      load4(beta + j, bt);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        oq[c] = (a[i][c] - ma) * ia * g[c] + bt[c];
        os[c] = (b[i][c] - mb) * ib * g[c] + bt[c];
      }
      store4(q + j, oq);
      store4(s + j, os);
    }
  }
}

__global__ void __launch_bounds__(kThreads)
hits_kernel(const int32_t* __restrict__ pred, const int32_t* __restrict__ truth, int T, int K,
            unsigned long long* __restrict__ hits) {
  pdl_wait_and_trigger();
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

template <typename TE, int kChunks>
cudaError_t ln_launch(const smoe_desc& d, const float* r, const float* d_l, const void* y,
               const float* gamma, const float* beta, void* qs, cudaStream_t s) {
  {
    auto kfn_ = ln_pair_kernel<TE, kChunks>;
    SMOE_LAUNCH(kfn_, d.T, kThreads, 0, s, r, d_l, static_cast<const TE*>(y), gamma, beta,
        static_cast<TE*>(qs), d.T, d.d);
  }
  return cudaSuccess;
}

// One CTA per token; the per-thread register arrays are sized to the 4-element chunks the
// row needs (d <= 1024 chunks * 4), which keeps several CTAs resident per SM.
template <typename TE>
cudaError_t ln_dispatch(const smoe_desc& d, const float* r, const float* d_l, const void* y,
                 const float* gamma, const float* beta, void* qs, cudaStream_t s) {
  const int chunks = ceil_div(d.d, 4 * kThreads);
  if (chunks <= 1) return ln_launch<TE, 1>(d, r, d_l, y, gamma, beta, qs, s);
  if (chunks <= 2) return ln_launch<TE, 2>(d, r, d_l, y, gamma, beta, qs, s);
  if (chunks <= 4) return ln_launch<TE, 4>(d, r, d_l, y, gamma, beta, qs, s);
  return ln_launch<TE, 8>(d, r, d_l, y, gamma, beta, qs, s);
}

cudaError_t launch_prefetch_ln(const smoe_desc& d, const float* r, const float* d_l,
                               const void* y, const float* gamma, const float* beta, void* qs,
                               cudaStream_t s) {
  if (d.dtype == SMOE_F32) return ln_dispatch<float>(d, r, d_l, y, gamma, beta, qs, s);
  return ln_dispatch<__nv_bfloat16>(d, r, d_l, y, gamma, beta, qs, s);
}

cudaError_t launch_hits(const smoe_desc& d, const int32_t* pred_idx, const int32_t* true_idx,
                        unsigned long long* hits, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(hits, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(ceil_div(d.T, kThreads), 1024));
  SMOE_LAUNCH(hits_kernel, grid, kThreads, 0, s, pred_idx, true_idx, d.T, d.K, hits);
  return cudaGetLastError();
}

}  // namespace smoe
