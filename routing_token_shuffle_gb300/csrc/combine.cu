// Weighted combine back into original token order ("Speculative MoE" §1: expert
// results return to the token's source; FoE: per-group results are summed).
//
// One CTA per token row, threads striding over 16-byte vectors; every element is
// accumulated in fp32 in the fixed order k = 0..K-1 then shared experts j = 0..S-1
// and written once: deterministic, no atomics.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 128;

template <typename TE>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint4* __restrict__ y_disp, const int32_t* __restrict__ pair_row,
               const float* __restrict__ w, const uint4* __restrict__ y_sh, uint4* __restrict__ y,
               int T, int K, int S, int nvec, int nrows, DeviceStatus* st) {
  pdl_wait_and_trigger();
  constexpr int V = Elem<TE>::kPerVec16;
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < K) {
    const int r = pair_row[(size_t)t * K + tid];
    const bool ok = (unsigned)r < (unsigned)nrows;
    if (!ok) record_error(st, kStatusData, kBadPairRow, (long long)t * K + tid);
    s_row[tid] = ok ? r : -1;
    s_w[tid] = w[(size_t)t * K + tid];
  }
  __syncthreads();
  const TE* tag = nullptr;
  for (int v = tid; v < nvec; v += kThreads) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int r = s_row[k];
      if (r < 0) continue;
      const uint4 u = __ldg(y_disp + (size_t)r * nvec + v);
      float f[V];
      unpack16(u, f, tag);
      const float wk = s_w[k];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(wk, f[i], acc[i]);
    }
    for (int j = 0; j < S; ++j) {
      const uint4 u = __ldg(y_sh + ((size_t)j * T + t) * nvec + v);
      float f[V];
      unpack16(u, f, tag);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += f[i];
    }
    y[(size_t)t * nvec + v] = pack16(acc, tag);
  }
}

}  // namespace

cudaError_t launch_combine(const smoe_desc& d, const void* y_disp, const int32_t* pair_row,
                           const float* w, const void* y_sh, void* y, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  const int nvec = (int)(d.d * elem_size(d) / 16);
  const int S = y_sh ? d.n_shared : 0;
  if (d.dtype == SMOE_F32)
    SMOE_LAUNCH(combine_kernel<float>, d.T, kThreads, 0, s, static_cast<const uint4*>(y_disp),
        pair_row, w, static_cast<const uint4*>(y_sh), static_cast<uint4*>(y), d.T, d.K, S, nvec,
        d.T * d.K, st);
  else
    SMOE_LAUNCH(combine_kernel<__nv_bfloat16>, d.T, kThreads, 0, s,
        static_cast<const uint4*>(y_disp), pair_row, w, static_cast<const uint4*>(y_sh),
        static_cast<uint4*>(y), d.T, d.K, S, nvec, d.T * d.K, st);
  return cudaGetLastError();
}

}  // namespace smoe
