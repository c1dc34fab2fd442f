// Weighted combine back into original token order ("Speculative MoE" §1: expert
// results return to the token's source; FoE: per-group results are summed).
//
// One CTA per token row, threads striding over 16-byte vectors, up to 8 rows' loads in
// flight per thread; every element is accumulated in fp32 in the fixed order
// k = 0..K-1 then shared experts j = 0..S-1 and written once: deterministic, no atomics.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 128;
constexpr int kBatch = 8;  // row loads in flight per thread

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
    // batches of kBatch rows: all of a batch's loads are issued before the first
    // accumulation, which still runs in the order k = 0, 1, ...
    for (int k0 = 0; k0 < K; k0 += kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int r = k0 + b < K ? s_row[k0 + b] : -1;
        u[b] = r >= 0 ? __ldg(y_disp + (size_t)r * nvec + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (k0 + b >= K || s_row[k0 + b] < 0) continue;
        float f[V];
        unpack16(u[b], f, tag);
        const float wk = s_w[k0 + b];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(wk, f[i], acc[i]);
      }
    }
    for (int j0 = 0; j0 < S; j0 += kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        u[b] = j0 + b < S ? __ldg(y_sh + ((size_t)(j0 + b) * T + t) * nvec + v)
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (j0 + b >= S) continue;
        float f[V];
        unpack16(u[b], f, tag);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += f[i];
      }
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
