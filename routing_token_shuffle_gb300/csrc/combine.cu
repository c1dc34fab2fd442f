// Weighted combine back into original token order ("Speculative MoE" §1: expert
// results return to the token's source; FoE: per-group results are summed).
//
// One CTA per token row, threads striding over 16-byte vectors, 8 row loads in flight
// per thread (several vectors at once when K is small); every element is accumulated in
// fp32 in the fixed order k = 0..K-1 then shared experts j = 0..S-1 and written once:
// deterministic, no atomics.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 128;
constexpr int kBatch = 8;  // row loads in flight per thread

// U vectors per thread and iteration, kBatch / U rows of each loaded before the first
// accumulation: with K = 2, U = 4 keeps 8 loads in flight per thread instead of 2. With
// shared experts one batch spans the routed and the shared rows (one round trip instead
// of two per vector when K + S <= 8); without, the plain routed loop is cheaper.
template <typename TE, int U, bool SH>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint4* __restrict__ y_disp, const int32_t* __restrict__ pair_row,
               const float* __restrict__ w, const uint4* __restrict__ y_sh, uint4* __restrict__ y,
               int T, int K, int S, int nvec, int nrows, DeviceStatus* st) {
  pdl_wait_and_trigger();
  constexpr int V = Elem<TE>::kPerVec16;
  constexpr int KB = kBatch / U;
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
  for (int v0 = tid; v0 < nvec; v0 += kThreads * U) {
    float acc[U][V];
#pragma unroll
    for (int uu = 0; uu < U; ++uu)
#pragma unroll
      for (int i = 0; i < V; ++i) acc[uu][i] = 0.0f;
    if constexpr (!SH) {
      // batches of KB rows: all of a batch's loads (for the U vectors) are issued before
      // the first accumulation, which still runs in the order k = 0, 1, ... per vector
      for (int k0 = 0; k0 < K; k0 += KB) {
        uint4 u[U][KB];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
          const int v = v0 + uu * kThreads;
#pragma unroll
          for (int b = 0; b < KB; ++b) {
            const int r = k0 + b < K ? s_row[k0 + b] : -1;
            u[uu][b] = (r >= 0 && v < nvec) ? __ldg(y_disp + (size_t)r * nvec + v)
                                            : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
#pragma unroll
          for (int b = 0; b < KB; ++b) {
            if (k0 + b >= K || s_row[k0 + b] < 0) continue;
            float f[V];
            unpack16(u[uu][b], f, tag);
            const float wk = s_w[k0 + b];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[uu][i] = fmaf(wk, f[i], acc[uu][i]);
          }
        }
      }
    } else {
      // batches of KB of the K + S rows (routed rows k = 0..K-1, then shared rows): all of a
      // batch's loads (for the U vectors) are issued before the first accumulation, which
      // still runs in the order k = 0..K-1 (weighted) then j = 0..S-1
      for (int q0 = 0; q0 < K + S; q0 += KB) {
        uint4 u[U][KB];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
          const int v = v0 + uu * kThreads;
#pragma unroll
          for (int b = 0; b < KB; ++b) {
            const int q = q0 + b;
            const uint4* src = nullptr;
            if (q < K) {
              const int r = s_row[q];
              if (r >= 0) src = y_disp + (size_t)r * nvec;
            } else if (q < K + S) {
              src = y_sh + ((size_t)(q - K) * T + t) * nvec;
            }
            u[uu][b] = (src != nullptr && v < nvec) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
#pragma unroll
          for (int b = 0; b < KB; ++b) {
            const int q = q0 + b;
            if (q >= K + S || (q < K && s_row[q] < 0)) continue;
            float f[V];
            unpack16(u[uu][b], f, tag);
            if (q < K) {
              const float wk = s_w[q];
#pragma unroll
              for (int i = 0; i < V; ++i) acc[uu][i] = fmaf(wk, f[i], acc[uu][i]);
            } else {
#pragma unroll
              for (int i = 0; i < V; ++i) acc[uu][i] += f[i];
            }
          }
        }
      }
    }
#pragma unroll
    for (int uu = 0; uu < U; ++uu) {
      const int v = v0 + uu * kThreads;
      if (v < nvec) y[(size_t)t * nvec + v] = pack16(acc[uu], tag);
    }
  }
}

// The combine follows the expert FFN's persistent down GEMM with programmatic launch; the
// down GEMM lets it be scheduled only as the GEMM's CTAs finish (pdl_trigger at its end),
// so its CTAs never sit resident beside the GEMM's.
template <typename TE>
cudaError_t launch_combine_t(const smoe_desc& d, const void* y_disp, const int32_t* pair_row,
                             const float* w, const void* y_sh, void* y, int S, int nvec,
                             DeviceStatus* st, cudaStream_t s) {
  const uint4* yd = static_cast<const uint4*>(y_disp);
  const uint4* ys = static_cast<const uint4*>(y_sh);
  uint4* yo = static_cast<uint4*>(y);
  const int rows = d.T * d.K;
  if (S > 0) {  // K + S > 2 always holds here (K >= 1)
    if (d.K + S <= 4)
      SMOE_LAUNCH((combine_kernel<TE, 2, true>), d.T, kThreads, 0, s, yd, pair_row, w, ys, yo, d.T,
                  d.K, S, nvec, rows, st);
    else
      SMOE_LAUNCH((combine_kernel<TE, 1, true>), d.T, kThreads, 0, s, yd, pair_row, w, ys, yo, d.T,
                  d.K, S, nvec, rows, st);
  } else if (d.K <= 2) {
    SMOE_LAUNCH((combine_kernel<TE, 4, false>), d.T, kThreads, 0, s, yd, pair_row, w, ys, yo, d.T,
                d.K, S, nvec, rows, st);
  } else if (d.K <= 4) {
    SMOE_LAUNCH((combine_kernel<TE, 2, false>), d.T, kThreads, 0, s, yd, pair_row, w, ys, yo, d.T,
                d.K, S, nvec, rows, st);
  } else {
    SMOE_LAUNCH((combine_kernel<TE, 1, false>), d.T, kThreads, 0, s, yd, pair_row, w, ys, yo, d.T,
                d.K, S, nvec, rows, st);
  }
  return cudaGetLastError();
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
    return launch_combine_t<float>(d, y_disp, pair_row, w, y_sh, y, S, nvec, st, s);
  return launch_combine_t<__nv_bfloat16>(d, y_disp, pair_row, w, y_sh, y, S, nvec, st, s);
}

}  // namespace smoe
