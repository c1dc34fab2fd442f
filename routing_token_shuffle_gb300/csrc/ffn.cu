// Grouped SwiGLU expert FFN over the expert-contiguous rows written by dispatch.
//
// Group g < E is routed expert g (rows expert_off[g] .. expert_off[g+1] of x_disp);
// group E + j is shared expert j, run on all T rows of x. The up projection writes
// H = silu(A W1^T) * (A W3^T) rounded to the element type; the down projection
// writes Y = H W2^T.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

// tile_start[g] = first tile of group g for a row-tile height bm; tile_start[G] = total.
// expert_off must be non-decreasing from 0 to at most T K; otherwise no tile is
// scheduled and the status word records the error.
__global__ void tile_table_kernel(const int32_t* __restrict__ expert_off, int E, int n_shared,
                                  int T, int TK, int bm, int32_t* __restrict__ tile_start,
                                  DeviceStatus* st) {
  const int lane = threadIdx.x;
  const int G = E + n_shared;
  bool bad = false;
  for (int g = lane; g < E; g += 32) {
    const int lo = expert_off[g], hi = expert_off[g + 1];
    bad |= lo < 0 || hi < lo || hi > TK;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (bad) {
    if (lane == 0) record_error(st, kStatusData, kBadPairRow, -1);
    for (int g = lane; g <= G; g += 32) tile_start[g] = 0;
    return;
  }
  int carry = 0;
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int g = g0 + lane;
    int rows = 0;
    if (g < E) rows = expert_off[g + 1] - expert_off[g];
    else if (g < G) rows = T;
    const int n = (rows + bm - 1) / bm;
    int incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (g < G) tile_start[g] = carry + incl - n;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tile_start[G] = carry;
}

struct GroupRows {
  int g, m0, rows;   // group, first row of this tile within the group, rows in the group
};

__device__ __forceinline__ bool find_tile(const int32_t* tile_start, int G, int tile, int bm,
                                          const int32_t* expert_off, int E, int T, GroupRows* out) {
  if (tile >= tile_start[G]) return false;
  int lo = 0, hi = G - 1;
  while (lo < hi) {  // last g with tile_start[g] <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  out->g = lo;
  out->m0 = (tile - tile_start[lo]) * bm;
  out->rows = lo < E ? expert_off[lo + 1] - expert_off[lo] : T;
  return true;
}

constexpr int kBM = 64, kBN = 64, kBK = 16;

// SIMT reference-speed grouped GEMM: 64x64 output tile per CTA, fp32 FMA.
// UP: out = H rows, computes both W1 and W3 tiles and applies SwiGLU.
template <typename TE, bool UP>
__global__ void __launch_bounds__(256)
ffn_simt_kernel(const TE* __restrict__ a_routed, const TE* __restrict__ a_shared,
                const int32_t* __restrict__ expert_off, const int32_t* __restrict__ tile_start,
                const TE* __restrict__ wa, const TE* __restrict__ wb, TE* __restrict__ out_routed,
                TE* __restrict__ out_shared, int E, int n_shared, int T, int TK, int N, int KD) {
  __shared__ float as[kBK][kBM + 4];
  __shared__ float b1s[kBK][kBN + 4];
  __shared__ float b3s[kBK][UP ? kBN + 4 : 1];
  GroupRows gr;
  if (!find_tile(tile_start, E + n_shared, blockIdx.x, kBM, expert_off, E, T, &gr)) return;
  const int n0 = blockIdx.y * kBN;
  const bool shared = gr.g >= E;
  const int j = gr.g - E;
  // A rows and output rows of this group
  const TE* A;
  TE* O;
  if (UP) {
    A = shared ? a_shared : a_routed + (size_t)expert_off[gr.g] * KD;
    O = out_routed + (size_t)(shared ? TK + j * T : expert_off[gr.g]) * N;  // H buffer
  } else {
    A = a_routed + (size_t)(shared ? TK + j * T : expert_off[gr.g]) * KD;   // H buffer
    O = shared ? out_shared + (size_t)j * T * N : out_routed + (size_t)expert_off[gr.g] * N;
  }
  const TE* B1 = wa + (size_t)gr.g * N * KD;
  const TE* B3 = UP ? wb + (size_t)gr.g * N * KD : nullptr;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc1[4][4] = {}, acc3[4][4] = {};
  for (int k0 = 0; k0 < KD; k0 += kBK) {
    for (int i = tid; i < kBM * kBK; i += 256) {
      const int r = i / kBK, k = i % kBK;
      const int gk = k0 + k;
      const int ar = gr.m0 + r;
      as[k][r] = (ar < gr.rows && gk < KD) ? Elem<TE>::to_f32(A[(size_t)ar * KD + gk]) : 0.0f;
      const int bn = n0 + r;
      b1s[k][r] = (bn < N && gk < KD) ? Elem<TE>::to_f32(B1[(size_t)bn * KD + gk]) : 0.0f;
      if (UP) b3s[k][r] = (bn < N && gk < KD) ? Elem<TE>::to_f32(B3[(size_t)bn * KD + gk]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float a[4], b1[4], b3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = as[k][ty * 4 + i];
        b1[i] = b1s[k][tx * 4 + i];
        if (UP) b3[i] = b3s[k][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc1[i][q] = fmaf(a[i], b1[q], acc1[i][q]);
          if (UP) acc3[i][q] = fmaf(a[i], b3[q], acc3[i][q]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = gr.m0 + ty * 4 + i;
    if (r >= gr.rows) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx * 4 + q;
      if (n >= N) continue;
      float v = acc1[i][q];
      if (UP) v = (v / (1.0f + expf(-v))) * acc3[i][q];
      O[(size_t)r * N + n] = Elem<TE>::from_f32(v);
    }
  }
}

template <typename TE>
cudaError_t run_ffn(const smoe_desc& d, const void* x_disp, const void* x,
                    const int32_t* expert_off, const void* w1, const void* w3, const void* w2,
                    void* y_disp, void* y_sh, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  int32_t* tiles = ws_ptr<int32_t>(ws, L.tiles);
  TE* hbuf = ws_ptr<TE>(ws, L.hbuf);
  const int TK = d.T * d.K;
  SMOE_COUNT_LAUNCH(1);
  tile_table_kernel<<<1, 32, 0, s>>>(expert_off, d.E, d.n_shared, d.T, TK, kBM, tiles,
                                     ws_ptr<DeviceStatus>(ws, L.status));
  const int max_tiles = ceil_div(TK, kBM) + d.E + d.n_shared * ceil_div(d.T, kBM);
  dim3 g_up(max_tiles, ceil_div(d.F, kBN));
  SMOE_COUNT_LAUNCH(1);
  ffn_simt_kernel<TE, true><<<g_up, 256, 0, s>>>(
      static_cast<const TE*>(x_disp), static_cast<const TE*>(x), expert_off, tiles,
      static_cast<const TE*>(w1), static_cast<const TE*>(w3), hbuf, nullptr, d.E, d.n_shared,
      d.T, TK, d.F, d.d);
  dim3 g_dn(max_tiles, ceil_div(d.d, kBN));
  SMOE_COUNT_LAUNCH(1);
  ffn_simt_kernel<TE, false><<<g_dn, 256, 0, s>>>(
      hbuf, nullptr, expert_off, tiles, static_cast<const TE*>(w2), nullptr,
      static_cast<TE*>(y_disp), static_cast<TE*>(y_sh), d.E, d.n_shared, d.T, TK, d.d, d.F);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_ffn(const smoe_desc& d, const void* x_disp, const void* x,
                              const int32_t* expert_off, const void* w1, const void* w3,
                              const void* w2, void* y_disp, void* y_sh, void* ws,
                              cudaStream_t s) {
  if (d.dtype == SMOE_F32)
    return run_ffn<float>(d, x_disp, x, expert_off, w1, w3, w2, y_disp, y_sh, ws, s);
  return run_ffn<__nv_bfloat16>(d, x_disp, x, expert_off, w1, w3, w2, y_disp, y_sh, ws, s);
}

}  // namespace smoe
