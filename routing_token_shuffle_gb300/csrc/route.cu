// Gate GEMM, softmax and grouped top-K.
//
// "Speculative MoE" §1: each token activates only its top-K experts. FoE grouped
// block: group h owns experts [h E/H, (h+1) E/H) and selects its own top-K/H from
// the router output of the full representation; the weights are the softmax over
// all experts taken at the selected indices.
//
// Selection: one warp per token, the token's fp32 logits spread over the lanes;
// each pick is a butterfly argmax under the total order (logit descending, expert
// index ascending), so equal logits (including +0 / -0) go to the lower index.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kSelWarps = 8;
constexpr int kMaxPerLane = 16;  // E <= 512

__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ logits, int T, int E, int K, int H, int renorm,
              int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
  float v[kMaxPerLane];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i)
    if (lane + 32 * i < E) sum += expf(v[i] - m);
#pragma unroll
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);

  const int per = E / H, kh = K / H;
  uint32_t taken = 0;
  float my_w = 0.0f;
  int my_idx = 0;
  for (int h = 0; h < H; ++h) {
    const int lo = h * per, hi = lo + per;
    for (int j = 0; j < kh; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e >= lo && e < hi && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == h * kh + j) {
        my_idx = bi;
        my_w = expf(bv - m) / sum;
      }
    }
  }
  if (renorm) {
    float s = lane < K ? my_w : 0.0f;
#pragma unroll
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    my_w = my_w / s;
  }
  if (lane < K) {
    topk_idx[(size_t)t * K + lane] = my_idx;
    topk_w[(size_t)t * K + lane] = my_w;
  }
}

// Tiled fp32-FMA gate GEMM: logits [rows, E] = x [rows, d] . w_gate[E, d]^T.
constexpr int kBM = 64, kBN = 64, kBK = 32;

template <typename TE>
__global__ void __launch_bounds__(256)
gate_gemm_kernel(const TE* __restrict__ x, const TE* __restrict__ wg, float* __restrict__ logits,
                 int rows, int d, int E) {
  __shared__ float xs[kBK][kBM + 4];
  __shared__ float gs[kBK][kBN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kBK) {
    for (int i = tid; i < kBM * kBK; i += 256) {
      const int r = i / kBK, k = i % kBK;
      const int gr = m0 + r, gk = k0 + k;
      xs[k][r] = (gr < rows && gk < d) ? Elem<TE>::to_f32(x[(size_t)gr * d + gk]) : 0.0f;
      const int ge = n0 + r;
      gs[k][r] = (ge < E && gk < d) ? Elem<TE>::to_f32(wg[(size_t)ge * d + gk]) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = xs[k][ty * 4 + i]; b[i] = gs[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = n0 + tx * 4 + j;
      if (e < E) logits[(size_t)r * E + e] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_route(const smoe_desc& d, int rows, const void* x, const void* w_gate,
                         const float* logits_in, float* logits_out, int32_t* topk_idx,
                         float* topk_w, cudaStream_t s) {
  const float* sel_in = logits_in;
  if (!sel_in) {
    dim3 grid(ceil_div(rows, kBM), ceil_div(d.E, kBN));
    SMOE_COUNT_LAUNCH(1);
    if (d.dtype == SMOE_F32)
      gate_gemm_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x),
                                                   static_cast<const float*>(w_gate), logits_out,
                                                   rows, d.d, d.E);
    else
      gate_gemm_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_gate),
          logits_out, rows, d.d, d.E);
    sel_in = logits_out;
  } else if (logits_out && logits_out != logits_in) {
    cudaError_t e = cudaMemcpyAsync(logits_out, logits_in, sizeof(float) * rows * d.E,
                                    cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
  }
  SMOE_COUNT_LAUNCH(1);
  select_kernel<<<ceil_div(rows, kSelWarps), kSelWarps * 32, 0, s>>>(sel_in, rows, d.E, d.K, d.H,
                                                                    d.renorm, topk_idx, topk_w);
  return cudaGetLastError();
}

}  // namespace smoe
