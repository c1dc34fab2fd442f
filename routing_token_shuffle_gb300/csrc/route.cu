// Gate GEMM, softmax and grouped top-K.
//
// "Speculative MoE" §1: each token activates only its top-K experts. FoE grouped
// block: group h owns experts [h E/H, (h+1) E/H) and selects its own top-K/H from
// the router output of the full representation; the weights are the softmax over
// all experts taken at the selected indices.
//
// bf16 layers: the gate GEMM runs on tcgen05 (M = 128 token rows, N = E rounded up to
// 16, K split over the CTAs of a cluster, or over KS CTAs in the two-launch path). With
// E <= 256 and K no larger than the lanes per token, route_fused_kernel reduces the split
// partials in distributed shared memory and selects in the same launch; otherwise each
// split writes fp32 partial logits and a selection kernel adds them in split order.
// fp32 layers keep an exact fp32-FMA gate GEMM: the tensor cores would round the
// operands to tf32 and move logits by ~1e-3, enough to flip routing decisions.
//
// Selection: 8 or 16 lanes per token (one warp per token when E > 256 or K > 16), the
// token's fp32 logits spread over those lanes; each pick is a butterfly argmax under the
// total order (logit descending, expert index ascending), so equal logits (including
// +0 / -0) go to the lower index. Grouped top-1 over 8 groups (FoE with H = K = 8) has
// its own static-index kernel.
#include <algorithm>

#include "tc_common.cuh"

namespace smoe {
namespace {

constexpr int kSelWarps = 8;

// kMaxPerLane logits per lane: E <= 32 * kMaxPerLane (4, 8 or 16).
template <int kMaxPerLane>
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ part, int KS, long long split_stride,
              float* __restrict__ logits_out, int T, int E, int K, int H, int renorm,
              int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, RouteSplitOut so) {
  pdl_wait_and_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  // rows from so.split on go to the second output set, renumbered from 0
  const bool second = t >= so.split;
  const int to = second ? t - so.split : t;
  if (second) {
    logits_out = so.logits;
    topk_idx = so.idx;
    topk_w = so.w;
  }
  // split s of every value is loaded before any of split s + 1 is added, so all of a
  // split's loads (and, unrolled, those of several splits) are in flight together
  float v[kMaxPerLane];
  const float* prow = part + (size_t)t * E + lane;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) v[i] = lane + 32 * i < E ? prow[32 * i] : -INFINITY;
#pragma unroll 4
  for (int s = 1; s < KS; ++s) {
    const float* ps = prow + (size_t)s * split_stride;
    float a[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) a[i] = lane + 32 * i < E ? ps[32 * i] : 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) v[i] += a[i];
  }
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    if (e < E && logits_out) logits_out[(size_t)to * E + e] = v[i];
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
    topk_idx[(size_t)to * K + lane] = my_idx;
    topk_w[(size_t)to * K + lane] = my_w;
  }
}

// Sub-warp selection: L lanes per token (32 / L tokens per warp), lane j holding experts
// j, j + L, j + 2L, ... The warp-per-token kernel spends most of its instructions on
// 5-step butterflies; with L = 8 or 16 lanes a pick takes 3 or 4 steps for 32 / L tokens
// at once, and the K weights are computed by K lanes together at the end. The picks,
// their order and the logits are the same as the warp kernel's (the same total order:
// logit descending, expert index ascending; the same split-order partial sums). Used
// when K <= L; pick k is held by lane k.
// Softmax and grouped top-K of one token held by L lanes (lane j holds experts j, j + L,
// j + 2L, ...; v[i] = -inf past E). Every lane of the warp must call it (the shuffles
// span the warp). Lane k < K returns pick k: its expert index and weight.
template <int L, int kPer>
__device__ __forceinline__ void select_sub_row(const float (&v)[kPer], int j, int E, int K, int H,
                                               int renorm, int& pick_i, float& pick_w) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int off = L >> 1; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (j + L * i < E) sum += expf(v[i] - m);
#pragma unroll
  for (int off = L >> 1; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);

  float my_v = -INFINITY;
  int my_i = 0;
  if (H == 1) {
    // ungrouped: a lane's best live value by strict > (its lower index wins a tie, its
    // indices grow with i), the butterfly over (logit desc, index asc), and the winner's
    // slot marked dead. A lane with nothing live reports (-inf, j), which loses to any
    // finite logit.
    uint32_t dead = 0;
    for (int q = 0; q < K; ++q) {
      float bv = -INFINITY;
      int bl = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        if (!(dead & (1u << i)) && v[i] > bv) {
          bv = v[i];
          bl = i;
        }
      }
      int bi = j + L * bl;
#pragma unroll
      for (int off = L >> 1; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if ((bi & (L - 1)) == j) dead |= 1u << (bi / L);
      if (j == q) { my_v = bv; my_i = bi; }
    }
  }
  const int per = E / H, kh = H == 1 ? 0 : K / H;
  uint32_t taken = 0;
  for (int h = 0; h < H && kh > 0; ++h) {
    const int lo = h * per, hi = lo + per;
    for (int q = 0; q < kh; ++q) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = j + L * i;
        if (e >= lo && e < hi && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = L >> 1; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (bi < E && (bi & (L - 1)) == j) taken |= 1u << (bi / L);
      if (j == h * kh + q) { my_v = bv; my_i = bi; }
    }
  }
  float w = j < K ? expf(my_v - m) / sum : 0.0f;
  if (renorm) {
    float sw = w;
#pragma unroll
    for (int off = L >> 1; off; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    w = w / sw;
  }
  pick_i = my_i;
  pick_w = w;
}

// Sub-warp selection: L lanes per token (32 / L tokens per warp), lane j holding experts
// j, j + L, j + 2L, ... The warp-per-token kernel spends most of its instructions on
// 5-step butterflies; with L = 8 or 16 lanes a pick takes 3 or 4 steps for 32 / L tokens
// at once, and the K weights are computed by K lanes together at the end. The picks,
// their order and the logits are the same as the warp kernel's (the same total order:
// logit descending, expert index ascending; the same split-order partial sums). Used
// when K <= L; pick k is held by lane k.
template <int L, int kPer>
__global__ void __launch_bounds__(256)
select_sub_kernel(const float* __restrict__ part, int KS, long long split_stride,
                  float* __restrict__ logits_out, int T, int E, int K, int H, int renorm,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, RouteSplitOut so) {
  pdl_wait_and_trigger();
  const int j = threadIdx.x & (L - 1);
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) / L);
  const bool valid = t < T;  // every lane stays for the shuffles
  const bool second = valid && t >= so.split;
  const int to = second ? t - so.split : t;
  if (second) {
    logits_out = so.logits;
    topk_idx = so.idx;
    topk_w = so.w;
  }
  float v[kPer];
  const float* prow = part + (size_t)(valid ? t : 0) * E + j;
#pragma unroll
  for (int i = 0; i < kPer; ++i) v[i] = (valid && j + L * i < E) ? prow[L * i] : -INFINITY;
#pragma unroll 4
  for (int s = 1; s < KS; ++s) {
    const float* ps = prow + (size_t)s * split_stride;
    float a[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) a[i] = (valid && j + L * i < E) ? ps[L * i] : 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] += a[i];
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = j + L * i;
    if (valid && e < E && logits_out) logits_out[(size_t)to * E + e] = v[i];
  }
  int my_i;
  float w;
  select_sub_row<L, kPer>(v, j, E, K, H, renorm, my_i, w);
  if (valid && j < K) {
    topk_idx[(size_t)to * K + j] = my_i;
    topk_w[(size_t)to * K + j] = w;
  }
}

// Grouped top-1 (K = H, one pick per group, as FoE's top-K/H = 1): with E = L * H * VPG,
// lane j's values i in [h VPG, (h+1) VPG) are exactly its experts of group h, so each
// group is one short local scan plus one butterfly, and every index is static. Same
// picks, order and weights as select_sub_kernel (within a lane the expert index grows
// with i, so strict > keeps the lower index; the butterfly breaks ties the same way).
// Grouped top-1 of one token held by L lanes, E = L * H_ * VPG: lane j's values i in
// [h VPG, (h + 1) VPG) are exactly its experts of group h. Every lane of the warp must
// call it. Lane h < H_ returns the pick of group h and its weight.
template <int L, int H_, int VPG>
__device__ __forceinline__ void select_group1_row(const float (&v)[H_ * VPG], int j, int renorm,
                                                  int& pick_i, float& pick_w) {
  constexpr int kPer = H_ * VPG, K = H_;
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int off = L >> 1; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) sum += expf(v[i] - m);
#pragma unroll
  for (int off = L >> 1; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  float my_v = -INFINITY;
  int my_i = 0;
#pragma unroll
  for (int h = 0; h < H_; ++h) {
    float bv = v[h * VPG];
    int bi = j + L * h * VPG;
#pragma unroll
    for (int u = 1; u < VPG; ++u) {
      if (v[h * VPG + u] > bv) {
        bv = v[h * VPG + u];
        bi = j + L * (h * VPG + u);
      }
    }
#pragma unroll
    for (int off = L >> 1; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (j == h) { my_v = bv; my_i = bi; }
  }
  float w = j < K ? expf(my_v - m) / sum : 0.0f;
  if (renorm) {
    float sw = w;
#pragma unroll
    for (int off = L >> 1; off; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    w = w / sw;
  }
  pick_i = my_i;
  pick_w = w;
}

template <int L, int H_, int VPG>
__global__ void __launch_bounds__(256)
select_group1_kernel(const float* __restrict__ part, int KS, long long split_stride,
                     float* __restrict__ logits_out, int T, int renorm,
                     int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                     RouteSplitOut so) {
  pdl_wait_and_trigger();
  constexpr int kPer = H_ * VPG, E = L * kPer, K = H_;
  const int j = threadIdx.x & (L - 1);
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) / L);
  const bool valid = t < T;  // every lane stays for the shuffles
  const bool second = valid && t >= so.split;
  const int to = second ? t - so.split : t;
  if (second) {
    logits_out = so.logits;
    topk_idx = so.idx;
    topk_w = so.w;
  }
  float v[kPer];
  const float* prow = part + (size_t)(valid ? t : 0) * E + j;
#pragma unroll
  for (int i = 0; i < kPer; ++i) v[i] = valid ? prow[L * i] : -INFINITY;
#pragma unroll 4
  for (int s = 1; s < KS; ++s) {
    const float* ps = prow + (size_t)s * split_stride;
    float a[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) a[i] = valid ? ps[L * i] : 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] += a[i];
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (valid && logits_out) logits_out[(size_t)to * E + j + L * i] = v[i];
  int my_i;
  float w;
  select_group1_row<L, H_, VPG>(v, j, renorm, my_i, w);
  if (valid && j < K) {
    topk_idx[(size_t)to * K + j] = my_i;
    topk_w[(size_t)to * K + j] = w;
  }
}

// ------------------------------------------------------------ fp32 gate GEMM
// Tiled fp32-FMA gate GEMM: logits [rows, E] = x [rows, d] . w_gate[E, d]^T.
constexpr int kBM = 64, kBN = 64, kBK = 32;

__global__ void __launch_bounds__(256)
gate_gemm_f32_kernel(const float* __restrict__ x, const float* __restrict__ wg,
                     float* __restrict__ logits, int rows, int d, int E) {
  pdl_wait_and_trigger();
  __shared__ float xs[kBK][kBM + 4];
  __shared__ float gs[kBK][kBN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kBK) {
    for (int i = tid; i < kBM * kBK; i += 256) {
      const int r = i / kBK, k = i % kBK;
      const int gr = m0 + r, gk = k0 + k;
      xs[k][r] = (gr < rows && gk < d) ? x[(size_t)gr * d + gk] : 0.0f;
      const int ge = n0 + r;
      gs[k][r] = (ge < E && gk < d) ? wg[(size_t)ge * d + gk] : 0.0f;
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

// ------------------------------------------------------------ bf16 gate GEMM
// One CTA per (128-row tile, K split). Warp 0: TMA producer (3-stage ring of
// A 128 x 64 and B E_pad x 64 bf16 tiles, 128-byte swizzle); warp 1: tcgen05.mma
// issuer (one N = E_pad MMA per 16-wide K step, two when E_pad > 256); warp 2: TMEM
// allocation; warps 4-7: write the split's fp32 partial logits, one row per thread.
constexpr int kGateMaxStages = 3;  // 2 when E > 256 (a 64 KB B stage)
constexpr uint32_t kGateA = 128 * 128;

struct GateArgs {
  float* part;              // [KS, rows, E]
  DeviceStatus* st;
  int rows, E, E_pad, nkb, KS;
  uint32_t idesc1, idesc2;  // N = min(E_pad, 256) and E_pad - 256
  uint32_t box_rows;        // B box rows (E_pad, or 256 when E_pad > 256)
  uint32_t b_stage;         // bytes of one B stage
  uint32_t tmem_cols;
  uint32_t stages;          // ring depth: 3, or 2 when a B stage is 64 KB
};

__global__ void __launch_bounds__(256, 1)
gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const GateArgs p) {
  pdl_wait_and_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  const uint32_t nst = p.stages;
  uint8_t* sB = base + nst * kGateA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + nst * p.b_stage);
  uint64_t* empty = full + kGateMaxStages;
  uint64_t* tfull = empty + kGateMaxStages;
  uint64_t* drain = tfull + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128, ks = blockIdx.y;
  const int kb0 = (int)((long long)ks * p.nkb / p.KS);
  const int kb1 = (int)((long long)(ks + 1) * p.nkb / p.KS);
  const bool two = p.E_pad > 256;
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < nst; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(drain, 1);
    *s_abort = 0;
    tc::mbar_init_fence();
    tc::tma_prefetch_map(&tmX);
    tc::tma_prefetch_map(&tmW);
  }
  if (warp == 2) {
    tc::tmem_alloc(s_tmem, p.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  volatile int* abort = s_abort;

  if (warp == 0 && lane == 0) {
    uint32_t it = 0;
    bool ok = true;
    const uint32_t tx = kGateA + (two ? 2u : 1u) * p.box_rows * 128u;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % nst, ph = (it / nst) & 1u;
      if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
      tc::mbar_expect_tx(&full[s], tx);
      tc::tma_load_2d(sA + s * kGateA, &tmX, &full[s], kb * 64, m0);
      tc::tma_load_2d(sB + s * p.b_stage, &tmW, &full[s], kb * 64, 0);
      if (two) tc::tma_load_2d(sB + s * p.b_stage + 256 * 128, &tmW, &full[s], kb * 64, 256);
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
      volatile int never = 0;
      const uint32_t first = it > nst ? it - nst : 0;
      for (uint32_t j = first; j < it; ++j)
        tc::mbar_wait(&full[j % nst], (j / nst) & 1u, &never);
    }
  } else if (warp == 1 && lane == 0) {
    uint32_t it = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % nst, ph = (it / nst) & 1u;
      if (!tc::mbar_wait(&full[s], ph, abort)) { ok = false; break; }
      tc::fence_after_sync();
      const uint64_t adesc = tc::sw128_kmajor_desc(tc::smem_u32(sA + s * kGateA));
      const uint64_t bdesc = tc::sw128_kmajor_desc(tc::smem_u32(sB + s * p.b_stage));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
        tc::mma_bf16(tmem, adesc + 2 * k, bdesc + 2 * k, p.idesc1, acc);
        if (two)
          tc::mma_bf16(tmem + 256, adesc + 2 * k, bdesc + 2 * k + ((256 * 128) >> 4), p.idesc2,
                       acc);
      }
      tc::commit(&empty[s]);
    }
    if (ok) {
      tc::commit(tfull);
    } else {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
    volatile int never = 0;
    tc::commit(drain);
    tc::mbar_wait(drain, 0, &never);
  } else if (warp >= 4) {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    if (tc::mbar_wait_warp(tfull, 0, abort)) {
      tc::fence_after_sync();
      const int row = m0 + r;
      float* out = p.part + ((size_t)ks * p.rows + row) * p.E;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
      const bool vec = (p.E & 3) == 0;
      for (int c = 0; c < p.E_pad; c += 32) {
        uint32_t v[32];
        tc::tmem_ld32(taddr + c, v);
        tc::tmem_ld_wait();
        if (row < p.rows) {
          if (vec && c + 32 <= p.E) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(out + c + 4 * i) =
                  make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c + i < p.E) out[c + i] = __uint_as_float(v[i]);
          }
        }
      }
    } else {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 2) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ------------------------------------------------------------ fused bf16 route
// Gate GEMM, softmax and grouped top-K in one launch. A cluster of CS CTAs owns one
// 128-row tile; CTA rank j accumulates the k-blocks [j nkb / CS, (j + 1) nkb / CS) of
// logits = x W_g^T in TMEM (M = 128, N = E_pad), with the same producer / MMA roles as
// gate_tc_kernel. Each rank's epilogue copies its partial logits into its own shared
// memory (the operand ring is free once its MMAs have completed); a cluster barrier
// (release / acquire) publishes them. Rank b then owns rows [b R, (b + 1) R), R = 128 /
// CS: its threads (512; 256 in the compact form) add the CS partials of those rows in
// rank order (the order in which the select kernels add the splits of the two-launch
// path), reading the other ranks' buffers through distributed shared memory, and select
// on the sums with L lanes per token (select_sub_row / select_group1_row: the same picks,
// order and weights as the select kernels). Partial logits never leave the chip, the
// reduction and the selection are spread over the cluster, and CS is chosen so that one
// wave of clusters covers the SMs.
//
// Shared-memory logit buffers (partials and sums) are row-major with a pitch of ncol + 4
// floats (ncol = E_pad rounded up to 32): a warp storing one 16-byte quad per row for 32
// rows touches every bank group once, a warp reading consecutive quads of one row is
// contiguous (locally and across the cluster), and the lanes of one token in the
// selection read consecutive words.
constexpr int kMaxFusedStages = 16;
// warps 0-7: producer, MMA, TMEM allocation, idle, 4 x TMEM readers; warps 8-15 join
// the reduction and the selection. With more row tiles than SMs the kernel runs 256
// threads and a 3-stage ring instead, so that two CTAs share an SM and one's selection
// overlaps the other's GEMM.
constexpr int kFusedThreads = 512;
constexpr int kFusedThreadsCompact = 256;

struct FusedRouteArgs {
  DeviceStatus* st;
  float* logits_out;  // nullable [rows, E]
  int32_t* topk_idx;  // [rows, K]
  float* topk_w;      // [rows, K]
  RouteSplitOut so;
  int rows, E, E_pad, nkb, K, H, renorm, CS;
  uint32_t idesc, b_stage, tmem_cols;
  uint32_t sum_off;   // byte offset of the summed-logit buffer (CS > 1)
  int stages;         // operand ring depth
  int threads;        // kFusedThreads, or kFusedThreadsCompact with more tiles than SMs
};

// byte offset of (row r, column c) in a logit buffer of the given pitch (floats)
__device__ __forceinline__ uint32_t row_off(int pitch, int r, int c) {
  return (uint32_t)((r * pitch + c) << 2);
}

// G1: grouped top-1 over 8 groups (E = L kPer, K = H = 8), else the general selection.
template <int L, int kPer, bool G1>
__global__ void __launch_bounds__(kFusedThreads, 1)
route_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const FusedRouteArgs p) {
  pdl_wait_and_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  const uint32_t nst = (uint32_t)p.stages;
  uint8_t* sB = base + nst * kGateA;
  // barriers after both the ring and the logit buffers
  const uint32_t ring = nst * (kGateA + p.b_stage);
  const int ncol = (p.E_pad + 31) & ~31;
  const int pitch = ncol + 4;
  const uint32_t bufs = p.CS > 1 ? p.sum_off + (uint32_t)pitch * (128u / p.CS) * 4u
                                 : (uint32_t)pitch * 512u;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + ((ring > bufs ? ring : bufs) + 7u) / 8u * 8u);
  uint64_t* empty = full + kMaxFusedStages;
  uint64_t* tfull = empty + kMaxFusedStages;
  uint64_t* drain = tfull + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t CS = (uint32_t)p.CS;
  const uint32_t rank = CS > 1 ? tc::cluster_rank() : 0u;
  const int m0 = (int)(blockIdx.x / CS) * 128;
  const int kb0 = (int)((long long)rank * p.nkb / CS);
  const int kb1 = (int)((long long)(rank + 1) * p.nkb / CS);
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < nst; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(drain, 1);
    *s_abort = 0;
    tc::mbar_init_fence();
    tc::tma_prefetch_map(&tmX);
    tc::tma_prefetch_map(&tmW);
  }
  if (warp == 2) {
    tc::tmem_alloc(s_tmem, p.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (CS > 1) tc::cluster_sync();  // every rank has started before any remote access
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  volatile int* abort = s_abort;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    uint32_t it = 0;
    bool ok = true;
    const uint32_t tx = kGateA + p.b_stage;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % nst, ph = (it / nst) & 1u;
      if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
      tc::mbar_expect_tx(&full[s], tx);
      tc::tma_load_2d(sA + s * kGateA, &tmX, &full[s], kb * 64, m0);
      tc::tma_load_2d(sB + s * p.b_stage, &tmW, &full[s], kb * 64, 0);
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
      volatile int never = 0;
      const uint32_t first = it > nst ? it - nst : 0;
      for (uint32_t j = first; j < it; ++j) tc::mbar_wait(&full[j % nst], (j / nst) & 1u, &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    uint32_t it = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % nst, ph = (it / nst) & 1u;
      if (!tc::mbar_wait(&full[s], ph, abort)) { ok = false; break; }
      tc::fence_after_sync();
      const uint64_t adesc = tc::sw128_kmajor_desc(tc::smem_u32(sA + s * kGateA));
      const uint64_t bdesc = tc::sw128_kmajor_desc(tc::smem_u32(sB + s * p.b_stage));
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16(tmem, adesc + 2 * k, bdesc + 2 * k, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
      tc::commit(&empty[s]);
    }
    if (ok) {
      tc::commit(tfull);
    } else {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
    volatile int never = 0;
    tc::commit(drain);
    tc::mbar_wait(drain, 0, &never);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- TMEM -> partials
    // (tcgen05.ld is warp-collective: the decision before it is warp-uniform)
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(tfull, 0, abort));
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
    tc::fence_after_sync();
    if (ok) {
      const int r = (warp & 3) * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      for (int c = 0; c < ncol; c += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + c, u);
        tc::tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<float4*>(base + row_off(pitch, r, c + 4 * g)) =
              make_float4(__uint_as_float(u[4 * g]), __uint_as_float(u[4 * g + 1]),
                          __uint_as_float(u[4 * g + 2]), __uint_as_float(u[4 * g + 3]));
      }
    }
  }
  // every rank's partials are in its shared memory: the cluster barrier publishes them
  tc::fence_before_sync();
  __syncthreads();
  if (CS > 1) tc::cluster_sync();
  tc::fence_after_sync();

  if (!*abort) {
    const int R = 128 / (int)CS;         // rows owned by this rank
    const int r0 = (int)rank * R;        // first of them within the tile
    const int E = p.E;
    // ------------------------------------------------------------------ sums of partials
    // item = (row rr, column quad c4), c4 fastest: the rank's rows, partials added in rank
    // order; logits_out written from the sums. With CS = 1 the partials are the sums.
    uint32_t sbuf = 0;  // byte offset of the sums from base
    int sr0 = r0;
    if (CS > 1) {
      sbuf = p.sum_off;
      sr0 = 0;
    }
    const int nq = ncol >> 2;
    for (int item = threadIdx.x; item < R * nq; item += (int)blockDim.x) {
      const int rr = item / nq, c4 = item % nq;
      float4 a;
      if (CS == 1) {
        a = *reinterpret_cast<const float4*>(base + row_off(pitch, rr, 4 * c4));
      } else {
        a = tc::ld_cluster_v4(tc::cluster_addr(base, 0) + row_off(pitch, r0 + rr, 4 * c4));
      }
      for (uint32_t j = 1; j < CS; ++j) {
        const float4 b = tc::ld_cluster_v4(tc::cluster_addr(base, j) + row_off(pitch, r0 + rr, 4 * c4));
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (CS > 1) *reinterpret_cast<float4*>(base + sbuf + row_off(pitch, rr, 4 * c4)) = a;
      const int t = m0 + r0 + rr;
      if (t < p.rows && p.logits_out) {
        float* lo = p.logits_out;
        int to = t;
        if (t >= p.so.split) {
          lo = p.so.logits;
          to = t - p.so.split;
        }
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (4 * c4 + u < E) lo[(size_t)to * E + 4 * c4 + u] = av[u];
      }
    }
    __syncthreads();
    // ------------------------------------------------------------------ selection
    const int j = threadIdx.x & (L - 1);
    for (int rr0 = 0; rr0 < R; rr0 += (int)blockDim.x / L) {
      const int rr = rr0 + (int)threadIdx.x / L;
      const bool in = rr < R;
      float v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = j + L * i;
        v[i] = (in && e < E) ? *reinterpret_cast<const float*>(
                                   base + sbuf + row_off(pitch, sr0 + rr, e))
                             : -INFINITY;
      }
      int pick_i;
      float pick_w;
      if constexpr (G1)
        select_group1_row<L, 8, kPer / 8>(v, j, p.renorm, pick_i, pick_w);
      else
        select_sub_row<L, kPer>(v, j, E, p.K, p.H, p.renorm, pick_i, pick_w);
      const int t = m0 + r0 + rr;
      if (in && t < p.rows && j < p.K) {
        int32_t* oi = p.topk_idx;
        float* ow = p.topk_w;
        int to = t;
        if (t >= p.so.split) {
          oi = p.so.idx;
          ow = p.so.w;
          to = t - p.so.split;
        }
        oi[(size_t)to * p.K + j] = pick_i;
        ow[(size_t)to * p.K + j] = pick_w;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (CS > 1) tc::cluster_sync();  // no rank leaves while another still reads its partials
  tc::fence_after_sync();
  if (warp == 2) tc::tmem_dealloc(tmem, p.tmem_cols);
}


}  // namespace

namespace {

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 152;
}

// The fused kernel takes bf16 layers with E <= 256 (one MMA of N = E rounded up to 16)
// and K no larger than the lanes per token of its selection (8 for E <= 128, else 16).
bool fused_route_ok(const smoe_desc& d) {
  return d.dtype == SMOE_BF16 && d.E <= 256 && d.K <= (d.E <= 128 ? 8 : 16);
}

// Cluster size: the largest power of two of k-splits that keeps one wave of clusters on
// the SMs, at most 8 (the portable cluster size) and with at least 2 k-blocks per split.
int fused_route_cs(const smoe_desc& d, int rows) {
  const int mt = ceil_div(rows, 128);
  const int nkb = ceil_div(d.d, 64);
  const int lim = std::min(std::min(device_sms() / std::max(mt, 1), nkb / 2), 8);
  int cs = 1;
  while (cs * 2 <= lim) cs *= 2;
  return cs;
}

template <int L, int kPer, bool G1 = false>
cudaError_t launch_fused(const CUtensorMap& tX, const CUtensorMap& tW, const FusedRouteArgs& a,
                         int tiles, size_t smem, cudaStream_t s) {
  auto kern = route_fused_kernel<L, kPer, G1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * a.CS);
  cfg.blockDim = dim3(a.threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.CS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.CS > 1 ? 2 : 1;
  SMOE_COUNT_LAUNCH(1);
  return cudaLaunchKernelEx(&cfg, kern, tX, tW, a);
}

cudaError_t launch_route_fused(const smoe_desc& d, int rows, const void* x, const void* w_gate,
                               float* logits_out, int32_t* topk_idx, float* topk_w, void* ws,
                               cudaStream_t s, RouteSplitOut so) {
  WsLayout L;
  ws_layout(d, &L);
  FusedRouteArgs a;
  a.st = ws_ptr<DeviceStatus>(ws, L.status);
  a.logits_out = logits_out;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.so = so;
  a.rows = rows;
  a.E = d.E;
  a.E_pad = (d.E + 15) / 16 * 16;
  a.nkb = ceil_div(d.d, 64);
  a.K = d.K;
  a.H = d.H;
  a.renorm = d.renorm;
  a.CS = fused_route_cs(d, rows);
  a.idesc = tc::instr_desc(false, 128, a.E_pad);
  a.b_stage = (uint32_t)a.E_pad * 128u;
  a.tmem_cols = 32;
  while (a.tmem_cols < (uint32_t)a.E_pad) a.tmem_cols <<= 1;
  // shared memory: the operand ring, as deep as fits (the loads of a split are few and
  // latency-bound, so every stage in flight counts), reused after the MMAs for the
  // 128-row partial buffer and (CS > 1) the R-row buffer of sums; then the barriers
  const uint32_t ncol = ((uint32_t)a.E_pad + 31u) & ~31u;
  const uint32_t stage = kGateA + a.b_stage;
  const uint32_t budget = 227u * 1024u - 1024u - 8u * (2u * kMaxFusedStages + 2u) - 16u;
  const int kb_split = ceil_div(a.nkb, a.CS);
  const bool compact = ceil_div(rows, 128) > device_sms();
  a.threads = compact ? kFusedThreadsCompact : kFusedThreads;
  a.stages = (int)std::min<uint32_t>(std::min<uint32_t>(budget / stage, kMaxFusedStages),
                                     (uint32_t)std::max(kb_split, 2));
  if (compact) a.stages = std::min(a.stages, 3);
  const uint32_t ring = (uint32_t)a.stages * stage;
  const uint32_t pitch = ncol + 4u;  // floats per row of a logit buffer
  a.sum_off = pitch * 512u;
  const uint32_t bufs = a.CS > 1 ? a.sum_off + pitch * (128u / (uint32_t)a.CS) * 4u : pitch * 512u;
  const uint32_t body = (std::max(ring, bufs) + 7u) / 8u * 8u;
  if (a.stages < 2 || body > budget) return cudaErrorInvalidValue;
  const size_t smem = 1024 + body + 8u * (2u * kMaxFusedStages + 2u) + 16u;
  alignas(64) CUtensorMap tX, tW;
  if (!encode_tmap_2d(&tX, x, false, rows, d.d, 128, 64)) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tW, w_gate, false, d.E, d.d, (uint32_t)a.E_pad, 64))
    return cudaErrorInvalidValue;
  const int tiles = ceil_div(rows, 128);
  if (d.H == 8 && d.K == 8) {  // grouped top-1 (FoE's top-K/H = 1)
    if (d.E == 64) return launch_fused<8, 8, true>(tX, tW, a, tiles, smem, s);
    if (d.E == 128) return launch_fused<8, 16, true>(tX, tW, a, tiles, smem, s);
    if (d.E == 256) return launch_fused<16, 16, true>(tX, tW, a, tiles, smem, s);
  }
  if (d.E <= 32) return launch_fused<8, 4>(tX, tW, a, tiles, smem, s);
  if (d.E <= 64) return launch_fused<8, 8>(tX, tW, a, tiles, smem, s);
  if (d.E <= 128) return launch_fused<8, 16>(tX, tW, a, tiles, smem, s);
  // 16 lanes per token and only the value slots the experts fill (E = 160: 10 of 16)
  if (d.E <= 160) return launch_fused<16, 10>(tX, tW, a, tiles, smem, s);
  return launch_fused<16, 16>(tX, tW, a, tiles, smem, s);
}

}  // namespace

int route_splits(const smoe_desc& d, int rows) {
  if (d.dtype == SMOE_F32) return 1;
  const int mt = ceil_div(rows, 128);
  const int nkb = ceil_div(d.d, 64);
  int ks = ceil_div(160, mt);   // enough (row tile, split) CTAs to cover the SMs once
  ks = std::min(ks, std::max(1, nkb / 2));
  return std::max(1, std::min(ks, 16));
}

cudaError_t launch_route(const smoe_desc& d, int rows, const void* x, const void* w_gate,
                         const float* logits_in, float* logits_out, int32_t* topk_idx,
                         float* topk_w, void* ws, cudaStream_t s, RouteSplitOut so) {
  if (!logits_in && fused_route_ok(d)) {
    const cudaError_t e =
        launch_route_fused(d, rows, x, w_gate, logits_out, topk_idx, topk_w, ws, s, so);
    if (e == cudaSuccess) return e;
    // a cluster shape the device cannot schedule (e.g. a partitioned GPU) is rejected at
    // launch, before anything runs: take the two-launch path instead
    if (e != cudaErrorInvalidClusterSize && e != cudaErrorLaunchOutOfResources) return e;
    (void)cudaGetLastError();
  }
  const float* part = logits_in;
  int KS = 1;
  if (!logits_in) {
    WsLayout L;
    ws_layout(d, &L);
    float* pbuf = ws_ptr<float>(ws, L.route_part);
    part = pbuf;
    if (d.dtype == SMOE_F32) {
      dim3 grid(ceil_div(rows, kBM), ceil_div(d.E, kBN));
      SMOE_LAUNCH(gate_gemm_f32_kernel, grid, 256, 0, s, static_cast<const float*>(x),
          static_cast<const float*>(w_gate), pbuf, rows, d.d, d.E);
    } else {
      KS = route_splits(d, rows);
      const int E_pad = (d.E + 15) / 16 * 16;
      GateArgs a;
      a.part = pbuf;
      a.st = ws_ptr<DeviceStatus>(ws, L.status);
      a.rows = rows;
      a.E = d.E;
      a.E_pad = E_pad;
      a.nkb = ceil_div(d.d, 64);
      a.KS = KS;
      a.idesc1 = tc::instr_desc(false, 128, std::min(E_pad, 256));
      a.idesc2 = E_pad > 256 ? tc::instr_desc(false, 128, E_pad - 256) : 0u;
      a.box_rows = E_pad > 256 ? 256u : (uint32_t)E_pad;
      a.b_stage = E_pad > 256 ? 65536u : (uint32_t)E_pad * 128u;
      a.tmem_cols = 32;
      while (a.tmem_cols < (uint32_t)E_pad) a.tmem_cols <<= 1;
      alignas(64) CUtensorMap tX, tW;
      if (!encode_tmap_2d(&tX, x, false, rows, d.d, 128, 64)) return cudaErrorInvalidValue;
      if (!encode_tmap_2d(&tW, w_gate, false, d.E, d.d, a.box_rows, 64))
        return cudaErrorInvalidValue;
      a.stages = E_pad > 256 ? 2u : 3u;
      const size_t smem = 1024 + a.stages * (kGateA + a.b_stage) + 128;
      cudaError_t e = cudaFuncSetAttribute(gate_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      dim3 grid(ceil_div(rows, 128), KS);
      SMOE_LAUNCH(gate_tc_kernel, grid, 256, smem, s, tX, tW, a);
    }
  }
  float* lo = logits_out == logits_in ? nullptr : logits_out;
  const long long stride = (long long)rows * d.E;
  if (d.H == 8 && d.K == 8 && (d.E == 64 || d.E == 128 || d.E == 256)) {
    const int grid = ceil_div(rows * 8, 256);
    if (d.E == 64)
      SMOE_LAUNCH((select_group1_kernel<8, 8, 1>), grid, 256, 0, s, part, KS, stride, lo, rows,
                  d.renorm, topk_idx, topk_w, so);
    else if (d.E == 128)
      SMOE_LAUNCH((select_group1_kernel<8, 8, 2>), grid, 256, 0, s, part, KS, stride, lo, rows,
                  d.renorm, topk_idx, topk_w, so);
    else
      SMOE_LAUNCH((select_group1_kernel<8, 8, 4>), grid, 256, 0, s, part, KS, stride, lo, rows,
                  d.renorm, topk_idx, topk_w, so);
    return cudaGetLastError();
  }
  if (d.K <= 8 && d.E <= 128) {
    const int grid = ceil_div(rows * 8, 256);
    if (d.E <= 32)
      SMOE_LAUNCH((select_sub_kernel<8, 4>), grid, 256, 0, s, part, KS, stride, lo, rows, d.E,
                  d.K, d.H, d.renorm, topk_idx, topk_w, so);
    else if (d.E <= 64)
      SMOE_LAUNCH((select_sub_kernel<8, 8>), grid, 256, 0, s, part, KS, stride, lo, rows, d.E,
                  d.K, d.H, d.renorm, topk_idx, topk_w, so);
    else
      SMOE_LAUNCH((select_sub_kernel<8, 16>), grid, 256, 0, s, part, KS, stride, lo, rows, d.E,
                  d.K, d.H, d.renorm, topk_idx, topk_w, so);
    return cudaGetLastError();
  }
  if (d.K <= 16 && d.E <= 160) {
    SMOE_LAUNCH((select_sub_kernel<16, 10>), ceil_div(rows * 16, 256), 256, 0, s, part, KS,
                stride, lo, rows, d.E, d.K, d.H, d.renorm, topk_idx, topk_w, so);
    return cudaGetLastError();
  }
  if (d.K <= 16 && d.E <= 256) {
    SMOE_LAUNCH((select_sub_kernel<16, 16>), ceil_div(rows * 16, 256), 256, 0, s, part, KS,
                stride, lo, rows, d.E, d.K, d.H, d.renorm, topk_idx, topk_w, so);
    return cudaGetLastError();
  }
  const dim3 grid(ceil_div(rows, kSelWarps)), block(kSelWarps * 32);
  if (d.E <= 128)
    SMOE_LAUNCH(select_kernel<4>, grid, block, 0, s, part, KS, stride, lo, rows, d.E, d.K, d.H,
        d.renorm, topk_idx, topk_w, so);
  else if (d.E <= 256)
    SMOE_LAUNCH(select_kernel<8>, grid, block, 0, s, part, KS, stride, lo, rows, d.E, d.K, d.H,
        d.renorm, topk_idx, topk_w, so);
  else
    SMOE_LAUNCH(select_kernel<16>, grid, block, 0, s, part, KS, stride, lo, rows, d.E, d.K, d.H,
        d.renorm, topk_idx, topk_w, so);
  return cudaGetLastError();
}

}  // namespace smoe
