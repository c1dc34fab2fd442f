// Predicted-partition lookup, stable counting sorts (token shuffle and expert
// dispatch), row gathers and local-activation counts.
//
// "Speculative MoE" §3.1 (s-TS: move each token ahead of time to the partition of
// its predicted experts), §4.1 (C_p = Pr(E_k | token) looked up by token id), §1
// (EP dispatch into the experts' devices), §2/§7 (local activation rate), and the
// FoE article's grouped layout for the source partition of a token copy.
//
// A counting sort is three launches with no inter-CTA waiting: per-tile bucket
// histograms, one CTA scanning the (bucket, tile) table, and a scatter that ranks
// each tile's elements stably (warp match + per-warp counts in shared memory). The
// shuffle's histogram columns are the predict kernel's 32-token CTAs (written
// directly, nothing to clear) and its scatter tiles 64 tokens; the dispatch's tiles are
// 256 to 1024 (token, expert) pairs, chosen per layer.
#include <algorithm>
#include <mutex>

#include <cuda.h>

#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBuckets = 512;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ------------------------------------------------------------------ predict
// 32 tokens per CTA (a 256-token shuffle tile spans 8 CTAs). The CTA stages the 32 C_p
// rows in shared memory with 16-byte loads all in flight at once, warp 0 lists each
// partition's experts in ascending order (warp match), then each warp scores 32 / P2
// tokens side by side (P2 = P rounded up to a power of two lanes per token): lane p
// adds its partition's row entries in that order (one fp32 add each, the oracle's
// order), and a butterfly argmax over the token's lanes with the order (score
// descending, partition ascending) picks pred[t]. The CTA's partition counts are added
// to its tile's histogram entries (which the launcher zeroes first).
constexpr int kPredTokens = kShufHistTokens;
constexpr int kShufScatter = 64;  // tokens per scatter CTA of the shuffle

// INTER: the inter-layer source of "Speculative MoE" §4.1 also votes. prev[t] is the
// token's cluster at the previous layer and table_a [P, P] the 2-gram table A; A's row
// maximum (first maximum) replaces the intra-layer pick when it is strictly larger than
// the intra-layer confidence (best partition score / K, an IEEE fp32 division).
template <bool INTER>
__global__ void __launch_bounds__(kThreads)
predict_hist_kernel(const int32_t* __restrict__ ids, const float* __restrict__ conf,
                    const int32_t* __restrict__ emap, int T, int E, int P, int vocab,
                    int32_t* __restrict__ pred, int32_t* __restrict__ hist, int ntiles,
                    int tile, DeviceStatus* st, const int32_t* __restrict__ prev,
                    const float* __restrict__ table_a, int K) {
  pdl_wait_and_trigger();
  extern __shared__ float s_rows[];          // [kPredTokens, E]
  __shared__ int s_map[kMaxBuckets];
  __shared__ int s_list[kMaxBuckets];
  __shared__ int s_start[33];
  __shared__ int s_fill[32];
  __shared__ int s_cnt[32];
  __shared__ int s_id[kPredTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kPredTokens;
  const int n = min(kPredTokens, T - t0);
  for (int e = tid; e < E; e += kThreads) {
    const int p = emap[e];
    const bool ok = (unsigned)p < (unsigned)P;
    if (!ok && blockIdx.x == 0) record_error(st, kStatusData, kBadExpertPart, e);
    s_map[e] = ok ? p : -1;
  }
  if (tid < 32) { s_cnt[tid] = 0; s_fill[tid] = 0; }
  if (tid < n) {
    const int id = ids[t0 + tid];
    const bool ok = (unsigned)id < (unsigned)vocab;
    if (!ok) record_error(st, kStatusData, kBadTokenId, t0 + tid);
    s_id[tid] = ok ? id : -1;
  }
  __syncthreads();
  if ((E & 3) == 0) {
    const int q = E >> 2;  // 16-byte vectors per row
    const int nv = n * q;
    float4* dst = reinterpret_cast<float4*>(s_rows);
#pragma unroll 4
    for (int k = tid; k < nv; k += kThreads) {
      const int i = k / q, c = k - i * q;
      const int id = s_id[i];
      dst[k] = id >= 0 ? __ldg(reinterpret_cast<const float4*>(conf + (size_t)id * E) + c)
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  } else {
#pragma unroll 4
    for (int k = tid; k < n * E; k += kThreads) {
      const int i = k / E, e = k - i * E;
      const int id = s_id[i];
      s_rows[k] = id >= 0 ? __ldg(conf + (size_t)id * E + e) : 0.0f;
    }
  }
  if (warp == 0) {
    // partition p's experts in ascending order: s_list[s_start[p] .. s_start[p+1])
    for (int c = 0; c < E; c += 32) {
      const int e = c + lane;
      const int p = e < E ? s_map[e] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (p >= 0 && (peers & lanemask_lt()) == 0) s_fill[p] += __popc(peers);
      __syncwarp();
    }
    const int cnt = lane < P ? s_fill[lane] : 0;
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    __syncwarp();
    if (lane < P) { s_start[lane] = incl - cnt; s_fill[lane] = incl - cnt; }
    if (lane == P - 1) s_start[P] = incl;
    __syncwarp();
    for (int c = 0; c < E; c += 32) {
      const int e = c + lane;
      const int p = e < E ? s_map[e] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      const int rank = __popc(peers & lanemask_lt());
      if (p >= 0) s_list[s_fill[p] + rank] = e;
      __syncwarp();
      if (p >= 0 && rank == 0) s_fill[p] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  int P2 = 1;
  while (P2 < P) P2 <<= 1;
  const int G = 32 / P2;                       // tokens per warp pass
  const int sub = lane / P2, pl = lane - sub * P2;
  for (int i0 = warp * G; i0 < n; i0 += kWarps * G) {
    const int i = i0 + sub;
    const bool tok = i < n;
    float sc = -INFINITY;
    if (tok && pl < P) {
      const float* row = s_rows + (size_t)i * E;
      const int j1 = s_start[pl + 1];
      float acc = 0.0f;
#pragma unroll 4
      for (int j = s_start[pl]; j < j1; ++j) acc = acc + row[s_list[j]];
      sc = acc;
    }
    int bi = pl;
    for (int off = P2 >> 1; off; off >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, sc, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (os > sc || (os == sc && oi < bi)) { sc = os; bi = oi; }
    }
    // an invalid id, or a NaN/inf row (outside the contract), gives partition 0
    const bool id_ok = tok && s_id[i] >= 0;
    int best = (id_ok && (unsigned)bi < (unsigned)P) ? bi : 0;
    if (INTER) {
      int c = 0;
      if (id_ok) {
        c = prev[t0 + i];
        if ((unsigned)c >= (unsigned)P) {
          if (pl == 0) record_error(st, kStatusData, kBadSrcPart, t0 + i);
          c = 0;
        }
      }
      float av = (id_ok && pl < P) ? table_a[c * P + pl] : -INFINITY;
      int ai = pl;
      for (int off = P2 >> 1; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, av, off);
        const int oi = __shfl_xor_sync(0xffffffffu, ai, off);
        if (ov > av || (ov == av && oi < ai)) { av = ov; ai = oi; }
      }
      const float conf_intra = sc / (float)K;
      if (id_ok && av > conf_intra && (unsigned)ai < (unsigned)P) best = ai;
    }
    if (tok && pl == 0) {
      pred[t0 + i] = best;
      atomicAdd(&s_cnt[best], 1);
    }
  }
  __syncthreads();
  // tile == kPredTokens: this CTA's counts are its own histogram column (no zeroing
  // needed); larger tiles: added into the tile's column, which the launcher zeroes
  if (tile == kPredTokens) {
    if (tid < P) hist[tid * ntiles + blockIdx.x] = s_cnt[tid];
  } else if (tid < P && s_cnt[tid] > 0) {
    atomicAdd(&hist[tid * ntiles + t0 / tile], s_cnt[tid]);
  }
}

size_t predict_smem(int E) { return sizeof(float) * kPredTokens * E; }

// ------------------------------------------------------------------ dispatch hist
// Pairs q = s K + k in shuffled-slot order; bucket = expert idx[perm[s], k].
__global__ void __launch_bounds__(kThreads)
dispatch_hist_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ perm, int T,
                     int K, int E, int32_t* __restrict__ bucket, int32_t* __restrict__ hist,
                     int ntiles, int tile, DeviceStatus* st) {
  pdl_wait_and_trigger();
  __shared__ int s_cnt[kMaxBuckets];
  const int tid = threadIdx.x;
  for (int b = tid; b < E; b += kThreads) s_cnt[b] = 0;
  __syncthreads();
  const long long n = (long long)T * K;
  const long long q0 = (long long)blockIdx.x * tile;
  const long long q1 = min(q0 + tile, n);
#pragma unroll 4
  for (long long q = q0 + tid; q < q1; q += kThreads) {
    const int s = (int)(q / K), k = (int)(q - (long long)s * K);
    const int t = perm ? perm[s] : s;
    int e = 0;
    if ((unsigned)t >= (unsigned)T) {
      record_error(st, kStatusData, kBadPerm, s);
    } else {
      e = idx[(size_t)t * K + k];
      if ((unsigned)e >= (unsigned)E) {
        record_error(st, kStatusData, kBadTopkIdx, (long long)t * K + k);
        e = 0;
      }
    }
    bucket[q] = e;
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int b = tid; b < E; b += kThreads) hist[b * ntiles + blockIdx.x] = s_cnt[b];
}

// ------------------------------------------------------------------ scan
// One CTA: exclusive scan of the bucket-major (bucket, tile) histogram, giving each
// tile's first output position per bucket; bucket_off[b] = start of bucket b.
__global__ void __launch_bounds__(1024)
scan_kernel(const int32_t* __restrict__ hist, int32_t* __restrict__ offs, int L, int B,
            int ntiles, int n, int32_t* __restrict__ bucket_off) {
  pdl_wait_and_trigger();
  // rounds of 4096 entries: each thread loads 4 consecutive counts with one 16-byte
  // load, the block scans the per-thread sums, a running carry links the rounds
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (int base = 0; base < L; base += 4096) {
    const int i = base + tid * 4;
    int v[4] = {0, 0, 0, 0};
    if (i + 3 < L) {
      const int4 q = *reinterpret_cast<const int4*>(hist + i);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j < L) v[j] = hist[i + j];
    }
    const int sum = v[0] + v[1] + v[2] + v[3];
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    int run = carry + x - sum + (warp > 0 ? s_warp[warp - 1] : 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i + j < L) offs[i + j] = run;
      run += v[j];
    }
    carry += s_warp[31];
    __syncthreads();
  }
  for (int b = tid; b < B; b += blockDim.x) bucket_off[b] = offs[b * ntiles];
  if (tid == 0) bucket_off[B] = n;
}

// ------------------------------------------------------------------ scatter
// Stable rank of every element of a tile within its bucket: chunks of kThreads
// elements in index order; inside a chunk, warps in order, inside a warp, lanes in
// order (warp match gives the peers of equal bucket). A scatter tile may span
// col_stride consecutive histogram columns: its running start per bucket is the scanned
// offset of its first column.
enum ScatterMode { kShuffle = 0, kDispatch = 1 };

template <int MODE, int MAXB = kMaxBuckets>
__global__ void __launch_bounds__(kThreads)
scatter_kernel(const int32_t* __restrict__ bucket, int n, int B, int ntiles, int tile,
               int col_stride, const int32_t* __restrict__ offs,
               // kShuffle: perm_out[pos] = i
               int32_t* __restrict__ perm_out,
               // kDispatch
               const int32_t* __restrict__ perm_in, int T, int K, int32_t* __restrict__ pair_row,
               int32_t* __restrict__ row_token, int32_t* __restrict__ row_src) {
  pdl_wait_and_trigger();
  __shared__ int s_run[MAXB];
  __shared__ int s_wc[kWarps][MAXB];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int b = tid; b < B; b += kThreads) {
    s_run[b] = offs[b * ntiles + blockIdx.x * col_stride];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_wc[w][b] = 0;
  }
  __syncthreads();
  const int base = blockIdx.x * tile;
  for (int c = 0; c < tile && base + c < n; c += kThreads) {
    const int i = base + c + tid;
    const bool valid = i < n && c + tid < tile;
    const int b = valid ? bucket[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    const int rank = __popc(peers & lanemask_lt());
    if (valid && rank == 0) s_wc[warp][b] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pos = s_run[b] + rank;
      for (int w = 0; w < warp; ++w) pos += s_wc[w][b];
      if (MODE == kShuffle) {
        perm_out[pos] = i;
      } else {
        const int s = i / K, k = i - s * K;
        const int t = perm_in ? perm_in[s] : s;
        const bool tok_ok = (unsigned)t < (unsigned)T;
        if (tok_ok) pair_row[(size_t)t * K + k] = pos;
        row_token[pos] = tok_ok ? t : -1;
        row_src[pos] = s;
      }
    }
    __syncthreads();
    for (int bb = tid; bb < B; bb += kThreads) {
      int sum = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        sum += s_wc[w][bb];
        s_wc[w][bb] = 0;
      }
      s_run[bb] += sum;
    }
    __syncthreads();
  }
  (void)lane;
}

// ------------------------------------------------------------------ row gather
// dst[r] = src[map[r]] for 16-byte-aligned rows; one warp per row, eight 16-byte
// loads in flight per lane (four for the last part of a row).
__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                   const int32_t* __restrict__ map, int nrows, int nsrc, int vec_per_row,
                   DeviceStatus* st) {
  pdl_wait_and_trigger();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nw = (gridDim.x * kThreads) >> 5;
  for (int r = gw; r < nrows; r += nw) {
    const int s = map[r];
    uint4* out = dst + (size_t)r * vec_per_row;
    if ((unsigned)s >= (unsigned)nsrc) {
      if (lane == 0) record_error(st, kStatusData, kBadPerm, r);
      for (int v = lane; v < vec_per_row; v += 32) out[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* in = src + (size_t)s * vec_per_row;
    int v = lane;
    for (; v + 224 < vec_per_row; v += 256) {
      uint4 t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) t[u] = __ldg(in + v + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) out[v + 32 * u] = t[u];
    }
    for (; v + 96 < vec_per_row; v += 128) {
      const uint4 a = __ldg(in + v), b = __ldg(in + v + 32), c = __ldg(in + v + 64),
                  d = __ldg(in + v + 96);
      out[v] = a; out[v + 32] = b; out[v + 64] = c; out[v + 96] = d;
    }
    for (; v < vec_per_row; v += 32) out[v] = __ldg(in + v);
  }
}

// The shuffle's row copy and the dispatch's row copy from one read of x ("Speculative
// MoE" §3.1 s-TS and §1 dispatch): for slot s and its token t = perm[s] (t = s without a
// shuffle), x_shuf[s] = x[t] and X_disp[pair_row[t, k]] = x[t] for k < K. The rows the
// dispatch would read back from x_shuf are written while x[t] is in registers. One warp
// per slot, eight 16-byte loads in flight per lane, each stored to the token's 1 + K rows.
__global__ void __launch_bounds__(kThreads)
shuffle_dispatch_rows_kernel(const uint4* __restrict__ x, uint4* __restrict__ x_shuf,
                             uint4* __restrict__ x_disp, const int32_t* __restrict__ perm,
                             const int32_t* __restrict__ pair_row, int T, int K, int vec,
                             DeviceStatus* st) {
  pdl_wait_and_trigger();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nw = (gridDim.x * kThreads) >> 5;
  const int TK = T * K;
  for (int s = gw; s < T; s += nw) {
    const int t = perm ? perm[s] : s;
    uint4* out0 = x_shuf ? x_shuf + (size_t)s * vec : nullptr;
    if ((unsigned)t >= (unsigned)T) {
      if (lane == 0) record_error(st, kStatusData, kBadPerm, s);
      if (out0)
        for (int v = lane; v < vec; v += 32) out0[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    int my_row = -1;  // lane k < K: the dispatched row of pair (t, k)
    if (lane < K) {
      const int r = pair_row[(size_t)t * K + lane];
      if ((unsigned)r < (unsigned)TK)
        my_row = r;
      else
        record_error(st, kStatusData, kBadPairRow, t * K + lane);
    }
    const uint4* in = x + (size_t)t * vec;
    // every lane takes every chunk (the shuffles below span the warp), whatever the row
    // length; lane + 32 u past the row does nothing
    for (int c0 = 0; c0 < vec; c0 += 256) {
      const int v0 = c0 + lane;
      uint4 tv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (v0 + 32 * u < vec) tv[u] = __ldg(in + v0 + 32 * u);
      if (out0) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v0 + 32 * u < vec) out0[v0 + 32 * u] = tv[u];
      }
      for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, my_row, k);
        if (r < 0) continue;
        uint4* o = x_disp + (size_t)r * vec;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v0 + 32 * u < vec) o[v0 + 32 * u] = tv[u];
      }
    }
  }
}

// ------------------------------------------------------------------ EP exchange
// "Speculative MoE" §1: under expert parallelism a token travels from its device to
// the devices of its K experts. Pairs q = t K + k in token order are bucketed by
// (dst device, src device): bucket = dst P + src, dst = map[idx[t, k]], src =
// src_part[t] or the contiguous split floor(t P / T). A stable counting sort over
// these P^2 buckets lays the pairs out as P concatenated receive buffers (device 0
// first), each holding its sources' segments in source order and, inside a segment,
// the source's (t, k) order.
constexpr int kMaxExchangeBuckets = 1024;   // P <= 32

__global__ void __launch_bounds__(kThreads)
exchange_hist_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ src_part,
                     const int32_t* __restrict__ emap, int T, int K, int E, int P,
                     int32_t* __restrict__ bucket, int32_t* __restrict__ hist, int ntiles,
                     int tile, DeviceStatus* st) {
  pdl_wait_and_trigger();
  __shared__ int s_cnt[kMaxExchangeBuckets];
  __shared__ int s_map[kMaxBuckets];
  const int tid = threadIdx.x;
  const int B = P * P;
  for (int b = tid; b < B; b += kThreads) s_cnt[b] = 0;
  for (int e = tid; e < E; e += kThreads) {
    const int p = emap[e];
    const bool ok = (unsigned)p < (unsigned)P;
    if (!ok && blockIdx.x == 0) record_error(st, kStatusData, kBadExpertPart, e);
    s_map[e] = ok ? p : 0;
  }
  __syncthreads();
  // T K <= INT_MAX / 2 (checked on the host)
  const int n = T * K;
  const int q0 = blockIdx.x * tile;
  const int q1 = min(q0 + tile, n);
#pragma unroll 4
  for (int q = q0 + tid; q < q1; q += kThreads) {
    const int t = q / K;
    int src;
    if (src_part) {
      src = src_part[t];
      if ((unsigned)src >= (unsigned)P) {
        record_error(st, kStatusData, kBadSrcPart, t);
        src = 0;
      }
    } else {
      src = (int)(((long long)t * P) / T);
    }
    int e = idx[q];
    if ((unsigned)e >= (unsigned)E) {
      record_error(st, kStatusData, kBadTopkIdx, q);
      e = 0;
    }
    const int b = s_map[e] * P + src;
    bucket[q] = b;
    atomicAdd(&s_cnt[b], 1);
  }
  __syncthreads();
  for (int b = tid; b < B; b += kThreads) hist[b * ntiles + blockIdx.x] = s_cnt[b];
}

// send_counts[p P + q] = pairs from device p to device q: the length of receive
// segment (dst q, src p).
__global__ void __launch_bounds__(kThreads)
send_counts_kernel(const int32_t* __restrict__ recv_off, int P, int32_t* __restrict__ counts) {
  pdl_wait_and_trigger();
  for (int i = threadIdx.x; i < P * P; i += kThreads) {
    const int p = i / P, q = i - p * P;
    counts[i] = recv_off[q * P + p + 1] - recv_off[q * P + p];
  }
}

// SRS ("Speculative MoE" §3.1): x_shuf[s] = sum_r x_parts[r][perm[s]], the R
// tensor-parallel partials added in fp32 in rank order and written in slot order.
// One warp per output row, 16-byte vectors, up to four ranks' loads in flight.
template <typename TE>
__global__ void __launch_bounds__(kThreads)
srs_kernel(const uint4* __restrict__ parts, uint4* __restrict__ out,
           const int32_t* __restrict__ perm, int T, int R, int vec_per_row,
           DeviceStatus* st) {
  pdl_wait_and_trigger();
  constexpr int V = Elem<TE>::kPerVec16;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nw = (gridDim.x * kThreads) >> 5;
  const size_t plane = (size_t)T * vec_per_row;
  for (int srow = gw; srow < T; srow += nw) {
    const int t = perm[srow];
    uint4* o = out + (size_t)srow * vec_per_row;
    if ((unsigned)t >= (unsigned)T) {
      if (lane == 0) record_error(st, kStatusData, kBadPerm, srow);
      for (int v = lane; v < vec_per_row; v += 32) o[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* in = parts + (size_t)t * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) {
      float acc[V];
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = 0.0f;
      int r = 0;
      for (; r + 4 <= R; r += 4) {
        uint4 u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = __ldg(in + (size_t)(r + i) * plane + v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float f[V];
          unpack16(u[i], f, (const TE*)nullptr);
#pragma unroll
          for (int j = 0; j < V; ++j) acc[j] += f[j];
        }
      }
      for (; r < R; ++r) {
        float f[V];
        unpack16(__ldg(in + (size_t)r * plane + v), f, (const TE*)nullptr);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] += f[j];
      }
      o[v] = pack16(acc, (const TE*)nullptr);
    }
  }
}

// SAG ("Speculative MoE" §3.1): rows held in slot order back to token order,
// dst[perm[s]] = src[s]; one warp per row, eight 16-byte loads in flight per lane.
__global__ void __launch_bounds__(kThreads)
scatter_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                    const int32_t* __restrict__ perm, int nrows, int vec_per_row,
                    DeviceStatus* st) {
  pdl_wait_and_trigger();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nw = (gridDim.x * kThreads) >> 5;
  for (int r = gw; r < nrows; r += nw) {
    const int t = perm[r];
    if ((unsigned)t >= (unsigned)nrows) {
      if (lane == 0) record_error(st, kStatusData, kBadPerm, r);
      continue;
    }
    const uint4* in = src + (size_t)r * vec_per_row;
    uint4* out = dst + (size_t)t * vec_per_row;
    int v = lane;
    for (; v + 224 < vec_per_row; v += 256) {
      uint4 u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = __ldg(in + v + 32 * i);
#pragma unroll
      for (int i = 0; i < 8; ++i) out[v + 32 * i] = u[i];
    }
    for (; v < vec_per_row; v += 32) out[v] = __ldg(in + v);
  }
}

// ------------------------------------------------------------------ token cluster
// cluster[t] = the partition holding the most of token t's experts, the lower partition
// on ties (a token's cluster, or device, at this layer).
__global__ void __launch_bounds__(kThreads)
token_cluster_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ emap, int T,
                     int K, int E, int P, int32_t* __restrict__ cluster, DeviceStatus* st) {
  pdl_wait_and_trigger();
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t >= T) return;
  const int32_t* row = idx + (size_t)t * K;
  int best_p = 0, best_c = -1;
  for (int k = 0; k < K; ++k) {
    const int e = row[k];
    if ((unsigned)e >= (unsigned)E) {
      record_error(st, kStatusData, kBadTopkIdx, (long long)t * K + k);
      continue;
    }
    const int p = emap[e];
    if ((unsigned)p >= (unsigned)P) {
      record_error(st, kStatusData, kBadExpertPart, e);
      continue;
    }
    int c = 0;
    for (int k2 = 0; k2 < K; ++k2) {
      const int e2 = row[k2];
      c += ((unsigned)e2 < (unsigned)E && emap[e2] == p);
    }
    if (c > best_c || (c == best_c && p < best_p)) {
      best_c = c;
      best_p = p;
    }
  }
  cluster[t] = best_p;
}

// ------------------------------------------------------------------ LAR
__device__ __forceinline__ int foe_source(int t, int h, int G, int H) {
  return H >= G ? (h * G) / H : h * (G / H) + (t % (G / H));
}

__global__ void __launch_bounds__(kThreads)
lar_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ src_part,
           const int32_t* __restrict__ emap, int T, int K, int E, int P, int H,
           unsigned long long* __restrict__ counts, DeviceStatus* st) {
  pdl_wait_and_trigger();
  __shared__ int s_map[kMaxBuckets];
  __shared__ unsigned long long s_red[3][kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kThreads) {
    const int p = emap[e];
    const bool ok = (unsigned)p < (unsigned)P;
    if (!ok && blockIdx.x == 0) record_error(st, kStatusData, kBadExpertPart, e);
    s_map[e] = ok ? p : -1;
  }
  __syncthreads();
  unsigned long long loc = 0, base = 0, mx = 0;
  const int kh = K / H;
  for (int t = blockIdx.x * kThreads + tid; t < T; t += gridDim.x * kThreads) {
    int src = -1;
    if (src_part) {
      src = src_part[t];
      if ((unsigned)src >= (unsigned)P) {
        record_error(st, kStatusData, kBadSrcPart, t);
        src = -1;
      }
    }
    const int bsrc = (int)(((long long)t * P) / T);
    const int32_t* row = idx + (size_t)t * K;
    int best = 0;
    for (int k = 0; k < K; ++k) {
      const int e = row[k];
      int dst = -1;
      if ((unsigned)e < (unsigned)E) dst = s_map[e];
      else record_error(st, kStatusData, kBadTopkIdx, (long long)t * K + k);
      const int sp = src_part ? src : foe_source(t, k / kh, P, H);
      loc += (dst >= 0 && dst == sp);
      base += (dst >= 0 && dst == bsrc);
      if (dst >= 0) {
        int c = 0;
        for (int k2 = 0; k2 < K; ++k2) {
          const int e2 = row[k2];
          c += ((unsigned)e2 < (unsigned)E && s_map[e2] == dst);
        }
        best = max(best, c);
      }
    }
    mx += best;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    loc += __shfl_xor_sync(0xffffffffu, loc, off);
    base += __shfl_xor_sync(0xffffffffu, base, off);
    mx += __shfl_xor_sync(0xffffffffu, mx, off);
  }
  if (lane == 0) { s_red[0][warp] = loc; s_red[1][warp] = base; s_red[2][warp] = mx; }
  __syncthreads();
  if (tid < 3) {
    unsigned long long v = 0;
    for (int w = 0; w < kWarps; ++w) v += s_red[tid][w];
    const int slot = tid == 0 ? 0 : (tid == 1 ? 2 : 3);
    atomicAdd(counts + slot, v);
  }
  if (blockIdx.x == 0 && tid == 0) atomicAdd(counts + 1, (unsigned long long)T * K);
}

int grid_for_rows(long long nrows) {
  static int sm_count = 0;
  if (sm_count == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (sm_count <= 0) sm_count = 152;
  }
  long long want = (nrows + kWarps - 1) / kWarps;
  long long cap = (long long)sm_count * 8;
  return (int)std::max<long long>(1, std::min(want, cap));
}

}  // namespace

// ------------------------------------------------------------------ launchers
int dispatch_sort_tile(const smoe_desc& d) {
  constexpr long long kWaveTiles = 2 * 152;   // two waves of a GB300's SMs
  constexpr long long kMaxTable = 4 * 4096;   // four scan rounds
  const long long n = (long long)d.T * d.K;
  int tile = kSortTile;
  while (tile > 256) {
    const long long nt = (n + tile / 2 - 1) / (tile / 2);
    if (nt > kWaveTiles || nt * d.E > kMaxTable) break;
    tile /= 2;
  }
  return tile;
}

cudaError_t launch_predict_shuffle(const smoe_desc& d, const int32_t* ids, const float* conf,
                                   const int32_t* emap, const void* x, int32_t* pred,
                                   int32_t* perm, int32_t* part_off, void* x_shuf, void* ws,
                                   cudaStream_t s, const int32_t* prev_cluster,
                                   const float* table_a) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  int32_t* hist = ws_ptr<int32_t>(ws, L.sort_hist);
  int32_t* offs = ws_ptr<int32_t>(ws, L.sort_off);
  // histogram columns of kPredTokens tokens (one per predict CTA, written directly);
  // scatter tiles of kShufScatter tokens
  const int ntiles = ceil_div(d.T, kPredTokens);
  constexpr int kStride = kShufScatter / kPredTokens;
  cudaError_t e = cudaFuncSetAttribute(predict_hist_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)predict_smem(d.E));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(predict_hist_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)predict_smem(d.E));
  if (e != cudaSuccess) return e;
  if (prev_cluster)
    SMOE_LAUNCH(predict_hist_kernel<true>, ntiles, kThreads, predict_smem(d.E), s, ids, conf,
        emap, d.T, d.E, d.P, d.vocab, pred, hist, ntiles, kPredTokens, st, prev_cluster, table_a,
        d.K);
  else
    SMOE_LAUNCH(predict_hist_kernel<false>, ntiles, kThreads, predict_smem(d.E), s, ids, conf,
        emap, d.T, d.E, d.P, d.vocab, pred, hist, ntiles, kPredTokens, st, nullptr, nullptr, d.K);
  SMOE_LAUNCH(scan_kernel, 1, 1024, 0, s, hist, offs, d.P * ntiles, d.P, ntiles, d.T, part_off);
  SMOE_LAUNCH(scatter_kernel<kShuffle>, ceil_div(d.T, kShufScatter), kThreads, 0, s, pred, d.T,
      d.P, ntiles, kShufScatter, kStride, offs, perm, nullptr, 0, 0, nullptr, nullptr, nullptr);
  if (x_shuf) {
    const int vec = (int)(d.d * elem_size(d) / 16);
    SMOE_LAUNCH(gather_rows_kernel, grid_for_rows(d.T), kThreads, 0, s,
        static_cast<const uint4*>(x), static_cast<uint4*>(x_shuf), perm, d.T, d.T, vec, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const smoe_desc& d, const int32_t* idx, const int32_t* perm,
                            const void* x_src, int32_t* expert_off, int32_t* pair_row,
                            int32_t* row_token, int32_t* row_slot, void* x_disp, void* ws,
                            cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  int32_t* hist = ws_ptr<int32_t>(ws, L.sort_hist);
  int32_t* offs = ws_ptr<int32_t>(ws, L.sort_off);
  int32_t* ws_rows = ws_ptr<int32_t>(ws, L.row_src);
  int32_t* row_src = row_slot ? row_slot : ws_rows;
  // per-pair buckets live in the second half of the workspace's row-source region
  int32_t* bucket = ws_rows + (size_t)d.T * d.K;
  const int n = d.T * d.K;
  const int tile = dispatch_sort_tile(d);
  const int ntiles = ceil_div(n, tile);
  SMOE_LAUNCH(dispatch_hist_kernel, ntiles, kThreads, 0, s, idx, perm, d.T, d.K, d.E, bucket, hist,
      ntiles, tile, st);
  SMOE_LAUNCH(scan_kernel, 1, 1024, 0, s, hist, offs, d.E * ntiles, d.E, ntiles, n, expert_off);
  SMOE_LAUNCH(scatter_kernel<kDispatch>, ntiles, kThreads, 0, s, bucket, n, d.E, ntiles, tile, 1,
      offs, nullptr, perm, d.T, d.K, pair_row, row_token, row_src);
  if (x_disp) {
    const int vec = (int)(d.d * elem_size(d) / 16);
    SMOE_LAUNCH(gather_rows_kernel, grid_for_rows(n), kThreads, 0, s,
        static_cast<const uint4*>(x_src), static_cast<uint4*>(x_disp), row_src, n, d.T, vec, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_shuffle_dispatch_rows(const smoe_desc& d, const void* x, const int32_t* perm,
                                        const int32_t* pair_row, void* x_shuf, void* x_disp,
                                        void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  const int vec = (int)(d.d * elem_size(d) / 16);
  SMOE_LAUNCH(shuffle_dispatch_rows_kernel, grid_for_rows(d.T), kThreads, 0, s,
      static_cast<const uint4*>(x), static_cast<uint4*>(x_shuf), static_cast<uint4*>(x_disp),
      perm, pair_row, d.T, d.K, vec, ws_ptr<DeviceStatus>(ws, L.status));
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const smoe_desc& d, const void* src, const int32_t* map,
                               int nrows, int nsrc, void* dst, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  const int vec = (int)(d.d * elem_size(d) / 16);
  SMOE_LAUNCH(gather_rows_kernel, grid_for_rows(nrows), kThreads, 0, s,
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), map, nrows, nsrc, vec,
      ws_ptr<DeviceStatus>(ws, L.status));
  return cudaGetLastError();
}

int exchange_sort_tile(const smoe_desc& d) {
  constexpr long long kWaveTiles = 2 * 152;
  constexpr long long kMaxTable = 4 * 4096;
  const long long n = (long long)d.T * d.K, B = (long long)d.P * d.P;
  int tile = kSortTile;
  while (tile > 256) {
    const long long nt = (n + tile / 2 - 1) / (tile / 2);
    if (nt > kWaveTiles || nt * B > kMaxTable) break;
    tile /= 2;
  }
  return tile;
}

cudaError_t launch_ep_exchange(const smoe_desc& d, const int32_t* idx, const int32_t* src_part,
                               const int32_t* emap, const void* x, int32_t* send_counts,
                               int32_t* recv_off, int32_t* pair_recv, int32_t* recv_token,
                               void* x_recv, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  int32_t* hist = ws_ptr<int32_t>(ws, L.sort_hist);
  int32_t* offs = ws_ptr<int32_t>(ws, L.sort_off);
  int32_t* rows = ws_ptr<int32_t>(ws, L.row_src);        // row -> pair index (unused here)
  int32_t* bucket = rows + (size_t)d.T * d.K;
  const int n = d.T * d.K, B = d.P * d.P;
  const int tile = exchange_sort_tile(d);
  const int ntiles = ceil_div(n, tile);
  SMOE_LAUNCH(exchange_hist_kernel, ntiles, kThreads, 0, s, idx, src_part, emap, d.T, d.K, d.E,
      d.P, bucket, hist, ntiles, tile, st);
  SMOE_LAUNCH(scan_kernel, 1, 1024, 0, s, hist, offs, B * ntiles, B, ntiles, n, recv_off);
  SMOE_LAUNCH((scatter_kernel<kDispatch, kMaxExchangeBuckets>), ntiles, kThreads, 0, s, bucket,
      n, B, ntiles, tile, 1, offs, nullptr, nullptr, d.T, d.K, pair_recv, recv_token, rows);
  SMOE_LAUNCH(send_counts_kernel, 1, kThreads, 0, s, recv_off, d.P, send_counts);
  if (x_recv) {
    const int vec = (int)(d.d * elem_size(d) / 16);
    SMOE_LAUNCH(gather_rows_kernel, grid_for_rows(n), kThreads, 0, s,
        static_cast<const uint4*>(x), static_cast<uint4*>(x_recv), recv_token, n, d.T, vec, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_srs(const smoe_desc& d, int R, const void* x_parts, const int32_t* perm,
                       void* x_shuf, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  const int vec = (int)(d.d * elem_size(d) / 16);
  if (d.dtype == SMOE_F32)
    SMOE_LAUNCH(srs_kernel<float>, grid_for_rows(d.T), kThreads, 0, s,
        static_cast<const uint4*>(x_parts), static_cast<uint4*>(x_shuf), perm, d.T, R, vec, st);
  else
    SMOE_LAUNCH(srs_kernel<__nv_bfloat16>, grid_for_rows(d.T), kThreads, 0, s,
        static_cast<const uint4*>(x_parts), static_cast<uint4*>(x_shuf), perm, d.T, R, vec, st);
  return cudaGetLastError();
}

cudaError_t launch_sag(const smoe_desc& d, const void* y_shuf, const int32_t* perm, void* y,
                       void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  const int vec = (int)(d.d * elem_size(d) / 16);
  SMOE_LAUNCH(scatter_rows_kernel, grid_for_rows(d.T), kThreads, 0, s,
      static_cast<const uint4*>(y_shuf), static_cast<uint4*>(y), perm, d.T, vec,
      ws_ptr<DeviceStatus>(ws, L.status));
  return cudaGetLastError();
}

cudaError_t launch_token_cluster(const smoe_desc& d, const int32_t* idx, const int32_t* emap,
                                 int32_t* cluster, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  SMOE_LAUNCH(token_cluster_kernel, ceil_div(d.T, kThreads), kThreads, 0, s, idx, emap, d.T, d.K,
              d.E, d.P, cluster, ws_ptr<DeviceStatus>(ws, L.status));
  return cudaGetLastError();
}

cudaError_t launch_lar(const smoe_desc& d, const int32_t* idx, const int32_t* src_part,
                       const int32_t* emap, unsigned long long* counts, void* ws,
                       cudaStream_t s) {
  WsLayout L;
  ws_layout(d, &L);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  cudaError_t e = cudaMemsetAsync(counts, 0, 4 * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(ceil_div(d.T, kThreads), 1024));
  SMOE_LAUNCH(lar_kernel, grid, kThreads, 0, s, idx, src_part, emap, d.T, d.K, d.E, d.P, d.H,
      counts, st);
  return cudaGetLastError();
}

}  // namespace smoe

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot allocate device memory at all: allocator-free embedded
// runtimes that reserve every byte at start-up, or hosts whose device memory pool
// is owned by another framework and may not be drawn from. For them the predict +
// shuffle step also exists without a caller workspace: its per-tile histogram and
// offsets live in the file-scope array below, which every GPU that loads the
// library keeps until the process exits.
namespace smoe {
namespace {

constexpr int kNoAllocMaxTiles = 4096;                        // T <= 4096 * kShufTile
constexpr int kNoAllocScratchInts = 2 * 32 * kNoAllocMaxTiles;  // hist + offs for P <= 32
static __device__ __align__(256) int32_t g_shuffle_scratch[kNoAllocScratchInts];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if there is none yet).
// Context ids are never reused within a process, so a context created after a reset
// of the device's primary context has a new id.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_shuffle_scratch in the current device's current context. It is
// looked up with that device current the first time a context calls, and again
// whenever the device's context has changed since (after cudaDeviceReset the module
// is loaded anew and the array can move). Host code must not use the symbol itself
// as a pointer.
int32_t* noalloc_scratch_ptr(int* err) {
  static std::mutex mu;
  static int32_t* ptrs[64] = {nullptr};
  static unsigned long long ctx_ids[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = set_last_error(SMOE_ERR_CUDA, "cudaGetDevice failed in the no-allocation shuffle");
    return nullptr;
  }
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    *err = set_last_error(SMOE_ERR_CUDA, "the current CUDA context could not be queried");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr || id == 0 || id != ctx_ids[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_shuffle_scratch);   // makes the context current too
    if (e != cudaSuccess || p == nullptr) {
      *err = set_last_error(SMOE_ERR_CUDA, "cudaGetSymbolAddress of the shuffle scratch failed");
      return nullptr;
    }
    if (id == 0 && !current_context_id(&id)) {
      *err = set_last_error(SMOE_ERR_CUDA, "the current CUDA context could not be queried");
      return nullptr;
    }
    ptrs[dev] = static_cast<int32_t*>(p);
    ctx_ids[dev] = id;
  }
  return ptrs[dev];
}

bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace smoe

extern "C" SMOE_API int smoe_predict_shuffle_noalloc(const smoe_desc* desc,
                                                     const int32_t* token_ids, const float* conf,
                                                     const int32_t* expert_part, const void* x,
                                                     int32_t* pred_part, int32_t* shuf_perm,
                                                     int32_t* part_off, void* x_shuf,
                                                     void* stream) {
  using namespace smoe;
  int rc = check_desc(desc);
  if (rc != SMOE_OK) return rc;
  const void* req[] = {token_ids, conf, expert_part, pred_part, shuf_perm, part_off};
  for (const void* p : req) {
    if (p == nullptr) return set_last_error(SMOE_ERR_ARG, "a required pointer is NULL");
    if (!aligned16_ptr(p)) return set_last_error(SMOE_ERR_ALIGN, "a pointer is not 16-byte aligned");
  }
  if (x_shuf != nullptr && (x == nullptr || !aligned16_ptr(x) || !aligned16_ptr(x_shuf)))
    return set_last_error(SMOE_ERR_ARG, "x_shuf needs a 16-byte aligned x");
  const int ntiles = ceil_div(desc->T, kShufTile);
  if (ntiles > kNoAllocMaxTiles)
    return set_last_error(SMOE_ERR_SHAPE,
                          "smoe_predict_shuffle_noalloc supports at most 1048576 tokens");
  int err = SMOE_OK;
  int32_t* scratch = noalloc_scratch_ptr(&err);
  if (scratch == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    cudaError_t e = cudaMemsetAsync(part_off, 0, sizeof(int32_t) * (desc->P + 1), s);
    return e == cudaSuccess ? SMOE_OK : set_last_error(SMOE_ERR_CUDA, cudaGetErrorString(e));
  }
  // The histogram part of the scratch is cleared at the start of every call (the
  // predict kernel adds into it); the offsets part is fully rewritten by the scan.
  // Device data errors are not reported by this variant: an out-of-range id is
  // treated as partition 0, as in smoe_predict_shuffle.
  int32_t* hist = scratch;
  int32_t* offs = scratch + 32 * kNoAllocMaxTiles;
  const smoe_desc& d = *desc;
  cudaError_t ce = cudaMemsetAsync(hist, 0, sizeof(int32_t) * d.P * ntiles, s);
  if (ce == cudaSuccess)
    ce = cudaFuncSetAttribute(predict_hist_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)predict_smem(d.E));
  if (ce != cudaSuccess) return set_last_error(SMOE_ERR_CUDA, cudaGetErrorString(ce));
  SMOE_LAUNCH_STATUS(predict_hist_kernel<false>, ceil_div(d.T, kPredTokens), kThreads,
      predict_smem(d.E), s, token_ids, conf, expert_part, d.T, d.E, d.P, d.vocab, pred_part, hist,
      ntiles, kShufTile, nullptr, nullptr, nullptr, d.K);
  SMOE_LAUNCH_STATUS(scan_kernel, 1, 1024, 0, s, hist, offs, d.P * ntiles, d.P, ntiles, d.T,
      part_off);
  SMOE_LAUNCH_STATUS(scatter_kernel<kShuffle>, ntiles, kThreads, 0, s, pred_part, d.T, d.P, ntiles,
      kShufTile, 1, offs, shuf_perm, nullptr, 0, 0, nullptr, nullptr, nullptr);
  if (x_shuf) {
    const int vec = (int)(d.d * elem_size(d) / 16);
    SMOE_LAUNCH_STATUS(gather_rows_kernel, grid_for_rows(d.T), kThreads, 0, s,
        static_cast<const uint4*>(x), static_cast<uint4*>(x_shuf), shuf_perm, d.T, d.T, vec,
        nullptr);
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SMOE_OK : set_last_error(SMOE_ERR_CUDA, cudaGetErrorString(e));
}
