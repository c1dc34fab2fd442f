// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), over the expert-contiguous rows written by dispatch.
//
// Group g < E is routed expert g (rows expert_off[g] .. expert_off[g+1] of x_disp);
// group E + j is shared expert j, run on all T rows of x. Two launches:
//   up:   H[r, n]  = silu(A W1^T)[r, n] * (A W3^T)[r, n]   (H rounded to the element type)
//   down: Y[r, n]  = (H W2^T)[r, n]
// Each is a persistent kernel, one CTA per SM, walking a tile list (group, n-tile,
// m-tile) with m fastest so that the CTAs working at the same time share weight
// tiles through L2. Inside a CTA:
//   warp 0  one thread issues TMA loads into a 4-stage shared-memory ring
//           (stage = A 128 x 128 B + B 256 x 128 B, 128-byte swizzle);
//   warp 1  one thread issues tcgen05.mma (M = 128, N = 256, K = 16 bf16 / 8 tf32)
//           into one of two TMEM accumulators of 256 fp32 columns;
//   warp 2  allocates and frees the 512 TMEM columns;
//   warps 4-7 drain an accumulator (tcgen05.ld, one TMEM lane = one row per thread),
//           apply SwiGLU (up) and store through a per-warp shared-memory staging tile
//           (coalesced 128-byte row segments), while the MMAs of the next tile run.
// In the up GEMM the B stage holds 128 rows of W1 followed by the same 128 rows of
// W3, so one N = 256 MMA produces the gate and up halves of the tile together.
// Expert segments are not padded: a tile reaching past its group's last row reads
// the following rows (or TMA's zero fill) and its stores are masked.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "tc_common.cuh"

namespace smoe {
namespace {

constexpr int kBM = 128;
constexpr int kStages = 4;
constexpr uint32_t kStageA = 128 * 128;  // 128 rows x 128 bytes
constexpr uint32_t kStageB = 256 * 128;  // 256 rows x 128 bytes
constexpr int kThreads = 256;
constexpr int kAccCols = 256;            // fp32 columns per accumulator
constexpr uint32_t kStageOut = 4 * 32 * 128;  // epilogue staging: 4 warps x 32 rows x 128 B
constexpr size_t kSmemBytes = 1024 + kStages * (kStageA + kStageB) + kStageOut + 256 +
                              4 * (kMaxGroups + 1 + 513 + 4);

// Epilogue stores. A thread owns one accumulator row, so a direct 16-byte store from a
// warp touches 32 rows and fills half of each 32-byte sector. Each epilogue warp instead
// stages its 32 rows x 128 bytes in shared memory (16-byte chunks XOR-swizzled by row,
// which keeps both the row-wise writes and the column-wise reads free of bank conflicts)
// and writes them back as 4 rows x 128 contiguous bytes per store instruction.
template <typename TE>
struct RowStager {
  static constexpr int kVec = 16 / (int)sizeof(TE);           // elements per 16 bytes
  static constexpr int kColsPerFlush = 128 / (int)sizeof(TE);  // columns per staged row
  uint8_t* buf;    // this warp's 32 x 128 bytes
  TE* out;         // output matrix, row pitch N elements
  long long row0;  // output row of the warp's first row
  int valid;       // leading rows of the 32 that belong to the group
  int N;

  // 32 values of this lane's row, columns [c, c + 32) (c a multiple of 32)
  __device__ __forceinline__ void put32(int lane, int c, const float* v) const {
    const int chunk0 = ((c % kColsPerFlush) * (int)sizeof(TE)) >> 4;
#pragma unroll
    for (int j = 0; j < 32 / kVec; ++j) {
      const int ch = chunk0 + j;
      *reinterpret_cast<uint4*>(buf + lane * 128 + ((ch ^ (lane & 7)) << 4)) =
          pack16(v + j * kVec, (const TE*)nullptr);
    }
  }
  // store the staged window, whose first column is col0
  __device__ __forceinline__ void flush(int lane, int col0) const {
    __syncwarp();
    const int ch = lane & 7;
    const int col = col0 + ch * kVec;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      const uint4 v = *reinterpret_cast<const uint4*>(buf + rr * 128 + ((ch ^ (rr & 7)) << 4));
      if (rr < valid && col + kVec <= N)
        *reinterpret_cast<uint4*>(out + (size_t)(row0 + rr) * N + col) = v;
    }
    __syncwarp();
  }
};

__device__ __forceinline__ int clamp_rows(int v) { return v < 0 ? 0 : (v > 32 ? 32 : v); }

// tile_start[g] = first m-tile of group g; tile_start[G] = total m-tiles. expert_off must
// be non-decreasing from 0 to at most T K; otherwise no tile is scheduled and the status
// word records the error.
__global__ void tile_table_kernel(const int32_t* __restrict__ expert_off, int E, int n_shared,
                                  int T, int TK, int bm, int32_t* __restrict__ tile_start,
                                  DeviceStatus* st, int32_t* __restrict__ g_flags, int g_n) {
  pdl_wait_and_trigger();
  const int lane = threadIdx.x;
  // gather mode: clear the ready flags and the chunk ticket of the up GEMM that follows
  for (int i = lane; i < g_n; i += 32) g_flags[i] = 0;
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

// In-GEMM row gather (see gather_worker): rows per completion counter.
constexpr int kGatherBlock = 64;

struct GemmArgs {
  const int32_t* expert_off;  // [E+1]
  const int32_t* tile_start;  // [G+1] m-tiles per group, prefix
  void* out;                  // up: H [TK + S T, F]; down: y_disp [TK, d]
  void* out_sh;               // down: y_shared [S, T, d]
  DeviceStatus* st;
  int E, G, T, TK;
  int N;                      // output columns: F (up) or d (down)
  int KD;                     // contraction length: d (up) or F (down)
  int NT;                     // n-tiles
  // gather mode (two-SM up GEMM): X_disp[r] = g_src[g_map[r]] is written by this kernel's
  // gather warps while it runs, in chunks of g_chunk rows (a power of two <= 32);
  // g_counts[b] counts the written rows of 64-row block b; *g_ticket numbers the chunks
  // taken. g_src == nullptr: X_disp is already in place.
  const uint4* g_src;
  const int32_t* g_map;
  uint4* g_dst;
  int32_t* g_ticket;
  int32_t* g_counts;
  int g_vec, g_nsrc, g_nchunks, g_chunk;
};

struct Tile {
  int g, m0, n0, rows;
  int a_row;          // first A row in its tensor map
  bool a_shared;      // A from the shared-input map (x) instead of the routed map
  int b_row;          // first B row
  long long out_row;  // first output row (in out, or in out_sh for a shared down tile)
  bool out_shared;
  bool swap;          // two-SM tile of a group's last <= 192 rows with swapped operands
  int N;              // MMA N: 256, or the swapped tile's tokens rounded up to 32
};

template <bool UP>
__device__ __forceinline__ void decode_tile(const int32_t* ts, const int32_t* eo,
                                            const GemmArgs& p, int t, Tile& r) {
  int lo = 0, hi = p.G - 1;
  while (lo < hi) {  // largest g whose first tile is <= t (empty groups are skipped)
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] * p.NT <= t) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int mt = ts[g + 1] - ts[g];
  const int local = t - ts[g] * p.NT;
  const int n_tile = local / mt, m_tile = local - n_tile * mt;
  r.g = g;
  r.m0 = m_tile * kBM;
  const bool shared = g >= p.E;
  const int j = g - p.E;
  r.rows = shared ? p.T : eo[g + 1] - eo[g];
  if (UP) {
    r.n0 = n_tile * 128;
    r.a_shared = shared;
    r.a_row = (shared ? 0 : eo[g]) + r.m0;
    r.b_row = g * p.N + r.n0;
    r.out_row = (long long)(shared ? p.TK + j * p.T : eo[g]) + r.m0;
    r.out_shared = false;
  } else {
    r.n0 = n_tile * 256;
    r.a_shared = false;
    r.a_row = (shared ? p.TK + j * p.T : eo[g]) + r.m0;
    r.b_row = g * p.N + r.n0;
    r.out_row = (shared ? (long long)j * p.T : (long long)eo[g]) + r.m0;
    r.out_shared = shared;
  }
}

template <bool UP, bool F32>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmA_sh,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmB3, const GemmArgs p) {
  // the down GEMM lets the combine be scheduled only as its CTAs finish (see the end)
  if (UP) pdl_wait_and_trigger(); else pdl_wait();
  using TE = typename std::conditional<F32, float, __nv_bfloat16>::type;
  constexpr int BK = F32 ? 32 : 64;           // elements per 128-byte row
  constexpr int kMmaK = F32 ? 8 : 16;          // elements per MMA
  constexpr int kMmaPerStage = BK / kMmaK;     // 4
  constexpr uint32_t kIdesc = tc::instr_desc(F32, kBM, 256);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kStages * kStageA;
  uint8_t* sOut = sB + kStages * kStageB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + kStageOut);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);
  int32_t* s_ts = reinterpret_cast<int32_t*>(s_abort + 1);
  int32_t* s_eo = s_ts + (p.G + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 128);
    }
    tc::mbar_init(drain, 1);
    *s_abort = 0;
    tc::mbar_init_fence();
    tc::tma_prefetch_map(&tmA);
    tc::tma_prefetch_map(&tmA_sh);
    tc::tma_prefetch_map(&tmB1);
    tc::tma_prefetch_map(&tmB3);
  }
  for (int i = threadIdx.x; i <= p.G; i += kThreads) s_ts[i] = p.tile_start[i];
  for (int i = threadIdx.x; i <= p.E; i += kThreads) s_eo[i] = p.expert_off[i];
  if (warp == 2) {
    tc::tmem_alloc(s_tmem, 2 * kAccCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int total = s_ts[p.G] * p.NT;
  const int nkb = (p.KD + BK - 1) / BK;
  volatile int* abort = s_abort;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      Tile tl;
      decode_tile<UP>(s_ts, s_eo, p, t, tl);
      const CUtensorMap* amap = tl.a_shared ? &tmA_sh : &tmA;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
        tc::mbar_expect_tx(&full[s], kStageA + kStageB);
        tc::tma_load_2d(sA + s * kStageA, amap, &full[s], kb * BK, tl.a_row);
        if (UP) {
          tc::tma_load_2d(sB + s * kStageB, &tmB1, &full[s], kb * BK, tl.b_row);
          tc::tma_load_2d(sB + s * kStageB + kStageB / 2, &tmB3, &full[s], kb * BK, tl.b_row);
        } else {
          tc::tma_load_2d(sB + s * kStageB, &tmB1, &full[s], kb * BK, tl.b_row);
        }
      }
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
      // let the copies already issued land before the CTA's shared memory goes away
      volatile int never = 0;
      const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
      for (uint32_t j = first; j < it; ++j)
        tc::mbar_wait(&full[j % kStages], (j / kStages) & 1u, &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tcount) {
      const uint32_t a = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!tc::mbar_wait(&tempty[a], aph ^ 1u, abort)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t d_tmem = tmem + a * kAccCols;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
        if (!tc::mbar_wait(&full[s], ph, abort)) { ok = false; break; }
        tc::fence_after_sync();
        const uint64_t adesc = tc::sw128_kmajor_desc(tc::smem_u32(sA + s * kStageA));
        const uint64_t bdesc = tc::sw128_kmajor_desc(tc::smem_u32(sB + s * kStageB));
#pragma unroll
        for (int k = 0; k < kMmaPerStage; ++k) {
          const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
          if (F32)
            tc::mma_tf32(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, acc);
          else
            tc::mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, acc);
        }
        tc::commit(&empty[s]);
      }
      if (!ok) break;
      tc::commit(&tfull[a]);
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
    // wait for every MMA this thread issued before TMEM is released
    volatile int never = 0;
    tc::commit(drain);
    tc::mbar_wait(drain, 0, &never);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    uint32_t tcount = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
      Tile tl;
      decode_tile<UP>(s_ts, s_eo, p, t, tl);
      const uint32_t a = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!tc::mbar_wait_warp(&tfull[a], aph, abort)) {
        *abort = 1;
        record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
        break;
      }
      tc::fence_after_sync();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + a * kAccCols;
      const RowStager<TE> rs{sOut + q * 4096, static_cast<TE*>(tl.out_shared ? p.out_sh : p.out),
                             tl.out_row + q * 32, clamp_rows(tl.rows - tl.m0 - q * 32), p.N};
      constexpr int kWin = RowStager<TE>::kColsPerFlush;
      if (UP) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(taddr + c, gv);
          tc::tmem_ld32(taddr + 128 + c, uv);
          tc::tmem_ld_wait();
          if (c == 96) {  // the accumulator is read out: the next tile's MMAs may start
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[a]);
          }
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float gg = __uint_as_float(gv[i]);
            h[i] = gg / (1.0f + __expf(-gg)) * __uint_as_float(uv[i]);
          }
          rs.put32(lane, c, h);
          if ((c + 32) % kWin == 0) rs.flush(lane, tl.n0 + c + 32 - kWin);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t yv[32];
          tc::tmem_ld32(taddr + c, yv);
          tc::tmem_ld_wait();
          if (c == 224) {
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[a]);
          }
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(yv[i]);
          rs.put32(lane, c, y);
          if ((c + 32) % kWin == 0) rs.flush(lane, tl.n0 + c + 32 - kWin);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (!UP && threadIdx.x == 0) pdl_trigger();
  if (warp == 2) tc::tmem_dealloc(tmem, 2 * kAccCols);
}

// ------------------------------------------------------------------ in-GEMM gather
// Gather mode hides the dispatch's row copy (X_disp[r] = x_src[row_slot[r]], a write-bound
// stream) under the up GEMM, which leaves DRAM mostly idle. Gather warps of every CTA take
// chunks of g_chunk rows (about 16 KB) from a global ticket, in row order (the order in
// which the tiles consume them), copy them and add their row count to the counter of
// their 64-row block; a TMA producer waits (bounded) until the blocks of its tile's own
// rows are complete, then orders the async proxy after the generic writes before
// loading. A claimed chunk is always being copied by a running CTA, and unclaimed chunks
// are claimed by any running CTA, the waiting one included, so no CTA waits on one that
// has not started.
__device__ __forceinline__ void gather_worker(const GemmArgs& p, int lane) {
  for (;;) {
    int c = 0;
    if (lane == 0) c = atomicAdd(p.g_ticket, 1);
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c >= p.g_nchunks) break;
    const int r0 = c * p.g_chunk;
    const int nr = min(p.g_chunk, p.TK - r0);
    const int my_src = lane < nr ? p.g_map[r0 + lane] : 0;
    for (int i = 0; i < nr; ++i) {
      const int srow = __shfl_sync(0xffffffffu, my_src, i);
      uint4* out = p.g_dst + (size_t)(r0 + i) * p.g_vec;
      if ((unsigned)srow >= (unsigned)p.g_nsrc) {
        if (lane == 0) record_error(p.st, kStatusData, kBadPerm, r0 + i);
        for (int v = lane; v < p.g_vec; v += 32) out[v] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint4* in = p.g_src + (size_t)srow * p.g_vec;
      for (int v = lane; v < p.g_vec; v += 32 * 8) {
        uint4 t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v + 32 * u < p.g_vec) t[u] = __ldg(in + v + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v + 32 * u < p.g_vec) out[v + 32 * u] = t[u];
      }
    }
    __threadfence();  // each lane's row writes, before the warp's count
    __syncwarp();
    if (lane == 0) atomicAdd(p.g_counts + r0 / kGatherBlock, nr);
  }
}

// Wait until rows [lo, hi) of X_disp are written (their 64-row blocks complete); false
// after the bounded wait (or when another role of the CTA gave up).
__device__ __forceinline__ bool wait_rows(const GemmArgs& p, int lo, int hi, volatile int* abort) {
  if (hi <= lo) return true;
  for (int b = lo / kGatherBlock; b <= (hi - 1) / kGatherBlock; ++b) {
    const int32_t* f = p.g_counts + b;
    const int want = min(kGatherBlock, p.TK - b * kGatherBlock);
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v >= want) continue;
    const unsigned long long t0 = tc::globaltimer();
    for (uint32_t i = 1;; ++i) {
      __nanosleep(64);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
      if (v >= want) break;
      if ((i & 63u) == 0 && (*abort || tc::globaltimer() - t0 > tc::kWaitTimeoutNs)) return false;
    }
  }
  // the rows were written through the generic proxy; TMA reads through the async proxy
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ------------------------------------------------------------------ two-SM variant
// A cluster of two CTAs (on the two SMs of a TPC) computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2: each CTA loads its own 128 rows of A and 128 rows of B, so
// each SM receives 32 KB per 64-wide k-block instead of 48 KB for the same MMA rate.
// B halves: up, 64 W1 rows then the same 64 W3 rows (leader: features n0 .. n0+63,
// peer: n0+64 .. n0+127), so that every accumulator row holds the gate and the up value
// of each of its features; down, the leader's and the peer's 128 of the 256 W2 rows.
// A group whose last rows fit in 192 ends with a swapped tile: the 256 MMA rows are the
// weight rows that would have been B (each CTA's own 128, loaded exactly as B) and the
// N = 32 .. 192 columns are the group's last tokens (N/2 per CTA, loaded with the 64-row
// box up to N = 128, the 128-row box above), so the tile's MMA work follows its tokens.
// It takes as long as a full tile (a fixed cost per MMA instruction) but does less tensor
// work, which under the power cap is clock: on the DeepSeek-V2-shaped layer (87 tails
// <= 128 rows and 71 remainders of 129-255 rows in 338 row tiles) swapping remainders up
// to 192 rows took the FFN 2.36 -> 2.31 ms. Past 192 rows the savings are small and the
// token-by-token epilogue of a wide swapped tile costs more than it saves (swapping every
// partial tile made the Qwen3- and Mixtral-shaped FFNs, whose remainders are 224-255
// rows, 40 % and 7 % slower).
// The accumulator of a swapped tile is transposed: TMEM lane = weight row (up: lanes 0-63
// the gate and 64-127 the up value of the CTA's 64 features; down: the CTA's 128 output
// columns), TMEM column = token; its epilogue writes the output token by token.
// The leader's thread issues the MMAs; stage bytes of both CTAs complete on the leader's
// `full` barrier; MMA completion is multicast to both CTAs' `empty` and `tfull`; both
// epilogues drain their own TMEM lanes and arrive on the leader's `tempty`.
// Ring of kPairStages stages, each two 64-wide k-blocks deep (A and B: 2 x 16 KB per CTA),
// so that a barrier round trip and a commit serve 8 MMAs: measured against 6 single
// k-block stages, the FFN took 3 % less time on the Mixtral shape, 2.5 % on the Qwen3
// shape and 0.4 % on the DeepSeek-V2 shape.
constexpr int kPairStages = 3;
// warps 0-7 as in the single-SM kernel; warps 2, 3 and 8-11 copy rows in gather mode
constexpr int kPairThreads = 384;
constexpr uint32_t kPairStage = 128 * 128;  // A half or B half: 128 rows x 128 bytes
constexpr size_t kPairSmemBytes = 1024 + kPairStages * 4 * kPairStage + kStageOut + 256 +
                                  4 * (kMaxGroups + 1 + 513 + 4);

template <bool UP>
__device__ __forceinline__ void decode_pair_tile(const int32_t* ts, const int32_t* eo,
                                                 const GemmArgs& p, int t, uint32_t rank,
                                                 Tile& r) {
  int lo = 0, hi = p.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] * p.NT <= t) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int mt = ts[g + 1] - ts[g];  // 256-row pairs of this group
  const int local = t - ts[g] * p.NT;
  const int n_tile = local / mt, m_pair = local - n_tile * mt;
  const bool shared = g >= p.E;
  const int j = g - p.E;
  r.g = g;
  r.rows = shared ? p.T : eo[g + 1] - eo[g];
  const int rem = r.rows - m_pair * 256;
  r.swap = rem <= 192;  // (see the two-SM variant's notes above)
  r.N = r.swap ? (rem + 31) & ~31 : 256;
  // this CTA's first operand row: its 128 of a 256-row tile, or its N/2 of the tokens
  r.m0 = m_pair * 256 + (int)rank * (r.swap ? r.N / 2 : 128);
  if (UP) {
    r.n0 = n_tile * 128;
    r.a_shared = shared;
    r.a_row = (shared ? 0 : eo[g]) + r.m0;
    r.b_row = g * p.N + r.n0 + (int)rank * 64;  // W1 and W3 rows of this CTA's 64 features
    r.out_row = (long long)(shared ? p.TK + j * p.T : eo[g]) + r.m0;
    r.out_shared = false;
  } else {
    r.n0 = n_tile * 256;
    r.a_shared = false;
    r.a_row = (shared ? p.TK + j * p.T : eo[g]) + r.m0;
    r.b_row = g * p.N + r.n0 + (int)rank * 128;
    r.out_row = (shared ? (long long)j * p.T : (long long)eo[g]) + r.m0;
    r.out_shared = shared;
  }
}

template <bool UP>
__global__ void __launch_bounds__(kPairThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,     // 128-row box
                         const __grid_constant__ CUtensorMap tmA_sh,  // 128-row box
                         const __grid_constant__ CUtensorMap tmA64,   // 64-row box
                         const __grid_constant__ CUtensorMap tmA_sh64,
                         const __grid_constant__ CUtensorMap tmB1,
                         const __grid_constant__ CUtensorMap tmB3, const GemmArgs p) {
  // the down GEMM lets the combine be scheduled only as its CTAs finish (see the end)
  if (UP) pdl_wait_and_trigger(); else pdl_wait();
  using TE = __nv_bfloat16;
  constexpr uint32_t kIdesc = tc::instr_desc(false, 256, 256);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + 2 * kPairStages * kPairStage;
  uint8_t* sOut = sB + 2 * kPairStages * kPairStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + kStageOut);
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);
  int32_t* s_ts = reinterpret_cast<int32_t*>(s_abort + 1);
  int32_t* s_eo = s_ts + (p.G + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 256);
    }
    tc::mbar_init(drain, 1);
    *s_abort = 0;
    tc::mbar_init_fence();
    tc::tma_prefetch_map(&tmA);
    tc::tma_prefetch_map(&tmA_sh);
    tc::tma_prefetch_map(&tmA64);
    tc::tma_prefetch_map(&tmA_sh64);
    tc::tma_prefetch_map(&tmB1);
    tc::tma_prefetch_map(&tmB3);
  }
  for (int i = threadIdx.x; i <= p.G; i += kPairThreads) s_ts[i] = p.tile_start[i];
  for (int i = threadIdx.x; i <= p.E; i += kPairThreads) s_eo[i] = p.expert_off[i];
  if (warp == 2) {
    tc::tmem_alloc_pair(s_tmem, 2 * kAccCols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers are initialised before any remote signal
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int total = s_ts[p.G] * p.NT;
  const int nkb = (p.KD + 63) / 64;
  volatile int* abort = s_abort;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs) {
      Tile tl;
      decode_pair_tile<UP>(s_ts, s_eo, p, t, rank, tl);
      // token rows: 128 (256-row tile) or a 64-row box holding the CTA's N/2 <= 64 tokens
      const bool box64 = tl.swap && tl.N <= 128;  // the CTA's N/2 tokens fit a 64-row box
      const CUtensorMap* amap = box64 ? (tl.a_shared ? &tmA_sh64 : &tmA64)
                                      : (tl.a_shared ? &tmA_sh : &tmA);
      const uint32_t tx = 2 * ((box64 ? kPairStage / 2 : kPairStage) + kPairStage);
      if (UP && p.g_src && !tl.a_shared &&
          !wait_rows(p, tl.a_row, min(tl.a_row + (box64 ? 64 : 128), s_eo[tl.g + 1]), abort)) {
        ok = false;
        break;
      }
      for (int kb2 = 0; kb2 < nkb; kb2 += 2, ++it) {
        const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1u;
        const int nj = min(2, nkb - kb2);
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
        const uint32_t leader_full = tc::cluster_addr(&full[s], 0);
        if (rank == 0) tc::mbar_expect_tx(&full[s], tx * nj);
        for (int j = 0; j < nj; ++j) {
          const int kb = kb2 + j;
          uint8_t* b = sB + (s * 2 + j) * kPairStage;
          tc::tma_load_2d_pair(sA + (s * 2 + j) * kPairStage, amap, leader_full, kb * 64, tl.a_row);
          tc::tma_load_2d_pair(b, &tmB1, leader_full, kb * 64, tl.b_row);
          if (UP) tc::tma_load_2d_pair(b + kPairStage / 2, &tmB3, leader_full, kb * 64, tl.b_row);
        }
      }
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs, ++tcount) {
      Tile tl;
      decode_pair_tile<UP>(s_ts, s_eo, p, t, rank, tl);
      // swapped tile: the weight rows (B stage) are the MMA's A, the tokens its B
      const uint32_t idesc = tl.swap ? tc::instr_desc(false, 256, tl.N) : kIdesc;
      const uint32_t a = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!tc::mbar_wait(&tempty[a], aph ^ 1u, abort)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t d_tmem = tmem + a * kAccCols;
      for (int kb2 = 0; kb2 < nkb; kb2 += 2, ++it) {
        const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1u;
        const int nj = min(2, nkb - kb2);
        if (!tc::mbar_wait(&full[s], ph, abort)) { ok = false; break; }
        tc::fence_after_sync();
        for (int j = 0; j < nj; ++j) {
          const uint64_t tok_desc = tc::sw128_kmajor_desc(tc::smem_u32(sA + (s * 2 + j) * kPairStage));
          const uint64_t w_desc = tc::sw128_kmajor_desc(tc::smem_u32(sB + (s * 2 + j) * kPairStage));
          const uint64_t adesc = tl.swap ? w_desc : tok_desc;
          const uint64_t bdesc = tl.swap ? tok_desc : w_desc;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                              (kb2 + j > 0 || k > 0) ? 1u : 0u);
        }
        tc::commit_pair(&empty[s], 0x3);
      }
      if (!ok) break;
      tc::commit_pair(&tfull[a], 0x3);
    }
    if (!ok) {
      *abort = 1;
      record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
    }
    volatile int never = 0;
    tc::commit_pair(drain, 0x1);
    tc::mbar_wait(drain, 0, &never);
  } else if (UP && p.g_src && (warp == 2 || warp == 3 || warp >= 8)) {
    // ---------------------------------------------------------------- row gather
    gather_worker(p, lane);
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    uint32_t tcount = 0;
    bool failed = false;
    for (int t = pair; t < total; t += npairs, ++tcount) {
      Tile tl;
      decode_pair_tile<UP>(s_ts, s_eo, p, t, rank, tl);
      const uint32_t a = tcount & 1u, aph = (tcount >> 1) & 1u;
      // A warp whose wait fails does not leave the loop: the swapped up epilogue
      // synchronises the four epilogue warps on named barrier 1, so a failed warp keeps
      // taking part in those barriers (and does nothing else) while the others, seeing
      // the abort flag, fail their own waits at once.
      if (!failed && !tc::mbar_wait_warp(&tfull[a], aph, abort)) {
        *abort = 1;
        record_error(p.st, kStatusTimeout, kTimeoutGemm, blockIdx.x);
        failed = true;
      }
      if (failed) {
        if (UP && tl.swap) {
          asm volatile("bar.sync 1, 128;" ::: "memory");
          for (int c0 = 0; c0 < tl.N; c0 += 32) {
            asm volatile("bar.sync 1, 128;" ::: "memory");
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        }
        continue;
      }
      tc::fence_after_sync();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + a * kAccCols;
      if (tl.swap) {
        // TMEM column c = token t0 + c of the tile (the leader's N/2 tokens, then the
        // peer's); this warp's lanes are weight rows 32q .. 32q + 31 of the CTA's 128
        const int half = tl.N >> 1;
        const int ntok = tl.rows - (tl.m0 - (int)rank * half);    // tokens in the tile
        const long long row0 = tl.out_row - (long long)rank * half;  // output row of t0
        TE* out = static_cast<TE*>(tl.out_shared ? p.out_sh : p.out);
        float* xchg = reinterpret_cast<float*>(sOut);  // up values [64 features][33]
        // the exchange buffer overlaps the staging rows of warps 0-2: every epilogue warp
        // has finished the previous tile's stores before any of it is overwritten
        if (UP) asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll 1
        for (int c0 = 0; c0 < tl.N; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(taddr + c0, v);
          tc::tmem_ld_wait();
          if (c0 + 32 >= tl.N) {  // read out: the next tile's MMAs may start
            tc::fence_before_sync();
            tc::mbar_arrive_cluster(tc::cluster_addr(&tempty[a], 0));
          }
          if (UP) {
            // warps 2-3 hold the up values of the features whose gates warps 0-1 hold
            if (q >= 2) {
#pragma unroll
              for (int i = 0; i < 32; ++i) xchg[((q - 2) * 32 + lane) * 33 + i] = __uint_as_float(v[i]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (q < 2) {
              const int col = tl.n0 + 64 * (int)rank + 32 * q + lane;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int tk = c0 + i;
                const float gg = __uint_as_float(v[i]);
                const float h = gg / (1.0f + __expf(-gg)) * xchg[(q * 32 + lane) * 33 + i];
                if (tk < ntok && col < p.N)
                  out[(size_t)(row0 + tk) * p.N + col] = Elem<TE>::from_f32(h);
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          } else {
            const int col = tl.n0 + 128 * (int)rank + 32 * q + lane;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int tk = c0 + i;
              if (tk < ntok && col < p.N)
                out[(size_t)(row0 + tk) * p.N + col] = Elem<TE>::from_f32(__uint_as_float(v[i]));
            }
          }
        }
        continue;
      }
      // rows 32q .. 32q+31 of the CTA's 128 over all 256 columns
      const int rsub = q;
      const int nhalf = 0;
      const int ncols = 256;
      const RowStager<TE> rs{sOut + q * 4096, static_cast<TE*>(tl.out_shared ? p.out_sh : p.out),
                             tl.out_row + rsub * 32, clamp_rows(tl.rows - tl.m0 - rsub * 32),
                             p.N};
      constexpr int kWin = RowStager<TE>::kColsPerFlush;
      if (UP) {
        // each 128-column block: the gate of 64 features, then the up of the same features
#pragma unroll 1
        for (int c0 = 0; c0 < ncols; c0 += 128) {
#pragma unroll 1
          for (int c = 0; c < 64; c += 32) {
            uint32_t gv[32], uv[32];
            tc::tmem_ld32(taddr + c0 + c, gv);
            tc::tmem_ld32(taddr + c0 + 64 + c, uv);
            tc::tmem_ld_wait();
            if (c0 + 128 == ncols && c == 32) {  // read out: the next tile's MMAs may start
              tc::fence_before_sync();
              tc::mbar_arrive_cluster(tc::cluster_addr(&tempty[a], 0));
            }
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gg = __uint_as_float(gv[i]);
              h[i] = gg / (1.0f + __expf(-gg)) * __uint_as_float(uv[i]);
            }
            rs.put32(lane, c, h);
          }
          rs.flush(lane, tl.n0 + 64 * nhalf + c0 / 2);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < ncols; c += 32) {
          uint32_t yv[32];
          tc::tmem_ld32(taddr + c, yv);
          tc::tmem_ld_wait();
          if (c + 32 == ncols) {
            tc::fence_before_sync();
            tc::mbar_arrive_cluster(tc::cluster_addr(&tempty[a], 0));
          }
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(yv[i]);
          rs.put32(lane, c, y);
          if ((c + 32) % kWin == 0) rs.flush(lane, tl.n0 + 128 * nhalf + c + 32 - kWin);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();
  tc::fence_after_sync();
  if (!UP && threadIdx.x == 0) pdl_trigger();
  if (warp == 2) tc::tmem_dealloc_pair(tmem, 2 * kAccCols);
}

template <bool UP>
cudaError_t launch_gemm_pair(const CUtensorMap& A, const CUtensorMap& Ash, const CUtensorMap& A64,
                             const CUtensorMap& Ash64, const CUtensorMap& B1,
                             const CUtensorMap& B3, const GemmArgs& args, long long tile_bound,
                             cudaStream_t s);

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <bool UP, bool F32>
cudaError_t launch_gemm(const CUtensorMap& A, const CUtensorMap& Ash, const CUtensorMap& B1,
                        const CUtensorMap& B3, const GemmArgs& args, long long tile_bound,
                        cudaStream_t s) {
  auto kern = grouped_gemm_kernel<UP, F32>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<long long>(sm_count(), std::max<long long>(tile_bound, 1));
  SMOE_LAUNCH(kern, grid, kThreads, kSmemBytes, s, A, Ash, B1, B3, args);
  return cudaGetLastError();
}

template <bool UP>
cudaError_t launch_gemm_pair(const CUtensorMap& A, const CUtensorMap& Ash, const CUtensorMap& A64,
                             const CUtensorMap& Ash64, const CUtensorMap& B1,
                             const CUtensorMap& B3, const GemmArgs& args, long long tile_bound,
                             cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<UP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kPairSmemBytes);
  if (e != cudaSuccess) return e;
  const int pairs = (int)std::min<long long>(sm_count() / 2, std::max<long long>(tile_bound, 1));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  SMOE_COUNT_LAUNCH(1);
  return cudaLaunchKernelEx(&cfg, kern, A, Ash, A64, Ash64, B1, B3, args);
}

// Two-SM tiles (with M = 128 tiles for a group's last <= 128 rows) pad like single-SM
// tiles and move less data per SM; below about 256 rows per expert the FFN streams
// weights and the single-SM tiles, with twice as many CTAs issuing loads, keep more
// bytes in flight.
constexpr int kPairMinRows = 256;
bool use_pair_tiles(const smoe_desc& d) {
  return d.dtype == SMOE_BF16 && (long long)d.T * d.K >= (long long)kPairMinRows * d.E;
}

}  // namespace

// The row copy runs inside the up GEMM on two-SM tiles with F <= 1024: the copied bytes
// per FFN flop are b / (6 F), so small experts gain most. Measured (dispatch + FFN, same
// session): F = 768 (Qwen3 shape) -6 %, F = 1536 (DeepSeek-V2) within 1 %, F = 14336
// (Mixtral) +2.5 %: there the power-capped GEMM loses more to the concurrent copy than
// the copy's own time.
bool ffn_gather_in_gemm(const smoe_desc& d) { return use_pair_tiles(d) && d.F <= 1024; }

namespace {

template <bool F32>
cudaError_t run_ffn(const smoe_desc& d, const void* x_disp, const void* x,
                    const int32_t* expert_off, const void* w1, const void* w3, const void* w2,
                    void* y_disp, void* y_sh, void* ws, cudaStream_t s, const FfnGather* gather) {
  WsLayout L;
  ws_layout(d, &L);
  int32_t* tiles = ws_ptr<int32_t>(ws, L.tiles);
  void* hbuf = ws_ptr<char>(ws, L.hbuf);
  DeviceStatus* st = ws_ptr<DeviceStatus>(ws, L.status);
  const int TK = d.T * d.K, G = d.E + d.n_shared;
  const uint32_t box_k = F32 ? 32 : 64;
  const bool pairs = !F32 && use_pair_tiles(d);
  const int bm = pairs ? 256 : kBM;
  if (gather && !ffn_gather_in_gemm(d)) {  // copy the rows first
    cudaError_t e = launch_gather_rows(d, gather->src, gather->map, TK, gather->nsrc,
                                       const_cast<void*>(x_disp), ws, s);
    if (e != cudaSuccess) return e;
    gather = nullptr;
  }
  // gather chunks of about 16 KB of rows: many warps copy the rows of the first tiles
  // in parallel
  const int row_bytes = (int)(d.d * elem_size(d));
  int chunk = 1;
  while (chunk < 32 && (chunk * 2) * row_bytes <= 16384) chunk *= 2;  // <= 32: a lane per row
  const int nchunks = ceil_div(TK, chunk), nblocks = ceil_div(TK, kGatherBlock);
  int32_t* gflags = ws_ptr<int32_t>(ws, L.gather_flags);  // [nblocks] counts, then the ticket
  SMOE_LAUNCH(tile_table_kernel, 1, 32, 0, s, expert_off, d.E, d.n_shared, d.T, TK, bm, tiles, st,
              gflags, gather ? nblocks + 1 : 0);

  const long long mtile_bound =
      ceil_div(TK, bm) + d.E + (long long)d.n_shared * ceil_div(d.T, bm);
  const uint64_t x_rows = d.n_shared ? d.T : TK;
  const void* x_src = d.n_shared ? x : x_disp;
  const uint64_t h_rows = (uint64_t)TK + (uint64_t)d.n_shared * d.T;
  GemmArgs up{expert_off, tiles, hbuf, nullptr, st, d.E, G, d.T, TK, d.F, d.d, ceil_div(d.F, 128)};
  if (gather) {
    up.g_src = static_cast<const uint4*>(gather->src);
    up.g_map = gather->map;
    up.g_dst = static_cast<uint4*>(const_cast<void*>(x_disp));
    up.g_counts = gflags;
    up.g_ticket = gflags + nblocks;
    up.g_vec = row_bytes / 16;
    up.g_nsrc = gather->nsrc;
    up.g_nchunks = nchunks;
    up.g_chunk = chunk;
  }
  GemmArgs dn{expert_off, tiles, y_disp, y_sh, st, d.E, G, d.T, TK, d.d, d.F, ceil_div(d.d, 256)};

  if (pairs) {
    // up: A = x_disp [TK, d] (shared experts: x [T, d]) in 128- and 64-row boxes;
    // B = W1, W3 [(E+S) F, d] in 64-row boxes
    alignas(64) CUtensorMap tA, tAsh, tA64, tAsh64, tB1, tB3;
    if (!encode_tmap_2d(&tA, x_disp, false, TK, d.d, 128, 64) ||
        !encode_tmap_2d(&tAsh, x_src, false, x_rows, d.d, 128, 64) ||
        !encode_tmap_2d(&tA64, x_disp, false, TK, d.d, 64, 64) ||
        !encode_tmap_2d(&tAsh64, x_src, false, x_rows, d.d, 64, 64) ||
        !encode_tmap_2d(&tB1, w1, false, (uint64_t)G * d.F, d.d, 64, 64) ||
        !encode_tmap_2d(&tB3, w3, false, (uint64_t)G * d.F, d.d, 64, 64))
      return cudaErrorInvalidValue;
    cudaError_t e =
        launch_gemm_pair<true>(tA, tAsh, tA64, tAsh64, tB1, tB3, up, mtile_bound * up.NT, s);
    if (e != cudaSuccess) return e;
    // down: A = H [TK + S T, F]; B = W2 [(E+S) d, F] in 128-row boxes
    alignas(64) CUtensorMap dA, dA64, dB;
    if (!encode_tmap_2d(&dA, hbuf, false, h_rows, d.F, 128, 64) ||
        !encode_tmap_2d(&dA64, hbuf, false, h_rows, d.F, 64, 64) ||
        !encode_tmap_2d(&dB, w2, false, (uint64_t)G * d.d, d.F, 128, 64))
      return cudaErrorInvalidValue;
    return launch_gemm_pair<false>(dA, dA, dA64, dA64, dB, dB, dn, mtile_bound * dn.NT, s);
  }

  alignas(64) CUtensorMap tA, tAsh, tB1, tB3;
  // up: A = x_disp [TK, d] (shared experts: x [T, d]); B = W1, W3 [(E+S) F, d]
  if (!encode_tmap_2d(&tA, x_disp, F32, TK, d.d, kBM, box_k) ||
      !encode_tmap_2d(&tAsh, x_src, F32, x_rows, d.d, kBM, box_k) ||
      !encode_tmap_2d(&tB1, w1, F32, (uint64_t)G * d.F, d.d, 128, box_k) ||
      !encode_tmap_2d(&tB3, w3, F32, (uint64_t)G * d.F, d.d, 128, box_k))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_gemm<true, F32>(tA, tAsh, tB1, tB3, up, mtile_bound * up.NT, s);
  if (e != cudaSuccess) return e;

  // down: A = H [TK + S T, F]; B = W2 [(E+S) d, F]
  alignas(64) CUtensorMap dA, dB;
  if (!encode_tmap_2d(&dA, hbuf, F32, h_rows, d.F, kBM, box_k) ||
      !encode_tmap_2d(&dB, w2, F32, (uint64_t)G * d.d, d.F, 256, box_k))
    return cudaErrorInvalidValue;
  return launch_gemm<false, F32>(dA, dA, dB, dB, dn, mtile_bound * dn.NT, s);
}

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

bool encode_tmap_2d(CUtensorMap* map, const void* base, bool fp32, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_last_error(SMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    return false;
  }
  const uint32_t esz = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows > 0 ? rows : 1};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error(SMOE_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor map");
    return false;
  }
  return true;
}

cudaError_t launch_expert_ffn(const smoe_desc& d, const void* x_disp, const void* x,
                              const int32_t* expert_off, const void* w1, const void* w3,
                              const void* w2, void* y_disp, void* y_sh, void* ws,
                              cudaStream_t s, const FfnGather* gather) {
  if (d.dtype == SMOE_F32)
    return run_ffn<true>(d, x_disp, x, expert_off, w1, w3, w2, y_disp, y_sh, ws, s, gather);
  return run_ffn<false>(d, x_disp, x, expert_off, w1, w3, w2, y_disp, y_sh, ws, s, gather);
}

}  // namespace smoe
