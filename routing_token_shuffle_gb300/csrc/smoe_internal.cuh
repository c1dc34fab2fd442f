// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "smoe.h"

namespace smoe {

// ---------------------------------------------------------------- status word
// The first 256 bytes of every workspace. Kernels that index with caller data
// record out-of-range elements here and skip them; smoe_get_status reads it.
enum : uint32_t { kStatusData = 1u, kStatusTimeout = 2u };

struct DeviceStatus {
  uint32_t flags;
  int32_t first_kind;        // which check failed first (see kBad*)
  long long first_index;     // element index of that failure
};

enum : int32_t {
  kBadTokenId = 1, kBadExpertPart = 2, kBadTopkIdx = 3, kBadPerm = 4, kBadPairRow = 5,
  kBadSrcPart = 6, kTimeoutGemm = 16, kTimeoutProbe = 17
};

__device__ __forceinline__ void record_error(DeviceStatus* st, uint32_t flag, int32_t kind,
                                             long long index) {
  if (st == nullptr) return;
  uint32_t old = atomicOr(&st->flags, flag);
  if (old == 0u) {
    st->first_kind = kind;
    st->first_index = index;
  }
}

// ---------------------------------------------------------------- elements
template <typename TE> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec16 = 4;
  __device__ __forceinline__ static float to_f32(float v) { return v; }
  __device__ __forceinline__ static float from_f32(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec16 = 8;
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector <-> 8/4 fp32 values
__device__ __forceinline__ void unpack16(const uint4& v, float* out, const float*) {
  out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
  out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float* out, const __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack16(const float* in, const float*) {
  return make_uint4(__float_as_uint(in[0]), __float_as_uint(in[1]), __float_as_uint(in[2]),
                    __float_as_uint(in[3]));
}
__device__ __forceinline__ uint4 pack16(const float* in, const __nv_bfloat16*) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- workspace
// Every entry point carves the same layout out of the caller's workspace, so one
// buffer of smoe_workspace_size bytes serves all of them.
struct WsLayout {
  size_t status;
  size_t sort_hist, sort_off;       // counting-sort histograms [buckets * tiles]
  size_t row_src;                   // [T K] slot of each dispatched row
  size_t tiles;                     // grouped-GEMM tile table
  size_t logits, idx, w, pred, perm, part_off, lar, expert_off, pair_row, row_token;
  size_t x_shuf, x_disp, hbuf, y_disp, y_sh;
  size_t x_dev, ids_dev, y_dev;     // staging for smoe_layer_forward_host
  size_t pf_qs, pf_logits, pf_idx;  // prefetch predictor: q and s rows, logits, routes
  size_t route_part;                // gate GEMM partial logits [KS, T, E]
  size_t gather_flags;              // in-GEMM row gather: chunk ready flags + ticket
  size_t total;
};

constexpr int kSortTile = 1024;     // largest tile (pairs) of the dispatch counting sort
// Tile of the dispatch counting sort for this layer (256, 512 or 1024 pairs): halved from
// 1024 while the tiles still fit two waves of a 152-SM GPU and the (expert, tile) table
// stays within four rounds of the scan, so that small batches spread over more SMs.
int dispatch_sort_tile(const smoe_desc& d);
// Tile of the expert-parallel exchange's counting sort over P^2 (dst, src) buckets, chosen
// by the same rule with P^2 buckets.
int exchange_sort_tile(const smoe_desc& d);
constexpr int kShufTile = 256;      // tokens per tile of the workspace-free shuffle's sort
constexpr int kShufHistTokens = 32; // tokens per histogram column of the shuffle sort
constexpr int kMaxGroups = 520;     // E + n_shared upper bound

bool ws_layout(const smoe_desc& d, WsLayout* out);
int set_last_error(int code, const char* msg);  // records msg for smoe_last_error, returns code
int check_desc(const smoe_desc* d);  // smoe_status

inline size_t elem_size(const smoe_desc& d) { return d.dtype == SMOE_F32 ? 4 : 2; }
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

template <typename T>
inline T* ws_ptr(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// Per-thread count of kernel launches (reported by smoe_kernel_launches).
extern thread_local unsigned long long g_kernel_launches;
#define SMOE_COUNT_LAUNCH(n) (::smoe::g_kernel_launches += (n))

// ---------------------------------------------------------------- dependent launch
// Every library kernel is launched with programmatic stream serialisation and starts with
// pdl_wait() (griddepcontrol.wait: the previous kernel in the stream has completed and its
// writes are visible) before touching global memory, then pdl_trigger() so that the next
// kernel's CTAs may be scheduled while this grid drains; the expert FFN's down GEMM
// triggers only at its end instead, because its CTAs hold every SM and a combine made
// resident beside them slowed the Qwen3-shaped step by ~24 us. Without a programmatic
// predecessor the wait returns at once.
__device__ __forceinline__ void pdl_wait_and_trigger() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The two halves, for a kernel that lets its dependents be scheduled only at its end
// (the expert FFN's down GEMM, whose CTAs hold every SM: the combine that follows is
// then launched as the GEMM's CTAs finish, instead of resident beside them).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  SMOE_COUNT_LAUNCH(1);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}


#define SMOE_LAUNCH(kern, grid, block, smem, stream, ...)                              \
  do {                                                                                 \
    cudaError_t le_ = ::smoe::launch_k(kern, dim3(grid), dim3(block), smem, stream,     \
                                       __VA_ARGS__);                                   \
    if (le_ != cudaSuccess) return le_;                                                \
  } while (0)


// The same for functions that return an smoe_status.
#define SMOE_LAUNCH_STATUS(kern, grid, block, smem, stream, ...)                       \
  do {                                                                                 \
    cudaError_t le_ = ::smoe::launch_k(kern, dim3(grid), dim3(block), smem, stream,     \
                                       __VA_ARGS__);                                   \
    if (le_ != cudaSuccess)                                                            \
      return ::smoe::set_last_error(SMOE_ERR_CUDA, cudaGetErrorString(le_));           \
  } while (0)

// ---------------------------------------------------------------- launchers
cudaError_t launch_timeout_probe(DeviceStatus* st, cudaStream_t s);

// Each returns cudaSuccess or the launch error; shapes are validated by the caller.
int route_splits(const smoe_desc& d, int rows);  // K splits of the tensor-core gate GEMM

// Rows from `split` on write their logits / indices / weights to these outputs instead,
// renumbered from 0 (one routing launch serves two row sets).
struct RouteSplitOut {
  int split;
  float* logits;
  int32_t* idx;
  float* w;
};

cudaError_t launch_route(const smoe_desc& d, int rows, const void* x, const void* w_gate,
                         const float* logits_in, float* logits_out, int32_t* topk_idx,
                         float* topk_w, void* ws, cudaStream_t s,
                         RouteSplitOut so = RouteSplitOut{0x7fffffff, nullptr, nullptr, nullptr});

// prev_cluster / table_a non-NULL: the inter-layer source also votes (see sort.cu).
cudaError_t launch_predict_shuffle(const smoe_desc& d, const int32_t* ids, const float* conf,
                                   const int32_t* emap, const void* x, int32_t* pred,
                                   int32_t* perm, int32_t* part_off, void* x_shuf, void* ws,
                                   cudaStream_t s, const int32_t* prev_cluster = nullptr,
                                   const float* table_a = nullptr);

cudaError_t launch_token_cluster(const smoe_desc& d, const int32_t* idx, const int32_t* emap,
                                 int32_t* cluster, void* ws, cudaStream_t s);

cudaError_t launch_lar(const smoe_desc& d, const int32_t* idx, const int32_t* src_part,
                       const int32_t* emap, unsigned long long* counts, void* ws,
                       cudaStream_t s);

// row_slot: nullable output [T K], the x_src row of each dispatched row (the workspace
// keeps it when NULL).
cudaError_t launch_dispatch(const smoe_desc& d, const int32_t* idx, const int32_t* perm,
                            const void* x_src, int32_t* expert_off, int32_t* pair_row,
                            int32_t* row_token, int32_t* row_slot, void* x_disp, void* ws,
                            cudaStream_t s);

// gather != nullptr: x_disp is an output, X_disp[r] = gather->src[gather->map[r]] for the
// T K dispatched rows, copied inside the up GEMM when ffn_gather_in_gemm (otherwise by a
// row-gather launch before it).
struct FfnGather {
  const void* src;     // [nsrc, d] rows (x_shuf or x)
  const int32_t* map;  // [T K] source row of each dispatched row
  int nsrc;
};
cudaError_t launch_expert_ffn(const smoe_desc& d, const void* x_disp, const void* x,
                              const int32_t* expert_off, const void* w1, const void* w3,
                              const void* w2, void* y_disp, void* y_sh, void* ws,
                              cudaStream_t s, const FfnGather* gather = nullptr);
// true when launch_expert_ffn with a gather copies the rows inside its up GEMM
bool ffn_gather_in_gemm(const smoe_desc& d);
// x_shuf[s] = x[perm[s]] (x_shuf nullable; perm NULL: the identity) and X_disp[pair_row[t,
// k]] = x[t], from one read of each row of x
cudaError_t launch_shuffle_dispatch_rows(const smoe_desc& d, const void* x, const int32_t* perm,
                                        const int32_t* pair_row, void* x_shuf, void* x_disp,
                                        void* ws, cudaStream_t s);
// dst[r] = src[map[r]] for nrows rows of d elements (16-byte vectors)
cudaError_t launch_gather_rows(const smoe_desc& d, const void* src, const int32_t* map,
                               int nrows, int nsrc, void* dst, void* ws, cudaStream_t s);

// Expert-parallel exchange plan and receive rows (sort.cu).
cudaError_t launch_ep_exchange(const smoe_desc& d, const int32_t* idx, const int32_t* src_part,
                               const int32_t* emap, const void* x, int32_t* send_counts,
                               int32_t* recv_off, int32_t* pair_recv, int32_t* recv_token,
                               void* x_recv, void* ws, cudaStream_t s);
// Shuffled reduce-scatter of R partials into slot order, and its inverse all-gather.
cudaError_t launch_srs(const smoe_desc& d, int R, const void* x_parts, const int32_t* perm,
                       void* x_shuf, void* ws, cudaStream_t s);
cudaError_t launch_sag(const smoe_desc& d, const void* y_shuf, const int32_t* perm, void* y,
                       void* ws, cudaStream_t s);
cudaError_t launch_combine(const smoe_desc& d, const void* y_disp, const int32_t* pair_row,
                           const float* w, const void* y_sh, void* y, void* ws, cudaStream_t s);

cudaError_t launch_prefetch_ln(const smoe_desc& d, const float* r, const float* d_l,
                               const void* y, const float* gamma, const float* beta, void* qs,
                               cudaStream_t s);

cudaError_t launch_hits(const smoe_desc& d, const int32_t* pred_idx, const int32_t* true_idx,
                        unsigned long long* hits, cudaStream_t s);

}  // namespace smoe
