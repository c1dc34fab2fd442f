// C entry points: host-side validation, workspace layout and launch sequencing.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "smoe_internal.cuh"

namespace smoe {

thread_local unsigned long long g_kernel_launches = 0;

namespace {
thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(SMOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The library carries sm_103a code only.
int check_device() {
  static std::atomic<int> cached[64];  // 0 unknown, 1 ok (zero-initialised: static storage)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const bool slot = dev >= 0 && dev < 64;
  if (slot && cached[dev].load(std::memory_order_relaxed) == 1) return SMOE_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(SMOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, major, minor);
  if (slot) cached[dev].store(1, std::memory_order_relaxed);
  return SMOE_OK;
}

#define SMOE_REQUIRE(cond, code, ...) \
  do {                                \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define SMOE_PTR(p) \
  do { \
    if ((p) == nullptr) return fail(SMOE_ERR_ARG, "%s must not be NULL", #p); \
    if (!aligned16(p)) return fail(SMOE_ERR_ALIGN, "%s is not 16-byte aligned", #p); \
  } while (0)

#define SMOE_OPT_PTR(p) \
  do { \
    if ((p) != nullptr && !aligned16(p)) return fail(SMOE_ERR_ALIGN, "%s is not 16-byte aligned", #p); \
  } while (0)

#define SMOE_CUDA(call) \
  do { \
    cudaError_t e_ = (call); \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

int check_ws(const smoe_desc* d, void* ws, size_t ws_bytes) {
  WsLayout L;
  ws_layout(*d, &L);
  if (ws == nullptr) return fail(SMOE_ERR_WORKSPACE, "workspace must not be NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(SMOE_ERR_ALIGN, "workspace is not 256-byte aligned");
  if (ws_bytes < L.total)
    return fail(SMOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, L.total);
  return SMOE_OK;
}

#define SMOE_CHECK(expr) \
  do { int rc_ = (expr); if (rc_ != SMOE_OK) return rc_; } while (0)

}  // namespace

int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

int check_desc(const smoe_desc* d) {
  SMOE_REQUIRE(d != nullptr, SMOE_ERR_ARG, "desc must not be NULL");
  SMOE_REQUIRE(d->dtype == SMOE_F32 || d->dtype == SMOE_BF16, SMOE_ERR_ARG, "bad dtype %d", d->dtype);
  SMOE_REQUIRE(d->renorm == 0 || d->renorm == 1, SMOE_ERR_ARG, "renorm must be 0 or 1");
  SMOE_REQUIRE(d->T >= 0 && d->d > 0 && d->E > 0 && d->K > 0 && d->H > 0 && d->F > 0 &&
                   d->n_shared >= 0 && d->P > 0 && d->vocab > 0,
               SMOE_ERR_SHAPE, "sizes must be positive (T may be 0)");
  SMOE_REQUIRE(d->K <= d->E, SMOE_ERR_SHAPE, "K=%d > E=%d", d->K, d->E);
  SMOE_REQUIRE(d->E % d->H == 0 && d->K % d->H == 0, SMOE_ERR_SHAPE,
               "H=%d must divide E=%d and K=%d", d->H, d->E, d->K);
  SMOE_REQUIRE(d->E <= 512 && d->K <= 32 && d->P <= 32 && d->n_shared <= 8, SMOE_ERR_SHAPE,
               "limits: E <= 512, K <= 32, P <= 32, n_shared <= 8");
  SMOE_REQUIRE(d->d % 8 == 0 && d->F % 8 == 0, SMOE_ERR_SHAPE, "d and F must be multiples of 8");
  SMOE_REQUIRE((long long)d->T * d->K <= (long long)INT_MAX / 2 &&
                   (long long)d->T * d->d <= (long long)INT_MAX * 8,
               SMOE_ERR_SHAPE, "T too large");
  return SMOE_OK;
}

bool ws_layout(const smoe_desc& d, WsLayout* L) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += round_up(bytes, 256);
    return o;
  };
  const size_t T = (size_t)d.T, K = (size_t)d.K, E = (size_t)d.E, P = (size_t)d.P;
  const size_t b = elem_size(d), dm = (size_t)d.d, F = (size_t)d.F, S = (size_t)d.n_shared;
  const size_t tile = (size_t)dispatch_sort_tile(d);
  const size_t ntT = (T + kShufHistTokens - 1) / kShufHistTokens, ntTK = (T * K + tile - 1) / tile;
  const size_t tile_x = (size_t)exchange_sort_tile(d);
  const size_t ntX = (T * K + tile_x - 1) / tile_x;      // EP exchange: P^2 buckets
  const size_t hist_n = std::max(std::max(P * ntT, E * ntTK), P * P * ntX) + 1;
  L->status = take(256);
  L->sort_hist = take(4 * hist_n);
  L->sort_off = take(4 * hist_n);
  L->row_src = take(4 * 2 * T * K);
  L->tiles = take(4 * (E + S + 1));
  L->logits = take(4 * T * E);
  L->idx = take(4 * T * K);
  L->w = take(4 * T * K);
  L->pred = take(4 * T);
  L->perm = take(4 * T);
  L->part_off = take(4 * (P + 1));
  L->lar = take(8 * 4);
  L->expert_off = take(4 * (E + 1));
  L->pair_row = take(4 * T * K);
  L->row_token = take(4 * T * K);
  L->x_shuf = take(T * dm * b);
  L->x_disp = take(T * K * dm * b);   // also receives the expert outputs (y_disp)
  L->y_disp = L->x_disp;
  L->hbuf = take((T * K + S * T) * F * b);
  L->y_sh = take(S * T * dm * b);
  L->x_dev = take(T * dm * b);
  L->ids_dev = take(4 * T);
  L->y_dev = take(T * dm * b);
  L->pf_qs = take(2 * T * dm * b);
  L->pf_logits = take(4 * 2 * T * E);
  L->pf_idx = take(4 * 2 * T * K);
  // the prefetch predictor routes 2T rows in one launch
  L->route_part = take(4 * E * std::max((size_t)route_splits(d, d.T) * T,
                                        (size_t)route_splits(d, 2 * d.T) * 2 * T));
  L->gather_flags = take(4 * ((T * K + 63) / 64 + 2));   // 64-row block counts + ticket
  L->total = off;
  return true;
}

}  // namespace smoe

using namespace smoe;

extern "C" {

SMOE_API size_t smoe_workspace_size(const smoe_desc* desc) {
  if (check_desc(desc) != SMOE_OK) return 0;
  WsLayout L;
  ws_layout(*desc, &L);
  return L.total;
}

SMOE_API const char* smoe_status_string(int status) {
  switch (status) {
    case SMOE_OK: return "ok";
    case SMOE_ERR_ARG: return "invalid argument";
    case SMOE_ERR_SHAPE: return "invalid shape";
    case SMOE_ERR_ALIGN: return "pointer not aligned";
    case SMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case SMOE_ERR_CUDA: return "CUDA error";
    case SMOE_ERR_DATA: return "device data out of range";
    case SMOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case SMOE_ERR_UNSUPPORTED: return "unsupported device or configuration";
    default: return "unknown status";
  }
}

SMOE_API const char* smoe_last_error(void) { return g_last_error.c_str(); }

SMOE_API unsigned long long smoe_kernel_launches(void) { return g_kernel_launches; }

SMOE_API int smoe_route(const smoe_desc* desc, const void* x, const void* w_gate,
                        const float* logits_in, float* logits_out, int32_t* topk_idx,
                        float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(topk_idx);
  SMOE_PTR(topk_w);
  SMOE_OPT_PTR(logits_out);
  if (logits_in) {
    SMOE_OPT_PTR(logits_in);
  } else {
    SMOE_PTR(x);
    SMOE_PTR(w_gate);
  }
  if (desc->T == 0) return SMOE_OK;
  if (!logits_in) SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaError_t e = launch_route(*desc, desc->T, x, w_gate, logits_in, logits_out, topk_idx, topk_w,
                               ws, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "route launch");
  return SMOE_OK;
}

SMOE_API int smoe_predict_shuffle(const smoe_desc* desc, const int32_t* token_ids,
                                  const float* conf, const int32_t* expert_part, const void* x,
                                  int32_t* pred_part, int32_t* shuf_perm, int32_t* part_off,
                                  void* x_shuf, void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(token_ids);
  SMOE_PTR(conf);
  SMOE_PTR(expert_part);
  SMOE_PTR(pred_part);
  SMOE_PTR(shuf_perm);
  SMOE_PTR(part_off);
  SMOE_OPT_PTR(x_shuf);
  if (x_shuf) SMOE_PTR(x);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    SMOE_CUDA(cudaMemsetAsync(part_off, 0, sizeof(int32_t) * (desc->P + 1), s));
    return SMOE_OK;
  }
  cudaError_t e = launch_predict_shuffle(*desc, token_ids, conf, expert_part, x, pred_part,
                                         shuf_perm, part_off, x_shuf, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "predict/shuffle launch");
  return SMOE_OK;
}

SMOE_API int smoe_token_cluster(const smoe_desc* desc, const int32_t* topk_idx,
                                const int32_t* expert_part, int32_t* cluster, void* ws,
                                size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(topk_idx);
  SMOE_PTR(expert_part);
  SMOE_PTR(cluster);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_token_cluster(*desc, topk_idx, expert_part, cluster, ws,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "token cluster launch");
  return SMOE_OK;
}

SMOE_API int smoe_predict_shuffle_inter(const smoe_desc* desc, const int32_t* token_ids,
                                        const float* conf, const int32_t* expert_part,
                                        const int32_t* prev_cluster, const float* table_a,
                                        const void* x, int32_t* pred_part, int32_t* shuf_perm,
                                        int32_t* part_off, void* x_shuf, void* ws,
                                        size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(token_ids);
  SMOE_PTR(conf);
  SMOE_PTR(expert_part);
  SMOE_PTR(prev_cluster);
  SMOE_PTR(table_a);
  SMOE_PTR(pred_part);
  SMOE_PTR(shuf_perm);
  SMOE_PTR(part_off);
  SMOE_OPT_PTR(x_shuf);
  if (x_shuf) SMOE_PTR(x);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    SMOE_CUDA(cudaMemsetAsync(part_off, 0, sizeof(int32_t) * (desc->P + 1), s));
    return SMOE_OK;
  }
  cudaError_t e = launch_predict_shuffle(*desc, token_ids, conf, expert_part, x, pred_part,
                                         shuf_perm, part_off, x_shuf, ws, s, prev_cluster, table_a);
  if (e != cudaSuccess) return cuda_fail(e, "predict/shuffle launch");
  return SMOE_OK;
}

SMOE_API int smoe_lar(const smoe_desc* desc, const int32_t* topk_idx, const int32_t* src_part,
                      const int32_t* expert_part, unsigned long long* counts, void* ws,
                      size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(topk_idx);
  SMOE_PTR(expert_part);
  SMOE_PTR(counts);
  SMOE_OPT_PTR(src_part);
  if (!src_part && desc->H < desc->P)
    SMOE_REQUIRE(desc->P % desc->H == 0, SMOE_ERR_SHAPE,
                 "the grouped source rule needs H | P when H < P (H=%d, P=%d)", desc->H, desc->P);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    SMOE_CUDA(cudaMemsetAsync(counts, 0, 4 * sizeof(unsigned long long), s));
    return SMOE_OK;
  }
  cudaError_t e = launch_lar(*desc, topk_idx, src_part, expert_part, counts, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "lar launch");
  return SMOE_OK;
}

SMOE_API int smoe_dispatch(const smoe_desc* desc, const int32_t* topk_idx,
                           const int32_t* shuf_perm, const void* x_src, int32_t* expert_off,
                           int32_t* pair_row, int32_t* row_token, int32_t* row_slot,
                           void* x_disp, void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(topk_idx);
  SMOE_OPT_PTR(shuf_perm);
  SMOE_PTR(expert_off);
  SMOE_PTR(pair_row);
  SMOE_PTR(row_token);
  SMOE_OPT_PTR(row_slot);
  SMOE_OPT_PTR(x_disp);
  if (x_disp) SMOE_PTR(x_src);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    SMOE_CUDA(cudaMemsetAsync(expert_off, 0, sizeof(int32_t) * (desc->E + 1), s));
    return SMOE_OK;
  }
  cudaError_t e = launch_dispatch(*desc, topk_idx, shuf_perm, x_src, expert_off, pair_row,
                                  row_token, row_slot, x_disp, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  return SMOE_OK;
}

SMOE_API int smoe_shuffle_dispatch_rows(const smoe_desc* desc, const void* x,
                                        const int32_t* shuf_perm, const int32_t* pair_row,
                                        void* x_shuf, void* x_disp, void* ws, size_t ws_bytes,
                                        void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(x);
  SMOE_OPT_PTR(shuf_perm);
  SMOE_PTR(pair_row);
  SMOE_OPT_PTR(x_shuf);
  SMOE_PTR(x_disp);
  SMOE_REQUIRE(x_shuf == nullptr || shuf_perm != nullptr, SMOE_ERR_ARG,
               "x_shuf needs shuf_perm");
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_shuffle_dispatch_rows(*desc, x, shuf_perm, pair_row, x_shuf, x_disp, ws,
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "shuffle/dispatch rows launch");
  return SMOE_OK;
}

SMOE_API int smoe_expert_ffn(const smoe_desc* desc, const void* x_disp, const void* x,
                             const int32_t* expert_off, const void* w1, const void* w3,
                             const void* w2, void* y_disp, void* y_shared, void* ws,
                             size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(x_disp);
  SMOE_PTR(expert_off);
  SMOE_PTR(w1);
  SMOE_PTR(w3);
  SMOE_PTR(w2);
  SMOE_PTR(y_disp);
  if (desc->n_shared > 0) {
    SMOE_PTR(x);
    SMOE_PTR(y_shared);
  }
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_expert_ffn(*desc, x_disp, x, expert_off, w1, w3, w2, y_disp, y_shared,
                                    ws, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "expert ffn launch");
  return SMOE_OK;
}

SMOE_API int smoe_expert_ffn_gather(const smoe_desc* desc, const void* x_src,
                                    const int32_t* row_slot, const void* x, void* x_disp,
                                    const int32_t* expert_off, const void* w1, const void* w3,
                                    const void* w2, void* y_disp, void* y_shared, void* ws,
                                    size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(x_src);
  SMOE_PTR(row_slot);
  SMOE_PTR(x_disp);
  SMOE_PTR(expert_off);
  SMOE_PTR(w1);
  SMOE_PTR(w3);
  SMOE_PTR(w2);
  SMOE_PTR(y_disp);
  if (desc->n_shared > 0) {
    SMOE_PTR(x);
    SMOE_PTR(y_shared);
  }
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  const FfnGather g{x_src, row_slot, desc->T};
  cudaError_t e = launch_expert_ffn(*desc, x_disp, x, expert_off, w1, w3, w2, y_disp, y_shared,
                                    ws, static_cast<cudaStream_t>(stream), &g);
  if (e != cudaSuccess) return cuda_fail(e, "expert ffn launch");
  return SMOE_OK;
}

SMOE_API int smoe_expert_ffn_gather_fused(const smoe_desc* desc) {
  if (check_desc(desc) != SMOE_OK) return 0;
  return ffn_gather_in_gemm(*desc) ? 1 : 0;
}

SMOE_API int smoe_combine(const smoe_desc* desc, const void* y_disp, const int32_t* pair_row,
                          const float* topk_w, const void* y_shared, void* y_out, void* ws,
                          size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(y_disp);
  SMOE_PTR(pair_row);
  SMOE_PTR(topk_w);
  SMOE_PTR(y_out);
  SMOE_OPT_PTR(y_shared);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_combine(*desc, y_disp, pair_row, topk_w, y_shared, y_out, ws,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return SMOE_OK;
}

SMOE_API int smoe_ep_exchange(const smoe_desc* desc, const int32_t* topk_idx,
                              const int32_t* src_part, const int32_t* expert_part,
                              const void* x, int32_t* send_counts, int32_t* recv_off,
                              int32_t* pair_recv, int32_t* recv_token, void* x_recv, void* ws,
                              size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(topk_idx);
  SMOE_PTR(expert_part);
  SMOE_OPT_PTR(src_part);
  SMOE_PTR(send_counts);
  SMOE_PTR(recv_off);
  SMOE_PTR(pair_recv);
  SMOE_PTR(recv_token);
  SMOE_OPT_PTR(x_recv);
  if (x_recv) SMOE_PTR(x);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    const int P = desc->P;
    SMOE_CUDA(cudaMemsetAsync(recv_off, 0, sizeof(int32_t) * (P * P + 1), s));
    SMOE_CUDA(cudaMemsetAsync(send_counts, 0, sizeof(int32_t) * P * P, s));
    return SMOE_OK;
  }
  cudaError_t e = launch_ep_exchange(*desc, topk_idx, src_part, expert_part, x, send_counts,
                                     recv_off, pair_recv, recv_token, x_recv, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "EP exchange launch");
  return SMOE_OK;
}

SMOE_API int smoe_srs(const smoe_desc* desc, int R, const void* x_parts,
                      const int32_t* shuf_perm, void* x_shuf, void* ws, size_t ws_bytes,
                      void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_REQUIRE(R >= 1 && R <= 64, SMOE_ERR_SHAPE, "R=%d must be in [1, 64]", R);
  SMOE_PTR(x_parts);
  SMOE_PTR(shuf_perm);
  SMOE_PTR(x_shuf);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_srs(*desc, R, x_parts, shuf_perm, x_shuf, ws,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "SRS launch");
  return SMOE_OK;
}

SMOE_API int smoe_sag(const smoe_desc* desc, const void* y_shuf, const int32_t* shuf_perm,
                      void* y, void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(y_shuf);
  SMOE_PTR(shuf_perm);
  SMOE_PTR(y);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaError_t e = launch_sag(*desc, y_shuf, shuf_perm, y, ws, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "SAG launch");
  return SMOE_OK;
}

static int layer_forward_impl(const smoe_desc* d, const smoe_layer_weights* W,
                              const smoe_layer_io* io, void* ws, cudaStream_t s) {
  WsLayout L;
  ws_layout(*d, &L);
  float* logits = io->logits ? io->logits : ws_ptr<float>(ws, L.logits);
  int32_t* idx = io->topk_idx ? io->topk_idx : ws_ptr<int32_t>(ws, L.idx);
  float* w = io->topk_w ? io->topk_w : ws_ptr<float>(ws, L.w);
  int32_t* pred = io->pred_part ? io->pred_part : ws_ptr<int32_t>(ws, L.pred);
  int32_t* perm = io->shuf_perm ? io->shuf_perm : ws_ptr<int32_t>(ws, L.perm);
  int32_t* part_off = io->part_off ? io->part_off : ws_ptr<int32_t>(ws, L.part_off);
  int32_t* expert_off = io->expert_off ? io->expert_off : ws_ptr<int32_t>(ws, L.expert_off);
  int32_t* pair_row = io->pair_row ? io->pair_row : ws_ptr<int32_t>(ws, L.pair_row);
  int32_t* row_token = io->row_token ? io->row_token : ws_ptr<int32_t>(ws, L.row_token);
  void* x_shuf = ws_ptr<char>(ws, L.x_shuf);
  void* x_disp = ws_ptr<char>(ws, L.x_disp);
  void* y_disp = ws_ptr<char>(ws, L.y_disp);
  void* y_sh = d->n_shared ? ws_ptr<char>(ws, L.y_sh) : nullptr;

  // where the FFN does not copy the dispatched rows inside its up GEMM, one pass over x
  // writes both x_shuf and X_disp after the dispatch's sort
  const bool rows_fused = !ffn_gather_in_gemm(*d);
  cudaError_t e = launch_route(*d, d->T, io->x, W->w_gate, nullptr, logits, idx, w, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "route launch");
  e = launch_predict_shuffle(*d, io->token_ids, W->conf, W->expert_part, io->x, pred, perm,
                             part_off, io->skip_shuffle || rows_fused ? nullptr : x_shuf, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "predict/shuffle launch");
  if (io->lar) {
    e = launch_lar(*d, idx, pred, W->expert_part, io->lar, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "lar launch");
  }
  const void* x_src = io->skip_shuffle ? io->x : x_shuf;
  // the dispatch sorts the pairs; then either one pass over x writes x_shuf and X_disp,
  // or the FFN copies the rows from x_shuf inside its up GEMM
  int32_t* row_slot = ws_ptr<int32_t>(ws, L.row_src);
  const int32_t* shuf = io->skip_shuffle ? nullptr : perm;
  e = launch_dispatch(*d, idx, shuf, x_src, expert_off, pair_row, row_token, row_slot, nullptr,
                      ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  if (rows_fused) {
    e = launch_shuffle_dispatch_rows(*d, io->x, shuf, pair_row, shuf ? x_shuf : nullptr, x_disp,
                                     ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "shuffle/dispatch rows launch");
  }
  const FfnGather g{x_src, row_slot, d->T};
  e = launch_expert_ffn(*d, x_disp, io->x, expert_off, W->w1, W->w3, W->w2, y_disp, y_sh, ws, s,
                        rows_fused ? nullptr : &g);
  if (e != cudaSuccess) return cuda_fail(e, "expert ffn launch");
  e = launch_combine(*d, y_disp, pair_row, w, y_sh, io->y, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return SMOE_OK;
}

static int check_weights(const smoe_layer_weights* W) {
  SMOE_REQUIRE(W != nullptr, SMOE_ERR_ARG, "weights must not be NULL");
  SMOE_PTR(W->w_gate);
  SMOE_PTR(W->w1);
  SMOE_PTR(W->w3);
  SMOE_PTR(W->w2);
  SMOE_PTR(W->conf);
  SMOE_PTR(W->expert_part);
  return SMOE_OK;
}

SMOE_API int smoe_layer_forward(const smoe_desc* desc, const smoe_layer_weights* weights,
                                const smoe_layer_io* io, void* ws, size_t ws_bytes,
                                void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_CHECK(check_weights(weights));
  SMOE_REQUIRE(io != nullptr, SMOE_ERR_ARG, "io must not be NULL");
  SMOE_PTR(io->x);
  SMOE_PTR(io->token_ids);
  SMOE_PTR(io->y);
  SMOE_OPT_PTR(io->logits);
  SMOE_OPT_PTR(io->topk_idx);
  SMOE_OPT_PTR(io->topk_w);
  SMOE_OPT_PTR(io->pred_part);
  SMOE_OPT_PTR(io->shuf_perm);
  SMOE_OPT_PTR(io->part_off);
  SMOE_OPT_PTR(io->expert_off);
  SMOE_OPT_PTR(io->pair_row);
  SMOE_OPT_PTR(io->row_token);
  SMOE_OPT_PTR(io->lar);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  return layer_forward_impl(desc, weights, io, ws, static_cast<cudaStream_t>(stream));
}

SMOE_API int smoe_layer_forward_host(const smoe_desc* desc, const smoe_layer_weights* weights,
                                     const void* x_host, const int32_t* ids_host, void* y_host,
                                     void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_CHECK(check_weights(weights));
  SMOE_REQUIRE(x_host && ids_host && y_host, SMOE_ERR_ARG, "host buffers must not be NULL");
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  WsLayout L;
  ws_layout(*desc, &L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)desc->T * desc->d * elem_size(*desc);
  void* x_dev = ws_ptr<char>(ws, L.x_dev);
  int32_t* ids_dev = ws_ptr<int32_t>(ws, L.ids_dev);
  void* y_dev = ws_ptr<char>(ws, L.y_dev);
  SMOE_CUDA(cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s));
  SMOE_CUDA(cudaMemcpyAsync(ids_dev, ids_host, sizeof(int32_t) * desc->T, cudaMemcpyHostToDevice, s));
  smoe_layer_io io;
  memset(&io, 0, sizeof(io));
  io.x = x_dev;
  io.token_ids = ids_dev;
  io.y = y_dev;
  SMOE_CHECK(layer_forward_impl(desc, weights, &io, ws, s));
  SMOE_CUDA(cudaMemcpyAsync(y_host, y_dev, xb, cudaMemcpyDeviceToHost, s));
  return SMOE_OK;
}

SMOE_API int smoe_moe_forward_routed(const smoe_desc* desc, const void* x,
                                     const int32_t* topk_idx, const float* topk_w,
                                     const void* w1, const void* w3, const void* w2, void* y,
                                     void* ws, size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_PTR(x);
  SMOE_PTR(topk_idx);
  SMOE_PTR(topk_w);
  SMOE_PTR(w1);
  SMOE_PTR(w3);
  SMOE_PTR(w2);
  SMOE_PTR(y);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  if (desc->T == 0) return SMOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsLayout L;
  ws_layout(*desc, &L);
  int32_t* expert_off = ws_ptr<int32_t>(ws, L.expert_off);
  int32_t* pair_row = ws_ptr<int32_t>(ws, L.pair_row);
  int32_t* row_token = ws_ptr<int32_t>(ws, L.row_token);
  void* x_disp = ws_ptr<char>(ws, L.x_disp);
  void* y_sh = desc->n_shared ? ws_ptr<char>(ws, L.y_sh) : nullptr;
  int32_t* row_slot = ws_ptr<int32_t>(ws, L.row_src);
  cudaError_t e = launch_dispatch(*desc, topk_idx, nullptr, x, expert_off, pair_row, row_token,
                                  row_slot, nullptr, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  const FfnGather g{x, row_slot, desc->T};
  e = launch_expert_ffn(*desc, x_disp, x, expert_off, w1, w3, w2, x_disp, y_sh, ws, s, &g);
  if (e != cudaSuccess) return cuda_fail(e, "expert ffn launch");
  e = launch_combine(*desc, x_disp, pair_row, topk_w, y_sh, y, ws, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return SMOE_OK;
}

SMOE_API int smoe_prefetch_predict(const smoe_desc* desc, const float* r, const float* d_l,
                                   const void* y, const float* gamma, const float* beta,
                                   const void* w_gate_next, float* logits_q, float* logits_s,
                                   int32_t* pred_idx, int32_t* true_idx,
                                   unsigned long long* hits, void* qs_out, void* ws,
                                   size_t ws_bytes, void* stream) {
  SMOE_CHECK(check_desc(desc));
  SMOE_REQUIRE(desc->d <= 8192, SMOE_ERR_SHAPE, "prefetch predictor supports d <= 8192");
  SMOE_PTR(r);
  SMOE_PTR(d_l);
  SMOE_PTR(y);
  SMOE_PTR(gamma);
  SMOE_PTR(beta);
  SMOE_PTR(w_gate_next);
  SMOE_PTR(pred_idx);
  SMOE_PTR(true_idx);
  SMOE_PTR(hits);
  SMOE_OPT_PTR(logits_q);
  SMOE_OPT_PTR(logits_s);
  SMOE_OPT_PTR(qs_out);
  SMOE_CHECK(check_ws(desc, ws, ws_bytes));
  SMOE_CHECK(check_device());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->T == 0) {
    SMOE_CUDA(cudaMemsetAsync(hits, 0, sizeof(unsigned long long), s));
    return SMOE_OK;
  }
  WsLayout L;
  ws_layout(*desc, &L);
  char* qs = qs_out ? static_cast<char*>(qs_out) : ws_ptr<char>(ws, L.pf_qs);
  float* lg = ws_ptr<float>(ws, L.pf_logits);
  float* wq = ws_ptr<float>(ws, L.pf_idx);
  const size_t T = desc->T;
  cudaError_t e = launch_prefetch_ln(*desc, r, d_l, y, gamma, beta, qs, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefetch layernorm launch");
  // q rows [0, T) and s rows [T, 2T) in one routing launch
  (void)lg;
  e = launch_route(*desc, 2 * desc->T, qs, w_gate_next, nullptr, logits_q, pred_idx, wq, ws, s,
                   RouteSplitOut{desc->T, logits_s, true_idx, wq + T * desc->K});
  if (e != cudaSuccess) return cuda_fail(e, "prefetch route launch");
  e = launch_hits(*desc, pred_idx, true_idx, hits, s);
  if (e != cudaSuccess) return cuda_fail(e, "hits launch");
  return SMOE_OK;
}

SMOE_API int smoe_selftest_device_timeout(void* ws, size_t ws_bytes, void* stream) {
  SMOE_REQUIRE(ws != nullptr, SMOE_ERR_ARG, "workspace must not be NULL");
  SMOE_REQUIRE(aligned16(ws), SMOE_ERR_ALIGN, "workspace must be 16-byte aligned");
  SMOE_REQUIRE(ws_bytes >= 256, SMOE_ERR_WORKSPACE, "workspace smaller than its status word");
  SMOE_CHECK(check_device());
  cudaError_t e = launch_timeout_probe(ws_ptr<DeviceStatus>(ws, 0),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "timeout probe launch");
  return SMOE_OK;
}

SMOE_API int smoe_get_status(void* ws, void* stream) {
  SMOE_REQUIRE(ws != nullptr, SMOE_ERR_ARG, "workspace must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SMOE_CUDA(cudaStreamSynchronize(s));
  DeviceStatus st;
  SMOE_CUDA(cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost));
  SMOE_CUDA(cudaMemset(ws, 0, sizeof(st)));
  if (st.flags & kStatusTimeout)
    return fail(SMOE_ERR_DEVICE_TIMEOUT, "device wait timed out (check %d, index %lld)",
                st.first_kind, st.first_index);
  if (st.flags & kStatusData)
    return fail(SMOE_ERR_DATA, "device data out of range (check %d, index %lld)", st.first_kind,
                st.first_index);
  return SMOE_OK;
}

}  // extern "C"
