/* The C ABI from plain C, with no Python or PyTorch in the process.
 *
 * Without arguments: host-side checks that need no GPU (workspace size, argument
 * validation). With "gpu": one small fp32 layer through smoe_layer_forward_host, its
 * routing outputs checked for their invariants and its output rows checked against a
 * direct C evaluation of the layer's definition (gate logits, softmax, top-K, SwiGLU
 * experts, weighted sum) on tokens whose top-K margin is not tiny. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "smoe.h"

enum { T = 64, D = 128, E = 8, K = 2, F = 256, P = 2, V = 97 };

static int failures = 0;
#define CHECK(cond, ...)                     \
  do {                                       \
    if (!(cond)) {                           \
      fprintf(stderr, "FAIL: " __VA_ARGS__); \
      fprintf(stderr, "\n");                 \
      ++failures;                            \
    }                                        \
  } while (0)

static unsigned long long rng_state = 12345;
static float uniform(void) { /* 64-bit LCG, top 24 bits */
  rng_state = rng_state * 6364136223846793005ULL + 1442695040888963407ULL;
  return (float)((rng_state >> 40) & 0xFFFFFF) / 16777216.0f;
}
static float normalish(void) { return (uniform() + uniform() + uniform() - 1.5f) * 2.0f; }

static void fill(float* p, size_t n, float scale) {
  for (size_t i = 0; i < n; ++i) p[i] = normalish() * scale;
}

static void* to_device(const void* h, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice);
  return d;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

int main(int argc, char** argv) {
  smoe_desc desc = {T, D, E, K, 1, F, 0, P, V, SMOE_F32, 0};
  size_t ws_bytes = smoe_workspace_size(&desc);
  CHECK(ws_bytes > 0, "workspace size of a valid descriptor");
  smoe_desc bad = desc;
  bad.K = E + 1;
  CHECK(smoe_workspace_size(&bad) == 0, "K > E must be rejected");
  CHECK(smoe_route(&desc, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == SMOE_ERR_ARG,
        "NULL pointers must be rejected before any CUDA call");
  CHECK(smoe_status_string(SMOE_ERR_SHAPE) != NULL, "status strings");
  if (argc < 2 || strcmp(argv[1], "gpu") != 0) {
    printf(failures ? "abi_demo host checks FAILED\n" : "abi_demo host checks ok\n");
    return failures ? 1 : 0;
  }

  /* weights and tables (device), activations and ids (pinned host) */
  float* wg = malloc(sizeof(float) * E * D);
  float* w1 = malloc(sizeof(float) * E * F * D);
  float* w3 = malloc(sizeof(float) * E * F * D);
  float* w2 = malloc(sizeof(float) * E * D * F);
  float* conf = malloc(sizeof(float) * V * E);
  int32_t emap[E];
  fill(wg, (size_t)E * D, 1.0f / sqrtf((float)D));
  fill(w1, (size_t)E * F * D, 1.0f / sqrtf((float)D));
  fill(w3, (size_t)E * F * D, 1.0f / sqrtf((float)D));
  fill(w2, (size_t)E * D * F, 1.0f / sqrtf((float)F));
  for (int v = 0; v < V; ++v) {
    float s = 0.0f;
    for (int e = 0; e < E; ++e) s += (conf[v * E + e] = uniform() + 0.01f);
    for (int e = 0; e < E; ++e) conf[v * E + e] *= (float)K / s;
  }
  for (int e = 0; e < E; ++e) emap[e] = e % P;
  float *x_h = NULL, *y_h = NULL;
  int32_t* ids_h = NULL;
  cudaMallocHost((void**)&x_h, sizeof(float) * T * D);
  cudaMallocHost((void**)&y_h, sizeof(float) * T * D);
  cudaMallocHost((void**)&ids_h, sizeof(int32_t) * T);
  fill(x_h, (size_t)T * D, 1.0f);
  for (int t = 0; t < T; ++t) ids_h[t] = (t * 7) % V;

  smoe_layer_weights W;
  W.w_gate = to_device(wg, sizeof(float) * E * D);
  W.w1 = to_device(w1, sizeof(float) * E * F * D);
  W.w3 = to_device(w3, sizeof(float) * E * F * D);
  W.w2 = to_device(w2, sizeof(float) * E * D * F);
  W.conf = to_device(conf, sizeof(float) * V * E);
  W.expert_part = to_device(emap, sizeof(emap));
  void* ws = NULL;
  CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess, "workspace allocation");
  cudaMemset(ws, 0, ws_bytes);
  int rc = smoe_layer_forward_host(&desc, &W, x_h, ids_h, y_h, ws, ws_bytes, NULL);
  CHECK(rc == SMOE_OK, "smoe_layer_forward_host: %s", smoe_last_error());
  cudaDeviceSynchronize();
  CHECK(smoe_get_status(ws, NULL) == SMOE_OK, "device status: %s", smoe_last_error());

  /* the layer's definition in double precision, token by token */
  int checked = 0;
  double worst = 0.0;
  for (int t = 0; t < T; ++t) {
    double logit[E], mx = -1e300, sum = 0.0;
    for (int e = 0; e < E; ++e) {
      double a = 0.0;
      for (int j = 0; j < D; ++j) a += (double)x_h[t * D + j] * wg[e * D + j];
      logit[e] = a;
      if (a > mx) mx = a;
    }
    for (int e = 0; e < E; ++e) sum += exp(logit[e] - mx);
    int pick[K];
    int taken[E] = {0};
    for (int k = 0; k < K; ++k) { /* largest logit first, lower index on ties */
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || logit[e] > logit[best])) best = e;
      pick[k] = best;
      taken[best] = 1;
    }
    double next = -1e300; /* the (K+1)-th logit: skip tokens near a routing tie */
    for (int e = 0; e < E; ++e)
      if (!taken[e] && logit[e] > next) next = logit[e];
    if (logit[pick[K - 1]] - next < 1e-3) continue;
    double y[D];
    memset(y, 0, sizeof(y));
    for (int k = 0; k < K; ++k) {
      const int e = pick[k];
      const double w = exp(logit[e] - mx) / sum;
      double h[F];
      for (int f = 0; f < F; ++f) {
        double a = 0.0, b = 0.0;
        for (int j = 0; j < D; ++j) {
          a += (double)x_h[t * D + j] * w1[((size_t)e * F + f) * D + j];
          b += (double)x_h[t * D + j] * w3[((size_t)e * F + f) * D + j];
        }
        h[f] = silu(a) * b;
      }
      for (int j = 0; j < D; ++j) {
        double o = 0.0;
        for (int f = 0; f < F; ++f) o += h[f] * w2[((size_t)e * D + j) * F + f];
        y[j] += w * o;
      }
    }
    double err = 0.0, ref = 0.0;
    for (int j = 0; j < D; ++j) {
      const double dlt = fabs((double)y_h[t * D + j] - y[j]);
      if (dlt > err) err = dlt;
      if (fabs(y[j]) > ref) ref = fabs(y[j]);
      CHECK(isfinite(y_h[t * D + j]), "non-finite output");
    }
    if (err / ref > worst) worst = err / ref;
    ++checked;
  }
  CHECK(checked > T / 2, "too few tokens checked (%d)", checked);
  CHECK(worst <= 2e-2, "max row relative error %.3e", worst);
  printf("abi_demo gpu: %d tokens checked, max row relative error %.2e, %s\n", checked, worst,
         failures ? "FAILED" : "ok");
  return failures ? 1 : 0;
}
