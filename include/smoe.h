/*
 * smoe.h -- C ABI of the single-GPU MoE-layer forward pass with speculative
 * token shuffling (GB300 / sm_103a).
 *
 * The layer, on one device:
 *   gate GEMM + softmax + (grouped) top-K          -> smoe_route
 *   C_p lookup -> predicted partition -> shuffle    -> smoe_predict_shuffle
 *   local activation rate alpha                     -> smoe_lar
 *   permute pairs into per-expert contiguous rows   -> smoe_dispatch
 *   x_shuf and the dispatched rows from one read    -> smoe_shuffle_dispatch_rows
 *   grouped SwiGLU expert FFN                       -> smoe_expert_ffn
 *   dispatch's row copy + expert FFN in one call    -> smoe_expert_ffn_gather
 *   weighted combine back into token order          -> smoe_combine
 *   EP all-to-all plan between simulated devices    -> smoe_ep_exchange
 *   shuffled reduce-scatter / all-gather (SRS, SAG) -> smoe_srs, smoe_sag
 *   all of the above in one call                    -> smoe_layer_forward
 *   next-layer route predictor q = LN(d + r)        -> smoe_prefetch_predict
 *
 * Sources (page title, section):
 *   "Speculative MoE" (research-notes page): §1 top-K gating and EP
 *     dispatch/combine; §2 and §7 local activation rate; §3.1 speculative token
 *     shuffling (s-TS) and Fig. 2; §4.1 token-expert confidence table C_p.
 *   "Federation of Experts (FoE)" (aitrends article): grouped MoE block -- group
 *     h owns experts [h E/H, (h+1) E/H) and takes its own top-k/H of the router
 *     output g[i]; cross-group results are summed; rho_foe = min(H/G, 1).
 *   "Speculating Experts Accelerates Inference for MoE" (gist.science summary):
 *     §2.A default vector d_l and quasi-hidden state q_l = LN_{l+1}(d_l + r_l).
 *
 * Conventions shared by every entry point
 *   - Memory: every pointer is a caller-owned DEVICE pointer unless the argument
 *     says host. The library allocates nothing; scratch space is the caller's
 *     workspace (size from smoe_workspace_size). Pointers must be 16-byte aligned
 *     (SMOE_ERR_ALIGN otherwise). Matrices are row-major and dense.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream; the return value covers
 *     host-side validation and launch errors only. Errors in device data (an id or
 *     index out of range) are recorded in the workspace status word, the offending
 *     element is skipped, and smoe_get_status reports them.
 *   - Workspace: 256-byte aligned; its first 256 bytes hold the device status
 *     word and must be zero before first use (allocate it zeroed);
 *     smoe_get_status clears it again.
 *   - Concurrency: calls that share a workspace must not overlap on the GPU.
 *   - Element type: desc->dtype selects fp32 or bf16 for activations x, weights
 *     and the outputs x_shuf/x_disp/y_disp/y; logits, weights w, C_p, r, d_l,
 *     gamma and beta are always fp32; indices are int32.
 *   - Shapes: 1 <= K <= E, H divides E and K, K/H <= E/H, 1 <= P,
 *     E <= 512, K <= 32, P <= 32, d and F multiples of 8, n_shared <= 8;
 *     T = 0 is a no-op.
 *   - Shared experts have weight indices E .. E+n_shared-1 and are never routed.
 *   - Expert weights: w1, w3 [E+n_shared, F, d]; w2 [E+n_shared, d, F].
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SMOE_API __attribute__((visibility("default")))
#else
#define SMOE_API
#endif

typedef enum smoe_status {
  SMOE_OK = 0,
  SMOE_ERR_ARG = -1,            /* null pointer or bad enum value */
  SMOE_ERR_SHAPE = -2,          /* shape relation violated */
  SMOE_ERR_ALIGN = -3,          /* pointer not 16-byte aligned */
  SMOE_ERR_WORKSPACE = -4,      /* workspace missing or smaller than smoe_workspace_size */
  SMOE_ERR_CUDA = -5,           /* a CUDA runtime call or launch failed */
  SMOE_ERR_DATA = -6,           /* device data out of range (reported by smoe_get_status) */
  SMOE_ERR_DEVICE_TIMEOUT = -7, /* a bounded device-side wait gave up */
  SMOE_ERR_UNSUPPORTED = -8     /* no sm_103a device / unsupported configuration */
} smoe_status;

typedef enum smoe_dtype { SMOE_F32 = 0, SMOE_BF16 = 1 } smoe_dtype;

/* Layer shape. T tokens, model dim d, E routed experts, K routed experts per token,
 * H expert groups (FoE; 1 = plain top-K), F expert hidden size, n_shared always-on
 * experts, P simulated expert-parallel partitions, vocab token-id range, dtype of
 * activations/weights/outputs, renorm = 1 divides the K weights by their sum. */
typedef struct smoe_desc {
  int32_t T, d, E, K, H, F, n_shared, P, vocab;
  int32_t dtype;
  int32_t renorm;
} smoe_desc;

/* Bytes of workspace that every entry point below accepts for this shape (one
 * buffer serves all of them). Returns 0 if the descriptor is invalid. */
SMOE_API size_t smoe_workspace_size(const smoe_desc* desc);

/* a1/a2 -- gate GEMM, softmax and grouped top-K ("Speculative MoE" §1: each token
 * activates its top-K experts; FoE grouped block: group h takes the top-K/H of
 * experts [h E/H, (h+1) E/H) from the same router output).
 *   x        [T, d] dtype      token activations (ignored if logits_in is set)
 *   w_gate   [E, d] dtype      router weight (ignored if logits_in is set)
 *   logits_in  nullable [T, E] fp32: route these logits instead of computing them
 *   logits_out nullable [T, E] fp32: the fp32 logits the selection was made on
 *   topk_idx [T, K] int32      group-major; within a group descending logit; equal
 *                              logits: the lower expert index wins
 *   topk_w   [T, K] fp32       softmax over all E logits, taken at topk_idx
 *                              (divided by their sum when desc->renorm = 1)
 *   ws       workspace (partial logits of the split gate GEMM); needed unless
 *            logits_in is set                                                        */
SMOE_API int smoe_route(const smoe_desc* desc, const void* x, const void* w_gate,
                        const float* logits_in, float* logits_out, int32_t* topk_idx,
                        float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* a3/a4 -- speculative token shuffle ("Speculative MoE" §3.1 s-TS and §4.1: a
 * token's experts are predicted from the token id through the confidence table
 * C_p = Pr(E_k | token); tokens are moved ahead of time to the partition of the
 * predicted experts).
 *   token_ids   [T] int32 in [0, vocab)
 *   conf        [vocab, E] fp32, C_p
 *   expert_part [E] int32 in [0, P), expert -> simulated partition
 *   x           nullable [T, d] dtype; required when x_shuf is set
 *   pred_part   [T] int32: argmax_p of sum_{e: expert_part[e]=p} C_p[id, e] (fp32 sum
 *               in ascending e; equal scores: lower p)
 *   shuf_perm   [T] int32: slot -> token, tokens grouped by pred_part, stable
 *   part_off    [P+1] int32: partition p owns slots [part_off[p], part_off[p+1])
 *   x_shuf      nullable [T, d] dtype: x_shuf[s] = x[shuf_perm[s]]
 * Out-of-range ids or map entries: the token gets partition 0 and the status word
 * records SMOE_ERR_DATA.                                                           */
SMOE_API int smoe_predict_shuffle(const smoe_desc* desc, const int32_t* token_ids,
                                  const float* conf, const int32_t* expert_part, const void* x,
                                  int32_t* pred_part, int32_t* shuf_perm, int32_t* part_off,
                                  void* x_shuf, void* ws, size_t ws_bytes, void* stream);

/* A token's cluster at this layer ("Speculative MoE" §4.1 inter-layer route prediction
 * models each token's sequence of clusters, i.e. devices, across layers): the partition
 * holding the most of its K routed experts, the lower partition on ties.
 *   topk_idx [T, K] int32, expert_part [E] int32, cluster [T] int32 out.             */
SMOE_API int smoe_token_cluster(const smoe_desc* desc, const int32_t* topk_idx,
                                const int32_t* expert_part, int32_t* cluster, void* ws,
                                size_t ws_bytes, void* stream);

/* a3/a4 with both prediction sources of "Speculative MoE" §4.1: the intra-layer C_p
 * lookup and the inter-layer 2-gram table A over the token's cluster sequence, adopting
 * the more confident one. Intra confidence = best partition score / K (fp32); inter
 * confidence = max_p table_a[prev_cluster[t], p]; A's pick (its first maximum) is
 * adopted only when strictly more confident.
 *   prev_cluster [T] int32 in [0, P): the token's cluster at the previous layer
 *   table_a      [P, P] fp32: A[c, p] = Pr(cluster p here | cluster c before)
 *   other arguments as smoe_predict_shuffle.                                         */
SMOE_API int smoe_predict_shuffle_inter(const smoe_desc* desc, const int32_t* token_ids,
                                        const float* conf, const int32_t* expert_part,
                                        const int32_t* prev_cluster, const float* table_a,
                                        const void* x, int32_t* pred_part, int32_t* shuf_perm,
                                        int32_t* part_off, void* x_shuf, void* ws,
                                        size_t ws_bytes, void* stream);

/* Workspace-free variant of smoe_predict_shuffle, for callers that cannot allocate
 * device memory: runtimes that reserve all their device memory at start-up and
 * forbid allocation afterwards, or hosts whose device memory pool belongs to another
 * framework that the library may not draw from. The pages have no counterpart; it
 * computes exactly what smoe_predict_shuffle computes, with the same arguments minus
 * the workspace.
 *   - Its histogram scratch is a 1 MB array inside the library that every GPU which
 *     loads the library holds until the process exits; T is limited to 1048576 tokens
 *     (4096 tiles of 256), larger T returns SMOE_ERR_SHAPE.
 *   - It allocates nothing and calls no allocating routine.
 *   - The first call in a CUDA context of a device (the device's primary context, and
 *     again after that context has been reset) looks up that array's device address
 *     with the device current; make that first call before any stream capture begins.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams, or different host threads) race and must be serialised by the caller.
 *     Each call clears the histogram part of the array before using it and rewrites
 *     the rest, so nothing carries over between calls.
 *   - Device data errors are not reported (there is no status word): an out-of-range
 *     token id or map entry gives partition 0, as in smoe_predict_shuffle.          */
SMOE_API int smoe_predict_shuffle_noalloc(const smoe_desc* desc, const int32_t* token_ids,
                                          const float* conf, const int32_t* expert_part,
                                          const void* x, int32_t* pred_part, int32_t* shuf_perm,
                                          int32_t* part_off, void* x_shuf, void* stream);

/* a5 -- local activation rate counts ("Speculative MoE" §2/§7: the fraction of
 * routed (token, expert) pairs whose expert sits on the token's device; FoE:
 * rho_moe = 1/G, rho_foe = min(H/G, 1)).
 *   topk_idx    [T, K] int32
 *   src_part    nullable [T] int32: the token's partition (the shuffle's pred_part).
 *               NULL selects FoE's layout: copy (t, h) of group h lives on
 *               floor(h P / H) if H >= P, else h (P/H) + (t mod P/H).
 *   expert_part [E] int32
 *   counts      [4] uint64, overwritten: {local, total = T K, base_local (contiguous
 *               split src = floor(t P / T)), max_local (sum_t max_p count)}.
 * Shared experts are not counted. alpha = local / total.                           */
SMOE_API int smoe_lar(const smoe_desc* desc, const int32_t* topk_idx, const int32_t* src_part,
                      const int32_t* expert_part, unsigned long long* counts, void* ws,
                      size_t ws_bytes, void* stream);

/* a6 -- expert permutation / dispatch ("Speculative MoE" §1: dispatch sends each
 * token to the devices of its K experts; here: into per-expert contiguous rows).
 * Pairs (t, k) are sorted by expert, stably in (slot s, k) order, where s is the
 * token's slot in the shuffle (s = t when shuf_perm is NULL).
 *   topk_idx   [T, K] int32 in [0, E)
 *   shuf_perm  nullable [T] int32 slot -> token
 *   x_src      [T, d] dtype rows in slot order (x_shuf, or x when shuf_perm is NULL)
 *   expert_off [E+1] int32: expert e owns rows [expert_off[e], expert_off[e+1])
 *   pair_row   [T, K] int32: row of pair (t, k)
 *   row_token  [T K] int32: token of each row
 *   row_slot   nullable [T K] int32: row of x_src feeding each row (its token's slot)
 *   x_disp     nullable [T K, d] dtype: x_disp[pair_row[t,k]] = x[t]               */
SMOE_API int smoe_dispatch(const smoe_desc* desc, const int32_t* topk_idx,
                           const int32_t* shuf_perm, const void* x_src, int32_t* expert_off,
                           int32_t* pair_row, int32_t* row_token, int32_t* row_slot,
                           void* x_disp, void* ws, size_t ws_bytes, void* stream);

/* a4 + a6 -- the shuffle's row copy and the dispatch's row copy from one read of x
 * ("Speculative MoE" §3.1 s-TS, Fig. 2, and §1 dispatch): for slot s and its token
 * t = shuf_perm[s] (t = s when shuf_perm is NULL),
 *   x_shuf[s] = x[t]  and  x_disp[pair_row[t, k]] = x[t] for k < K,
 * the same rows smoe_predict_shuffle(x_shuf) and smoe_dispatch(x_src = x_shuf, x_disp)
 * write, with every row of x read once instead of x_shuf being read back K times.
 *   x          [T, d] dtype
 *   shuf_perm  nullable [T] int32 slot -> token (smoe_predict_shuffle's output)
 *   pair_row   [T, K] int32 (smoe_dispatch's output for the same shuf_perm)
 *   x_shuf     nullable [T, d] dtype (needs shuf_perm)
 *   x_disp     [T K, d] dtype
 * A slot whose token is out of range gives a zero x_shuf row; a pair_row entry outside
 * [0, T K) is skipped; both record SMOE_ERR_DATA.                                    */
SMOE_API int smoe_shuffle_dispatch_rows(const smoe_desc* desc, const void* x,
                                        const int32_t* shuf_perm, const int32_t* pair_row,
                                        void* x_shuf, void* x_disp, void* ws, size_t ws_bytes,
                                        void* stream);

/* a7/a8 -- grouped SwiGLU expert FFN: for every expert e and each of its rows,
 * y = (silu(x W1_e^T) * (x W3_e^T)) W2_e^T, bf16/tf32 tensor-core products with fp32
 * accumulation, the hidden activation rounded to dtype. Shared expert j runs on all
 * T rows of x.
 *   x_disp     [T K, d] dtype (from smoe_dispatch)
 *   x          nullable [T, d] dtype (needed when n_shared > 0)
 *   expert_off [E+1] int32 (from smoe_dispatch)
 *   w1, w3     [E+n_shared, F, d] dtype;  w2 [E+n_shared, d, F] dtype
 *   y_disp     [T K, d] dtype
 *   y_shared   nullable [n_shared, T, d] dtype (needed when n_shared > 0)          */
SMOE_API int smoe_expert_ffn(const smoe_desc* desc, const void* x_disp, const void* x,
                             const int32_t* expert_off, const void* w1, const void* w3,
                             const void* w2, void* y_disp, void* y_shared, void* ws,
                             size_t ws_bytes, void* stream);

/* a6 + a7/a8 -- the dispatch's row copy and the expert FFN in one call: X_disp[r] =
 * x_src[row_slot[r]] for the T K dispatched rows, then the FFN of smoe_expert_ffn on
 * them. Where smoe_expert_ffn_gather_fused says so (bf16 two-SM tiles, at least 256 rows
 * per expert on average, F <= 1024) the copy runs inside the up GEMM, chunk by chunk
 * ahead of the tiles that read it, so the write-bound copy overlaps the tensor-core
 * work; otherwise it runs as a separate copy first.
 * Same results as smoe_dispatch(x_disp) followed by smoe_expert_ffn.
 *   x_src      [T, d] dtype rows (x_shuf, or x without a shuffle)
 *   row_slot   [T K] int32 in [0, T) (smoe_dispatch's row_slot output)
 *   x_disp     [T K, d] dtype, written (the gathered rows); may be the same buffer as
 *              y_disp, which the down GEMM writes after the up GEMM has read it
 *   x, expert_off, w1, w3, w2, y_disp, y_shared as in smoe_expert_ffn.
 * An out-of-range row_slot entry gives a zero row and SMOE_ERR_DATA in the status; a
 * copy that is not published within the device wait limit gives SMOE_ERR_DEVICE_TIMEOUT. */
SMOE_API int smoe_expert_ffn_gather(const smoe_desc* desc, const void* x_src,
                                    const int32_t* row_slot, const void* x, void* x_disp,
                                    const int32_t* expert_off, const void* w1, const void* w3,
                                    const void* w2, void* y_disp, void* y_shared, void* ws,
                                    size_t ws_bytes, void* stream);

/* 1 when smoe_expert_ffn_gather copies the rows inside the up GEMM for this layer shape,
 * 0 when it copies them before the FFN (or the descriptor is invalid). Host only. */
SMOE_API int smoe_expert_ffn_gather_fused(const smoe_desc* desc);

/* Expert-parallel exchange between P simulated devices ("Speculative MoE" §1: under
 * expert parallelism each token is sent from its device to the devices of its K
 * experts, and the results are sent back). On one GPU nothing crosses a link: this
 * builds the all-to-all plan and the P receive buffers in this GPU's memory.
 * Token t sits on device src_part[t] (the s-TS predicted partition), or on the
 * contiguous split floor(t P / T) when src_part is NULL; pair (t, k) goes to device
 * expert_part[topk_idx[t, k]]. Receive rows are sorted by (dst, src, t, k): the P
 * receive buffers are concatenated, device 0 first, each holding its sources'
 * segments in source order, each segment in the source's (t, k) order -- what an
 * all2allv delivers from send buffers laid out by (dst, t, k).
 *   topk_idx    [T, K] int32 in [0, E)
 *   src_part    nullable [T] int32 in [0, P)
 *   expert_part [E] int32 in [0, P)
 *   x           nullable [T, d] dtype (needed when x_recv is given)
 *   send_counts [P, P] int32: pairs from device p (row) to device q (column); the
 *               diagonal are the pairs that stay local (the alpha count of the same
 *               sources); every off-diagonal pair moves d elements each way
 *   recv_off    [P*P + 1] int32: segment (dst q, src p) is rows
 *               recv_off[q P + p] .. recv_off[q P + p + 1]
 *   pair_recv   [T, K] int32: receive row of pair (t, k); passing it as pair_row to
 *               smoe_combine with the expert outputs in receive order gives the
 *               combine after the return all-to-all
 *   recv_token  [T K] int32: token of each receive row
 *   x_recv      nullable [T K, d] dtype: x_recv[r] = x[recv_token[r]]
 * P <= 32. Out-of-range indices or map entries are counted as device 0 / expert 0 and
 * recorded in the status word.                                                        */
SMOE_API int smoe_ep_exchange(const smoe_desc* desc, const int32_t* topk_idx,
                              const int32_t* src_part, const int32_t* expert_part,
                              const void* x, int32_t* send_counts, int32_t* recv_off,
                              int32_t* pair_recv, int32_t* recv_token, void* x_recv, void* ws,
                              size_t ws_bytes, void* stream);

/* Shuffled reduce-scatter, SRS ("Speculative MoE" §3.1: the tensor-parallel all-reduce
 * after attention is replaced by a reduce-scatter that also moves each token to the
 * device predicted for it). x_shuf[s] = sum_{r=0}^{R-1} x_parts[r][shuf_perm[s]],
 * added in fp32 in rank order and written in the layer dtype; device p's share is slots
 * part_off[p] .. part_off[p+1] of the shuffle.
 *   x_parts   [R, T, d] dtype, the R partial sums; 1 <= R <= 64
 *   shuf_perm [T] int32 slot -> token (smoe_predict_shuffle's output)
 *   x_shuf    [T, d] dtype                                                          */
SMOE_API int smoe_srs(const smoe_desc* desc, int R, const void* x_parts,
                      const int32_t* shuf_perm, void* x_shuf, void* ws, size_t ws_bytes,
                      void* stream);

/* Shuffled all-gather, SAG ("Speculative MoE" §3.1: the way back to token order):
 * y[shuf_perm[s]] = y_shuf[s].
 *   y_shuf [T, d] dtype in slot order, shuf_perm [T] int32 (a permutation), y [T, d].
 * A shuf_perm entry out of range is skipped and recorded in the status word.       */
SMOE_API int smoe_sag(const smoe_desc* desc, const void* y_shuf, const int32_t* shuf_perm,
                      void* y, void* ws, size_t ws_bytes, void* stream);

/* a9 -- combine ("Speculative MoE" §1: results return to the token's source;
 * FoE: per-group results are summed): y[t] = sum_{k=0}^{K-1} w[t,k] y_disp[pair_row[t,k]]
 * + sum_j y_shared[j, t], accumulated in fp32 in exactly that order, one writer per
 * output row (deterministic, no atomics).
 *   y_disp [T K, d], pair_row [T, K], topk_w [T, K] fp32, y_shared nullable
 *   [n_shared, T, d], y_out [T, d] dtype. An out-of-range pair_row entry is skipped
 *   and recorded in the status word.                                                */
SMOE_API int smoe_combine(const smoe_desc* desc, const void* y_disp, const int32_t* pair_row,
                          const float* topk_w, const void* y_shared, void* y_out, void* ws,
                          size_t ws_bytes, void* stream);

/* Weights and tables of one layer (device pointers). */
typedef struct smoe_layer_weights {
  const void* w_gate;           /* [E, d] dtype */
  const void* w1;               /* [E+n_shared, F, d] dtype */
  const void* w3;               /* [E+n_shared, F, d] dtype */
  const void* w2;               /* [E+n_shared, d, F] dtype */
  const float* conf;            /* [vocab, E] fp32, C_p */
  const int32_t* expert_part;   /* [E] int32 */
} smoe_layer_weights;

/* Inputs and outputs of one layer call (device pointers). Every optional output,
 * when non-NULL, receives the intermediate of the same name described above; when
 * NULL that intermediate lives in the workspace. */
typedef struct smoe_layer_io {
  const void* x;                /* [T, d] dtype */
  const int32_t* token_ids;     /* [T] */
  void* y;                      /* [T, d] dtype, layer output */
  float* logits;                /* optional [T, E] */
  int32_t* topk_idx;            /* optional [T, K] */
  float* topk_w;                /* optional [T, K] */
  int32_t* pred_part;           /* optional [T] */
  int32_t* shuf_perm;           /* optional [T] */
  int32_t* part_off;            /* optional [P+1] */
  int32_t* expert_off;          /* optional [E+1] */
  int32_t* pair_row;            /* optional [T, K] */
  int32_t* row_token;           /* optional [T K] */
  unsigned long long* lar;      /* optional [4], as smoe_lar with src_part = pred_part */
  int32_t skip_shuffle;         /* 1: dispatch straight from x (no s-TS shuffle) */
} smoe_layer_io;

/* The whole layer: route -> predict/shuffle -> (lar) -> dispatch -> expert FFN ->
 * combine, on one stream, in that order. */
SMOE_API int smoe_layer_forward(const smoe_desc* desc, const smoe_layer_weights* weights,
                                const smoe_layer_io* io, void* ws, size_t ws_bytes,
                                void* stream);

/* The whole layer from HOST buffers: copies x_host [T, d] and ids_host [T] (pinned
 * host memory for asynchronous copies) into the workspace, runs smoe_layer_forward
 * and copies y back to y_host [T, d], all on `stream`. Returns after enqueueing; the
 * caller synchronises the stream before reading y_host. */
SMOE_API int smoe_layer_forward_host(const smoe_desc* desc, const smoe_layer_weights* weights,
                                     const void* x_host, const int32_t* ids_host, void* y_host,
                                     void* ws, size_t ws_bytes, void* stream);

/* a10 -- next-layer prefetch predictor ("Speculating Experts ..." §2.A): the
 * quasi-hidden state q = LN(d_l + r) stands in for the next router input
 * s = LN(r + y); both are rounded to dtype and routed by w_gate_next with the layer's
 * rule (desc->K, desc->H); hits = sum_t |pred_t intersect true_t|.
 *   r [T, d] fp32 residual; d_l [d] fp32 default vector; y [T, d] dtype layer output;
 *   gamma, beta [d] fp32 (LayerNorm over d, biased variance, eps 1e-5);
 *   w_gate_next [E, d] dtype; logits_q, logits_s nullable [T, E] fp32;
 *   pred_idx, true_idx [T, K] int32; hits [1] uint64, overwritten;
 *   qs_out nullable [2, T, d] dtype: the q rows then the s rows (else kept in ws).
 * Requires d <= 8192 (the LayerNorm holds a row in registers); else SMOE_ERR_SHAPE.  */
SMOE_API int smoe_prefetch_predict(const smoe_desc* desc, const float* r, const float* d_l,
                                   const void* y, const float* gamma, const float* beta,
                                   const void* w_gate_next, float* logits_q, float* logits_s,
                                   int32_t* pred_idx, int32_t* true_idx,
                                   unsigned long long* hits, void* qs_out, void* ws,
                                   size_t ws_bytes, void* stream);

/* The MoE body with routes supplied by the caller: dispatch (token order, no shuffle),
 * grouped SwiGLU FFN (shared experts included) and combine. With the routes predicted
 * by smoe_prefetch_predict this is speculative execution ("Speculating Experts ..."
 * §2.B: the predicted experts run instead of the router's true ones).
 *   x [T, d] dtype; topk_idx [T, K] int32 in [0, E); topk_w [T, K] fp32;
 *   w1, w3, w2 as smoe_expert_ffn; y [T, d] dtype out.                                */
SMOE_API int smoe_moe_forward_routed(const smoe_desc* desc, const void* x,
                                     const int32_t* topk_idx, const float* topk_w,
                                     const void* w1, const void* w3, const void* w2, void* y,
                                     void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, returns SMOE_OK, SMOE_ERR_DATA or SMOE_ERR_DEVICE_TIMEOUT from
 * the workspace status word, and clears it. */
SMOE_API int smoe_get_status(void* ws, void* stream);

/* Self-test of the device-side failure path (the pages have no counterpart): one
 * kernel waits on an mbarrier that nothing arrives at; the wait is the bounded wait
 * every kernel uses (2 s), so it gives up, records a device timeout in the status word
 * of `ws` and returns. The context stays usable; the next smoe_get_status(ws) returns
 * SMOE_ERR_DEVICE_TIMEOUT. ws: any workspace of at least 256 bytes, zeroed status word. */
SMOE_API int smoe_selftest_device_timeout(void* ws, size_t ws_bytes, void* stream);

/* Static description of a status code. */
SMOE_API const char* smoe_status_string(int status);

/* Message of the last failing call on this host thread ("" if none). */
SMOE_API const char* smoe_last_error(void);

/* Number of kernels this host thread has launched through the library so far
 * (a monotone counter; the difference across a call is that call's launches). */
SMOE_API unsigned long long smoe_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* SMOE_H */
