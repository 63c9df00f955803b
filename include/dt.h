/* dt.h - C ABI of the GB300 dynamic draft-tree library (libdt.so).
 *
 * The library runs the batched hot path of dynamic draft-tree speculative
 * decoding between the draft and the target model forwards:
 *
 *   EAGLE-2 ("EAGLE-2 完全拆解：动态草稿树如何让投机解码上下文感知"):
 *     vocab softmax + top-K per expanded node, path value as the product of
 *     confidences (kept as a sum of logs), frontier top-k expansion
 *     (§"扩展阶段"), global top-m rerank with shallow-first ties giving a
 *     connected subtree, flattening with an ancestor-only mask (§"重排阶段"),
 *     greedy and speculative-sampling acceptance along the tree with a bonus
 *     token (§"先把投机解码的账本摆清楚", §"无损性为什么没有被动态树破坏").
 *   CAST ("Inference-Cost-Aware Dynamic Tree Construction for Efficient
 *     Inference in Large Language Models", §关键设计 1-4): cost-table driven
 *     width, depth and verify-count pruning.
 *   Graft ("Draft Less, Retrieve More: Hybrid Tree Construction for
 *     Speculative Decoding", method steps (1)-(3)): confidence checkpoints,
 *     retrieval graft from a GPU-resident adjacency matrix M[V][8], online
 *     refresh of M from the target rows.
 *
 * Conventions (every entry point):
 *   - Every array argument is a DEVICE pointer, allocated and owned by the
 *     caller, unless the comment says "host". The library keeps no pointer
 *     past the call.
 *   - Calls are asynchronous on the caller's stream. A handle holds one draft
 *     tree; using one handle from two streams at once is a race.
 *   - Return value: DT_OK (0) or a negative DT_ERR_* code. DT_ERR_ARG means
 *     the host-side argument check failed and nothing was launched;
 *     dt_last_error_string() (thread-local) says why. DT_ERR_CUDA is a launch
 *     or runtime error.
 *   - Errors found on the device (bad logits, bad tokens, a bounded wait that
 *     ran out) are OR-ed into the handle's sticky status word; read it with
 *     dt_get_status(), which synchronises the given stream. Kernels never trap.
 *   - Row-major contiguous layouts; logits rows are `ld` elements apart.
 *   - Only dt_create allocates (device workspace sized from the config
 *     maxima). Hot calls allocate nothing.
 *
 * Limits (checked, DT_ERR_ARG otherwise): 2 <= V < 2^31, 1 <= K <= 32,
 * K <= V, 1 <= W <= 32, W*K <= 1024, 1 <= D_max <= 16, 1 <= P_max <= 512,
 * 1 <= B_max <= 4096.
 */
#ifndef DT_H_
#define DT_H_

#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { DT_OK = 0, DT_ERR_ARG = -1, DT_ERR_CUDA = -2, DT_ERR_DEVICE = -3, DT_ERR_DEVICE_TIMEOUT = -4 };
enum { DT_BF16 = 0, DT_F32 = 1 };
enum { DT_GREEDY = 0, DT_SAMPLE = 1 };
/* OR-ed into the verify mode: padding-free target rows. Request b's used rows are packed after those
 * of requests 0..b-1: row (b, i) is row row_off[b] + i of the logits buffer, with
 * row_off[b] = n_pos[0] + ... + n_pos[b-1] (dt_tree_meta.row_off), so a ragged batch's target
 * forward computes and stores sum_b n_pos[b] rows instead of B * P. */
enum { DT_VERIFY_PACKED = 2 };
enum {
  DT_POLICY_CAST_WIDTH_DEPTH = 0, /* CAST width n_d and grow/stop after layer d */
  DT_POLICY_CAST_VERIFY = 1,      /* CAST batch-wide verify count m            */
  DT_POLICY_GRAFT_CHECKPOINT = 2, /* Graft confidence checkpoint after layer d */
  DT_POLICY_NONE = 3              /* no pruning (EAGLE-2): dt_expand_prune_select only */
};
/* Bits of the device status word. */
enum {
  DT_DEV_BAD_LOGITS = 1,   /* a row read by a kernel holds NaN or +inf, or has no finite entry */
  DT_DEV_BAD_TOKEN = 2,    /* a token id outside [0, V) where a token was required            */
  DT_DEV_BAD_TREE = 4,     /* selection not parent-closed, or a tree deeper than D_path - 1    */
  DT_DEV_TIMEOUT = 8,      /* a bounded wait on an asynchronous copy ran out                   */
  DT_DEV_INTERNAL = 16,    /* an internal iteration bound was hit                              */
  DT_DEV_KV_FULL = 32      /* dt_commit_kv: a request's rows would pass the cache's capacity   */
};
/* dt_config.flags */
enum { DT_FLAG_TEST_TIMEOUT = 1 }; /* test only: the expansion row scans (dt_expand_layer and the
                                      calls built on it, dt_block_expand) give their first bounded
                                      copy wait a limit of zero, so it runs out; the verify streaming
                                      pass behaves as if its reads had timed out (reads nothing).
                                      Either way empty results and DT_DEV_TIMEOUT, no fault */

typedef struct dt_handle dt_handle;

typedef struct {
  int32_t B_max;  /* largest batch                                                  */
  int32_t V;      /* vocabulary size                                                */
  int32_t K;      /* per-node top-K (children per expanded node)                    */
  int32_t W;      /* largest frontier width k (nodes expanded per layer)            */
  int32_t D_max;  /* largest number of draft layers (the root is depth 0)          */
  int32_t P_max;  /* largest verify positions per request (root + nodes)            */
  int32_t dtype;  /* DT_BF16 or DT_F32: element type of every logits buffer         */
  int32_t flags;  /* DT_FLAG_*                                                      */
} dt_config;

/* Read-only view of the handle's draft tree (device pointers into the workspace).
 * Node-id layout: root = 0; layer 1 = ids 1..K; layer d >= 2 = ids
 * base(d) .. base(d)+W*K-1 with base(d) = 1 + K + (d-2)*W*K; the child of
 * rank r of frontier slot f in layer d is base(d) + f*K + r. Frontier slots
 * hold the selected frontier nodes in ascending id. Invalid slots have
 * token -1, parent -1, logc = value = -inf. Values are log path values
 * (sum of log confidences), fp32. */
typedef struct {
  int32_t B, K, W, D_max, N, LW; /* N = nodes per request, LW = W*K slots per layer (>= K)   */
  int32_t depth;                 /* layers built so far                                        */
  const int32_t* token;          /* [B_max][N]                                                 */
  const int32_t* parent;         /* [B_max][N] node id of the parent, -1 for root/invalid     */
  const int32_t* node_depth;     /* [B_max][N] layer of the slot                               */
  const float* logc;             /* [B_max][N] log confidence                                  */
  const float* value;            /* [B_max][N] log path value                                  */
  const int32_t* layer_order;    /* [B_max][D_max+1][LW] layer d's valid ids by (value desc,
                                    id asc), -1 padded                                         */
  const int32_t* layer_count;    /* [B_max][D_max+1] valid nodes per layer                     */
  const int32_t* frontier;       /* [B_max][W] ids of the current frontier, -1 padded          */
  const int32_t* frontier_count; /* [B_max]                                                    */
} dt_tree_view;

/* CAST / Graft pruning parameters (host struct; the tables are device arrays). */
typedef struct {
  /* CAST (cost tables f(B, c, n) for the running batch size B) */
  const double* S_T;  /* device [M_rows][N_cols]: target cost; column n-1 holds input length n */
  const double* S_D;  /* device [M_rows][N_cols]: draft cost                                   */
  int32_t M_rows, N_cols;
  double L;           /* context grid step: row = min(floor(c / L), M_rows - 1)                */
  int64_t n0;         /* prefix (context) length                                              */
  double C1, C2, C3;  /* width, depth and verify-count thresholds                             */
  int32_t R;          /* FIFO length of the depth ratio buffer, 1..16                         */
  int32_t width_cap;  /* largest width n_d, <= min(W, N_cols)                                  */
  int32_t m_cap;      /* largest verify count m, <= N_cols                                     */
  int32_t D_max;      /* last layer: no growth after it                                        */
  /* Graft */
  int32_t n_ckpt;        /* number of checkpoints, 0..16 (a block drafter may gate every position) */
  int32_t ckpt_layer[16];/* checkpoint layer indices (layer index 0 = draft layer 1)            */
  double tau[16];        /* confidence thresholds: request continues iff exp(max value) > tau   */
  int32_t k_draft[16];   /* draft nodes kept when stopped at checkpoint s                       */
  int32_t K_total;      /* K_max: draft + retrieved nodes per request                         */
  /* CAST, per-request rule (CAST page §局限与展望: padded equal-length batches are a limit of the
   * batch rule): nonzero = every request applies the width/depth and verify-count rules to its own
   * utilities, context, FIFO and stop; width, stop and m are then [B] outputs. */
  int32_t per_request;
} dt_prune_params;

/* Outputs of dt_cast_prune (device pointers; NULL where a policy does not write). */
typedef struct {
  int32_t* width; /* [1]  CAST_WIDTH_DEPTH: n_d ([B] with per_request)                     */
  int32_t* stop;  /* [B]  CAST_WIDTH_DEPTH: 1 = do not grow (batch-wide, or per request with
                          per_request: a stopped request stays stopped); GRAFT: per request,
                          set once a request stops                                          */
  int32_t* m;     /* [1]  CAST_VERIFY: m ([B] with per_request); [B] GRAFT: K_draft of each
                          request (set on stop)                                             */
  int32_t* stage; /* [B]  GRAFT: checkpoint index that stopped the request, n_ckpt if none  */
} dt_prune_out;

/* Template anchors (Graft page: root-grafted G_ret^root and tail-grafted G_ret^tail templates). */
enum { DT_ANCHOR_ROOT = 0, DT_ANCHOR_TAIL = 1 };
/* Retrieval template (host arrays), nodes in breadth-first order:
 * parent[u] in [-1, u) (-1 = the template root), rank[u] in [0, 8): x_u = M[x_parent][rank]. n <= 256.
 * anchor: DT_ANCHOR_ROOT = the template root is the tree's root; DT_ANCHOR_TAIL = it is the deepest
 * kept draft node (ties: value desc, then id asc), the end of the kept draft path (a block drafter's
 * kept prefix). Any shape a caller designs or learns fits these arrays. */
typedef struct {
  int32_t n;
  const int32_t* parent;
  const int32_t* rank;
  int32_t anchor;
} dt_template;

/* Flattened verify tree (device arrays, caller-owned), P positions per request. */
typedef struct {
  int32_t P;             /* positions per request = row stride of every [B][P] array     */
  int32_t D_path;        /* width of a retrieve row (>= deepest position + 1)            */
  int32_t* tokens;       /* [B][P] token, -1 for an invalid node or an unused position   */
  int32_t* parents;      /* [B][P] parent position, -1 for the root / unused             */
  int32_t* depth;        /* [B][P] depth (root 0), -1 unused                             */
  int32_t* node_id;      /* [B][P] draft-tree node id, -1 for retrieved / unused          */
  uint8_t* mask;         /* [B][P][P] 1 iff column is an ancestor-or-self of the row     */
  int32_t* position_ids; /* [B][P] pos_offset + depth, -1 unused                        */
  int32_t* retrieve;     /* [B][P][D_path] root-to-leaf positions, -1 padded              */
  int32_t* n_leaves;     /* [B]                                                           */
  int32_t* n_pos;        /* [B] positions in use                                          */
  int32_t* row_off;      /* [B+1] or NULL: exclusive prefix sums of n_pos (row_off[B] = total),
                            the packed target-row offsets of DT_VERIFY_PACKED                */
} dt_tree_meta;

const char* dt_last_error_string(void);

/* Create a handle and its workspace (the only allocating call). */
int dt_create(const dt_config* cfg, dt_handle** out);
int dt_destroy(dt_handle* h);
int dt_get_tree(const dt_handle* h, dt_tree_view* out);
/* Synchronise `s`, then OR-ed DT_DEV_* bits since the last clear; returns DT_ERR_DEVICE or
 * DT_ERR_DEVICE_TIMEOUT when bits are set, DT_OK otherwise. */
int dt_get_status(dt_handle* h, cudaStream_t s, int32_t* device_bits);
int dt_clear_status(dt_handle* h, cudaStream_t s);

/* Start a round for B <= B_max requests: root node = root_token[b] (depth 0, value 0), every
 * other slot invalid, the frontier = {root}, CAST state reset (FIFO = {1}). */
int dt_tree_reset(dt_handle* h, int32_t B, const int32_t* root_token, cudaStream_t s);

/* a2 (EAGLE-2 §扩展阶段): choose the frontier of the next layer: for request b, the first
 * w_b nodes of the newest layer in (value desc, id asc) order, slotted in ascending id. Right
 * after dt_tree_reset the newest layer is layer 0 = {root}: the call then gives the frontier of
 * layer 1 (the root in slot 0, its token in frontier_token[b][0]).
 * w_b = min(width, W, nodes in the layer), 0 where stop[b] != 0. width: device [width_len]
 * with width_len 1 (batch-wide) or B, or NULL for W. stop: device [B] or NULL.
 * frontier_token: device [B][W] out (tokens of the slots, -1 padded) or NULL. */
int dt_select_frontier(dt_handle* h, const int32_t* width, int32_t width_len, const int32_t* stop,
                       int32_t* frontier_token, cudaStream_t s);

/* a1 + a2 (EAGLE-2 §置信度…, §value 公式, §扩展阶段): expand the current frontier into the
 * next layer. logits: device [B][F][V] of dtype, row (b, f) at element (b*F + f)*ld, the draft
 * row of frontier slot f (F = 1 for layer 1, rows f >= frontier_count[b] are not read).
 * Per row: m = max, S = sum exp(x - m), the K largest logits (ties: lower id) become children
 * with log c = x - m - log S and value = value(parent) + log c; then the new layer is ordered
 * by (value desc, id asc). A NaN/+inf row or a row without a finite entry sets
 * DT_DEV_BAD_LOGITS. */
int dt_expand_layer(dt_handle* h, const void* logits, int64_t ld, int32_t F, cudaStream_t s);

/* a3/a4: CAST (width/depth after the newest layer, or verify count) or Graft checkpoint.
 * CAST width (page 2 §关键设计 2): u_k = (1/B) sum_b sum_{s<=k} exp(value of the s-th node of
 * b's newest layer), c_k = S_D[row][k-1] / S_T[row][0] with row from ctx = n0 + widths so far;
 * k0 = 1, for k = 2..min(width_cap, candidates): k0 = k if c_k <= c_k0 or
 * (u_k - u_k0)/(c_k - c_k0) >= C1; n_d = k0 -> out->width[0].
 * CAST depth (§关键设计 3): after layer d >= 2 push u(d)/u(d-1) into a FIFO of length R
 * (initial {1}); grow iff d < D_max and mean(FIFO) * u_{n_d} / c_{n_d} >= C2; out->stop[b] = !grow.
 * CAST verify (§关键设计 4): same rule over all nodes of each request in the total order with
 * c_k = S_T[row(n0)][k-1] / S_T[row(n0)][0], C3, cap m_cap -> out->m[0].
 * Graft (page 3 step (1)): for every running request, if the newest layer index is checkpoint s
 * and not exp(max value) > tau[s]: stop[b] = 1, stage[b] = s, m[b] = k_draft[s]; a request that
 * reaches D_max gets stage n_ckpt and m = K_total. */
int dt_cast_prune(dt_handle* h, int32_t policy, const dt_prune_params* p, const dt_prune_out* out,
                  cudaStream_t s);

/* a1 + a2, then a3/a4, then the next frontier, as one call: exactly
 *   dt_expand_layer(h, logits, ld, F, s);
 *   policy DT_POLICY_CAST_WIDTH_DEPTH: dt_cast_prune_select(h, p, out, frontier_token, s)
 *     (after the last layer, D_max: dt_cast_prune(h, policy, p, out, s) alone);
 *   policy DT_POLICY_GRAFT_CHECKPOINT: dt_cast_prune(h, policy, p, out, s), then
 *     dt_select_frontier(h, width, width_len, out->stop, frontier_token, s);
 *   policy DT_POLICY_NONE (EAGLE-2, no pruning): dt_select_frontier(h, width, width_len, NULL,
 *     frontier_token, s);
 * no frontier is selected once the tree has D_max layers. width: device [width_len] (1 or B) or
 * NULL for W; p and out may be NULL for DT_POLICY_NONE. */
int dt_expand_prune_select(dt_handle* h, const void* logits, int64_t ld, int32_t F, int32_t policy,
                           const dt_prune_params* p, const dt_prune_out* out, const int32_t* width,
                           int32_t width_len, int32_t* frontier_token, cudaStream_t s);

/* Block drafters (Graft page, extension direction 1; weakness 4: token-level confidence inside the
 * block): draft layers 1..L in one call from a block drafter's rows. logits: device [B][L][V] of dtype,
 * row (b, j) at element (b*L + j)*ld, the drafter's distribution for block position j + 1 (the same
 * whatever tokens are picked at earlier positions). Layer j + 1 = the top-K tokens of row j (log c,
 * ties and the DT_DEV_BAD_LOGITS rule as in dt_expand_layer), children of the block token at position
 * j (the root for j = 0), the block token being the top node of its layer (value desc, id asc), i.e.
 * the top-1 of its row; they occupy frontier slot 0's ids. Values: value(parent) + log c. With p and
 * out (Graft checkpoint parameters and outputs, as dt_cast_prune with DT_POLICY_GRAFT_CHECKPOINT):
 * the checkpoint rule after every layer; a request stopped after layer j keeps layers 1..j only
 * (deeper slots invalid) and has no frontier; one that passes layer L gets stage n_ckpt and m =
 * K_total (layer L plays the part of p->D_max); stop, stage and m are written for every request.
 * p == NULL: no gate, L layers. Needs the tree right after dt_tree_reset, 1 <= L <= D_max and
 * B * L <= B_max * max(W, P_max). The tree then has L layers; the frontier is the block token of
 * layer L - 1 (the root if L = 1). One row pass over the B*L rows (the expansion's kernel design);
 * the last row of a request to finish builds its layers, values, layer orders and gates. */
int dt_block_expand(dt_handle* h, const void* logits, int64_t ld, int32_t L, const dt_prune_params* p,
                    const dt_prune_out* out, cudaStream_t s);

/* Sampled drafts (EAGLE-2 page, §先把投机解码的账本摆清楚: drafted tokens drawn from the draft
 * distribution q and tested with min(1, p/q)): dt_expand_layer with the K children of each expanded
 * node drawn from softmax(row) without replacement, i.e. the first K tokens by x_v + G_v (ties: lower
 * id), G_v = -log(-log u_v), u_v = (k + 1/2) 2^-23 with k the top 23 bits of word v & 3 of
 * Philox4x32-10(key seed; counter (round lo, round hi, 0x40000000 + 4096 b + node, v >> 2)); the
 * children are in draw order (rank r = the r-th draw), log c = log softmax(row)[token]. Each expanded
 * node records its row's slot and softmax statistics for dt_verify_sampled. Needs N <= 4096.
 * For dt_verify_sampled the rows of every layer must stay in one buffer draft_rows [D_max][B][W][ld_d]:
 * pass logits = draft_rows + (d - 1) * B * W * ld_d and F = W for layer d (layer 1 too; rows past the
 * frontier are not read). */
int dt_expand_layer_sampled(dt_handle* h, const void* logits, int64_t ld, int32_t F, uint64_t seed, uint64_t round,
                            cudaStream_t s);

/* a3 + a2 in one launch: exactly dt_cast_prune(h, DT_POLICY_CAST_WIDTH_DEPTH, p, out, s) followed by
 * dt_select_frontier(h, out->width, 1, out->stop, frontier_token, s): CAST width and grow/stop after
 * the newest layer, then the next layer's frontier (none for stopped requests). One kernel instead of
 * two dependent ones between the draft forwards. */
int dt_cast_prune_select(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out, int32_t* frontier_token,
                         cudaStream_t s);

/* a3 (verify count) + a5 in two launches instead of three: exactly
 * dt_cast_prune(h, DT_POLICY_CAST_VERIFY, p, out, s) followed by
 * dt_rerank(h, out->m, 1, p->m_cap, selected, s). selected: device [B][p->m_cap]. */
int dt_cast_verify_rerank(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out, int32_t* selected,
                          cudaStream_t s);

/* a5 (EAGLE-2 §重排阶段): top-m_b valid non-root nodes in (value desc, depth asc, id asc) order,
 * written in ascending id. m: device [m_len] (m_len 1 = batch-wide, or B), NULL = m_cap.
 * selected: device [B][m_cap], -1 padded. */
int dt_rerank(dt_handle* h, const int32_t* m, int32_t m_len, int32_t m_cap, int32_t* selected,
              cudaStream_t s);

/* a6 (Graft step (2)): gather the retrieval envelope, the first e = min(tpl->n, R_cap) template nodes,
 * from M (device [B][V][8] int32, -1 = unset): token(u) = M[b][token(parent(u))][rank(u)], the template
 * root's token being that of the anchor; -1 when the parent is invalid or the entry unset. The cut to
 * K_ret = K_total - kept draft nodes is made by dt_build_tree_meta. With DT_ANCHOR_ROOT the call
 * depends on the root tokens and M only (selected may be NULL): it can be issued right after
 * dt_tree_reset, on a second stream, while the draft layers are built (step (2): retrieval adds no
 * serial stage). With DT_ANCHOR_TAIL it needs the kept draft nodes, selected (device [B][m_cap], as
 * written by dt_rerank), and follows the rerank.
 * ret_token/ret_parent: device [B][R_cap] (parent = template parent index, -1 the template root, -2
 * unused); ret_count: device [B] (= e); ret_anchor: device [B] (the anchor's node id, 0 = the root) or
 * NULL. */
int dt_graft_retrieve(dt_handle* h, const int32_t* M, const dt_template* tpl, int32_t R_cap, const int32_t* selected,
                      int32_t m_cap, int32_t* ret_token, int32_t* ret_parent, int32_t* ret_count,
                      int32_t* ret_anchor, cudaStream_t s);

/* a7 (EAGLE-2 §重排阶段; Graft step (3)): flatten and build the verify metadata. Position 0 is
 * the root, then selected nodes (device [B][m_cap], ascending id, -1 padded), then retrieved
 * nodes (ret_*: device, NULL when there is no graft) in template order: the first
 * min(ret_count[b], K_total - selected nodes) of them (all ret_count[b] when K_total <= 0), the
 * template root's children hanging from the position of draft node ret_anchor[b] (NULL: the root;
 * an anchor that is not selected sets DT_DEV_BAD_TREE and the root is used). pos_offset: device [B]
 * or NULL (0). Needs 1 + m_cap <= meta->P; a request whose root + selected + retrieved nodes
 * exceed P sets DT_DEV_BAD_TREE and keeps the first P positions. meta->row_off, when not NULL,
 * receives the packed row offsets (DT_VERIFY_PACKED). */
int dt_build_tree_meta(dt_handle* h, const int32_t* selected, int32_t m_cap, const int32_t* ret_token,
                       const int32_t* ret_parent, const int32_t* ret_count, const int32_t* ret_anchor,
                       int32_t R_cap, int32_t K_total, const int32_t* pos_offset, const dt_tree_meta* meta,
                       cudaStream_t s);

/* a8 + a9 (EAGLE-2 §先把投机解码的账本摆清楚, §无损性…): verify against the target rows
 * logits: device [B][P][V], row (b, i) at element (b*P + i)*ld, the target row after position i;
 * with mode | DT_VERIFY_PACKED: device [sum_b n_pos[b]][V], row (b, i) at element
 * (n_pos[0] + ... + n_pos[b-1] + i)*ld: a ragged batch without padding (CAST page §局限与展望).
 * DT_GREEDY: longest leaf path whose tokens equal the argmax (ties: lower id) of their parent's
 * row (ties: first path), bonus = argmax of the last accepted position's row.
 * DT_SAMPLE: from the root, children in position order are accepted with probability
 * P_res(x) (point-mass proposals), P_res = softmax(row) with rejected tokens removed,
 * u = Philox4x32-10(key seed; counter (round, 512*b + j, 0x80000000)) top 24 bits; the bonus is
 * a Gumbel-max draw from the final residual (23-bit uniforms, counter (round, 512*b + i, v>>2),
 * word v&3). accept_len: [B]; accept_path: [B][D_path] positions (root first, -1 padded);
 * bonus: [B]; top8: [B][P][8] top-8 ids of each used row (NULL = skip). */
int dt_verify(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
              uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path, int32_t* bonus,
              int32_t* top8, cudaStream_t s);

/* The two halves of dt_verify, for callers that time or schedule them apart (same arguments).
 * dt_verify_rows (a8): the streaming pass over the used target rows (one read of each), leaving each
 * row piece's statistics in the handle's workspace: the argmax key, the top-8 keys when with_top8,
 * and for DT_SAMPLE the max and sum exp(x - max).
 * dt_verify_accept (a9 + the bonus): merges the pieces of the rows it needs and runs the acceptance
 * walk; with top8 non-NULL it also writes the top-8 ids of every used row (then dt_verify_rows must
 * have had with_top8 = 1). It must follow dt_verify_rows with the same meta, logits and mode on the
 * same stream, with no other call of this handle between them. */
int dt_verify_rows(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                   int32_t with_top8, cudaStream_t s);
int dt_verify_accept(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                     uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path, int32_t* bonus,
                     int32_t* top8, cudaStream_t s);

/* Verify of a tree of sampled drafts (EAGLE-2 page, §先把投机解码的账本摆清楚, §无损性…): every drawn
 * node must be in the tree (dt_rerank with m = every node: dropping drawn nodes by value is not
 * lossless). From the root, the children of the current position, in position order (= draw order),
 * are tested: child j, drawn from q_j = q without the earlier children (renormalised), q = softmax of
 * the row its parent's children were drawn from, against the residual r_j (r_0 = softmax(target row)):
 * accepted with probability min(1, r_j(t)/q_j(t)), u as in dt_verify; on rejection r_{j+1} =
 * norm(max(0, r_j - q_j)) (one pass over both rows per rejection). An accepted child becomes the
 * current position; when all children are rejected, or there are none, the bonus is the Gumbel-max
 * draw of dt_verify from the last residual (token 0 if the residual is empty). mode: 0 or
 * DT_VERIFY_PACKED (target row layout as dt_verify). draft_rows: the [D_max][B][W][ld_d] buffer of
 * dt_expand_layer_sampled. Per-element arithmetic in fp32, sums and the tests in fp64. Two launches
 * (the streaming pass over the target rows, then one CTA per request). */
int dt_verify_sampled(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                      const void* draft_rows, int64_t ld_d, uint64_t seed, uint64_t round, int32_t* accept_len,
                      int32_t* accept_path, int32_t* bonus, cudaStream_t s);

/* a10 (Graft step (3)): M[b][token_i][0..7] = top8[b][i][0..7] for every used position i with a
 * valid token; when a token repeats the highest position wins. M: device [B][V][8]. */
int dt_adj_update(dt_handle* h, int32_t* M, const dt_tree_meta* meta, const int32_t* top8,
                  cudaStream_t s);

/* After a9 (EAGLE-2 §一段更贴近实现的流程: commit the accepted tokens' KV, discard the rejected
 * candidates'; §工程实现里的几个难点: the tree's KV is temporary while it is verified): append to each
 * request's KV cache the rows of the root and of the accepted positions, in path order.
 *   tmp_kv: device bytes, row of position i of request b at b * tmp_req_stride + i * tmp_pos_stride
 *           (the verify forward's temporary KV, P positions per request); read only.
 *   cache:  device bytes, row j of request b at b * cache_req_stride + j * cache_pos_stride, L_max
 *           rows per request; rows cache_len[b] .. cache_len[b] + accept_len[b] are written.
 *   row_bytes: bytes of one row (one token's keys and values of every layer). Every pointer, stride and
 *           row_bytes must be a multiple of 16 bytes (DT_ERR_ARG otherwise).
 *   tmp_row_off: device [B+1] int32 or NULL. Not NULL: the temporary KV is packed like the target rows
 *           of DT_VERIFY_PACKED: the row of position i of request b is at (tmp_row_off[b] + i) *
 *           tmp_pos_stride (tmp_req_stride is ignored; dt_tree_meta.row_off gives the offsets).
 *   cache_len: device [B] int32, in/out: increased by accept_len[b] + 1.
 *   accept_len, accept_path: device, as written by dt_verify ([B], [B][D_path]).
 * A request whose rows would pass L_max, or whose accept_len + 1 exceeds D_path, commits nothing,
 * keeps its cache_len and sets DT_DEV_KV_FULL; a path position outside [0, P) sets DT_DEV_BAD_TREE.
 * Two launches (the copy, then the lengths). */
int dt_commit_kv(dt_handle* h, const void* tmp_kv, int64_t tmp_pos_stride, int64_t tmp_req_stride, int32_t P,
                 void* cache, int64_t cache_pos_stride, int64_t cache_req_stride, int32_t L_max, int64_t row_bytes,
                 int32_t* cache_len, const int32_t* accept_len, const int32_t* accept_path, int32_t D_path,
                 const int32_t* tmp_row_off, cudaStream_t s);

/* Standalone row log-softmax top-K that allocates nothing. This entry point has no counterpart in
 * the method's pages: it is the expansion's row pass (EAGLE-2 §扩展阶段: the children of a node
 * are the top-K tokens of softmax(row), c = draft probability) offered without a handle, for
 * callers that cannot allocate device memory at the point of the call: dt_create's workspace
 * comes from cudaMalloc, which synchronises the device and fails once the process has handed all
 * of its memory to other pools (a serving engine that reserves HBM for its KV cache at start-up).
 *   logits: device [rows][ld] (DT_BF16 or DT_F32 per dtype), element-aligned; V <= ld.
 *   logp:   device [rows][K] fp32, log softmax(row)[ids], descending.
 *   ids:    device [rows][K] int32 token ids; equal logits go to the lower id.
 *   status: device int32 or NULL; DT_DEV_* bits are OR-ed into it (never cleared here).
 * Scratch: file-scope device arrays of fixed size, about 1.1 MB per device: 4096 row-segment
 * partial results and 1024 per-row arrival counters. Hence rows <= 1024 (DT_ERR_ARG beyond).
 * The counters must be zero when a call starts: they are zero when the library is loaded and each
 * call leaves them zero. The partials need no initial value.
 * The first call on each device does a one-time set-up (cudaGetSymbolAddress of the scratch,
 * the SM count, the kernels' shared-memory limit), cached per device index for the life of the
 * process; make that first call outside any stream capture. A device reset (cudaDeviceReset)
 * invalidates that set-up and is not supported: calls after it may fail with DT_ERR_CUDA. Every call on a device shares the one scratch: two calls that may overlap in time
 * (different streams with no ordering between them) race and corrupt each other's results;
 * issue them on one stream or order them with events. */
int dt_row_topk_static(const void* logits, int64_t ld, int32_t rows, int32_t V, int32_t K, int32_t dtype,
                       float* logp, int32_t* ids, int32_t* status, cudaStream_t s);

#ifdef __cplusplus
}
#endif

#endif /* DT_H_ */
