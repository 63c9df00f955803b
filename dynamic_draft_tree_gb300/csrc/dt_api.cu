// Host side of the C ABI: argument checks, the workspace, and kernel launches.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "dt_internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(DT_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Carver {
  size_t off = 0;
  template <typename T>
  size_t take(size_t count) {
    off = (off + 255) / 256 * 256;
    const size_t at = off;
    off += count * sizeof(T);
    return at;
  }
};

}  // namespace

extern "C" {

const char* dt_last_error_string(void) { return g_err; }

int dt_create(const dt_config* cfg, dt_handle** out) {
  if (!cfg || !out) return fail(DT_ERR_ARG, "dt_create: null argument");
  const dt_config c = *cfg;
  if (c.V < 2) return fail(DT_ERR_ARG, "V must be >= 2");
  if (c.K < 1 || c.K > dt::kMaxK || c.K > c.V) return fail(DT_ERR_ARG, "K must be in [1, min(32, V)]");
  if (c.W < 1 || c.W > dt::kMaxW) return fail(DT_ERR_ARG, "W must be in [1, 32]");
  if (c.W * c.K > dt::kCandCap) return fail(DT_ERR_ARG, "W*K must be <= 1024");
  if (c.D_max < 1 || c.D_max > dt::kMaxD) return fail(DT_ERR_ARG, "D_max must be in [1, 16]");
  if (c.P_max < 1 || c.P_max > dt::kMaxP) return fail(DT_ERR_ARG, "P_max must be in [1, 512]");
  if (c.B_max < 1 || c.B_max > 4096) return fail(DT_ERR_ARG, "B_max must be in [1, 4096]");
  if (c.dtype != DT_BF16 && c.dtype != DT_F32) return fail(DT_ERR_ARG, "dtype must be DT_BF16 or DT_F32");

  dt_handle* h = new (std::nothrow) dt_handle();
  if (!h) return fail(DT_ERR_ARG, "out of host memory");
  h->cfg = c;
  h->LW = c.W * c.K;
  h->N = 1 + c.K + (c.D_max - 1) * h->LW;
  if (h->LW < c.K) h->LW = c.K;
  h->B = 0;
  h->depth = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "cudaGetDevice");
  }
  e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }

  e = dt::init_tree_attributes();
  if (e == cudaSuccess) e = dt::init_verify_attributes();
  if (e == cudaSuccess) e = dt::init_select_attributes();
  if (e == cudaSuccess) e = dt::init_meta_attributes();
  if (e == cudaSuccess) e = dt::init_block_attributes();
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "cudaFuncSetAttribute");
  }

  const size_t BN = (size_t)c.B_max * h->N;
  const size_t rows_max = (size_t)c.B_max * std::max(c.W, c.P_max);
  // the streaming passes place elements with 64-bit products (rows x V) x warps
  const double place = (double)rows_max * (double)c.V * (double)dt::stream_grid(h) * 8.0;
  if (place >= 9.0e18) {
    delete h;
    return fail(DT_ERR_ARG, "B_max * max(W, P_max) * V too large for 64-bit row placement");
  }
  Carver cv;
  const size_t o_token = cv.take<int32_t>(BN), o_parent = cv.take<int32_t>(BN), o_depth = cv.take<int32_t>(BN);
  const size_t o_logc = cv.take<float>(BN), o_value = cv.take<float>(BN), o_dd = cv.take<float2>(BN);
  const size_t o_eslot = cv.take<int32_t>(BN), o_estat = cv.take<float4>(BN);
  const size_t o_lorder = cv.take<int32_t>((size_t)c.B_max * (c.D_max + 1) * h->LW);
  const size_t o_lval = cv.take<float>((size_t)c.B_max * (c.D_max + 1) * h->LW);
  const size_t o_ltok = cv.take<int32_t>((size_t)c.B_max * (c.D_max + 1) * h->LW);
  const size_t o_lcount = cv.take<int32_t>((size_t)c.B_max * (c.D_max + 1));
  const size_t o_front = cv.take<int32_t>((size_t)c.B_max * c.W);
  const size_t o_fval = cv.take<float>((size_t)c.B_max * c.W);
  const size_t o_fcount = cv.take<int32_t>(c.B_max);
  // one partial per (row, segment) of a row-scan launch; launches clamp their segment count to it
  const size_t partial_cap = rows_max * 8 + (size_t)h->num_sms * 64;
  const size_t o_part = cv.take<dt::Partial>(partial_cap);
  const size_t o_rowc = cv.take<int32_t>(rows_max);
  const size_t o_rtau = cv.take<unsigned long long>(rows_max);
  const size_t o_reqc = cv.take<int32_t>(c.B_max);
  const size_t o_rstat = cv.take<dt::RowStat>((size_t)c.B_max * c.P_max);
  const size_t o_slin = cv.take<double>((size_t)c.B_max * c.P_max);
  const size_t o_scnt = cv.take<int32_t>(c.B_max);
  const size_t o_sids = cv.take<int32_t>((size_t)c.B_max * c.P_max);
  const size_t o_cast = cv.take<dt::CastState>(1);
  const size_t o_castr = cv.take<dt::CastState>(c.B_max);
  const size_t o_walk = cv.take<dt::WalkState>(c.B_max);
  const size_t o_bkey = cv.take<unsigned long long>(c.B_max);
  const size_t o_bcnt = cv.take<int32_t>(c.B_max);
  const size_t o_status = cv.take<int32_t>(1);
  const size_t total = cv.off;

  void* base = nullptr;
  e = cudaMalloc(&base, total);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "cudaMalloc(workspace)");
  }
  e = cudaMemset(base, 0, total);
  if (e != cudaSuccess) {
    cudaFree(base);
    delete h;
    return cuda_fail(e, "cudaMemset(workspace)");
  }
  char* bp = static_cast<char*>(base);
  dt::Workspace& w = h->ws;
  w.token = reinterpret_cast<int32_t*>(bp + o_token);
  w.parent = reinterpret_cast<int32_t*>(bp + o_parent);
  w.node_depth = reinterpret_cast<int32_t*>(bp + o_depth);
  w.logc = reinterpret_cast<float*>(bp + o_logc);
  w.value = reinterpret_cast<float*>(bp + o_value);
  w.node_dd = reinterpret_cast<float2*>(bp + o_dd);
  w.exp_slot = reinterpret_cast<int32_t*>(bp + o_eslot);
  w.exp_stat = reinterpret_cast<float4*>(bp + o_estat);
  w.layer_order = reinterpret_cast<int32_t*>(bp + o_lorder);
  w.layer_val = reinterpret_cast<float*>(bp + o_lval);
  w.layer_tok = reinterpret_cast<int32_t*>(bp + o_ltok);
  w.layer_count = reinterpret_cast<int32_t*>(bp + o_lcount);
  w.frontier = reinterpret_cast<int32_t*>(bp + o_front);
  w.frontier_val = reinterpret_cast<float*>(bp + o_fval);
  w.frontier_count = reinterpret_cast<int32_t*>(bp + o_fcount);
  w.partials = reinterpret_cast<dt::Partial*>(bp + o_part);
  w.partial_cap = (int64_t)partial_cap;
  w.row_counter = reinterpret_cast<int32_t*>(bp + o_rowc);
  w.row_tau = reinterpret_cast<unsigned long long*>(bp + o_rtau);
  w.row_counter_cap = (int64_t)rows_max;
  w.req_counter = reinterpret_cast<int32_t*>(bp + o_reqc);
  w.row_stats = reinterpret_cast<dt::RowStat*>(bp + o_rstat);
  w.sorted_lin = reinterpret_cast<double*>(bp + o_slin);
  w.sorted_cnt = reinterpret_cast<int32_t*>(bp + o_scnt);
  w.sorted_ids = reinterpret_cast<int32_t*>(bp + o_sids);
  w.cast = reinterpret_cast<dt::CastState*>(bp + o_cast);
  w.cast_req = reinterpret_cast<dt::CastState*>(bp + o_castr);
  w.walk = reinterpret_cast<dt::WalkState*>(bp + o_walk);
  w.bonus_key = reinterpret_cast<unsigned long long*>(bp + o_bkey);
  w.bonus_counter = reinterpret_cast<int32_t*>(bp + o_bcnt);
  w.status = reinterpret_cast<int32_t*>(bp + o_status);
  h->alloc = base;
  h->alloc_bytes = total;
  *out = h;
  return DT_OK;
}

int dt_destroy(dt_handle* h) {
  if (!h) return fail(DT_ERR_ARG, "dt_destroy: null handle");
  cudaError_t e = cudaFree(h->alloc);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
  return DT_OK;
}

int dt_get_tree(const dt_handle* h, dt_tree_view* v) {
  if (!h || !v) return fail(DT_ERR_ARG, "dt_get_tree: null argument");
  v->B = h->B;
  v->K = h->cfg.K;
  v->W = h->cfg.W;
  v->D_max = h->cfg.D_max;
  v->N = h->N;
  v->LW = h->LW;
  v->depth = h->depth;
  v->token = h->ws.token;
  v->parent = h->ws.parent;
  v->node_depth = h->ws.node_depth;
  v->logc = h->ws.logc;
  v->value = h->ws.value;
  v->layer_order = h->ws.layer_order;
  v->layer_count = h->ws.layer_count;
  v->frontier = h->ws.frontier;
  v->frontier_count = h->ws.frontier_count;
  return DT_OK;
}

int dt_get_status(dt_handle* h, cudaStream_t s, int32_t* bits) {
  if (!h || !bits) return fail(DT_ERR_ARG, "dt_get_status: null argument");
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, h->ws.status, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_get_status");
  *bits = v;
  if (v & DT_DEV_TIMEOUT) return fail(DT_ERR_DEVICE_TIMEOUT, "device status 0x%x (a bounded wait ran out)", v);
  if (v) return fail(DT_ERR_DEVICE, "device status 0x%x", v);
  return DT_OK;
}

int dt_clear_status(dt_handle* h, cudaStream_t s) {
  if (!h) return fail(DT_ERR_ARG, "dt_clear_status: null handle");
  cudaError_t e = cudaMemsetAsync(h->ws.status, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_clear_status");
  return DT_OK;
}

int dt_tree_reset(dt_handle* h, int32_t B, const int32_t* root_token, cudaStream_t s) {
  if (!h || !root_token) return fail(DT_ERR_ARG, "dt_tree_reset: null argument");
  if (B < 1 || B > h->cfg.B_max) return fail(DT_ERR_ARG, "B=%d outside [1, B_max=%d]", B, h->cfg.B_max);
  h->B = B;
  h->depth = 0;
  cudaError_t e = dt::launch_tree_reset(h, root_token, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_tree_reset");
  return DT_OK;
}

int dt_select_frontier(dt_handle* h, const int32_t* width, int32_t width_len, const int32_t* stop,
                       int32_t* frontier_token, cudaStream_t s) {
  if (!h) return fail(DT_ERR_ARG, "dt_select_frontier: null handle");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_select_frontier: no tree (call dt_tree_reset)");
  if (h->depth >= h->cfg.D_max) return fail(DT_ERR_ARG, "dt_select_frontier: tree at D_max");
  if (width && width_len != 1 && width_len != h->B) return fail(DT_ERR_ARG, "width_len must be 1 or B");
  cudaError_t e = dt::launch_select_frontier(h, width, width_len, stop, frontier_token, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_select_frontier");
  return DT_OK;
}

int dt_expand_layer(dt_handle* h, const void* logits, int64_t ld, int32_t F, cudaStream_t s) {
  if (!h || !logits) return fail(DT_ERR_ARG, "dt_expand_layer: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_expand_layer: no tree (call dt_tree_reset)");
  if (h->depth >= h->cfg.D_max) return fail(DT_ERR_ARG, "dt_expand_layer: tree already has D_max layers");
  if (F < 1 || F > h->cfg.W) return fail(DT_ERR_ARG, "F=%d outside [1, W=%d]", F, h->cfg.W);
  if (ld < h->cfg.V) return fail(DT_ERR_ARG, "ld=%lld < V", (long long)ld);
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  cudaError_t e = dt::launch_expand(h, logits, ld, F, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_expand_layer");
  return DT_OK;
}

// Host checks shared by the CAST width/depth entry points.
static int check_cast_width_params(const dt_handle* h, const dt_prune_params* p, const dt_prune_out* out) {
  if (!p->S_T || !p->S_D) return fail(DT_ERR_ARG, "cost tables missing");
  if (p->M_rows < 1 || p->N_cols < 1) return fail(DT_ERR_ARG, "table shape must be positive");
  if (!(p->L > 0.0)) return fail(DT_ERR_ARG, "L must be > 0");
  if (p->n0 < 0) return fail(DT_ERR_ARG, "n0 must be >= 0");
  if (p->width_cap < 1 || p->width_cap > h->cfg.W || p->width_cap > p->N_cols)
    return fail(DT_ERR_ARG, "width_cap must be in [1, min(W, N_cols)]");
  if (p->R < 1 || p->R > dt::kMaxFifo) return fail(DT_ERR_ARG, "R must be in [1, 16]");
  if (!out->width || !out->stop) return fail(DT_ERR_ARG, "width and stop outputs required");
  return DT_OK;
}

static int check_policy_args(const dt_handle* h, int32_t policy, const dt_prune_params* p, const dt_prune_out* out,
                             const int32_t* width, int32_t width_len) {
  if (width && width_len != 1 && width_len != h->B) return fail(DT_ERR_ARG, "width_len must be 1 or B");
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH) {
    if (!p || !out) return fail(DT_ERR_ARG, "CAST pruning needs params and outputs");
    return check_cast_width_params(h, p, out);
  }
  if (policy == DT_POLICY_GRAFT_CHECKPOINT) {
    if (!p || !out) return fail(DT_ERR_ARG, "the Graft checkpoint needs params and outputs");
    if (p->n_ckpt < 0 || p->n_ckpt > 16) return fail(DT_ERR_ARG, "n_ckpt must be in [0, 16]");
    if (!out->stop) return fail(DT_ERR_ARG, "stop output required");
    return DT_OK;
  }
  if (policy != DT_POLICY_NONE)
    return fail(DT_ERR_ARG, "policy must be DT_POLICY_NONE, DT_POLICY_CAST_WIDTH_DEPTH or "
                            "DT_POLICY_GRAFT_CHECKPOINT");
  return DT_OK;
}

int dt_expand_prune_select(dt_handle* h, const void* logits, int64_t ld, int32_t F, int32_t policy,
                           const dt_prune_params* p, const dt_prune_out* out, const int32_t* width,
                           int32_t width_len, int32_t* frontier_token, cudaStream_t s) {
  if (!h || !logits) return fail(DT_ERR_ARG, "dt_expand_prune_select: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_expand_prune_select: no tree (call dt_tree_reset)");
  if (h->depth >= h->cfg.D_max) return fail(DT_ERR_ARG, "dt_expand_prune_select: tree already has D_max layers");
  if (F < 1 || F > h->cfg.W) return fail(DT_ERR_ARG, "F=%d outside [1, W=%d]", F, h->cfg.W);
  if (ld < h->cfg.V) return fail(DT_ERR_ARG, "ld=%lld < V", (long long)ld);
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  const int rc = check_policy_args(h, policy, p, out, width, width_len);
  if (rc != DT_OK) return rc;
  cudaError_t e = dt::launch_expand_ex(h, logits, ld, F, policy, p, out, width, width_len, frontier_token, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_expand_prune_select");
  return DT_OK;
}

int dt_expand_layer_sampled(dt_handle* h, const void* logits, int64_t ld, int32_t F, uint64_t seed, uint64_t round,
                            cudaStream_t s) {
  if (!h || !logits) return fail(DT_ERR_ARG, "dt_expand_layer_sampled: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_expand_layer_sampled: no tree (call dt_tree_reset)");
  if (h->depth >= h->cfg.D_max) return fail(DT_ERR_ARG, "dt_expand_layer_sampled: tree already has D_max layers");
  if (F < 1 || F > h->cfg.W) return fail(DT_ERR_ARG, "F=%d outside [1, W=%d]", F, h->cfg.W);
  if (ld < h->cfg.V) return fail(DT_ERR_ARG, "ld=%lld < V", (long long)ld);
  if (h->N > 4096) return fail(DT_ERR_ARG, "sampled drafts need at most 4096 nodes per request (draw counter)");
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  cudaError_t e = dt::launch_expand(h, logits, ld, F, s, true, seed, round);
  if (e != cudaSuccess) return cuda_fail(e, "dt_expand_layer_sampled");
  return DT_OK;
}

int dt_block_expand(dt_handle* h, const void* logits, int64_t ld, int32_t L, const dt_prune_params* p,
                    const dt_prune_out* out, cudaStream_t s) {
  if (!h || !logits) return fail(DT_ERR_ARG, "dt_block_expand: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_block_expand: no tree (call dt_tree_reset)");
  if (h->depth != 0) return fail(DT_ERR_ARG, "dt_block_expand: the tree must be right after dt_tree_reset");
  if (L < 1 || L > h->cfg.D_max) return fail(DT_ERR_ARG, "L=%d outside [1, D_max=%d]", L, h->cfg.D_max);
  if ((int64_t)h->B * L > h->ws.row_counter_cap) return fail(DT_ERR_ARG, "B*L exceeds B_max*max(W, P_max)");
  if (ld < h->cfg.V) return fail(DT_ERR_ARG, "ld=%lld < V", (long long)ld);
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  if (p) {
    if (!out || !out->stop) return fail(DT_ERR_ARG, "dt_block_expand: the gates need out->stop");
    if (p->n_ckpt < 0 || p->n_ckpt > 16) return fail(DT_ERR_ARG, "n_ckpt must be in [0, 16]");
  }
  cudaError_t e = dt::launch_block_expand(h, logits, ld, L, p, out, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_block_expand");
  return DT_OK;
}

int dt_cast_prune(dt_handle* h, int32_t policy, const dt_prune_params* p, const dt_prune_out* out,
                  cudaStream_t s) {
  if (!h || !p || !out) return fail(DT_ERR_ARG, "dt_cast_prune: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_cast_prune: no tree (call dt_tree_reset)");
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH || policy == DT_POLICY_CAST_VERIFY) {
    if (!p->S_T || (policy == DT_POLICY_CAST_WIDTH_DEPTH && !p->S_D))
      return fail(DT_ERR_ARG, "cost tables missing");
    if (p->M_rows < 1 || p->N_cols < 1) return fail(DT_ERR_ARG, "table shape must be positive");
    if (!(p->L > 0.0)) return fail(DT_ERR_ARG, "L must be > 0");
    if (p->n0 < 0) return fail(DT_ERR_ARG, "n0 must be >= 0");
  }
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH) {
    if (h->depth < 1) return fail(DT_ERR_ARG, "no layer to prune");
    if (p->width_cap < 1 || p->width_cap > h->cfg.W || p->width_cap > p->N_cols)
      return fail(DT_ERR_ARG, "width_cap must be in [1, min(W, N_cols)]");
    if (p->R < 1 || p->R > dt::kMaxFifo) return fail(DT_ERR_ARG, "R must be in [1, 16]");
    if (!out->width || !out->stop) return fail(DT_ERR_ARG, "width and stop outputs required");
  } else if (policy == DT_POLICY_CAST_VERIFY) {
    if (p->m_cap < 1 || p->m_cap > p->N_cols || p->m_cap > h->cfg.P_max - 1)
      return fail(DT_ERR_ARG, "m_cap must be in [1, min(N_cols, P_max-1)]");
    if (!out->m) return fail(DT_ERR_ARG, "m output required");
  } else if (policy == DT_POLICY_GRAFT_CHECKPOINT) {
    if (h->depth < 1) return fail(DT_ERR_ARG, "no layer to check");
    if (p->n_ckpt < 0 || p->n_ckpt > 16) return fail(DT_ERR_ARG, "n_ckpt must be in [0, 16]");
    if (!out->stop) return fail(DT_ERR_ARG, "stop output required");
  } else {
    return fail(DT_ERR_ARG, "unknown policy %d", policy);
  }
  cudaError_t e = dt::launch_cast_prune(h, policy, p, out, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_cast_prune");
  return DT_OK;
}

int dt_cast_verify_rerank(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out, int32_t* selected,
                          cudaStream_t s) {
  if (!h || !p || !out || !selected) return fail(DT_ERR_ARG, "dt_cast_verify_rerank: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_cast_verify_rerank: no tree (call dt_tree_reset)");
  if (!p->S_T) return fail(DT_ERR_ARG, "cost tables missing");
  if (p->M_rows < 1 || p->N_cols < 1) return fail(DT_ERR_ARG, "table shape must be positive");
  if (!(p->L > 0.0)) return fail(DT_ERR_ARG, "L must be > 0");
  if (p->n0 < 0) return fail(DT_ERR_ARG, "n0 must be >= 0");
  if (p->m_cap < 1 || p->m_cap > p->N_cols || p->m_cap > h->cfg.P_max - 1)
    return fail(DT_ERR_ARG, "m_cap must be in [1, min(N_cols, P_max-1)]");
  if (!out->m) return fail(DT_ERR_ARG, "m output required");
  cudaError_t e = dt::launch_cast_verify_rerank(h, p, out, selected, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_cast_verify_rerank");
  return DT_OK;
}

int dt_cast_prune_select(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out, int32_t* frontier_token,
                         cudaStream_t s) {
  if (!h || !p || !out) return fail(DT_ERR_ARG, "dt_cast_prune_select: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_cast_prune_select: no tree (call dt_tree_reset)");
  if (h->depth < 1) return fail(DT_ERR_ARG, "no layer to prune");
  const int rc = check_cast_width_params(h, p, out);
  if (rc != DT_OK) return rc;
  cudaError_t e = dt::launch_cast_prune_select(h, p, out, frontier_token, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_cast_prune_select");
  return DT_OK;
}

int dt_rerank(dt_handle* h, const int32_t* m, int32_t m_len, int32_t m_cap, int32_t* selected, cudaStream_t s) {
  if (!h || !selected) return fail(DT_ERR_ARG, "dt_rerank: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_rerank: no tree (call dt_tree_reset)");
  if (m_cap < 1 || m_cap > h->N - 1) return fail(DT_ERR_ARG, "m_cap must be in [1, N-1]");
  if (m && m_len != 1 && m_len != h->B) return fail(DT_ERR_ARG, "m_len must be 1 or B");
  cudaError_t e = dt::launch_rerank(h, m, m_len, m_cap, selected, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_rerank");
  return DT_OK;
}

int dt_graft_retrieve(dt_handle* h, const int32_t* M, const dt_template* tpl, int32_t R_cap, const int32_t* selected,
                      int32_t m_cap, int32_t* ret_token, int32_t* ret_parent, int32_t* ret_count,
                      int32_t* ret_anchor, cudaStream_t s) {
  if (!h || !M || !tpl || !ret_token || !ret_parent || !ret_count)
    return fail(DT_ERR_ARG, "dt_graft_retrieve: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_graft_retrieve: no tree (call dt_tree_reset)");
  if (tpl->n < 0 || tpl->n > 256) return fail(DT_ERR_ARG, "template size must be in [0, 256]");
  if (tpl->n > 0 && (!tpl->parent || !tpl->rank)) return fail(DT_ERR_ARG, "template arrays missing");
  for (int u = 0; u < tpl->n; ++u) {
    if (tpl->parent[u] < -1 || tpl->parent[u] >= u) return fail(DT_ERR_ARG, "template parent[%d] invalid", u);
    if (tpl->rank[u] < 0 || tpl->rank[u] >= 8) return fail(DT_ERR_ARG, "template rank[%d] invalid", u);
  }
  if (tpl->anchor != DT_ANCHOR_ROOT && tpl->anchor != DT_ANCHOR_TAIL)
    return fail(DT_ERR_ARG, "template anchor must be DT_ANCHOR_ROOT or DT_ANCHOR_TAIL");
  if (tpl->anchor == DT_ANCHOR_TAIL && (!selected || m_cap < 1 || m_cap > h->N - 1))
    return fail(DT_ERR_ARG, "a tail-anchored template needs selected and m_cap in [1, N-1]");
  if (R_cap < 1 || R_cap > dt::kMaxP) return fail(DT_ERR_ARG, "R_cap must be in [1, 512]");
  cudaError_t e = dt::launch_graft_retrieve(h, M, tpl, R_cap, selected, m_cap, ret_token, ret_parent, ret_count,
                                            ret_anchor, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_graft_retrieve");
  return DT_OK;
}

int dt_build_tree_meta(dt_handle* h, const int32_t* selected, int32_t m_cap, const int32_t* ret_token,
                       const int32_t* ret_parent, const int32_t* ret_count, const int32_t* ret_anchor,
                       int32_t R_cap, int32_t K_total, const int32_t* pos_offset, const dt_tree_meta* meta,
                       cudaStream_t s) {
  if (!h || !selected || !meta) return fail(DT_ERR_ARG, "dt_build_tree_meta: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_build_tree_meta: no tree (call dt_tree_reset)");
  if (!meta->tokens || !meta->parents || !meta->depth || !meta->node_id || !meta->mask ||
      !meta->position_ids || !meta->retrieve || !meta->n_leaves || !meta->n_pos)
    return fail(DT_ERR_ARG, "dt_build_tree_meta: a meta array is null");
  if (meta->P < 1 || meta->P > h->cfg.P_max) return fail(DT_ERR_ARG, "meta P must be in [1, P_max]");
  if (meta->D_path < 1 || meta->D_path > 64) return fail(DT_ERR_ARG, "D_path must be in [1, 64]");
  if (m_cap < 0 || m_cap > h->N - 1) return fail(DT_ERR_ARG, "m_cap out of range");
  const bool graft = ret_token != nullptr;
  if (graft && (!ret_parent || !ret_count || R_cap < 1)) return fail(DT_ERR_ARG, "retrieval arrays incomplete");
  if (1 + m_cap > meta->P) return fail(DT_ERR_ARG, "1 + m_cap exceeds P");
  cudaError_t e = dt::launch_build_meta(h, selected, m_cap, ret_token, ret_parent, ret_count,
                                        graft ? ret_anchor : nullptr, graft ? R_cap : 0, K_total, pos_offset, meta,
                                        s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_build_tree_meta");
  return DT_OK;
}

static int check_verify_args(const dt_handle* h, const char* who, const dt_tree_meta* meta, const void* logits,
                             int64_t ld, int32_t mode) {
  if (!meta || !logits) return fail(DT_ERR_ARG, "%s: null argument", who);
  if (h->B < 1) return fail(DT_ERR_ARG, "%s: no tree (call dt_tree_reset)", who);
  const int32_t base_mode = mode & ~DT_VERIFY_PACKED;
  if (base_mode != DT_GREEDY && base_mode != DT_SAMPLE)
    return fail(DT_ERR_ARG, "mode must be DT_GREEDY or DT_SAMPLE, optionally | DT_VERIFY_PACKED");
  if (meta->P < 1 || meta->P > h->cfg.P_max) return fail(DT_ERR_ARG, "meta P must be in [1, P_max]");
  if (meta->D_path < 1 || meta->D_path > 64) return fail(DT_ERR_ARG, "D_path must be in [1, 64]");
  if (ld < h->cfg.V) return fail(DT_ERR_ARG, "ld < V");
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  if ((int64_t)h->B * meta->P > (int64_t)h->ws.row_counter_cap) return fail(DT_ERR_ARG, "B*P too large");
  return DT_OK;
}

int dt_verify_rows(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                   int32_t with_top8, cudaStream_t s) {
  if (!h) return fail(DT_ERR_ARG, "dt_verify_rows: null handle");
  const int rc = check_verify_args(h, "dt_verify_rows", meta, logits, ld, mode);
  if (rc != DT_OK) return rc;
  cudaError_t e = dt::launch_verify_rows(h, meta, logits, ld, mode, with_top8 ? 1 : 0, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_verify_rows");
  return DT_OK;
}

int dt_verify_accept(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                     uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path, int32_t* bonus,
                     int32_t* top8, cudaStream_t s) {
  if (!h || !accept_len || !accept_path || !bonus) return fail(DT_ERR_ARG, "dt_verify_accept: null argument");
  const int rc = check_verify_args(h, "dt_verify_accept", meta, logits, ld, mode);
  if (rc != DT_OK) return rc;
  cudaError_t e = dt::launch_verify_accept(h, meta, logits, ld, mode, seed, round, accept_len, accept_path, bonus,
                                           top8, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_verify_accept");
  return DT_OK;
}

int dt_verify(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
              uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path, int32_t* bonus,
              int32_t* top8, cudaStream_t s) {
  if (!h || !accept_len || !accept_path || !bonus) return fail(DT_ERR_ARG, "dt_verify: null argument");
  const int rc = check_verify_args(h, "dt_verify", meta, logits, ld, mode);
  if (rc != DT_OK) return rc;
  cudaError_t e = dt::launch_verify(h, meta, logits, ld, mode, seed, round, accept_len, accept_path, bonus, top8, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_verify");
  return DT_OK;
}

int dt_verify_sampled(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int32_t mode,
                      const void* draft_rows, int64_t ld_d, uint64_t seed, uint64_t round, int32_t* accept_len,
                      int32_t* accept_path, int32_t* bonus, cudaStream_t s) {
  if (!h || !accept_len || !accept_path || !bonus || !draft_rows)
    return fail(DT_ERR_ARG, "dt_verify_sampled: null argument");
  if (mode != 0 && mode != DT_VERIFY_PACKED) return fail(DT_ERR_ARG, "mode must be 0 or DT_VERIFY_PACKED");
  const int rc = check_verify_args(h, "dt_verify_sampled", meta, logits, ld, DT_SAMPLE | mode);
  if (rc != DT_OK) return rc;
  if (ld_d < h->cfg.V) return fail(DT_ERR_ARG, "ld_d < V");
  const size_t esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  if (!aligned(draft_rows, esz)) return fail(DT_ERR_ARG, "draft rows not aligned to their element size");
  cudaError_t e = dt::launch_verify_sampled(h, meta, logits, ld, mode, draft_rows, ld_d, seed, round, accept_len,
                                            accept_path, bonus, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_verify_sampled");
  return DT_OK;
}

int dt_adj_update(dt_handle* h, int32_t* M, const dt_tree_meta* meta, const int32_t* top8, cudaStream_t s) {
  if (!h || !M || !meta || !top8) return fail(DT_ERR_ARG, "dt_adj_update: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_adj_update: no tree (call dt_tree_reset)");
  if (meta->P < 1 || meta->P > h->cfg.P_max) return fail(DT_ERR_ARG, "meta P must be in [1, P_max]");
  if (!aligned(M, 16) || !aligned(top8, 16)) return fail(DT_ERR_ARG, "M and top8 must be 16-byte aligned");
  cudaError_t e = dt::launch_adj_update(h, M, meta, top8, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_adj_update");
  return DT_OK;
}

int dt_commit_kv(dt_handle* h, const void* tmp_kv, int64_t tmp_pos_stride, int64_t tmp_req_stride, int32_t P,
                 void* cache, int64_t cache_pos_stride, int64_t cache_req_stride, int32_t L_max, int64_t row_bytes,
                 int32_t* cache_len, const int32_t* accept_len, const int32_t* accept_path, int32_t D_path,
                 const int32_t* tmp_row_off, cudaStream_t s) {
  if (!h || !tmp_kv || !cache || !cache_len || !accept_len || !accept_path)
    return fail(DT_ERR_ARG, "dt_commit_kv: null argument");
  if (h->B < 1) return fail(DT_ERR_ARG, "dt_commit_kv: no tree (call dt_tree_reset)");
  if (P < 1 || L_max < 1 || D_path < 1 || D_path > 64) return fail(DT_ERR_ARG, "P, L_max >= 1 and D_path in [1, 64]");
  if (row_bytes < 16) return fail(DT_ERR_ARG, "row_bytes must be >= 16");
  if (!aligned(tmp_kv, 16) || !aligned(cache, 16) || tmp_pos_stride % 16 || tmp_req_stride % 16 ||
      cache_pos_stride % 16 || cache_req_stride % 16 || row_bytes % 16)
    return fail(DT_ERR_ARG, "dt_commit_kv: pointers, strides and row_bytes must be multiples of 16 bytes");
  if (tmp_pos_stride < row_bytes || cache_pos_stride < row_bytes ||
      (!tmp_row_off && tmp_req_stride < tmp_pos_stride * P) || cache_req_stride < cache_pos_stride * L_max)
    return fail(DT_ERR_ARG, "dt_commit_kv: strides smaller than the rows they hold");
  if (!aligned(cache_len, 4) || !aligned(accept_len, 4) || !aligned(accept_path, 4) || !aligned(tmp_row_off, 4))
    return fail(DT_ERR_ARG, "dt_commit_kv: int32 arrays must be 4-byte aligned");
  cudaError_t e = dt::launch_commit_kv(h, tmp_kv, tmp_pos_stride, tmp_req_stride, P, cache, cache_pos_stride,
                                       cache_req_stride, L_max, row_bytes, cache_len, accept_len, accept_path,
                                       D_path, tmp_row_off, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_commit_kv");
  return DT_OK;
}

int dt_row_topk_static(const void* logits, int64_t ld, int32_t rows, int32_t V, int32_t K, int32_t dtype,
                       float* logp, int32_t* ids, int32_t* status, cudaStream_t s) {
  if (!logits || !logp || !ids) return fail(DT_ERR_ARG, "dt_row_topk_static: null argument");
  if (rows < 1 || rows > dt::kStaticRows)
    return fail(DT_ERR_ARG, "rows=%d outside [1, %d] (size of the static scratch)", rows, dt::kStaticRows);
  if (V < 2) return fail(DT_ERR_ARG, "V must be >= 2");
  if (K < 1 || K > dt::kMaxK || K > V) return fail(DT_ERR_ARG, "K must be in [1, min(32, V)]");
  if (dtype != DT_BF16 && dtype != DT_F32) return fail(DT_ERR_ARG, "dtype must be DT_BF16 or DT_F32");
  if (ld < V) return fail(DT_ERR_ARG, "ld=%lld < V", (long long)ld);
  const size_t esz = dtype == DT_BF16 ? 2 : 4;
  if (!aligned(logits, esz)) return fail(DT_ERR_ARG, "logits not aligned to its element size");
  if (!aligned(logp, 4) || !aligned(ids, 4) || !aligned(status, 4))
    return fail(DT_ERR_ARG, "logp, ids and status must be 4-byte aligned");
  cudaError_t e = dt::launch_row_topk_static(logits, ld, rows, V, K, dtype, logp, ids, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "dt_row_topk_static");
  return DT_OK;
}

}  // extern "C"
