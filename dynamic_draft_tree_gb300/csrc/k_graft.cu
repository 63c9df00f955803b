// Graft retrieval graft and adjacency-matrix refresh.
//
// Graft page, step (2): from the root token x_t, x_u = M[x_{F(u)}, r_u] over the retrieval
// template, cut to K_ret = K_max - K_draft nodes; the matrix lives on the GPU and retrieval is a
// row gather. Step (3): after verification, every verified token's row of M is refreshed with the
// top-k successors of the target's next-token distribution at that position.
#include <algorithm>

#include "dt_internal.cuh"

namespace dt {
namespace {

constexpr int kMaxTpl = 256;

struct TemplateDev {
  int32_t n, levels;
  int16_t parent[kMaxTpl];
  int8_t rank[kMaxTpl];
  int8_t level[kMaxTpl];
};

struct RetrieveArgs {
  Workspace ws;
  TemplateDev tpl;
  const int32_t* M;
  const int32_t* m_draft;
  int K_total, R_cap, N, D, V;
  int32_t* ret_token;
  int32_t* ret_parent;
  int32_t* ret_count;
};

// One CTA per request; template levels are resolved in order (a node's parent is one level up).
__global__ void __launch_bounds__(kMaxTpl) graft_retrieve_kernel(RetrieveArgs a) {
  pdl_begin();
  __shared__ int32_t tok[kMaxTpl];
  __shared__ int32_t s_kret;
  const int b = blockIdx.x;
  const int u = threadIdx.x;
  const Workspace& ws = a.ws;
  if (u == 0) {
    int nodes = 0;
    for (int d = 1; d <= a.D; ++d) nodes += ws.layer_count[(int64_t)b * (a.D + 1) + d];
    const int kept = min(a.m_draft[b], nodes);
    s_kret = max(0, min(min(a.K_total - kept, a.tpl.n), a.R_cap));
  }
  __syncthreads();
  const int kret = s_kret;
  const int root = ws.token[(int64_t)b * a.N];
  for (int lvl = 1; lvl <= a.tpl.levels; ++lvl) {
    if (u < kret && a.tpl.level[u] == lvl) {
      const int p = a.tpl.parent[u];
      const int pt = p < 0 ? root : tok[p];
      int t = -1;
      if (pt >= 0 && pt < a.V) t = __ldg(a.M + ((int64_t)b * a.V + pt) * 8 + a.tpl.rank[u]);
      else if (pt >= a.V) set_status(ws.status, DT_DEV_BAD_TOKEN);
      tok[u] = t;
    }
    __syncthreads();
  }
  for (int i = u; i < a.R_cap; i += blockDim.x) {
    const bool used = i < kret;
    a.ret_token[(int64_t)b * a.R_cap + i] = used ? tok[i] : -1;
    a.ret_parent[(int64_t)b * a.R_cap + i] = used ? (int32_t)a.tpl.parent[i] : -2;
  }
  if (u == 0) a.ret_count[b] = kret;
}

struct AdjArgs {
  Workspace ws;
  int32_t* M;
  const int32_t* top8;
  const int32_t* tokens;
  const int32_t* n_pos;
  int P, V;
};

// One CTA per request: the highest position of each distinct valid token writes its row.
__global__ void __launch_bounds__(kMaxP) adj_update_kernel(AdjArgs a) {
  pdl_begin();
  __shared__ int32_t tok[kMaxP];
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  const int np = min(a.n_pos[b], a.P);
  if (i < np) tok[i] = a.tokens[(int64_t)b * a.P + i];
  __syncthreads();
  if (i >= np) return;
  const int t = tok[i];
  if (t < 0) return;
  if (t >= a.V) {
    set_status(a.ws.status, DT_DEV_BAD_TOKEN);
    return;
  }
  for (int j = i + 1; j < np; ++j)
    if (tok[j] == t) return;
  const int4* src = reinterpret_cast<const int4*>(a.top8 + ((int64_t)b * a.P + i) * 8);
  int4* dst = reinterpret_cast<int4*>(a.M + ((int64_t)b * a.V + t) * 8);
  dst[0] = src[0];
  dst[1] = src[1];
}

}  // namespace

cudaError_t launch_graft_retrieve(dt_handle* h, const int32_t* M, const int32_t* m_draft, int K_total,
                                  const dt_template* tpl, int R_cap, int32_t* ret_token, int32_t* ret_parent,
                                  int32_t* ret_count, cudaStream_t s) {
  RetrieveArgs a;
  a.ws = h->ws;
  a.tpl.n = tpl->n;
  int levels = 0;
  for (int u = 0; u < tpl->n; ++u) {
    const int p = tpl->parent[u];
    a.tpl.parent[u] = (int16_t)p;
    a.tpl.rank[u] = (int8_t)tpl->rank[u];
    a.tpl.level[u] = (int8_t)(p < 0 ? 1 : a.tpl.level[p] + 1);
    levels = std::max(levels, (int)a.tpl.level[u]);
  }
  a.tpl.levels = levels;
  a.M = M;
  a.m_draft = m_draft;
  a.K_total = K_total;
  a.R_cap = R_cap;
  a.N = h->N;
  a.D = h->cfg.D_max;
  a.V = h->cfg.V;
  a.ret_token = ret_token;
  a.ret_parent = ret_parent;
  a.ret_count = ret_count;
  launch_k(graft_retrieve_kernel, dim3(h->B), dim3(kMaxTpl), 0, s, a);
  return cudaGetLastError();
}

cudaError_t launch_adj_update(dt_handle* h, int32_t* M, const dt_tree_meta* meta, const int32_t* top8,
                              cudaStream_t s) {
  AdjArgs a;
  a.ws = h->ws;
  a.M = M;
  a.top8 = top8;
  a.tokens = meta->tokens;
  a.n_pos = meta->n_pos;
  a.P = meta->P;
  a.V = h->cfg.V;
  launch_k(adj_update_kernel, dim3(h->B), dim3(kMaxP), 0, s, a);
  return cudaGetLastError();
}

}  // namespace dt
