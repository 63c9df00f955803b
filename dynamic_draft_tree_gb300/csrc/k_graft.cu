// Graft retrieval graft and adjacency-matrix refresh.
//
// Graft page, step (2): from the root token x_t, x_u = M[x_{F(u)}, r_u] over the retrieval
// template, cut to K_ret = K_max - K_draft nodes; the matrix lives on the GPU and retrieval is a
// row gather. Root-centred retrieval can run while the tree is drafted (it needs the root and M
// only); the cut is applied when the tree is flattened. The page contrasts root- and tail-grafted
// templates; a tail-anchored template hangs from the end of the kept draft path. Step (3): after verification, every verified token's row of M is refreshed with the
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
  const int32_t* selected;  // [B][m_cap] kept draft nodes (tail anchor only)
  int m_cap, anchor_mode, R_cap, N, V;
  int32_t* ret_token;
  int32_t* ret_parent;
  int32_t* ret_count;
  int32_t* ret_anchor;
};

// One CTA per request. The anchor (the template root): the root, or the deepest kept draft node with
// ties to the higher value, then the lower id. Template levels are resolved in order (a node's parent
// is one level up); the whole envelope min(n, R_cap) is gathered, the cut to K_ret being the meta
// builder's.
__global__ void __launch_bounds__(kMaxTpl) graft_retrieve_kernel(RetrieveArgs a) {
  pdl_begin();
  __shared__ int32_t tok[kMaxTpl];
  __shared__ int32_t s_anchor;
  const int b = blockIdx.x;
  const int u = threadIdx.x;
  const Workspace& ws = a.ws;
  const int n = min(a.tpl.n, a.R_cap);
  if (u < 32) {
    int anchor = 0;
    if (a.anchor_mode == DT_ANCHOR_TAIL) {
      // key: depth (8 bits) | ordered value (32 bits) | 2^24 - 1 - id (24 bits); the root's key is the
      // smallest a node can have at depth 0, so any kept node wins over it
      uint64_t best = ((uint64_t)f2ord(0.0f) << 24) | 0xFFFFFFull;
      for (int j = u; j < a.m_cap; j += 32) {
        const int id = a.selected[(int64_t)b * a.m_cap + j];
        if (id <= 0 || id >= a.N) continue;
        const int64_t gi = (int64_t)b * a.N + id;
        const uint64_t k = ((uint64_t)(uint32_t)ws.node_depth[gi] << 56) | ((uint64_t)f2ord(ws.value[gi]) << 24) |
                           (uint64_t)(0xFFFFFFu - (uint32_t)id);
        best = k > best ? k : best;
      }
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = x > best ? x : best;
      }
      anchor = (int)(0xFFFFFFu - (uint32_t)(best & 0xFFFFFFull));
    }
    if (u == 0) s_anchor = anchor;
  }
  __syncthreads();
  const int anchor = s_anchor;
  const int root = ws.token[(int64_t)b * a.N + anchor];
  for (int lvl = 1; lvl <= a.tpl.levels; ++lvl) {
    if (u < n && a.tpl.level[u] == lvl) {
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
    const bool used = i < n;
    a.ret_token[(int64_t)b * a.R_cap + i] = used ? tok[i] : -1;
    a.ret_parent[(int64_t)b * a.R_cap + i] = used ? (int32_t)a.tpl.parent[i] : -2;
  }
  if (u == 0) {
    a.ret_count[b] = n;
    if (a.ret_anchor) a.ret_anchor[b] = anchor;
  }
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

cudaError_t launch_graft_retrieve(dt_handle* h, const int32_t* M, const dt_template* tpl, int R_cap,
                                  const int32_t* selected, int m_cap, int32_t* ret_token, int32_t* ret_parent,
                                  int32_t* ret_count, int32_t* ret_anchor, cudaStream_t s) {
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
  a.anchor_mode = tpl->anchor;
  a.selected = selected;
  a.m_cap = tpl->anchor == DT_ANCHOR_TAIL ? m_cap : 0;
  a.R_cap = R_cap;
  a.N = h->N;
  a.V = h->cfg.V;
  a.ret_token = ret_token;
  a.ret_parent = ret_parent;
  a.ret_count = ret_count;
  a.ret_anchor = ret_anchor;
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
