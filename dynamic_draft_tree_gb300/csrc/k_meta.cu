// Flattening and tree-attention metadata.
//
// EAGLE-2 page §"重排阶段": the selected connected subtree is flattened to a token list and a
// tree attention mask lets each node see only its ancestors. Graft page step (3): the kept draft
// nodes and the grafted retrieval nodes are flattened to K_max tokens with standard position IDs,
// ancestor mask and candidate path (retrieve) indices.
#include <algorithm>

#include "dt_internal.cuh"

namespace dt {
namespace {

struct MetaArgs {
  Workspace ws;
  int N, m_cap, R_cap;
  const int32_t* selected;
  const int32_t* ret_token;
  const int32_t* ret_parent;
  const int32_t* ret_count;
  const int32_t* ret_anchor;  // [B] draft node the template root stands for, or null (the root)
  int K_total;                // > 0: at most K_total - selected nodes retrieved ones are used
  const int32_t* pos_offset;
  dt_tree_meta meta;
};

// Retrieved nodes request b uses when it keeps n selected draft nodes.
__device__ __forceinline__ int used_retrieved(const MetaArgs& a, int b, int n) {
  int rc = a.ret_count ? max(0, min(a.ret_count[b], a.R_cap)) : 0;
  if (a.K_total > 0) rc = min(rc, max(0, a.K_total - n));
  return rc;
}

constexpr int kMetaThreads = 512;
constexpr int kWords = kMaxP / 32;

// One CTA per request.
__global__ void __launch_bounds__(kMetaThreads) build_meta_kernel(MetaArgs a) {
  pdl_begin();
  extern __shared__ __align__(16) int16_t pos_of[];  // [N] node id -> position, -1 if not placed
  __shared__ int32_t tok[kMaxP], par[kMaxP], dep[kMaxP], nid[kMaxP];
  __shared__ uint32_t anc[kMaxP][kWords];
  __shared__ int32_t has_child[kMaxP];
  __shared__ int32_t leaf_idx[kMaxP];
  __shared__ int32_t s_nsel, s_npos, s_bad, s_rc, s_off;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const Workspace& ws = a.ws;
  const int P = a.meta.P;
  const int Dp = a.meta.D_path;

  for (int i = tid; i < a.N; i += blockDim.x) pos_of[i] = -1;
  if (tid == 0) {
    s_nsel = a.m_cap;
    s_bad = 0;
    s_off = 0;
  }
  for (int i = tid; i < P; i += blockDim.x) has_child[i] = 0;
  __syncthreads();
  // selected nodes: the entries before the first -1 (all loaded at once, the first -1 found by a min)
  for (int j = tid; j < a.m_cap; j += blockDim.x)
    if (a.selected[(int64_t)b * a.m_cap + j] < 0) atomicMin(&s_nsel, j);
  __syncthreads();
  if (tid == 0) {
    const int n = s_nsel;
    const int rc = used_retrieved(a, b, n);
    s_rc = rc;
    s_npos = min(P, 1 + n + rc);
    if (1 + n + rc > P) s_bad = 1;  // positions would not fit: flagged, the extra ones dropped
  }
  __syncthreads();
  const int nsel = s_nsel, npos = s_npos;
  if (a.meta.row_off) {
    // packed row offset: the positions of requests 0..b-1, counted as their own CTAs count them (root +
    // the selected entries before the first -1 + the retrieved nodes, at most P); one warp per request
    const int lane = tid & 31;
    for (int bb = tid >> 5; bb < b; bb += kMetaThreads / 32) {
      int n = a.m_cap;
      for (int c = 0; c < a.m_cap; c += 32) {
        const bool neg = c + lane < a.m_cap && a.selected[(int64_t)bb * a.m_cap + c + lane] < 0;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, neg);
        if (m) {
          n = c + __ffs(m) - 1;
          break;
        }
      }
      if (lane == 0) atomicAdd(&s_off, min(P, 1 + n + used_retrieved(a, bb, n)));
    }
  }
  if (tid == 0) pos_of[0] = 0;
  for (int j = tid; j < nsel; j += blockDim.x) {
    const int id = a.selected[(int64_t)b * a.m_cap + j];
    if (id > 0 && id < a.N) pos_of[id] = (int16_t)(1 + j);
  }
  __syncthreads();

  // token, parent position, node id
  for (int p = tid; p < P; p += blockDim.x) {
    int t = -1, pp = -1, id = -1;
    if (p == 0) {
      t = ws.token[(int64_t)b * a.N];
      id = 0;
    } else if (p <= nsel) {
      id = a.selected[(int64_t)b * a.m_cap + (p - 1)];
      if (id > 0 && id < a.N) {
        t = ws.token[(int64_t)b * a.N + id];
        const int parent_id = ws.parent[(int64_t)b * a.N + id];
        pp = parent_id >= 0 ? pos_of[parent_id] : -1;
        if (pp < 0 || pp >= p) {  // selection is not parent-closed
          s_bad = 1;
          pp = 0;
        }
      } else {
        s_bad = 1;
        pp = 0;
      }
    } else if (p < npos) {
      const int u = p - nsel - 1;
      t = a.ret_token[(int64_t)b * a.R_cap + u];
      const int rp = a.ret_parent[(int64_t)b * a.R_cap + u];
      int ap = 0;  // position of the template root: the root, or the anchor draft node
      if (a.ret_anchor) {
        const int an = a.ret_anchor[b];
        if (an > 0) {
          ap = an < a.N ? pos_of[an] : -1;
          if (ap < 0) {  // the anchor was not kept
            s_bad = 1;
            ap = 0;
          }
        }
      }
      pp = rp < 0 ? ap : nsel + 1 + rp;
      if (pp >= p) {
        s_bad = 1;
        pp = 0;
      }
    }
    tok[p] = t;
    par[p] = pp;
    nid[p] = id;
  }
  __syncthreads();
  // depth and ancestor bitset by walking to the root (parents precede children)
  for (int p = tid; p < P; p += blockDim.x) {
#pragma unroll
    for (int w = 0; w < kWords; ++w) anc[p][w] = 0u;
    if (p >= npos) {
      dep[p] = -1;
      continue;
    }
    int q = p, d = 0;
    while (true) {
      anc[p][q >> 5] |= 1u << (q & 31);
      if (q == 0) break;
      q = par[q];
      ++d;
      if (d > kMaxP) {
        s_bad = 1;
        break;
      }
    }
    dep[p] = d;
    if (p > 0) atomicOr(&has_child[par[p]], 1);
  }
  __syncthreads();
  // leaves in increasing position: exclusive prefix count of leaf flags (serial over <= 512 flags
  // by warp 0 with ballots)
  if (tid < 32) {
    int base = 0;
    for (int c = 0; c < P; c += 32) {
      const int p = c + tid;
      const bool leaf = p < npos && !has_child[p];
      const unsigned m = __ballot_sync(0xFFFFFFFFu, leaf);
      if (leaf) leaf_idx[p] = base + __popc(m & ((1u << tid) - 1u));
      else if (p < P) leaf_idx[p] = -1;
      base += __popc(m);
    }
    if (tid == 0) a.meta.n_leaves[b] = base;
  }
  __syncthreads();

  // ---- outputs ----
  const int64_t rb = (int64_t)b * P;
  const int po = a.pos_offset ? a.pos_offset[b] : 0;
  for (int p = tid; p < P; p += blockDim.x) {
    a.meta.tokens[rb + p] = p < npos ? tok[p] : -1;
    a.meta.parents[rb + p] = p < npos ? par[p] : -1;
    a.meta.depth[rb + p] = dep[p];
    a.meta.node_id[rb + p] = p < npos ? nid[p] : -1;
    a.meta.position_ids[rb + p] = p < npos ? po + dep[p] : -1;
  }
  // mask [P][P] bytes
  uint8_t* mask = a.meta.mask + rb * P;
  const int64_t mbytes = (int64_t)P * P;
  for (int e = tid; e < (int)mbytes; e += blockDim.x) {  // P*P <= 2^18: 32-bit index arithmetic
    const int i = e / P, j = e - i * P;
    mask[e] = (uint8_t)((anc[i][j >> 5] >> (j & 31)) & 1u);
  }
  // retrieve rows
  int32_t* ret = a.meta.retrieve + rb * Dp;
  for (int64_t e = tid; e < (int64_t)P * Dp; e += blockDim.x) ret[e] = -1;
  __syncthreads();
  for (int p = tid; p < npos; p += blockDim.x) {
    const int li = leaf_idx[p];
    if (li < 0) continue;
    const int d = dep[p];
    if (d + 1 > Dp) {
      s_bad = 1;
      continue;
    }
    int q = p;
    for (int k = d; k >= 0; --k) {
      ret[(int64_t)li * Dp + k] = q;
      q = par[q];
    }
  }
  __syncthreads();
  if (tid == 0) {
    a.meta.n_pos[b] = npos;
    if (a.meta.row_off) {
      a.meta.row_off[b] = s_off;
      if (b == (int)gridDim.x - 1) a.meta.row_off[b + 1] = s_off + npos;
    }
    if (s_bad) set_status(ws.status, DT_DEV_BAD_TREE);
  }
}

}  // namespace

cudaError_t init_meta_attributes() {
  // node -> position map of the largest tree: 16384 int16 entries
  return cudaFuncSetAttribute(build_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 2);
}

cudaError_t launch_build_meta(dt_handle* h, const int32_t* selected, int m_cap, const int32_t* ret_token,
                              const int32_t* ret_parent, const int32_t* ret_count, const int32_t* ret_anchor,
                              int R_cap, int K_total, const int32_t* pos_offset, const dt_tree_meta* meta,
                              cudaStream_t s) {
  MetaArgs a;
  a.ws = h->ws;
  a.N = h->N;
  a.m_cap = m_cap;
  a.R_cap = R_cap;
  a.selected = selected;
  a.ret_token = ret_token;
  a.ret_parent = ret_parent;
  a.ret_count = ret_token ? ret_count : nullptr;
  a.ret_anchor = ret_token ? ret_anchor : nullptr;
  a.K_total = ret_token ? K_total : 0;
  a.pos_offset = pos_offset;
  a.meta = *meta;
  const size_t smem = ((size_t)h->N * sizeof(int16_t) + 15) / 16 * 16;
  launch_k(build_meta_kernel, dim3(h->B), dim3(kMetaThreads), smem, s, a);
  return cudaGetLastError();
}

}  // namespace dt
