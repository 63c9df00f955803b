// Selection kernels: global rerank, CAST width/depth/verify-count pruning, Graft checkpoints.
//
// EAGLE-2 page §"重排阶段": sort every node by value, take the top-m, shallow nodes first on
// ties, which keeps the selection a connected subtree (V_child <= V_parent).
// CAST page §关键设计 2-4: marginal utility (u_k - u_k0)/(c_k - c_k0) against C1 (width) and C3
// (verify count), FIFO gain buffer against C2 (depth); costs from the S_T/S_D lookup tables.
// Graft page step (1): c_d = exp(max_j S_{d,j}) against tau_d at the checkpoints.
#include <algorithm>

#include "cast_block.cuh"

namespace dt {
namespace {

struct SortArgs {
  Workspace ws;
  int N, LW, D, depth, mode;  // mode 0: rerank -> selected; 1: linear values of the top m_cap
  const int32_t* m;
  int m_len, m_cap;
  int32_t* selected;
};

constexpr int kSortThreads = 512;

// One CTA per request: the valid non-root nodes in the total order (value desc, id asc), which puts
// shallower nodes first on equal values since ids grow with depth. Every layer is already sorted by
// the expansion (layer_order), so a node's rank is its place in its own layer plus, for every other
// layer, the number of keys above it there (binary search): no full sort is needed.
__global__ void __launch_bounds__(kSortThreads) sort_nodes_kernel(SortArgs a) {
  pdl_begin();
  extern __shared__ __align__(16) uint64_t keys[];  // [depth][LW]: layer d's valid keys at (d-1)*LW
  __shared__ int cnt[kMaxD + 1];
  __shared__ int32_t sel[kMaxP];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Workspace& ws = a.ws;
  // every node's key in one round of loads (slot (d-1)*LW + p holds layer d's p-th node, 0 if none or
  // invalid); then warp d-1 compacts layer d's valid keys in place, order preserved
  for (int f = tid; f < a.depth * a.LW; f += blockDim.x) {
    const int d = 1 + f / a.LW, p = f % a.LW;
    const int64_t lb = (int64_t)b * (a.D + 1) + d;
    uint64_t k = 0ull;
    const int64_t li = lb * a.LW + p;
    const int lc = ws.layer_count[lb];
    const int id = ws.layer_order[li];  // read with the count: not used past it
    const int tok = ws.layer_tok[li];
    const float v = ws.layer_val[li];
    if (p < lc && id > 0 && id < a.N && tok >= 0) k = make_key(v, (uint32_t)id);
    keys[f] = k;
  }
  __syncthreads();
  for (int d = 1 + warp; d <= a.depth; d += kSortThreads / 32) {
    uint64_t* g = keys + (int64_t)(d - 1) * a.LW;
    int c = 0;
    for (int p0 = 0; p0 < a.LW; p0 += 32) {
      const uint64_t k = p0 + lane < a.LW ? g[p0 + lane] : 0ull;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, k != 0ull);
      __syncwarp();
      if (k != 0ull) g[c + __popc(m & ((1u << lane) - 1u))] = k;  // c + rank <= p0 + lane: no overtaking
      c += __popc(m);
    }
    if (lane == 0) cnt[d] = c;
  }
  __syncthreads();
  int n = 0;
  for (int d = 1; d <= a.depth; ++d) n += cnt[d];
  int limit;
  if (a.mode == 0) {
    int mb = a.m ? a.m[a.m_len == 1 ? 0 : b] : a.m_cap;
    limit = max(0, min(min(mb, a.m_cap), n));
  } else {
    limit = min(n, a.m_cap);
  }
  double* lin = ws.sorted_lin + (int64_t)b * a.m_cap;
  for (int f = tid; f < a.depth * a.LW; f += blockDim.x) {
    const int d = 1 + f / a.LW, p = f % a.LW;
    if (p >= cnt[d]) continue;
    const uint64_t k = keys[f];
    int rank = p;
    for (int e = 1; e <= a.depth && rank < limit; ++e) {
      if (e == d) continue;
      const uint64_t* g = keys + (int64_t)(e - 1) * a.LW;
      int lo = 0, hi = cnt[e];  // keys above k in layer e
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (g[mid] > k) lo = mid + 1;
        else hi = mid;
      }
      rank += lo;
    }
    if (rank >= limit) continue;
    if (a.mode == 0) {
      sel[rank] = (int32_t)key_id(k);
    } else {
      lin[rank] = (double)expf(key_value(k));
      ws.sorted_ids[(int64_t)b * a.m_cap + rank] = (int32_t)key_id(k);
    }
  }
  if (a.mode == 0) {
    __syncthreads();
    // selected ids, ascending: rank each of the first `limit` ids among themselves
    int32_t* out = a.selected + (int64_t)b * a.m_cap;
    for (int i = tid; i < limit; i += blockDim.x) {
      const int32_t id = sel[i];
      int r = 0;
      for (int j = 0; j < limit; ++j) r += sel[j] < id;
      out[r] = id;
    }
    for (int i = limit + tid; i < a.m_cap; i += blockDim.x) out[i] = -1;
  } else {
    for (int i = limit + tid; i < a.m_cap; i += blockDim.x) lin[i] = 0.0;
    if (tid == 0) ws.sorted_cnt[b] = limit;
  }
}

// CAST width + depth after layer d (1 CTA).
__global__ void __launch_bounds__(kPruneThreads) cast_width_depth_kernel(PruneArgs a) {
  pdl_begin();
  cast_width_depth_block(a);
}

// CAST verify count from the per-request sorted linear values (1 CTA).
__global__ void __launch_bounds__(kPruneThreads) cast_verify_kernel(PruneArgs a) {
  pdl_begin();
  __shared__ double items[kMaxP + 1];
  __shared__ double cost[kMaxP + 2];
  __shared__ double part[32 * kItemChunk];
  __shared__ double u[kMaxP + 2];
  __shared__ uint64_t cimg[kMaxP + 2], qimg[kMaxP + 2];
  __shared__ int s_maxn, s_k0;
  const Workspace& ws = a.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = (int)(blockDim.x >> 5);
  const double* lin = ws.sorted_lin;
  const int mcap = a.p.m_cap;
  // No barrier before the loads: the last two warps compute the cost vector, the third-last the
  // largest count, while batch_items reads the linear values of every slot up to m_cap (the sort
  // left 0 past each request's count); its first barrier publishes all of it.
  if (warp >= nwarps - 2) {
    const int row = table_row((double)a.p.n0, a.p.L, a.p.M_rows);
    for (int k = 1 + (tid - (nwarps - 2) * 32); k <= mcap; k += 64)
      cost[k] = a.p.S_T[(int64_t)row * a.p.N_cols + (k - 1)] / a.p.S_T[(int64_t)row * a.p.N_cols];
  }
  if (warp == nwarps - 3) {
    int mc = 0;
    for (int b = lane; b < a.B; b += 32) mc = max(mc, ws.sorted_cnt[b]);
    mc = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)max(mc, 0));
    if (lane == 0) s_maxn = mc;
  }
  batch_items(items, part, mcap, a.B, [&](int b, int s) { return lin[(int64_t)b * a.p.m_cap + s]; });
  const int cap = min(a.p.m_cap, s_maxn);
  int m = 0;
  if (cap > 0) m = selection_rule(items, cost, a.p.C3, cap, u, cimg, qimg, &s_k0, [](int) {});
  if (tid == 0) a.out.m[0] = m;
  if (a.sel) {  // the rerank, as dt_rerank(m) would write it: each request's top-m ids, ascending
    const int lane = tid & 31;
    for (int b = tid >> 5; b < a.B; b += blockDim.x >> 5) {
      const int mb = max(0, min(min(m, a.p.m_cap), ws.sorted_cnt[b]));
      const int32_t* ids = ws.sorted_ids + (int64_t)b * a.p.m_cap;
      int32_t* out = a.sel + (int64_t)b * a.p.m_cap;
      for (int i = lane; i < a.p.m_cap; i += 32) {
        if (i < mb) {
          const int32_t id = ids[i];
          int r = 0;
          for (int j = 0; j < mb; ++j) r += ids[j] < id;
          out[r] = id;
        } else {
          out[i] = -1;
        }
      }
    }
  }
}

// CAST width + depth, per-request rule: one warp per request applies the batch rule to the request
// alone (a batch of one: its items are its own sorted path values, the batch mean of one value being
// that value), with its own state (context sum, FIFO, last utility) and its own stop; then, with
// select, its next frontier. A request stopped at an earlier layer stays stopped.
constexpr int kReqWarps = 8;
__global__ void __launch_bounds__(32 * kReqWarps) cast_width_depth_req_kernel(PruneArgs a) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kReqWarps + (threadIdx.x >> 5);
  if (b >= a.B) return;
  const Workspace& ws = a.ws;
  CastState* cst = ws.cast_req + b;
  int f_id = -1, f_tok = -1, f_avail = 0;
  float f_val = -INFINITY;
  if (a.select) f_avail = frontier_candidates(ws, b, a.N, a.W, a.LW, a.D, a.d, f_id, f_tok, f_val);
  const bool stopped = a.d > 1 && a.out.stop[b] != 0;
  int n = 0;
  bool grow = false;
  if (!stopped) {
    const int wcap = min(a.p.width_cap, a.LW);
    const int64_t lb = (int64_t)b * (a.D + 1) + a.d;
    const int cnt = ws.layer_count[lb];
    const float v = lane < a.LW ? ws.layer_val[lb * a.LW + lane] : 0.0f;  // read with the count
    const int row = table_row((double)(a.p.n0 + cst->ctx_sum), a.p.L, a.p.M_rows);
    const int cap = min(a.p.width_cap, cnt);
    const int k = lane + 1;  // lane k - 1 holds u_k and c_k
    const double item = (lane < wcap && lane < cnt) ? 0.0 + (double)expf(v) : 0.0;
    double ck = 0.0;
    if (k <= wcap) ck = a.p.S_D[(int64_t)row * a.p.N_cols + (k - 1)] / a.p.S_T[(int64_t)row * a.p.N_cols];
    double x = k <= cap ? item : 0.0;  // u_k: inclusive prefix (the batch rule's scan)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    x += 0.0;
    const uint64_t cimg = d2ord(ck), qimg = d2ord(x - a.p.C1 * ck);
    if (cap > 0) {
      int k0 = 1;
      uint64_t c0 = __shfl_sync(0xFFFFFFFFu, cimg, 0), q0 = __shfl_sync(0xFFFFFFFFu, qimg, 0);
      for (int kk = 2; kk <= cap; ++kk) {
        const uint64_t c = __shfl_sync(0xFFFFFFFFu, cimg, kk - 1), q = __shfl_sync(0xFFFFFFFFu, qimg, kk - 1);
        if (c <= c0 || q >= q0) {
          k0 = kk;
          c0 = c;
          q0 = q;
        }
      }
      n = k0;
    }
    const double un = __shfl_sync(0xFFFFFFFFu, x, max(n, 1) - 1);
    const double cn = __shfl_sync(0xFFFFFFFFu, ck, max(n, 1) - 1);
    int g = 0;
    if (lane == 0 && cap > 0) {
      CastState cs = *cst;
      const int len = cs.fifo_len;
      const double up = cs.u_prev;
      const bool app = up >= 0.0;  // this layer appends a ratio
      double kept = 0.0;
      for (int j = app && len >= a.p.R ? 1 : 0; j < len; ++j) kept += cs.fifo[j];
      const int nlen = app ? (len < a.p.R ? len + 1 : len) : len;
      bool gg;
      if (nlen <= 0) {
        gg = false;  // the mean of an empty FIFO is NaN
      } else if (app && up > 0.0) {
        gg = (kept * up + un) * un >= a.p.C2 * cn * (double)nlen * up;
      } else if (app) {  // u_prev = 0: the ratio is not finite; the quotient form as written
        const double alpha = (kept + un / up) / (double)nlen;
        gg = alpha * un >= a.p.C2 * cn;
      } else {
        gg = kept * un >= a.p.C2 * cn * (double)nlen;
      }
      g = ((a.d < a.p.D_max) && gg) ? 1 : 0;
      if (app) {
        const double ratio = un / up;
        int l2 = len;
        if (l2 < a.p.R) {
          cs.fifo[l2++] = ratio;
        } else {
          for (int j = 1; j < l2; ++j) cs.fifo[j - 1] = cs.fifo[j];
          cs.fifo[l2 - 1] = ratio;
        }
        cs.fifo_len = l2;
      }
      cs.u_prev = un;
      cs.u_layer = un;
      cs.ctx_sum += n;
      *cst = cs;
    }
    grow = __shfl_sync(0xFFFFFFFFu, g, 0) != 0;
  }
  if (lane == 0) {
    a.out.width[b] = n;
    a.out.stop[b] = grow ? 0 : 1;
  }
  if (a.select)  // the next layer's frontier, as dt_select_frontier(width[b], stop[b]) would choose it
    select_frontier_write(ws, b, a.W, max(0, min(min(grow ? n : 0, a.W), f_avail)), f_id, f_tok, f_val, a.ftok);
}

// CAST verify count, per-request rule: one warp per request runs the selection over the request's own
// sorted path values (a batch of one), then, with sel, writes its top-m_b ids in ascending order.
__global__ void __launch_bounds__(32) cast_verify_req_kernel(PruneArgs a) {
  pdl_begin();
  __shared__ uint64_t cimg[kMaxP + 2], qimg[kMaxP + 2];
  const int b = blockIdx.x, lane = threadIdx.x;
  const Workspace& ws = a.ws;
  const int mcap = a.p.m_cap;
  const double* lin = ws.sorted_lin + (int64_t)b * mcap;
  const int cnt = ws.sorted_cnt[b];
  const int cap = min(mcap, cnt);
  const int row = table_row((double)a.p.n0, a.p.L, a.p.M_rows);
  const double t0 = a.p.S_T[(int64_t)row * a.p.N_cols];
  double carry = 0.0;
  for (int c0 = 0; c0 < cap; c0 += 32) {  // u_k, chunk by chunk (the batch rule's scan)
    const int k = c0 + lane + 1;
    double x = k <= cap ? (0.0 + (0.0 + lin[k - 1])) : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    x += carry;
    if (k <= cap) {
      const double ck = a.p.S_T[(int64_t)row * a.p.N_cols + (k - 1)] / t0;
      cimg[k] = d2ord(ck);
      qimg[k] = d2ord(x - a.p.C3 * ck);
    }
    carry = __shfl_sync(0xFFFFFFFFu, x, 31);
  }
  __syncwarp();
  int m = 0;
  if (lane == 0 && cap > 0) {
    int k0 = 1;
    uint64_t c0 = cimg[1], q0 = qimg[1];
    for (int k = 2; k <= cap; ++k) {
      const uint64_t ck = cimg[k], qk = qimg[k];
      if (ck <= c0 || qk >= q0) {
        k0 = k;
        c0 = ck;
        q0 = qk;
      }
    }
    m = k0;
  }
  m = __shfl_sync(0xFFFFFFFFu, m, 0);
  if (lane == 0) a.out.m[b] = m;
  if (a.sel) {  // the rerank, as dt_rerank(m[b]) would write it: the request's top-m ids, ascending
    const int mb = max(0, min(m, cnt));
    const int32_t* ids = ws.sorted_ids + (int64_t)b * mcap;
    int32_t* out = a.sel + (int64_t)b * mcap;
    for (int i = lane; i < mcap; i += 32) {
      if (i < mb) {
        const int32_t id = ids[i];
        int r = 0;
        for (int j = 0; j < mb; ++j) r += ids[j] < id;
        out[r] = id;
      } else {
        out[i] = -1;
      }
    }
  }
}

// Graft checkpoint after layer d: one thread per request.
__global__ void graft_checkpoint_kernel(PruneArgs a) {
  pdl_begin();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < a.B) graft_checkpoint_one(a, b);
}

}  // namespace

cudaError_t init_select_attributes() {
  // the largest tree: 16 layers of W*K <= 1024 keys of 8 bytes
  return cudaFuncSetAttribute(sort_nodes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxD * kCandCap * 8);
}

static cudaError_t launch_sort(dt_handle* h, int mode, const int32_t* m, int m_len, int m_cap, int32_t* selected,
                               cudaStream_t s) {
  SortArgs a;
  a.ws = h->ws;
  a.N = h->N;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.depth = h->depth;
  a.mode = mode;
  a.m = m;
  a.m_len = m_len;
  a.m_cap = m_cap;
  a.selected = selected;
  const size_t smem = (size_t)std::max(1, h->depth) * h->LW * sizeof(uint64_t);
  launch_k(sort_nodes_kernel, dim3(h->B), dim3(kSortThreads), smem, s, a);
  return cudaGetLastError();
}

cudaError_t launch_rerank(dt_handle* h, const int32_t* m, int m_len, int m_cap, int32_t* selected,
                          cudaStream_t s) {
  return launch_sort(h, 0, m, m_len, m_cap, selected, s);
}

cudaError_t launch_cast_prune(dt_handle* h, int policy, const dt_prune_params* p, const dt_prune_out* out,
                              cudaStream_t s) {
  PruneArgs a;
  a.ws = h->ws;
  a.p = *p;
  a.out = *out;
  a.B = h->B;
  a.N = h->N;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.d = h->depth;
  a.policy = policy;
  a.W = h->cfg.W;
  a.select = 0;
  a.ftok = nullptr;
  a.sel = nullptr;
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH) {
    if (p->per_request)
      launch_k(cast_width_depth_req_kernel, dim3((h->B + kReqWarps - 1) / kReqWarps), dim3(32 * kReqWarps), 0, s, a);
    else
      launch_k(cast_width_depth_kernel, dim3(1), dim3(prune_threads(h->B)), 0, s, a);
    return cudaGetLastError();
  }
  if (policy == DT_POLICY_CAST_VERIFY) {
    cudaError_t e = launch_sort(h, 1, nullptr, 1, p->m_cap, nullptr, s);
    if (e != cudaSuccess) return e;
    if (p->per_request)
      launch_k(cast_verify_req_kernel, dim3(h->B), dim3(32), 0, s, a);
    else
      launch_k(cast_verify_kernel, dim3(1), dim3(prune_threads(h->B)), 0, s, a);
    return cudaGetLastError();
  }
  launch_k(graft_checkpoint_kernel, dim3((h->B + 127) / 128), dim3(128), 0, s, a);
  return cudaGetLastError();
}

cudaError_t launch_cast_prune_select(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out,
                                     int32_t* frontier_token, cudaStream_t s) {
  PruneArgs a;
  a.ws = h->ws;
  a.p = *p;
  a.out = *out;
  a.B = h->B;
  a.N = h->N;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.d = h->depth;
  a.policy = DT_POLICY_CAST_WIDTH_DEPTH;
  a.W = h->cfg.W;
  a.select = 1;
  a.ftok = frontier_token;
  a.sel = nullptr;
  if (p->per_request)
    launch_k(cast_width_depth_req_kernel, dim3((h->B + kReqWarps - 1) / kReqWarps), dim3(32 * kReqWarps), 0, s, a);
  else
    launch_k(cast_width_depth_kernel, dim3(1), dim3(prune_threads(h->B)), 0, s, a);
  return cudaGetLastError();
}

cudaError_t launch_cast_verify_rerank(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out,
                                     int32_t* selected, cudaStream_t s) {
  cudaError_t e = launch_sort(h, 1, nullptr, 1, p->m_cap, nullptr, s);
  if (e != cudaSuccess) return e;
  PruneArgs a;
  a.ws = h->ws;
  a.p = *p;
  a.out = *out;
  a.B = h->B;
  a.N = h->N;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.d = h->depth;
  a.policy = DT_POLICY_CAST_VERIFY;
  a.W = h->cfg.W;
  a.select = 0;
  a.ftok = nullptr;
  a.sel = selected;
  if (p->per_request)
    launch_k(cast_verify_req_kernel, dim3(h->B), dim3(32), 0, s, a);
  else
    launch_k(cast_verify_kernel, dim3(1), dim3(prune_threads(h->B)), 0, s, a);
  return cudaGetLastError();
}

}  // namespace dt
