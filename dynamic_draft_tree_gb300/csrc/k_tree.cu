// Tree construction kernels: reset, frontier selection, layer expansion.
//
// EAGLE-2 page, §"置信度为什么可以近似接受率" (c = draft probability of the token),
// §"value 公式" (value = product of confidences on the path, kept as a sum of logs) and
// §"扩展阶段" (expand the top-k nodes of the newest layer; every expanded node adds its
// top-K vocabulary children; value(child) = value(parent) * c).
#include <algorithm>

#include "rowscan.cuh"

namespace dt {
namespace {

__device__ __forceinline__ int layer_of(int id, int K, int LW) {
  if (id == 0) return 0;
  if (id <= K) return 1;
  return 2 + (id - 1 - K) / LW;
}

__global__ void tree_reset_kernel(Workspace ws, const int32_t* __restrict__ root, int B, int N, int K, int LW,
                                  int D, int V) {
  pdl_begin();
  const int64_t total = (int64_t)B * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / N), id = (int)(i % N);
    if (id == 0) {
      const int r = root[b];
      if (r < 0 || r >= V) set_status(ws.status, DT_DEV_BAD_TOKEN);
      ws.token[i] = r;
      ws.logc[i] = 0.0f;
      ws.value[i] = 0.0f;
    } else {
      ws.token[i] = -1;
      ws.logc[i] = -INFINITY;
      ws.value[i] = -INFINITY;
    }
    ws.parent[i] = -1;
    ws.node_depth[i] = layer_of(id, K, LW);
  }
  // layer orders invalid, except layer 0 = {root}: id 0, value 0, the root token (so that the
  // frontier of layer 1 is selected like any other)
  const int64_t lo_total = (int64_t)B * (D + 1) * LW;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < lo_total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t lb = i / LW;
    if (lb % (D + 1) == 0 && i % LW == 0) {
      ws.layer_order[i] = 0;
      ws.layer_val[i] = 0.0f;
      ws.layer_tok[i] = root[lb / (D + 1)];
    } else {
      ws.layer_order[i] = -1;
    }
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)B * (D + 1);
       i += (int64_t)gridDim.x * blockDim.x)
    ws.layer_count[i] = (i % (D + 1)) == 0 ? 1 : 0;
  const int W = LW / K;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)B * W;
       i += (int64_t)gridDim.x * blockDim.x) {
    ws.frontier[i] = (i % W) == 0 ? 0 : -1;
    ws.frontier_val[i] = (i % W) == 0 ? 0.0f : -INFINITY;
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < B; i += (int64_t)gridDim.x * blockDim.x)
    ws.frontier_count[i] = 1;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < B; i += (int64_t)gridDim.x * blockDim.x) {
    CastState* cs = ws.cast_req + i;  // per-request rule: FIFO = {1}, no ratio yet, no context yet
    for (int j = 0; j < kMaxFifo; ++j) cs->fifo[j] = 0.0;
    cs->fifo[0] = 1.0;
    cs->fifo_len = 1;
    cs->u_prev = -1.0;
    cs->ctx_sum = 0;
    cs->u_layer = 0.0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    CastState* cs = ws.cast;
    for (int j = 0; j < kMaxFifo; ++j) cs->fifo[j] = 0.0;
    cs->fifo[0] = 1.0;
    cs->fifo_len = 1;
    cs->u_prev = -1.0;  // none yet
    cs->ctx_sum = 0;
    cs->u_layer = 0.0;
  }
}

// One warp per request: the first w nodes of layer d in (value desc, id asc) order, slotted by id.
__global__ void select_frontier_kernel(Workspace ws, int B, int N, int K, int W, int LW, int D, int d,
                                       const int32_t* __restrict__ width, int width_len,
                                       const int32_t* __restrict__ stop, int32_t* __restrict__ ftok) {
  pdl_begin();
  const int warps = blockDim.x >> 5;
  const int b = blockIdx.x * warps + (threadIdx.x >> 5);
  if (b >= B) return;
  int w = width ? width[width_len == 1 ? 0 : b] : W;
  if (stop && stop[b]) w = 0;
  select_frontier_warp(ws, b, N, W, LW, D, d, w, ftok);
}

struct ExpandArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int F, B, N, K, W, LW, D, d, V;
  int Smax;      // pieces per row at most
  int32_t base;  // first id of layer d
  uint32_t first_wait_cap;
  GumbelCtx draw;  // sampled drafts: seed and round of the draw noise (c2 set per row)
};

// Balanced over the active rows (request b expands min(frontier_count[b], F) nodes); see the
// balanced row pass in rowscan.cuh.
// GUMBEL: sampled drafts, the K children are the first K tokens of x + G (draws without replacement
// from softmax(x)), in draw order; each expanded node records its slot and its row's statistics for the
// sampled verify.
template <typename T, bool GUMBEL>
__global__ void __launch_bounds__(kRowThreads, 4) expand_kernel(ExpandArgs a) {
  pdl_begin();
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ ScanSmem sm;
  __shared__ RowPlan plan;
  const int tid = threadIdx.x;
  Workspace& ws = a.ws;
  auto cnt = [&](int b) -> int { return min(max(ws.frontier_count[b], 0), a.F); };
  if (tid < 32) {
    RowPlan p;
    plan_rows(p, a.B, a.V, a.Smax, (int)sizeof(T), cnt, GUMBEL ? 1 : 2);
    if (tid == 0) plan = p;
    if (blockIdx.x == 0)  // a frontier wider than the launch's F is a caller error
      for (int b = tid; b < a.B; b += 32)
        if (ws.frontier_count[b] > a.F) set_status(ws.status, DT_DEV_BAD_TREE);
  }
  __syncthreads();
  const RowPlan p = plan;
  if ((int)blockIdx.x >= p.G) return;

  // the parent's id and value are loaded when a piece starts (no dependent load in the finish)
  int pid = -1;
  float pval = 0.0f;
  auto row_of = [&](int b, int f) -> const T* {
    pid = ws.frontier[(int64_t)b * a.W + f];
    pval = ws.frontier_val[(int64_t)b * a.W + f];
    return reinterpret_cast<const T*>(a.logits) + ((int64_t)b * a.F + f) * a.ld;
  };
  // last piece of row (b, f): write the K children of frontier slot f
  auto finish = [&](int b, int f, const SoftmaxStat& st) {
    const float M = st.m;
    if (tid == 0 && (st.nan || !(M > -INFINITY) || M == INFINITY || !(st.s_hi > 0.0f) || st.s_hi == INFINITY))
      set_status(ws.status, DT_DEV_BAD_LOGITS);
    if (tid < a.K) {
      const uint64_t k = sm.topk[tid];
      const int id = a.base + f * a.K + tid;
      const int64_t gi = (int64_t)b * a.N + id;
      // log c = (x - M) - log S and value = value(parent) + log c, each kept as a double-float until
      // the final rounding
      float dh, dl;
      float x = key_value(k);
      if (GUMBEL) {  // the key holds x + G: the token's own logit
        const uint32_t t = key_id(k);
        const T* rowp = reinterpret_cast<const T*>(a.logits) + ((int64_t)b * a.F + f) * a.ld;
        x = k != 0ull && t < (uint32_t)a.V ? Elt<T>::load(rowp + t) : -INFINITY;
      }
      log_softmax_dd(st, x, dh, dl);
      const float lc = __fadd_rn(dh, dl);
      float vh = pval, vl = 0.0f;
      ff_add(vh, vl, dh, dl);
      ws.token[gi] = (int32_t)key_id(k);
      ws.parent[gi] = pid;
      ws.logc[gi] = lc;
      ws.value[gi] = __fadd_rn(vh, vl);
      if (GUMBEL && tid == 0) {  // the row the node's children were drawn from, for the sampled verify
        ws.exp_slot[(int64_t)b * a.N + pid] = f;
        ws.exp_stat[(int64_t)b * a.N + pid] = make_float4(st.m, st.s_hi, st.s_lo, 0.0f);
      }
      __threadfence();  // the children reach L2 before this row's arrival below
    }
    __syncthreads();
    const int active = cnt(b);
    if (tid == 0) {
      const int prev = atomicAdd(&ws.req_counter[b], 1);
      sm.last = (prev == active - 1);
    }
    __syncthreads();
    if (sm.last) {  // last row of the request: order the new layer by (value desc, id asc)
      if (tid == 0) ws.req_counter[b] = 0;
      const int n = active * a.K;
      const int64_t lo = ((int64_t)b * (a.D + 1) + a.d) * a.LW;
      // keys staged in the candidate buffer (n <= W*K <= 1024 = kCandCap), the tokens after it (the
      // stage memory holds both); the layer's values and tokens are written in order next to the ids
      int32_t* tok_s = reinterpret_cast<int32_t*>(sm.cand + kCandCap);
      for (int i = tid; i < n; i += blockDim.x) {
        const int64_t gi = (int64_t)b * a.N + a.base + i;
        sm.cand[i] = make_key(__ldcg(&ws.value[gi]), (uint32_t)(a.base + i));
        tok_s[i] = __ldcg(&ws.token[gi]);
      }
      __syncthreads();
      for (int i = tid; i < n; i += blockDim.x) {
        const uint64_t k = sm.cand[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += (sm.cand[j] > k);
        ws.layer_order[lo + rank] = (int32_t)key_id(k);
        ws.layer_val[lo + rank] = key_value(k);
        ws.layer_tok[lo + rank] = tok_s[i];
      }
      if (tid == 0) ws.layer_count[(int64_t)b * (a.D + 1) + a.d] = n;
    }
  };
  auto noise = [&](int b, int f) -> GumbelCtx {
    GumbelCtx g = a.draw;
    g.c2 = 0x40000000u + 4096u * (uint32_t)b + (uint32_t)pid;
    return g;
  };
  scan_pieces<T, true, GUMBEL>(p, a.V, a.K, a.B, ws.partials, ws.row_counter, ws.row_tau, sm, dyn_smem,
                               a.first_wait_cap, ws.status, row_of, cnt, finish, noise);
}

}  // namespace

int row_pass_grid(const dt_handle* h) {
  // one wave: 4 CTAs per SM (128 registers and 56 KB of shared memory each), within the piece-slot capacity
  const int64_t g = std::min<int64_t>((int64_t)h->num_sms * 4, 4096);
  return (int)std::max<int64_t>(1, g);
}

int row_pass_smax(int K) { return std::min(64, kCandCap / K); }

static size_t row_smem_bytes() { return (size_t)kScanSmemBytes; }

template <typename T, bool G>
static cudaError_t set_expand_attributes(int smem) {
  cudaError_t e = cudaFuncSetAttribute(expand_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // all of the unified L1 as shared memory, so that 4 CTAs fit on an SM
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expand_kernel<T, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t init_tree_attributes() {
  const int smem = (int)row_smem_bytes();
  cudaError_t e = set_expand_attributes<uint16_t, false>(smem);
  if (e == cudaSuccess) e = set_expand_attributes<float, false>(smem);
  if (e == cudaSuccess) e = set_expand_attributes<uint16_t, true>(smem);
  if (e == cudaSuccess) e = set_expand_attributes<float, true>(smem);
  return e;
}

cudaError_t launch_tree_reset(dt_handle* h, const int32_t* root, cudaStream_t s) {
  const int64_t total = (int64_t)h->B * h->N;
  int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)h->num_sms * 4);
  if (blocks < 1) blocks = 1;
  launch_k(tree_reset_kernel, dim3(blocks), dim3(256), 0, s, h->ws, root, h->B, h->N, h->cfg.K, h->LW, h->cfg.D_max, h->cfg.V);
  return cudaGetLastError();
}

cudaError_t launch_select_frontier(dt_handle* h, const int32_t* width, int width_len, const int32_t* stop,
                                   int32_t* frontier_token, cudaStream_t s) {
  const int warps = 8;
  const int blocks = (h->B + warps - 1) / warps;
  launch_k(select_frontier_kernel, dim3(blocks), dim3(warps * 32), 0, s, h->ws, h->B, h->N, h->cfg.K, h->cfg.W, h->LW,
                                                        h->cfg.D_max, h->depth, width, width_len, stop,
                                                        frontier_token);
  return cudaGetLastError();
}

cudaError_t launch_expand(dt_handle* h, const void* logits, int64_t ld, int F, cudaStream_t s, bool draw,
                          uint64_t seed, uint64_t round) {
  const int d = h->depth + 1;
  ExpandArgs a;
  a.ws = h->ws;
  a.logits = logits;
  a.ld = ld;
  a.F = F;
  a.B = h->B;
  a.N = h->N;
  a.K = h->cfg.K;
  a.W = h->cfg.W;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.d = d;
  a.V = h->cfg.V;
  a.Smax = row_pass_smax(h->cfg.K);
  a.base = d == 1 ? 1 : 1 + h->cfg.K + (d - 2) * h->LW;
  a.first_wait_cap = (h->cfg.flags & DT_FLAG_TEST_TIMEOUT) ? 0u : kSpinCap;
  a.draw = GumbelCtx{(uint32_t)seed, (uint32_t)(seed >> 32), (uint32_t)round, (uint32_t)(round >> 32), 0u};
  const unsigned grid = (unsigned)row_pass_grid(h);
  const size_t smem = row_smem_bytes();
  if (h->cfg.dtype == DT_BF16) {
    if (draw) launch_k(expand_kernel<uint16_t, true>, dim3(grid), dim3(kRowThreads), smem, s, a);
    else launch_k(expand_kernel<uint16_t, false>, dim3(grid), dim3(kRowThreads), smem, s, a);
  } else {
    if (draw) launch_k(expand_kernel<float, true>, dim3(grid), dim3(kRowThreads), smem, s, a);
    else launch_k(expand_kernel<float, false>, dim3(grid), dim3(kRowThreads), smem, s, a);
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) h->depth = d;
  return e;
}

// The expansion followed by the policy's pruning and the next frontier (the same kernels as the
// separate calls: after CAST's pruning the fused prune + select kernel).
cudaError_t launch_expand_ex(dt_handle* h, const void* logits, int64_t ld, int F, int policy,
                             const dt_prune_params* p, const dt_prune_out* out, const int32_t* width,
                             int width_len, int32_t* frontier_token, cudaStream_t s) {
  cudaError_t e = launch_expand(h, logits, ld, F, s);
  if (e != cudaSuccess) return e;
  const bool select = h->depth < h->cfg.D_max;  // no frontier after the last layer
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH)
    return select ? launch_cast_prune_select(h, p, out, frontier_token, s)
                  : launch_cast_prune(h, DT_POLICY_CAST_WIDTH_DEPTH, p, out, s);
  const int32_t* stop = nullptr;
  if (policy == DT_POLICY_GRAFT_CHECKPOINT) {
    e = launch_cast_prune(h, DT_POLICY_GRAFT_CHECKPOINT, p, out, s);
    if (e != cudaSuccess) return e;
    stop = out->stop;
  }
  return select ? launch_select_frontier(h, width, width_len, stop, frontier_token, s) : cudaSuccess;
}

}  // namespace dt
