// Block drafters: all draft layers of a block in one launch.
//
// Graft page, extension direction 1 (grafting for block drafters such as DFlash, which drafts 16
// tokens in one pass) and weakness 4 (token-level confidence inside the block instead of whole-block
// decisions; tree-shaped expansion inside the block). The drafter's row j is its distribution for
// block position j + 1 and does not depend on the tokens picked before it, so every row is read in
// one row pass. Layer j + 1 holds row j's top-K tokens as children of the block token at position j
// (the root for j = 0); the block token of a layer is its top node, the top-1 of its row. Values
// follow EAGLE-2 (value = value(parent) + log c, the Graft score S_j), and the Graft checkpoint rule
// (step (1)) gates each layer.
#include <algorithm>

#include "rowscan.cuh"

namespace dt {
namespace {

struct BlockArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int B, N, K, W, LW, D, L, V;
  int Smax;  // pieces per row at most
  uint32_t first_wait_cap;
  int gate;  // apply the Graft checkpoints
  dt_prune_params p;
  dt_prune_out out;
};

__device__ __forceinline__ int layer_base(int d, int K, int LW) { return d == 1 ? 1 : 1 + K + (d - 2) * LW; }

// Layers 1..L of request b from its rows' children (token, parent, log c written by the row pass,
// log c also as a double-float in node_dd): one warp, layer by layer. Lane r < K holds child r.
__device__ void build_block_layers(const BlockArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  Workspace ws = a.ws;
  const int64_t nb = (int64_t)b * a.N;
  float S = 0.0f;       // value of the block token above the current layer (the root: 0)
  int chain = 0;        // its id
  float S_prev = 0.0f;  // value of the block token above the last built layer
  int chain_prev = 0;
  int stop_d = 0;       // layer after which a gate stopped the request (0: none)
  if (a.gate && lane == 0) a.out.stop[b] = 0;
  for (int d = 1; d <= a.L; ++d) {
    const int base = layer_base(d, a.K, a.LW);
    const int64_t gi = nb + base + lane;
    float v = -INFINITY;
    uint64_t key = 0ull;
    int32_t tok = -1;
    if (lane < a.K) {
      const float2 dd = __ldcg(&ws.node_dd[gi]);
      float vh = S, vl = 0.0f;
      ff_add(vh, vl, dd.x, dd.y);
      v = __fadd_rn(vh, vl);
      tok = __ldcg(&ws.token[gi]);
      key = make_key(v, (uint32_t)(base + lane));
      ws.value[gi] = v;
    }
    // place of each child in (value desc, id asc) order
    int rank = 0;
    uint64_t top = key;
    for (int r = 0; r < a.K; ++r) {
      const uint64_t o = __shfl_sync(0xFFFFFFFFu, key, r);
      rank += o > key;
      top = o > top ? o : top;
    }
    const int64_t lo = ((int64_t)b * (a.D + 1) + d) * a.LW;
    if (lane < a.K) {
      ws.layer_order[lo + rank] = base + lane;
      ws.layer_val[lo + rank] = v;
      ws.layer_tok[lo + rank] = tok;
    }
    // the row pass made child 0 (the top-1 of the row) the parent of the next layer: it must be the
    // layer's top node
    if (lane == 0) {
      ws.layer_count[(int64_t)b * (a.D + 1) + d] = a.K;
      if ((int)key_id(top) != base) set_status(ws.status, DT_DEV_INTERNAL);
    }
    S_prev = S;
    chain_prev = chain;
    S = __shfl_sync(0xFFFFFFFFu, v, 0);
    chain = base;
    if (a.gate) {  // Graft step (1) after layer d (the same test as the per-layer checkpoint kernel)
      int stopped = 0;
      if (lane == 0) {
        const int li = d - 1;
        for (int s = 0; s < a.p.n_ckpt && !stopped; ++s) {
          if (a.p.ckpt_layer[s] != li) continue;
          const double c = (double)expf(S);
          if (!(c > a.p.tau[s])) {
            stopped = 1;
            a.out.stop[b] = 1;
            if (a.out.stage) a.out.stage[b] = s;
            if (a.out.m) a.out.m[b] = a.p.k_draft[s];
          }
        }
        if (!stopped && d == a.L) {
          a.out.stop[b] = 1;
          if (a.out.stage) a.out.stage[b] = a.p.n_ckpt;
          if (a.out.m) a.out.m[b] = a.p.K_total;
        }
      }
      stopped = __shfl_sync(0xFFFFFFFFu, stopped, 0);
      if (stopped) {
        stop_d = d;
        break;
      }
    }
  }
  // layers past a stop: the row pass wrote their children, which the truncated tree does not have
  if (stop_d > 0) {
    for (int d = stop_d + 1; d <= a.L; ++d) {
      const int64_t gi = nb + layer_base(d, a.K, a.LW) + lane;
      if (lane < a.K) {
        ws.token[gi] = -1;
        ws.parent[gi] = -1;
        ws.logc[gi] = -INFINITY;
        ws.value[gi] = -INFINITY;
      }
    }
  }
  // frontier: the block token that produced layer L, none for a stopped request
  if (lane == 0) {
    const bool running = stop_d == 0 || stop_d == a.L;
    ws.frontier[(int64_t)b * a.W] = running ? chain_prev : -1;
    ws.frontier_val[(int64_t)b * a.W] = running ? S_prev : -INFINITY;
    ws.frontier_count[b] = running ? 1 : 0;
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 4) block_expand_kernel(BlockArgs a) {
  pdl_begin();
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ ScanSmem sm;
  __shared__ RowPlan plan;
  const int tid = threadIdx.x;
  Workspace& ws = a.ws;
  auto cnt = [&](int b) -> int { return a.L; };
  if (tid < 32) {
    RowPlan p;
    plan_rows(p, a.B, a.V, a.Smax, (int)sizeof(T), cnt);
    if (tid == 0) plan = p;
  }
  __syncthreads();
  const RowPlan p = plan;
  if ((int)blockIdx.x >= p.G) return;
  auto row_of = [&](int b, int j) -> const T* {
    return reinterpret_cast<const T*>(a.logits) + ((int64_t)b * a.L + j) * a.ld;
  };
  // last piece of row (b, j): the K children of layer j + 1 (values once the layers above are known)
  auto finish = [&](int b, int j, const SoftmaxStat& st) {
    const float M = st.m;
    if (tid == 0 && (st.nan || !(M > -INFINITY) || M == INFINITY || !(st.s_hi > 0.0f) || st.s_hi == INFINITY))
      set_status(ws.status, DT_DEV_BAD_LOGITS);
    if (tid < a.K) {
      const uint64_t k = sm.topk[tid];
      const int d = j + 1;
      const int64_t gi = (int64_t)b * a.N + layer_base(d, a.K, a.LW) + tid;
      float dh, dl;
      log_softmax_dd(st, key_value(k), dh, dl);
      ws.token[gi] = (int32_t)key_id(k);
      ws.parent[gi] = d == 1 ? 0 : layer_base(d - 1, a.K, a.LW);
      ws.logc[gi] = __fadd_rn(dh, dl);
      ws.node_dd[gi] = make_float2(dh, dl);
      __threadfence();  // the children reach L2 before this row's arrival below
    }
    __syncthreads();
    if (tid == 0) {
      const int prev = atomicAdd(&ws.req_counter[b], 1);
      sm.last = (prev == a.L - 1);
    }
    __syncthreads();
    if (sm.last) {  // the request's last row: build its layers
      if (tid == 0) ws.req_counter[b] = 0;
      if (tid < 32) build_block_layers(a, b);
    }
  };
  scan_pieces<T, true>(p, a.V, a.K, a.B, ws.partials, ws.row_counter, ws.row_tau, sm, dyn_smem, a.first_wait_cap,
                       ws.status, row_of, cnt, finish, [](int, int) { return GumbelCtx{}; });
}

}  // namespace

cudaError_t init_block_attributes() {
  const int smem = (int)kScanSmemBytes;
  cudaError_t e =
      cudaFuncSetAttribute(block_expand_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(block_expand_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(block_expand_kernel<uint16_t>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(block_expand_kernel<float>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t launch_block_expand(dt_handle* h, const void* logits, int64_t ld, int L, const dt_prune_params* p,
                                const dt_prune_out* out, cudaStream_t s) {
  BlockArgs a;
  a.ws = h->ws;
  a.logits = logits;
  a.ld = ld;
  a.B = h->B;
  a.N = h->N;
  a.K = h->cfg.K;
  a.W = h->cfg.W;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.L = L;
  a.V = h->cfg.V;
  a.Smax = row_pass_smax(h->cfg.K);
  a.first_wait_cap = (h->cfg.flags & DT_FLAG_TEST_TIMEOUT) ? 0u : kSpinCap;
  a.gate = p != nullptr;
  if (p) {
    a.p = *p;
    a.out = *out;
  } else {
    a.p = dt_prune_params{};
    a.out = dt_prune_out{};
  }
  const unsigned grid = (unsigned)row_pass_grid(h);
  if (h->cfg.dtype == DT_BF16)
    launch_k(block_expand_kernel<uint16_t>, dim3(grid), dim3(kRowThreads), (size_t)kScanSmemBytes, s, a);
  else
    launch_k(block_expand_kernel<float>, dim3(grid), dim3(kRowThreads), (size_t)kScanSmemBytes, s, a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) h->depth = L;
  return e;
}

}  // namespace dt
