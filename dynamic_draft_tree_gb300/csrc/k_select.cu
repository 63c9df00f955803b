// Selection kernels: global rerank, CAST width/depth/verify-count pruning, Graft checkpoints.
//
// EAGLE-2 page §"重排阶段": sort every node by value, take the top-m, shallow nodes first on
// ties, which keeps the selection a connected subtree (V_child <= V_parent).
// CAST page §关键设计 2-4: marginal utility (u_k - u_k0)/(c_k - c_k0) against C1 (width) and C3
// (verify count), FIFO gain buffer against C2 (depth); costs from the S_T/S_D lookup tables.
// Graft page step (1): c_d = exp(max_j S_{d,j}) against tau_d at the checkpoints.
#include <algorithm>

#include "dt_internal.cuh"

namespace dt {
namespace {

// Descending bitonic sort of n_pad (power of two) 64-bit keys in shared memory.
__device__ void block_bitonic_desc(uint64_t* keys, int n_pad) {
  for (int size = 2; size <= n_pad; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < n_pad / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a < b) == desc) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
    }
  }
  __syncthreads();
}

struct SortArgs {
  Workspace ws;
  int N, depth, n_pad, mode;  // mode 0: rerank -> selected; 1: linear values of the top m_cap
  const int32_t* m;
  int m_len, m_cap;
  int32_t* selected;
};

// One CTA per request: all valid non-root nodes in the total order.
__global__ void __launch_bounds__(1024) sort_nodes_kernel(SortArgs a) {
  extern __shared__ __align__(16) uint64_t keys[];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const Workspace& ws = a.ws;
  // slot i holds node i+1 (empty key 0 for invalid slots, which sort last)
  int mine = 0;
  for (int i = tid; i < a.n_pad; i += blockDim.x) {
    uint64_t k = 0ull;
    const int id = i + 1;
    if (id < a.N) {
      const int64_t gi = (int64_t)b * a.N + id;
      if (ws.token[gi] >= 0) {
        k = make_key(ws.value[gi], (uint32_t)id);
        ++mine;
      }
    }
    keys[i] = k;
  }
  __shared__ int s_n;
  if (tid == 0) s_n = 0;
  __syncthreads();
  if (mine) atomicAdd(&s_n, mine);  // one atomic per thread
  __syncthreads();
  const int n = s_n;
  block_bitonic_desc(keys, a.n_pad);
  if (a.mode == 0) {
    int mb = a.m ? a.m[a.m_len == 1 ? 0 : b] : a.m_cap;
    mb = max(0, min(min(mb, a.m_cap), n));
    // selected ids, ascending: rank each of the first mb ids among themselves
    int32_t* out = a.selected + (int64_t)b * a.m_cap;
    for (int i = tid; i < mb; i += blockDim.x) {
      const uint32_t id = key_id(keys[i]);
      int rank = 0;
      for (int j = 0; j < mb; ++j) rank += key_id(keys[j]) < id;
      out[rank] = (int32_t)id;
    }
    for (int i = mb + tid; i < a.m_cap; i += blockDim.x) out[i] = -1;
  } else {
    double* lin = ws.sorted_lin + (int64_t)b * a.m_cap;
    for (int i = tid; i < a.m_cap; i += blockDim.x)
      lin[i] = i < n ? (double)expf(key_value(keys[i])) : 0.0;
    if (tid == 0) ws.sorted_cnt[b] = min(n, a.m_cap);
  }
}

__device__ __forceinline__ int table_row(double c, double L, int M_rows) {
  const double q = floor(c / L);
  return q >= (double)(M_rows - 1) ? M_rows - 1 : (int)q;
}

// Marginal-utility selection over k = 1..cap (thread-serial; cap <= 512).
__device__ int selection_rule(const double* items, const double* cost, double thr, int cap) {
  // du = items[k0] + ... + items[k-1], accumulated in that order as k advances
  int k0 = 1;
  double du = 0.0;
  for (int k = 2; k <= cap; ++k) {
    du += items[k - 1];
    // marginal utility du / (c_k - c_k0) >= thr, written without the division (c_k > c_k0 here)
    if (cost[k] <= cost[k0] || du >= thr * (cost[k] - cost[k0])) {
      k0 = k;
      du = 0.0;
    }
  }
  return k0;
}

struct PruneArgs {
  Workspace ws;
  dt_prune_params p;
  dt_prune_out out;
  int B, N, LW, D, d, policy;
};

// Batch-averaged utility items[s] = (1/B) sum_b v_b(s), s < cap, with v_b(s) given by `vb`.
// One warp per item; lanes take requests b = lane, lane + 32, ... and reduce in a fixed order, so
// the result is deterministic.
template <typename F>
__device__ __forceinline__ void batch_items(double* items, int cap, int B, F vb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int s = warp; s < cap; s += nw) {
    double acc = 0.0;
    for (int b = lane; b < B; b += 32) acc += vb(b, s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) items[s] = acc / (double)B;
  }
}

// CAST width + depth after layer d (1 CTA).
__global__ void cast_width_depth_kernel(PruneArgs a) {
  __shared__ double items[kMaxW * kMaxK + 1];
  __shared__ double cost[kMaxW * kMaxK + 2];
  __shared__ int maxcand;
  const Workspace& ws = a.ws;
  const int tid = threadIdx.x;
  if (tid == 0) maxcand = 0;
  __syncthreads();
  for (int b = tid; b < a.B; b += blockDim.x) atomicMax(&maxcand, ws.layer_count[(int64_t)b * (a.D + 1) + a.d]);
  __syncthreads();
  const int cap = min(a.p.width_cap, maxcand);
  CastState* cs = ws.cast;
  // normalised draft cost of k frontier nodes at the current context: c_k = S_D[row][k-1] / S_T[row][0]
  const int row = table_row((double)(a.p.n0 + cs->ctx_sum), a.p.L, a.p.M_rows);
  const double t1 = a.p.S_T[(int64_t)row * a.p.N_cols];
  for (int k = 1 + tid; k <= cap; k += blockDim.x) cost[k] = a.p.S_D[(int64_t)row * a.p.N_cols + (k - 1)] / t1;
  // items[s] = (1/B) sum_b exp(value of the s-th node of b's layer), missing nodes count 0
  batch_items(items, cap, a.B, [&](int b, int s) {
    const int64_t lb = (int64_t)b * (a.D + 1) + a.d;
    if (s >= ws.layer_count[lb]) return 0.0;
    const int id = ws.layer_order[lb * a.LW + s];
    return (double)expf(ws.value[(int64_t)b * a.N + id]);
  });
  __syncthreads();
  if (tid != 0) return;
  if (cap <= 0) {
    a.out.width[0] = 0;
    for (int b = 0; b < a.B; ++b) a.out.stop[b] = 1;
    return;
  }
  const int n = selection_rule(items, cost, a.p.C1, cap);
  double u = 0.0;
  for (int s = 0; s < n; ++s) u += items[s];
  if (cs->u_prev >= 0.0) {
    int len = cs->fifo_len;
    if (len < a.p.R) {
      cs->fifo[len++] = u / cs->u_prev;
    } else {
      for (int j = 1; j < len; ++j) cs->fifo[j - 1] = cs->fifo[j];
      cs->fifo[len - 1] = u / cs->u_prev;
    }
    cs->fifo_len = len;
  }
  double alpha = 0.0;
  for (int j = 0; j < cs->fifo_len; ++j) alpha += cs->fifo[j];
  alpha /= (double)cs->fifo_len;
  const bool grow = (a.d < a.p.D_max) && (alpha * u >= a.p.C2 * cost[n]);  // alpha * u / c_n >= C2
  cs->u_prev = u;
  cs->u_layer = u;
  cs->ctx_sum += n;
  a.out.width[0] = n;
  for (int b = 0; b < a.B; ++b) a.out.stop[b] = grow ? 0 : 1;
}

// CAST verify count from the per-request sorted linear values (1 CTA).
__global__ void cast_verify_kernel(PruneArgs a) {
  __shared__ double items[kMaxP + 1];
  __shared__ double cost[kMaxP + 2];
  __shared__ int maxn;
  const Workspace& ws = a.ws;
  const int tid = threadIdx.x;
  if (tid == 0) maxn = 0;
  __syncthreads();
  for (int b = tid; b < a.B; b += blockDim.x) atomicMax(&maxn, ws.sorted_cnt[b]);
  __syncthreads();
  const int cap = min(a.p.m_cap, maxn);
  const double* lin = ws.sorted_lin;
  const int row = table_row((double)a.p.n0, a.p.L, a.p.M_rows);
  const double t1 = a.p.S_T[(int64_t)row * a.p.N_cols];
  for (int k = 1 + tid; k <= cap; k += blockDim.x) cost[k] = a.p.S_T[(int64_t)row * a.p.N_cols + (k - 1)] / t1;
  batch_items(items, cap, a.B, [&](int b, int s) { return lin[(int64_t)b * a.p.m_cap + s]; });
  __syncthreads();
  if (tid != 0) return;
  a.out.m[0] = cap <= 0 ? 0 : selection_rule(items, cost, a.p.C3, cap);
}

// Graft checkpoint after layer d: one thread per request.
__global__ void graft_checkpoint_kernel(PruneArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  if (a.out.stop[b]) return;
  const Workspace& ws = a.ws;
  const int li = a.d - 1;
  for (int s = 0; s < a.p.n_ckpt; ++s) {
    if (a.p.ckpt_layer[s] != li) continue;
    const int64_t lb = (int64_t)b * (a.D + 1) + a.d;
    double c = 0.0;
    if (ws.layer_count[lb] > 0) c = (double)expf(ws.value[(int64_t)b * a.N + ws.layer_order[lb * a.LW]]);
    if (!(c > a.p.tau[s])) {
      a.out.stop[b] = 1;
      if (a.out.stage) a.out.stage[b] = s;
      if (a.out.m) a.out.m[b] = a.p.k_draft[s];
      return;
    }
  }
  if (a.d >= a.p.D_max) {
    a.out.stop[b] = 1;
    if (a.out.stage) a.out.stage[b] = a.p.n_ckpt;
    if (a.out.m) a.out.m[b] = a.p.K_total;
  }
}

int next_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace

cudaError_t init_select_attributes() {
  // largest node count: 1 + 32 + 15 * 1024 slots -> 16384 keys of 8 bytes
  return cudaFuncSetAttribute(sort_nodes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 8);
}

static cudaError_t launch_sort(dt_handle* h, int mode, const int32_t* m, int m_len, int m_cap, int32_t* selected,
                               cudaStream_t s) {
  SortArgs a;
  a.ws = h->ws;
  a.N = h->N;
  a.depth = h->depth;
  a.n_pad = next_pow2(std::max(2, h->N - 1));
  a.mode = mode;
  a.m = m;
  a.m_len = m_len;
  a.m_cap = m_cap;
  a.selected = selected;
  const size_t smem = (size_t)a.n_pad * sizeof(uint64_t);
  const int threads = std::min(1024, std::max(32, a.n_pad / 2));
  sort_nodes_kernel<<<h->B, threads, smem, s>>>(a);
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
  if (policy == DT_POLICY_CAST_WIDTH_DEPTH) {
    cast_width_depth_kernel<<<1, 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  if (policy == DT_POLICY_CAST_VERIFY) {
    cudaError_t e = launch_sort(h, 1, nullptr, 1, p->m_cap, nullptr, s);
    if (e != cudaSuccess) return e;
    cast_verify_kernel<<<1, 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  graft_checkpoint_kernel<<<(h->B + 127) / 128, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dt
