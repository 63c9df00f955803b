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
  const int64_t lo_total = (int64_t)B * (D + 1) * LW;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < lo_total;
       i += (int64_t)gridDim.x * blockDim.x)
    ws.layer_order[i] = -1;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)B * (D + 1);
       i += (int64_t)gridDim.x * blockDim.x)
    ws.layer_count[i] = (i % (D + 1)) == 0 ? 1 : 0;
  const int W = LW / K;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)B * W;
       i += (int64_t)gridDim.x * blockDim.x)
    ws.frontier[i] = (i % W) == 0 ? 0 : -1;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < B; i += (int64_t)gridDim.x * blockDim.x)
    ws.frontier_count[i] = 1;
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
  const int warps = blockDim.x >> 5;
  const int b = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  int w = width ? width[width_len == 1 ? 0 : b] : W;
  if (stop && stop[b]) w = 0;
  const int avail = ws.layer_count[(int64_t)b * (D + 1) + d];
  w = max(0, min(min(w, W), avail));
  int id = -1;
  if (lane < w) id = ws.layer_order[((int64_t)b * (D + 1) + d) * LW + lane];
  // slot = rank of my id among the chosen ids
  int slot = 0;
  for (int j = 0; j < w; ++j) {
    const int o = __shfl_sync(0xFFFFFFFFu, id, j);
    slot += (o < id);
  }
  if (lane < W) {
    ws.frontier[(int64_t)b * W + lane] = -1;
    if (ftok) ftok[(int64_t)b * W + lane] = -1;
  }
  __syncwarp();
  if (lane < w) {
    ws.frontier[(int64_t)b * W + slot] = id;
    if (ftok) ftok[(int64_t)b * W + slot] = ws.token[(int64_t)b * N + id];
  }
  if (lane == 0) ws.frontier_count[b] = w;
}

struct ExpandArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int F, S, B, N, K, W, LW, D, d, V;
  int64_t seg_len;
  int32_t base;  // first id of layer d
  uint32_t first_wait_cap;
};

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 3) expand_kernel(ExpandArgs a) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ ScanSmem sm;
  const int r = blockIdx.x / a.S;
  const int seg = blockIdx.x % a.S;
  const int b = r / a.F, f = r % a.F;
  const int tid = threadIdx.x;
  Workspace& ws = a.ws;
  const int fc = ws.frontier_count[b];
  const int active = min(fc, a.F);
  if (f >= active) {  // no node in this slot: the row is not read
    if (f == 0 && seg == 0 && tid == 0 && fc > a.F) set_status(ws.status, DT_DEV_BAD_TREE);
    return;
  }

  const T* row = reinterpret_cast<const T*>(a.logits) + (int64_t)r * a.ld;
  const int64_t s0 = (int64_t)seg * a.seg_len;
  const int64_t s1 = min((int64_t)a.V, s0 + a.seg_len);
  SegOut so = scan_segment<T, true>(row, s0, s1, a.K, sm, dyn_smem, a.first_wait_cap);

  Partial* part = ws.partials + (int64_t)r * a.S;
  for (int i = tid; i < a.K; i += blockDim.x) part[seg].keys[i] = i < so.nkeys ? sm.cand[i] : 0ull;
  if (tid == 0) {
    part[seg].m = so.m;
    part[seg].s = so.s;
    if (so.timed_out) set_status(ws.status, DT_DEV_TIMEOUT);
    if (so.internal) set_status(ws.status, DT_DEV_INTERNAL);
    __threadfence();
    const int prev = atomicAdd(&ws.row_counter[r], 1);
    sm.last = (prev == a.S - 1);
  }
  __syncthreads();
  if (!sm.last) return;

  // ---- last segment of the row: merge the partials and write the K children ----
  __threadfence();
  if (tid == 0) ws.row_counter[r] = 0;
  const int nk = a.S * a.K;
  for (int i = tid; i < nk; i += blockDim.x) {
    const uint64_t k = __ldcg(&part[i / a.K].keys[i % a.K]);
    sm.cand[i] = k;
  }
  if (tid < kMaxK) sm.topk[tid] = 0ull;
  __syncthreads();
  // empty keys are 0 and rank below every real key
  merge_sorted_lists(sm, a.S, a.K);
  float M;
  double Ssum;
  bool nan;
  merge_softmax(part, a.S, sm, M, Ssum, nan);
  if (tid == 0 && (nan || !(M > -INFINITY) || M == INFINITY || !(Ssum > 0.0)))
    set_status(ws.status, DT_DEV_BAD_LOGITS);
  const int pid = ws.frontier[(int64_t)b * a.W + f];
  const float pval = ws.value[(int64_t)b * a.N + pid];
  // log S = e * ln 2 + log(mantissa), mantissa in [1, 2): the exponent split is exact and the fp32
  // log of the mantissa is accurate to ~1e-7 absolute (no fp64 transcendental on the tail)
  double logS;
  {
    const unsigned long long bits = (unsigned long long)__double_as_longlong(Ssum);
    const int e = (int)((bits >> 52) & 0x7FF) - 1023;
    const double mant = __longlong_as_double((long long)((bits & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull));
    logS = (double)e * 0.6931471805599453 + (double)logf((float)mant);
    if (!(Ssum > 0.0) || Ssum != Ssum || e == 1024) logS = log(Ssum);  // zero, NaN, inf: let log decide
  }
  if (tid < a.K) {
    const uint64_t k = sm.topk[tid];
    const int id = a.base + f * a.K + tid;
    const int64_t gi = (int64_t)b * a.N + id;
    const float x = key_value(k);
    const double lc = ((double)x - (double)M) - logS;
    ws.token[gi] = (int32_t)key_id(k);
    ws.parent[gi] = pid;
    ws.logc[gi] = (float)lc;
    ws.value[gi] = (float)((double)pval + lc);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&ws.req_counter[b], 1);
    sm.last = (prev == active - 1);
  }
  __syncthreads();
  if (!sm.last) return;

  // ---- last row of the request: order the new layer by (value desc, id asc) ----
  __threadfence();
  if (tid == 0) ws.req_counter[b] = 0;
  const int n = active * a.K;
  int32_t* order = ws.layer_order + ((int64_t)b * (a.D + 1) + a.d) * a.LW;
  // keys staged in the candidate buffer (n <= W*K <= 1024 = kCandCap)
  for (int i = tid; i < n; i += blockDim.x) {
    const int id = a.base + i;
    sm.cand[i] = make_key(__ldcg(&ws.value[(int64_t)b * a.N + id]), (uint32_t)id);
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const uint64_t k = sm.cand[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += (sm.cand[j] > k);
    order[rank] = (int32_t)key_id(k);
  }
  if (tid == 0) ws.layer_count[(int64_t)b * (a.D + 1) + a.d] = n;
}

}  // namespace

int choose_segments(const dt_handle* h, int64_t rows, int64_t V, int elt_bytes) {
  // Enough CTAs for one full wave (3 resident per SM) with segments as long as possible, so that
  // every warp streams through its ring for many stages; at least ~8 KB of work per CTA.
  const int64_t row_bytes = V * elt_bytes;
  int64_t S = ((int64_t)h->num_sms * 3 + rows - 1) / rows;
  const int64_t max_by_len = (row_bytes + 8191) / 8192;
  if (S > max_by_len) S = max_by_len;
  const int64_t max_by_keys = kCandCap / h->cfg.K;
  if (S > max_by_keys) S = max_by_keys;
  if (S > 64) S = 64;
  const int64_t max_by_buf = h->ws.partial_cap / (rows > 0 ? rows : 1);  // partials buffer capacity
  if (S > max_by_buf) S = max_by_buf;
  if (S < 1) S = 1;
  return (int)S;
}

static int64_t seg_len_for(int64_t V, int S) {
  int64_t L = (V + S - 1) / S;
  L = (L + 7) / 8 * 8;
  return L;
}

static size_t row_smem_bytes() { return (size_t)kScanSmemBytes; }

cudaError_t init_tree_attributes() {
  const int smem = (int)row_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(expand_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expand_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t launch_tree_reset(dt_handle* h, const int32_t* root, cudaStream_t s) {
  const int64_t total = (int64_t)h->B * h->N;
  int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)h->num_sms * 4);
  if (blocks < 1) blocks = 1;
  tree_reset_kernel<<<blocks, 256, 0, s>>>(h->ws, root, h->B, h->N, h->cfg.K, h->LW, h->cfg.D_max, h->cfg.V);
  return cudaGetLastError();
}

cudaError_t launch_select_frontier(dt_handle* h, const int32_t* width, int width_len, const int32_t* stop,
                                   int32_t* frontier_token, cudaStream_t s) {
  const int warps = 8;
  const int blocks = (h->B + warps - 1) / warps;
  select_frontier_kernel<<<blocks, warps * 32, 0, s>>>(h->ws, h->B, h->N, h->cfg.K, h->cfg.W, h->LW,
                                                        h->cfg.D_max, h->depth, width, width_len, stop,
                                                        frontier_token);
  return cudaGetLastError();
}

cudaError_t launch_expand(dt_handle* h, const void* logits, int64_t ld, int F, cudaStream_t s) {
  const int d = h->depth + 1;
  const int esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  const int64_t rows = (int64_t)h->B * F;
  const int S = choose_segments(h, rows, h->cfg.V, esz);
  ExpandArgs a;
  a.ws = h->ws;
  a.logits = logits;
  a.ld = ld;
  a.F = F;
  a.S = S;
  a.B = h->B;
  a.N = h->N;
  a.K = h->cfg.K;
  a.W = h->cfg.W;
  a.LW = h->LW;
  a.D = h->cfg.D_max;
  a.d = d;
  a.V = h->cfg.V;
  a.seg_len = seg_len_for(h->cfg.V, S);
  a.base = d == 1 ? 1 : 1 + h->cfg.K + (d - 2) * h->LW;
  a.first_wait_cap = (h->cfg.flags & DT_FLAG_TEST_TIMEOUT) ? 0u : kSpinCap;
  const unsigned grid = (unsigned)(rows * S);
  const size_t smem = row_smem_bytes();
  if (h->cfg.dtype == DT_BF16)
    expand_kernel<uint16_t><<<grid, kRowThreads, smem, s>>>(a);
  else
    expand_kernel<float><<<grid, kRowThreads, smem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) h->depth = d;
  return e;
}

}  // namespace dt
