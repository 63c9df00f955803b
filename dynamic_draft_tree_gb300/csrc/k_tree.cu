// Tree construction kernels: reset, frontier selection, layer expansion.
//
// EAGLE-2 page, §"置信度为什么可以近似接受率" (c = draft probability of the token),
// §"value 公式" (value = product of confidences on the path, kept as a sum of logs) and
// §"扩展阶段" (expand the top-k nodes of the newest layer; every expanded node adds its
// top-K vocabulary children; value(child) = value(parent) * c).
#include <algorithm>

#include <cstring>

#include "cast_block.cuh"
#include "rowstream.cuh"

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

struct StreamArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int F, B, K, V, maxp;
  int64_t Gtot;   // warps of the grid
  int test_timeout;
};

// Streaming pass of an expansion: request b's frontier slots f < min(frontier_count[b], F) are its
// rows; every warp leaves the softmax statistics and top-K keys of the row pieces it reads.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm) expand_stream_kernel(StreamArgs a) {
  pdl_begin();
  __shared__ WarpRing rings[kStreamWarps];
  WarpRing& rg = rings[threadIdx.x >> 5];
  Workspace& ws = a.ws;
  const int lane = threadIdx.x & 31;
  auto cnt = [&](int b) -> int { return min(max(ws.frontier_count[b], 0), a.F); };
  auto row_of = [&](int b, int f) -> const T* {
    return reinterpret_cast<const T*>(a.logits) + ((int64_t)b * a.F + f) * a.ld;
  };
  if (blockIdx.x == 0 && threadIdx.x < 32)  // a frontier wider than the launch's F is a caller error
    for (int b = lane; b < a.B; b += 32)
      if (ws.frontier_count[b] > a.F) set_status(ws.status, DT_DEV_BAD_TREE);
  if (a.test_timeout) {  // test only: as if every read had given up (empty pieces)
    auto skip = [&](int b, int f) -> const T* { return nullptr; };
    stream_rows<T, true>(a.B, a.V, a.K, a.maxp, a.Gtot, rg, nullptr, cnt, skip,
                         [&](int64_t, int64_t, int, int, const PieceOut&) {});
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(ws.status, DT_DEV_TIMEOUT);
    return;
  }
  stream_rows<T, true>(a.B, a.V, a.K, a.maxp, a.Gtot, rg, ws.row_tau, cnt, row_of,
                       [&](int64_t j, int64_t g, int b, int f, const PieceOut& o) {
                         publish_partial(ws.partials + j + g, rg, o, a.K);
                         if (lane == 0 && o.internal) set_status(ws.status, DT_DEV_INTERNAL);
                       });
}

constexpr int kFinishWarps = 16;
constexpr int kFinishThreads = 32 * kFinishWarps;
constexpr int kFinishNodes = 4096;  // new-layer nodes of the requests of one finishing CTA
enum { kFinishPlain = 0, kFinishEagle = 1, kFinishCast = 2, kFinishGraft = 3 };

struct FinishArgs {
  Workspace ws;
  int F, B, N, K, W, LW, D, d, V, maxp, esz, vecel;
  int64_t Gtot;                 // warps of the streaming launch
  int32_t base;                 // first id of layer d
  int rpc;                      // requests per CTA
  int mode;                     // kFinish*
  int select;                   // choose the next layer's frontier (never after D_max)
  const int32_t* width;         // EAGLE / Graft frontier width, device [width_len] or null (W)
  int width_len;
  int32_t* ftok;                // frontier tokens [B][W] or null
  PruneArgs pa;                 // CAST / Graft parameters and outputs
};

__host__ __device__ __forceinline__ size_t finish_smem_bytes(int maxp, int K, int rpc, int LW) {
  return (size_t)kFinishWarps * maxp * K * 8 + (size_t)kFinishWarps * kMaxK * 8 + (size_t)rpc * LW * 12;
}

// Finishing pass of an expansion (requests [c * rpc, c * rpc + rpc) per CTA): each warp merges the
// pieces of a row into its softmax statistics and top-K (the children of frontier slot f: log c =
// x - m - log S and value = value(parent) + log c), then the new layer of every request is ordered by
// (value desc, id asc) and, by mode, the next frontier is chosen (EAGLE), the Graft checkpoint is
// tested first, or CAST's width and depth pruning runs on the whole batch (one CTA).
__global__ void __launch_bounds__(kFinishThreads) expand_finish_kernel(FinishArgs a) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t fsm[];
  uint64_t* mbuf = reinterpret_cast<uint64_t*>(fsm);                // [warp][maxp * K] merge scratch
  uint64_t* mtop = mbuf + (size_t)kFinishWarps * a.maxp * a.K;      // [warp][kMaxK] merged row
  uint64_t* nkey = mtop + (size_t)kFinishWarps * kMaxK;             // [rpc][LW] new nodes' keys
  int32_t* ntok = reinterpret_cast<int32_t*>(nkey + (size_t)a.rpc * a.LW);  // [rpc][LW] their tokens
  __shared__ int s_cnt[33], s_pre[34], s_valid[33];
  __shared__ int64_t s_base0, s_A;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Workspace& ws = a.ws;
  const int b_lo = blockIdx.x * a.rpc, b_hi = min(a.B, b_lo + a.rpc), nreq = b_hi - b_lo;
  auto cnt = [&](int b) -> int { return min(max(ws.frontier_count[b], 0), a.F); };
  if (warp == 0) {
    const int64_t A = warp_total_rows(a.B, cnt);
    const int64_t base0 = warp_rows_before(b_lo, cnt);
    const int c = lane < nreq ? cnt(b_lo + lane) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    s_cnt[lane] = c;
    s_pre[lane + 1] = incl;
    s_valid[lane] = 0;
    if (lane == 0) {
      s_pre[0] = 0;
      s_A = A;
      s_base0 = base0;
    }
  }
  __syncthreads();
  const int64_t A = s_A;
  const int64_t G = stream_warps(A, a.V, a.esz, a.Gtot, a.maxp);
  const int nr = s_pre[nreq];
  for (int r = warp; r < nr; r += kFinishWarps) {
    int c = 0;
    while (s_pre[c + 1] <= r) ++c;
    const int f = r - s_pre[c], b = b_lo + c;
    const int64_t j = s_base0 + s_pre[c] + f;
    const int pid = ws.frontier[(int64_t)b * a.W + f];
    const float pval = ws.frontier_val[(int64_t)b * a.W + f];
    const RowPieces rp = row_pieces(j, a.V, A, G, a.vecel);
    uint64_t* top = mtop + (size_t)warp * kMaxK;
    float M, sh, sl;
    if (rp.S > a.maxp) {  // never: the streaming plan bounds the pieces of a row
      if (lane == 0) set_status(ws.status, DT_DEV_INTERNAL);
      if (lane < a.K) top[lane] = 0ull;
      M = -INFINITY;
      sh = sl = 0.0f;
      __syncwarp();
    } else {
      warp_merge_row(ws.partials + rp.slot0, rp.S, a.K, mbuf + (size_t)warp * a.maxp * a.K, top, true, M, sh, sl);
    }
    if (lane == 0) {
      ws.row_tau[j] = 0ull;  // every piece of the row has finished with it
      if (sh != sh || !(M > -INFINITY) || M == INFINITY || !(sh > 0.0f) || sh == INFINITY)
        set_status(ws.status, DT_DEV_BAD_LOGITS);
    }
    if (lane < a.K) {
      // log S as a double-float: S = mant * 2^e with mant in [1, 2) (exact scaling), log S =
      // e * ln2 (Cody-Waite split: e * LN2_HI is exact for |e| < 2^9) + log(mant_hi) + mant_lo / mant_hi
      constexpr float LN2_HI = 0.693145751953125f, LN2_LO = 1.4286068203094173e-06f;
      float lh, ll;
      if (sh > 0.0f && sh < INFINITY) {
        const int e = (int)((__float_as_uint(sh) >> 23) & 0xFF) - 127;
        const float scale = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
        const float mh = __fmul_rn(sh, scale), ml = __fmul_rn(sl, scale);
        const float lm = __fadd_rn(logf(mh), __fdiv_rn(ml, mh));
        two_sum(__fmul_rn((float)e, LN2_HI), fmaf((float)e, LN2_LO, lm), lh, ll);
      } else {
        lh = logf(sh);
        ll = 0.0f;
      }
      const uint64_t k = top[lane];
      const int id = a.base + f * a.K + lane;
      const int64_t gi = (int64_t)b * a.N + id;
      const int slot = c * a.LW + f * a.K + lane;
      if (k == 0ull) {  // the row has fewer than K finite logits: no child in this slot
        ws.token[gi] = -1;
        ws.parent[gi] = -1;
        ws.logc[gi] = -INFINITY;
        ws.value[gi] = -INFINITY;
        nkey[slot] = 0ull;
        ntok[slot] = -1;
      } else {
        const float x = key_value(k);
        // log c = (x - M) - log S and value = value(parent) + log c, each kept as a double-float
        // until the final rounding
        float dh, dl;
        two_sum(x, -M, dh, dl);
        ff_add(dh, dl, -lh, -ll);
        const float lc = __fadd_rn(dh, dl);
        float vh = pval, vl = 0.0f;
        ff_add(vh, vl, dh, dl);
        const float v = __fadd_rn(vh, vl);
        const int32_t tok = (int32_t)key_id(k);
        ws.token[gi] = tok;
        ws.parent[gi] = pid;
        ws.logc[gi] = lc;
        ws.value[gi] = v;
        nkey[slot] = make_key(v, (uint32_t)id);
        ntok[slot] = tok;
        atomicAdd(&s_valid[c], 1);
      }
    }
    __syncwarp();
  }
  __syncthreads();
  // the new layer of every request in (value desc, id asc) order; slots without a child sort last
  const int ntot = s_pre[nreq] * a.K;
  for (int t = tid; t < ntot; t += blockDim.x) {
    int c = 0;
    while (s_pre[c + 1] * a.K <= t) ++c;
    const int p = t - s_pre[c] * a.K;
    const int n = s_cnt[c] * a.K;
    const uint64_t* ks = nkey + (size_t)c * a.LW;
    const uint64_t k = ks[p];
    if (k == 0ull) continue;
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += ks[q] > k;
    const int b = b_lo + c;
    const int64_t lo = ((int64_t)b * (a.D + 1) + a.d) * a.LW;
    ws.layer_order[lo + rank] = (int32_t)key_id(k);
    ws.layer_val[lo + rank] = key_value(k);
    ws.layer_tok[lo + rank] = ntok[(size_t)c * a.LW + p];
  }
  if (tid < nreq) ws.layer_count[(int64_t)(b_lo + tid) * (a.D + 1) + a.d] = s_valid[tid];
  if (a.mode == kFinishPlain) return;
  __syncthreads();  // the new layer is complete (global writes of this CTA are visible to it)
  if (a.mode == kFinishCast) {
    cast_width_depth_block(a.pa);
    return;
  }
  for (int b = b_lo + warp; b < b_hi; b += kFinishWarps) {
    int w = a.width ? a.width[a.width_len == 1 ? 0 : b] : a.W;
    if (a.mode == kFinishGraft) {
      if (lane == 0) graft_checkpoint_one(a.pa, b);
      __syncwarp();
      if (a.pa.out.stop[b]) w = 0;
    }
    if (a.select) select_frontier_warp(ws, b, a.N, a.W, a.LW, a.D, a.d, w, a.ftok);
  }
}

}  // namespace

int stream_grid(const dt_handle* h) { return std::max(1, h->num_sms * kStreamCtasPerSm); }

static size_t finish_smem_max() { return finish_smem_bytes(kMaxPieces, 512 / kMaxPieces, kFinishNodes, 1); }

cudaError_t init_tree_attributes() {
  const int smem = (int)finish_smem_max();
  cudaError_t e = cudaFuncSetAttribute(expand_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // all of the unified L1 as cache for the streaming passes (they use a few KB of shared memory)
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expand_stream_kernel<uint16_t>, cudaFuncAttributePreferredSharedMemoryCarveout, 10);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expand_stream_kernel<float>, cudaFuncAttributePreferredSharedMemoryCarveout, 10);
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

// Whether the fused CAST pruning fits the finishing kernel: the whole batch in one CTA.
bool expand_fuses_cast(const dt_handle* h) {
  return h->B <= 32 && (int64_t)h->B * h->LW <= kFinishNodes;
}

cudaError_t launch_expand_rows(dt_handle* h, const void* logits, int64_t ld, int F, cudaStream_t s) {
  StreamArgs sa;
  sa.ws = h->ws;
  sa.logits = logits;
  sa.ld = ld;
  sa.F = F;
  sa.B = h->B;
  sa.K = h->cfg.K;
  sa.V = h->cfg.V;
  sa.maxp = stream_max_pieces(h->cfg.K);
  const unsigned grid = (unsigned)stream_grid(h);
  sa.Gtot = (int64_t)grid * kStreamWarps;
  sa.test_timeout = (h->cfg.flags & DT_FLAG_TEST_TIMEOUT) ? 1 : 0;
  if (h->cfg.dtype == DT_BF16)
    launch_k(expand_stream_kernel<uint16_t>, dim3(grid), dim3(kStreamThreads), 0, s, sa);
  else
    launch_k(expand_stream_kernel<float>, dim3(grid), dim3(kStreamThreads), 0, s, sa);
  return cudaGetLastError();
}

cudaError_t launch_expand_finish(dt_handle* h, int F, int policy, const dt_prune_params* p,
                                 const dt_prune_out* out, const int32_t* width, int width_len,
                                 int32_t* frontier_token, cudaStream_t s) {
  const int d = h->depth + 1;
  const int K = h->cfg.K;
  const int esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  FinishArgs fa;
  fa.ws = h->ws;
  fa.F = F;
  fa.B = h->B;
  fa.N = h->N;
  fa.K = K;
  fa.W = h->cfg.W;
  fa.LW = h->LW;
  fa.D = h->cfg.D_max;
  fa.d = d;
  fa.V = h->cfg.V;
  fa.maxp = stream_max_pieces(K);
  fa.esz = esz;
  fa.vecel = 16 / esz;
  fa.Gtot = (int64_t)stream_grid(h) * kStreamWarps;
  fa.base = d == 1 ? 1 : 1 + K + (d - 2) * h->LW;
  fa.select = d < h->cfg.D_max ? 1 : 0;
  fa.width = width;
  fa.width_len = width_len;
  fa.ftok = frontier_token;
  PruneArgs& pa = fa.pa;
  memset(&pa, 0, sizeof(pa));
  pa.ws = h->ws;
  if (p) pa.p = *p;
  if (out) pa.out = *out;
  pa.B = h->B;
  pa.N = h->N;
  pa.LW = h->LW;
  pa.D = h->cfg.D_max;
  pa.d = d;
  pa.policy = policy;
  pa.W = h->cfg.W;
  pa.select = fa.select;
  pa.ftok = frontier_token;
  pa.sel = nullptr;
  int mode = kFinishPlain;
  bool cast_after = false;
  if (policy == DT_POLICY_NONE) mode = kFinishEagle;
  else if (policy == DT_POLICY_GRAFT_CHECKPOINT) mode = kFinishGraft;
  else if (policy == DT_POLICY_CAST_WIDTH_DEPTH) {
    if (expand_fuses_cast(h)) mode = kFinishCast;
    else cast_after = true;
  }
  fa.mode = mode;
  fa.rpc = mode == kFinishCast ? h->B : std::max(1, std::min(std::min(h->B, 32), kFinishNodes / h->LW));
  const int fgrid = (h->B + fa.rpc - 1) / fa.rpc;
  const size_t smem = finish_smem_bytes(fa.maxp, K, fa.rpc, h->LW);
  launch_k(expand_finish_kernel, dim3(fgrid), dim3(kFinishThreads), smem, s, fa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  h->depth = d;
  if (cast_after) {  // the batch does not fit one finishing CTA: the pruning kernel follows
    e = launch_cast_prune(h, DT_POLICY_CAST_WIDTH_DEPTH, p, out, s);
    if (e != cudaSuccess || !fa.select) return e;
    return launch_select_frontier(h, out->width, 1, out->stop, frontier_token, s);
  }
  return cudaSuccess;
}

cudaError_t launch_expand_ex(dt_handle* h, const void* logits, int64_t ld, int F, int policy,
                             const dt_prune_params* p, const dt_prune_out* out, const int32_t* width,
                             int width_len, int32_t* frontier_token, cudaStream_t s) {
  cudaError_t e = launch_expand_rows(h, logits, ld, F, s);
  if (e != cudaSuccess) return e;
  return launch_expand_finish(h, F, policy, p, out, width, width_len, frontier_token, s);
}

cudaError_t launch_expand(dt_handle* h, const void* logits, int64_t ld, int F, cudaStream_t s) {
  return launch_expand_ex(h, logits, ld, F, DT_EXPAND_ONLY, nullptr, nullptr, nullptr, 0, nullptr, s);
}

}  // namespace dt
