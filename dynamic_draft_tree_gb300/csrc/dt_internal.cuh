// Internal declarations shared by the libdt translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dt.h"

namespace dt {

constexpr int kMaxK = 32;
constexpr int kMaxW = 32;
constexpr int kMaxD = 16;
constexpr int kMaxP = 512;
constexpr int kMaxFifo = 16;
constexpr int kScanWarps = 4;        // warps of a row-scan CTA
constexpr int kRowThreads = 32 * kScanWarps;
constexpr int kStageBytes = 4096;   // one TMA bulk copy into a warp's ring
constexpr int kWarpStages = 3;      // ring depth per warp
constexpr int kWarpCand = 128;      // per-warp candidate buffer
constexpr int kCandCap = 1024;      // CTA merge / sort buffer (keys)
constexpr int kScanSmemBytes = kScanWarps * kWarpStages * kStageBytes;  // dynamic shared memory
static_assert(kCandCap * (8 + 4) <= kScanSmemBytes, "layer sort keys + tokens must fit the stage memory");
constexpr int kStaticRows = 1024;      // rows per call of the static-scratch row top-K
constexpr int kStaticPartials = 4096;  // row segments per call of the static-scratch row top-K

// Per-(row, segment) partial result of a row scan.
struct Partial {
  float m;           // segment max (or -inf)
  float s_hi, s_lo;  // sum exp(x - m) over the segment as an unevaluated sum of two floats
  int32_t pad;
  uint64_t keys[kMaxK];  // segment top-K keys, descending; 0 = empty
};

// Per-row statistics left by the verify row pass.
struct RowStat {
  float m;       // row max
  int32_t amax;  // argmax token (lowest id among maxima)
  double s;      // sum exp(x - m)
};

// CAST running state of the tree in flight.
struct CastState {
  double fifo[kMaxFifo];
  int32_t fifo_len;
  int32_t pad;
  double u_prev;
  int64_t ctx_sum;
  double u_layer;     // u_{n_d} of the newest pruned layer
};

// Sampled walk result handed to the bonus kernel.
struct WalkState {
  int64_t row;        // its row of the target logits (padded or packed layout)
  int32_t cur;        // position whose residual is sampled
  int32_t n_rej;      // rejected tokens at that position
  int32_t rej[kMaxP];
};

struct Workspace {
  // tree
  int32_t* token;
  int32_t* parent;
  int32_t* node_depth;
  float* logc;
  float* value;
  float2* node_dd;       // [B_max][N] log c of a block layer's child as a double-float (block expansion)
  int32_t* exp_slot;     // [B_max][N] sampled drafts: frontier slot of each expanded node's row
  float4* exp_stat;      // [B_max][N] sampled drafts: (max, sum hi, sum lo) of that row's softmax
  int32_t* layer_order;
  float* layer_val;      // [B_max][D_max+1][LW] value of layer_order's node at the same place
  int32_t* layer_tok;    // [B_max][D_max+1][LW] token of layer_order's node at the same place
  int32_t* layer_count;
  int32_t* frontier;
  float* frontier_val;   // [B_max][W] value of each frontier node (read with the frontier)
  int32_t* frontier_count;
  // row scans
  Partial* partials;
  int64_t partial_cap;
  int32_t* row_counter;
  int64_t row_counter_cap;
  unsigned long long* row_tau;  // [row_counter_cap] best K-th key published by a row's pieces (0 = none)
  int32_t* req_counter;
  RowStat* row_stats;
  // selection scratch
  double* sorted_lin;    // [B_max][P_max] linear values of each request's top nodes
  int32_t* sorted_cnt;   // [B_max]
  int32_t* sorted_ids;   // [B_max][P_max] ids of each request's top nodes in rank order
  CastState* cast;
  CastState* cast_req;   // [B_max] per-request CAST state (per_request rule)
  WalkState* walk;
  unsigned long long* bonus_key;  // [B_max]
  int32_t* bonus_counter;         // [B_max]
  int32_t* status;
};

}  // namespace dt

struct dt_handle {
  dt_config cfg;
  int32_t N;       // nodes per request
  int32_t LW;      // slots per layer
  int32_t B;       // batch of the tree in flight
  int32_t depth;   // layers built
  int num_sms;
  dt::Workspace ws;
  void* alloc;     // single device allocation backing the workspace
  size_t alloc_bytes;
};

namespace dt {

// Launches `kernel` on `s` with programmatic stream serialization allowed (see pdl_begin).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- launchers implemented in the kernel translation units (host functions) ----
cudaError_t launch_tree_reset(dt_handle* h, const int32_t* root, cudaStream_t s);
cudaError_t launch_select_frontier(dt_handle* h, const int32_t* width, int width_len, const int32_t* stop,
                                   int32_t* frontier_token, cudaStream_t s);
cudaError_t launch_expand(dt_handle* h, const void* logits, int64_t ld, int F, cudaStream_t s, bool draw = false,
                          uint64_t seed = 0, uint64_t round = 0);
// Expansion followed, by policy, by no pruning (DT_POLICY_NONE), the Graft checkpoint or CAST's width
// and depth pruning, then the next frontier (not after D_max).
cudaError_t launch_expand_ex(dt_handle* h, const void* logits, int64_t ld, int F, int policy,
                             const dt_prune_params* p, const dt_prune_out* out, const int32_t* width,
                             int width_len, int32_t* frontier_token, cudaStream_t s);
// CTAs of a streaming row pass (one wave).
int stream_grid(const dt_handle* h);
cudaError_t launch_cast_prune(dt_handle* h, int policy, const dt_prune_params* p, const dt_prune_out* out,
                              cudaStream_t s);
cudaError_t launch_rerank(dt_handle* h, const int32_t* m, int m_len, int m_cap, int32_t* selected,
                          cudaStream_t s);
cudaError_t launch_cast_verify_rerank(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out,
                                     int32_t* selected, cudaStream_t s);
cudaError_t launch_cast_prune_select(dt_handle* h, const dt_prune_params* p, const dt_prune_out* out,
                                     int32_t* frontier_token, cudaStream_t s);
cudaError_t launch_graft_retrieve(dt_handle* h, const int32_t* M, const dt_template* tpl, int R_cap,
                                  const int32_t* selected, int m_cap, int32_t* ret_token, int32_t* ret_parent,
                                  int32_t* ret_count, int32_t* ret_anchor, cudaStream_t s);
cudaError_t launch_build_meta(dt_handle* h, const int32_t* selected, int m_cap, const int32_t* ret_token,
                              const int32_t* ret_parent, const int32_t* ret_count, const int32_t* ret_anchor,
                              int R_cap, int K_total, const int32_t* pos_offset, const dt_tree_meta* meta,
                              cudaStream_t s);
cudaError_t launch_verify_sampled(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                                  const void* draft, int64_t ld_d, uint64_t seed, uint64_t round,
                                  int32_t* accept_len, int32_t* accept_path, int32_t* bonus, cudaStream_t s);
cudaError_t launch_block_expand(dt_handle* h, const void* logits, int64_t ld, int L, const dt_prune_params* p,
                                const dt_prune_out* out, cudaStream_t s);
cudaError_t launch_verify(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                          uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path,
                          int32_t* bonus, int32_t* top8, cudaStream_t s);
cudaError_t launch_verify_rows(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                               int with_top8, cudaStream_t s);
cudaError_t launch_verify_accept(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld,
                                 int mode, uint64_t seed, uint64_t round, int32_t* accept_len,
                                 int32_t* accept_path, int32_t* bonus, int32_t* top8, cudaStream_t s);
cudaError_t launch_adj_update(dt_handle* h, int32_t* M, const dt_tree_meta* meta, const int32_t* top8,
                              cudaStream_t s);
// Expansion row pass: CTAs per launch (one wave) and the most pieces a row may be cut into when its
// partial lists hold K keys.
int row_pass_grid(const dt_handle* h);
int row_pass_smax(int K);

cudaError_t launch_commit_kv(dt_handle* h, const void* tmp_kv, int64_t tmp_pos_stride, int64_t tmp_req_stride, int P,
                             void* cache, int64_t cache_pos_stride, int64_t cache_req_stride, int L_max,
                             int64_t row_bytes, int32_t* cache_len, const int32_t* accept_len,
                             const int32_t* accept_path, int D_path, const int32_t* tmp_row_off,
                             cudaStream_t s);
cudaError_t launch_row_topk_static(const void* logits, int64_t ld, int rows, int V, int K, int dtype, float* logp,
                                   int32_t* ids, int32_t* status, cudaStream_t s);

// One-time kernel attributes (dynamic shared memory limits), set by dt_create so that no launch
// path calls a non-stream API (launches stay capturable in CUDA graphs).
cudaError_t init_tree_attributes();
cudaError_t init_verify_attributes();
cudaError_t init_select_attributes();
cudaError_t init_meta_attributes();
cudaError_t init_block_attributes();


}  // namespace dt

// ---------------------------------------------------------------- device helpers ----
#ifdef __CUDACC__
namespace dt {

__device__ __forceinline__ uint32_t f2ord(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 orders as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}
// Total-order key: larger key = larger value, then smaller id. 0 is below every real key.
__device__ __forceinline__ uint64_t make_key(float v, uint32_t id) {
  return ((uint64_t)f2ord(v) << 32) | (uint64_t)(~id);
}
__device__ __forceinline__ float key_value(uint64_t k) { return ord2f((uint32_t)(k >> 32)); }
__device__ __forceinline__ uint32_t key_id(uint64_t k) { return ~(uint32_t)k; }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 2^x on the SFU (ex2.approx, flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) { atomicOr(status, bits); }

// Unevaluated sums of two floats (hi + lo, |lo| <= ulp(hi) / 2): exact error-free transformations
// (Knuth's TwoSum, Dekker's FastTwoSum) give about 48 bits of precision with fp32 operations only.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}
// (h, l) += (h2, l2)
__device__ __forceinline__ void ff_add(float& h, float& l, float h2, float l2) {
  float s, e;
  two_sum(h, h2, s, e);
  e = __fadd_rn(e, __fadd_rn(l, l2));
  h = __fadd_rn(s, e);
  l = __fsub_rn(e, __fsub_rn(h, s));
}

// Frontier of the next layer for request b (one warp): the first w nodes of layer d in (value desc,
// id asc) order (layer_order), slotted in ascending id. Lane l < w holds the l-th node (id, token,
// value); select_frontier_write slots and stores them.
__device__ __forceinline__ void select_frontier_write(const Workspace& ws, int b, int W, int w, int id, int tok,
                                                      float val, int32_t* __restrict__ ftok) {
  const int lane = threadIdx.x & 31;
  int slot = 0;  // rank of my id among the chosen ids
  for (int j = 0; j < w; ++j) {
    const int o = __shfl_sync(0xFFFFFFFFu, id, j);
    slot += (o < id);
  }
  if (lane < W) {
    ws.frontier[(int64_t)b * W + lane] = -1;
    ws.frontier_val[(int64_t)b * W + lane] = -INFINITY;
    if (ftok) ftok[(int64_t)b * W + lane] = -1;
  }
  __syncwarp();
  if (lane < w) {
    ws.frontier[(int64_t)b * W + slot] = id;
    ws.frontier_val[(int64_t)b * W + slot] = val;
    if (ftok) ftok[(int64_t)b * W + slot] = tok;
  }
  if (lane == 0) ws.frontier_count[b] = w;
}
// Loads the candidates of request b's frontier (the first min(W, nodes) nodes of layer d) into lanes:
// id, token and value come from the layer's sorted arrays in one round of loads.
__device__ __forceinline__ int frontier_candidates(const Workspace& ws, int b, int N, int W, int LW, int D, int d,
                                                   int& id, int& tok, float& val) {
  const int lane = threadIdx.x & 31;
  const int64_t lb = (int64_t)b * (D + 1) + d;
  const int avail = ws.layer_count[lb];
  id = -1;
  tok = -1;
  val = -INFINITY;
  if (lane < W) {  // read with the count: entries past it are not used
    const int i = ws.layer_order[lb * LW + lane];
    const int t = ws.layer_tok[lb * LW + lane];
    const float v = ws.layer_val[lb * LW + lane];
    if (lane < min(avail, W) && i >= 0) {
      id = i;
      tok = t;
      val = v;
    }
  }
  return avail;
}
__device__ __forceinline__ void select_frontier_warp(const Workspace& ws, int b, int N, int W, int LW, int D, int d,
                                                     int w_req, int32_t* __restrict__ ftok) {
  int id, tok;
  float val;
  const int avail = frontier_candidates(ws, b, N, W, LW, D, d, id, tok, val);
  select_frontier_write(ws, b, W, max(0, min(min(w_req, W), avail)), id, tok, val, ftok);
}

// Programmatic dependent launch. Every kernel of the path starts with pdl_begin(): it waits until the
// previous kernel in the stream has completed and its writes are visible (a no-op when the kernel was
// launched without the attribute), then lets the next kernel's CTAs be scheduled, so that the next
// launch overlaps this kernel instead of following it. Nothing is read or written before the wait.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src);
  uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}

// Descending bitonic sort of one 64-bit key per lane across a warp.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t k) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t o = shfl_xor_u64(k, stride);
      bool up = ((lane & size) == 0);        // this block sorts descending
      bool lower = ((lane & stride) == 0);   // lower index of the pair
      bool take_max = (lower == up);
      k = take_max ? (k > o ? k : o) : (k < o ? k : o);
    }
  }
  return k;
}

// Philox4x32-10 (Salmon et al., SC'11), written from the published round function.
struct Philox4 {
  uint32_t v[4];
};
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  Philox4 out;
  out.v[0] = c0;
  out.v[1] = c1;
  out.v[2] = c2;
  out.v[3] = c3;
  return out;
}

}  // namespace dt
#endif
