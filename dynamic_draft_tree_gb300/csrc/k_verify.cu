// Tree verification: one read of the target rows, then the acceptance walk.
//
// EAGLE-2 page §"先把投机解码的账本摆清楚": accept the candidate with probability
// min(1, p/q), on rejection resample from norm(max(0, p - q)); §"无损性为什么没有被动态树破坏":
// the tree only changes the proposals, the rule keeps the target distribution; greedy decoding
// is deterministic. The candidates here are deterministic (top-K / top-m), so each candidate's
// proposal is a point mass: accept x with probability P_res(x), drop x from the residual on a
// rejection. Graft page step (3): every verified row also yields its top-k successor ids.
#include <algorithm>

#include "rowstream.cuh"

namespace dt {
namespace {

struct StreamArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int B, P, V, K, maxp;
  int64_t Gtot;           // warps of the grid
  const int32_t* tokens;  // meta [B][P]
  const int32_t* n_pos;   // meta [B]
  int packed;             // logits rows packed (row (b, i) = the pass's row j) instead of [B][P]
  int test_timeout;
};

// Streaming pass of the verify: request b's rows are its used positions i < n_pos[b] (a position
// without a valid token is counted but not read), numbered in request order, which is the packed
// layout's row order; every warp leaves the statistics and top-K keys (K = 1, or 8 for the Graft
// refresh) of the row pieces it reads.
template <typename T, bool SOFTMAX>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm) verify_stream_kernel(StreamArgs a) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t stream_smem[];
  WarpStream& wsm = reinterpret_cast<WarpStream*>(stream_smem)[threadIdx.x >> 5];
  WarpRing& rg = wsm.rg;
  Workspace& ws = a.ws;
  const int lane = threadIdx.x & 31;
  auto cnt = [&](int b) -> int { return min(max(a.n_pos[b], 0), a.P); };
  auto row_of = [&](int b, int i, int64_t j) -> const T* {
    const int64_t r = (int64_t)b * a.P + i;
    if (a.test_timeout || a.tokens[r] < 0) return nullptr;  // invalid token: row not needed
    return reinterpret_cast<const T*>(a.logits) + (a.packed ? j : r) * a.ld;
  };
  if (a.test_timeout && blockIdx.x == 0 && threadIdx.x == 0) set_status(ws.status, DT_DEV_TIMEOUT);
  stream_rows<T, SOFTMAX>(a.B, a.V, a.K, a.maxp, a.Gtot, wsm, ws.row_tau, cnt, row_of,
                          [&](int64_t j, int64_t g, int b, int i, const PieceOut& o) {
                            publish_partial(ws.partials + j + g, rg, o, a.K);
                            if (lane == 0 && o.internal) set_status(ws.status, DT_DEV_INTERNAL);
                            if (lane == 0 && o.bad) set_status(ws.status, DT_DEV_BAD_LOGITS);
                          });
}

struct WalkArgs {
  Workspace ws;
  dt_tree_meta meta;
  const void* logits;
  int64_t ld;
  int B, P, V, dtype, mode, packed;
  int K, maxp, esz, vecel;  // pieces of the streaming pass: keys per piece, pieces per row at most
  int64_t Gtot;             // warps of the streaming launch
  uint32_t key0, key1, r0, r1;
  int32_t* accept_len;
  int32_t* accept_path;
  int32_t* bonus;
  int32_t* top8;            // [B][P][8] or null
};

__device__ __forceinline__ float load_logit(const void* logits, int dtype, int64_t idx) {
  if (dtype == DT_BF16)
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t*>(logits) + idx) << 16);
  return __ldg(reinterpret_cast<const float*>(logits) + idx);
}

constexpr int kWalkThreads = 256;

// Exact residual mass of row `r` without the tokens rej[0..n_rej): fixed-point sum of
// exp(x - M) (2^-46 units), so that subtracting the rejected terms cannot cancel. The integer sum
// does not depend on the order of its terms; the row is read with 16-byte loads, four per thread in
// flight (the elements before the first 16-byte boundary and after the last one singly).
static __device__ __noinline__ double residual_rescan(const WalkArgs& a, int64_t r, float M, const int32_t* rej, int n_rej) {
  __shared__ unsigned long long acc;
  if (threadIdx.x == 0) acc = 0ull;
  __syncthreads();
  unsigned long long part = 0ull;
  const float scale = 70368744177664.0f;  // 2^46
  auto term = [&](float x) -> unsigned long long {
    return (unsigned long long)__float2ull_rn(ex2((x - M) * kLog2e) * scale);
  };
  const int esz = a.dtype == DT_BF16 ? 2 : 4;
  const int per = 16 / esz;  // elements per vector
  const char* row = reinterpret_cast<const char*>(a.logits) + r * a.ld * esz;
  const int64_t head = min((int64_t)a.V, (int64_t)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) / esz));
  const int64_t nvec = ((int64_t)a.V - head) / per;
  const int64_t tail0 = head + nvec * per;
  for (int64_t v = threadIdx.x; v < head; v += blockDim.x) part += term(load_logit(a.logits, a.dtype, r * a.ld + v));
  for (int64_t v = tail0 + threadIdx.x; v < a.V; v += blockDim.x)
    part += term(load_logit(a.logits, a.dtype, r * a.ld + v));
  const uint4* vp = reinterpret_cast<const uint4*>(row + head * esz);
  const int64_t bd = blockDim.x;
  for (int64_t q0 = threadIdx.x; q0 < nvec; q0 += 4 * bd) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (q0 + u * bd < nvec) w[u] = __ldg(vp + q0 + u * bd);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (q0 + u * bd >= nvec) break;
      const uint32_t wd[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (esz == 2) {
          part += term(bf16_lo(wd[c]));
          part += term(bf16_hi(wd[c]));
        } else {
          part += term(__uint_as_float(wd[c]));
        }
      }
    }
  }
  atomicAdd(&acc, part);
  __syncthreads();
  unsigned long long tot = acc;
  for (int j = 0; j < n_rej; ++j) {
    const float e = ex2((load_logit(a.logits, a.dtype, r * a.ld + rej[j]) - M) * kLog2e);
    tot -= (unsigned long long)__float2ull_rn(e * scale);
  }
  __syncthreads();
  return (double)tot * 1.4210854715202004e-14;  // 2^-46
}

// One CTA per request. The statistics of the target rows come from the streaming pass's pieces:
// greedy verify merges every used row's argmax first (the top-8 ids for the Graft refresh are merged
// before the walk by verify_top8_kernel);
// sampling merges the softmax statistics of each row the walk visits.
__global__ void __launch_bounds__(kWalkThreads) verify_walk_kernel(WalkArgs a) {
  pdl_begin();
  __shared__ uint64_t s_mbuf[256];  // merge scratch of warp 0 (pieces x keys <= 32 x 8)
  __shared__ uint64_t s_mtop[kMaxK];
  __shared__ uint64_t s_key[kMaxP];
  __shared__ int64_t s_A, s_base;
  __shared__ float s_m;
  __shared__ double s_S;
  __shared__ int32_t s_first_child[kMaxP], s_next_sib[kMaxP];
  __shared__ int32_t s_path[kMaxP];
  __shared__ int32_t s_rej[kMaxP];
  __shared__ int32_t s_tok[kMaxP], s_par[kMaxP], s_amax[kMaxP], s_depth[kMaxP];
  __shared__ uint8_t s_reach[kMaxP], s_haschild[kMaxP];
  __shared__ unsigned long long s_best;
  __shared__ int32_t s_cur, s_len, s_nrej, s_state, s_nkids, s_jpos;
  __shared__ double s_sres;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int P = a.P;
  const int Dp = a.meta.D_path;
  const Workspace& ws = a.ws;
  const int64_t rb = (int64_t)b * P;
  const int npos = min(a.meta.n_pos[b], P);

  const int lane = tid & 31, warp = tid >> 5;
  auto cnt = [&](int bb) -> int { return min(max(a.meta.n_pos[bb], 0), a.P); };
  // stage the flattened tree (coalesced, independent loads); warp 0 places this request's rows in the
  // streaming pass's row order
  if (warp == 0) {
    const int64_t A = warp_total_rows(a.B, cnt);
    const int64_t base = warp_rows_before(b, cnt);
    if (lane == 0) {
      s_A = A;
      s_base = base;
    }
  }
  for (int p = tid; p < P; p += blockDim.x) {
    const bool used = p < npos;
    s_tok[p] = used ? a.meta.tokens[rb + p] : -1;
    s_par[p] = used ? a.meta.parents[rb + p] : -1;
    s_depth[p] = used ? a.meta.depth[rb + p] : -1;
    s_haschild[p] = 0;
    s_key[p] = 0ull;
  }
  __syncthreads();
  const int64_t rowA = s_A, rowbase = s_base;
  const int64_t lrow0 = a.packed ? rowbase : rb;  // logits row of position 0
  const int64_t G = stream_warps(rowA, a.V, a.esz, a.Gtot, a.maxp);
  const PieceMap pm(rowA, a.V, G, a.vecel);
  for (int p = tid; p < npos; p += blockDim.x) ws.row_tau[rowbase + p] = 0ull;  // the pass is over
  if (a.mode == DT_GREEDY) {
    // argmax of every used row: the best of its pieces' keys (one load per piece; the top-8 output of
    // the Graft refresh is merged by verify_top8_kernel before this walk)
    for (int p = tid; p < npos; p += blockDim.x) {
      if (s_tok[p] < 0) continue;
      const RowPieces rp = pm.row(rowbase + p);
      uint64_t best = 0ull;
      for (int q0 = 0; q0 < rp.S; q0 += 8) {  // independent loads, eight at a time
        uint64_t k8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) k8[u] = q0 + u < rp.S ? ws.partials[rp.slot0 + q0 + u].keys[0] : 0ull;
#pragma unroll
        for (int u = 0; u < 8; ++u) best = k8[u] > best ? k8[u] : best;
      }
      s_key[p] = best;
    }
    __syncthreads();
    for (int p = tid; p < npos; p += blockDim.x) {
      if (s_tok[p] >= 0 && s_key[p] == 0ull) set_status(ws.status, DT_DEV_BAD_LOGITS);  // no finite entry
      s_amax[p] = (s_tok[p] >= 0 && s_key[p] != 0ull) ? (int32_t)key_id(s_key[p]) : -1;
      if (p > 0 && s_par[p] >= 0) s_haschild[s_par[p]] = 1;
    }
    if (tid == 0) s_best = 0ull;
    __syncthreads();
    // reach[p]: every position on the path root..p matches the argmax of its parent's row
    for (int p = tid; p < npos; p += blockDim.x) {
      bool ok = true;
      for (int q = p, guard = 0; q > 0 && ok && guard < kMaxP; q = s_par[q], ++guard) {
        const int pq = s_par[q];
        ok = pq >= 0 && s_tok[q] >= 0 && s_tok[q] == s_amax[pq];
      }
      s_reach[p] = ok ? 1 : 0;
    }
    __syncthreads();
    // every leaf: its accepted count is the depth of its deepest reachable ancestor; the largest
    // count wins, ties go to the leaf of lowest position (retrieve rows are in leaf order)
    for (int p = tid; p < npos; p += blockDim.x) {
      if (s_haschild[p]) continue;
      int q = p, guard = 0;
      while (q > 0 && !s_reach[q] && guard++ < kMaxP) q = s_par[q];
      if (q < 0) q = 0;
      const int cnt = s_depth[q];
      const unsigned long long key = ((unsigned long long)(cnt + 1) << 32) |
                                     ((unsigned long long)(0xFFFFu - (uint32_t)p) << 16) | (uint32_t)q;
      atomicMax(&s_best, key);
    }
    __syncthreads();
    const int cnt = (int)(s_best >> 32) - 1;
    const int last = (int)(s_best & 0xFFFFull);
    if (tid == 0) {
      for (int j = 0; j < Dp; ++j) s_path[j] = -1;
      int q = last;
      for (int j = cnt; j >= 0 && j < Dp; --j) {
        s_path[j] = q;
        q = s_par[q];
      }
      a.accept_len[b] = cnt;
      a.bonus[b] = s_amax[last];
    }
    __syncthreads();
    for (int j = tid; j < Dp; j += blockDim.x) a.accept_path[(int64_t)b * Dp + j] = s_path[j];
    return;
  }

  // ---- speculative sampling walk ----
  if (tid == 0) {
    for (int p = 0; p < P; ++p) {
      s_first_child[p] = -1;
      s_next_sib[p] = -1;
    }
    for (int p = npos - 1; p >= 1; --p) {  // children in increasing position
      const int q = s_par[p];
      if (q >= 0 && q < P) {
        s_next_sib[p] = s_first_child[q];
        s_first_child[q] = p;
      }
    }
    s_cur = 0;
    s_len = 0;
    s_path[0] = 0;
  }
  __syncthreads();
  for (int guard = 0; guard < kMaxP; ++guard) {
    const int cur = s_cur;
    if (warp == 0) {  // the softmax statistics of the row at the current position, from its pieces
      const RowPieces rp = pm.row(rowbase + cur);
      float M = -INFINITY, sh = 0.0f, sl = 0.0f;
      if (s_tok[cur] < 0 || rp.S > a.maxp) {
        if (lane == 0) set_status(ws.status, s_tok[cur] < 0 ? DT_DEV_BAD_TOKEN : DT_DEV_INTERNAL);
      } else {
        warp_merge_row(ws.partials + rp.slot0, rp.S, a.K, s_mbuf, 256, s_mtop, true, M, sh, sl);
      }
      if (lane == 0) {
        if (sh != sh || !(M > -INFINITY) || M == INFINITY || !(sh > 0.0f) || sh == INFINITY)
          set_status(ws.status, DT_DEV_BAD_LOGITS);
        s_m = M;
        s_S = (double)sh + (double)sl;
      }
    }
    __syncthreads();
    RowStat st;
    st.m = s_m;
    st.s = s_S;
    st.amax = -1;
    const double S = st.s;
    // the children of cur in position order, each one's e = exp(x_t - M) and acceptance uniform
    // loaded in parallel; the tests then only compare them (one thread, in order)
    if (tid == 0) {
      int n = 0;
      for (int c = s_first_child[cur]; c >= 0 && n < kMaxP; c = s_next_sib[c]) s_amax[n++] = c;
      s_nkids = n;
      s_nrej = 0;
      s_sres = S;
    }
    __syncthreads();
    const int nk = s_nkids;
    float2* ev = reinterpret_cast<float2*>(s_key);  // (e, u) per child (s_key serves the greedy walk only)
    for (int j = tid; j < nk; j += blockDim.x) {
      const int c = s_amax[j];
      const int t = s_tok[c];
      float e = 0.0f;
      if (t >= 0 && t < a.V) e = ex2((load_logit(a.logits, a.dtype, (lrow0 + cur) * a.ld + t) - st.m) * kLog2e);
      const Philox4 w = philox4x32_10(a.r0, a.r1, (uint32_t)(512 * b + c), 0x80000000u, a.key0, a.key1);
      ev[j] = make_float2(e, (float)(w.v[0] >> 8) * 5.9604644775390625e-08f);  // u: 24 bits x 2^-24, exact
    }
    __syncthreads();
    double s_ref = S;
    int child = -1;
    bool moved = false;
    for (int j0 = 0, pass = 0; pass <= kMaxP; ++pass) {
      if (tid == 0) {
        // 0: every child tested; 1: child j accepted; 4: the running residual lost too much to
        // cancellation before child j
        int state = 0, j = j0, nrej = s_nrej;
        double sres = s_sres;
        for (; j < nk; ++j) {
          const int t = s_tok[s_amax[j]];
          bool skip = t < 0;
          if (t >= a.V) {
            set_status(ws.status, DT_DEV_BAD_TOKEN);
            skip = true;
          }
          for (int r = 0; r < nrej && !skip; ++r) skip = s_rej[r] == t;
          if (skip) continue;
          if (sres < s_ref * 0.125) {
            state = 4;
            break;
          }
          const float2 eu = ev[j];
          if ((double)eu.y * sres < (double)eu.x) {  // u < e / S_res = P_res(x), without the division
            state = 1;
            break;
          }
          s_rej[nrej++] = t;
          sres -= (double)eu.x;
        }
        s_nrej = nrej;
        s_sres = sres;
        s_state = state;
        s_jpos = j;
      }
      __syncthreads();
      const int state = s_state;
      j0 = s_jpos;
      if (state == 4) {  // recompute the residual exactly, then test the same child again
        const double v = residual_rescan(a, lrow0 + cur, st.m, s_rej, s_nrej);
        if (tid == 0) s_sres = v;
        s_ref = v;
        __syncthreads();
        continue;
      }
      if (state == 1) {
        moved = true;
        child = s_amax[j0];
      }
      break;
    }
    if (moved) {
      if (tid == 0) {
        s_len = s_len + 1;
        s_path[s_len] = child;
        s_cur = child;
      }
      __syncthreads();
      continue;
    }
    // residual draw happens in the bonus kernel
    if (tid == 0) {
      WalkState* wsb = ws.walk + b;
      wsb->row = lrow0 + cur;
      wsb->cur = cur;
      wsb->n_rej = s_nrej;
      for (int j = 0; j < s_nrej; ++j) wsb->rej[j] = s_rej[j];
      ws.bonus_key[b] = 0ull;
      a.accept_len[b] = s_len;
    }
    __syncthreads();
    for (int j = tid; j < Dp; j += blockDim.x) a.accept_path[(int64_t)b * Dp + j] = j <= s_len ? s_path[j] : -1;
    return;
  }
  if (tid == 0) set_status(ws.status, DT_DEV_INTERNAL);
}

// The top-8 ids of every used row from its pieces (Graft page step (3): every verified row refreshes M
// with its top-k successors), one warp per row over many CTAs, rows numbered as in the streaming
// pass; launched before the walk, which then needs only each row's argmax.
constexpr int kTop8Warps = 8;
__global__ void __launch_bounds__(32 * kTop8Warps) verify_top8_kernel(WalkArgs a) {
  pdl_begin();
  __shared__ uint64_t s_mbuf[kTop8Warps][256];
  __shared__ uint64_t s_mtop[kTop8Warps][kMaxK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t j = (int64_t)blockIdx.x * kTop8Warps + warp;
  auto cnt = [&](int bb) -> int { return min(max(a.meta.n_pos[bb], 0), a.P); };
  const int64_t A = warp_total_rows(a.B, cnt);
  if (j >= A) return;
  int b, i;
  warp_find_row(a.B, j, cnt, b, i);
  if (b >= a.B) return;
  const int64_t r = (int64_t)b * a.P + i;
  if (a.meta.tokens[r] < 0) {
    if (lane < 8) a.top8[r * 8 + lane] = -1;
    return;
  }
  const PieceMap pm(A, a.V, stream_warps(A, a.V, a.esz, a.Gtot, a.maxp), a.vecel);
  const RowPieces rp = pm.row(j);
  if (rp.S > a.maxp) {  // never: the streaming plan bounds the pieces of a row
    if (lane == 0) set_status(a.ws.status, DT_DEV_INTERNAL);
    return;
  }
  float M, sh, sl;
  warp_merge_row(a.ws.partials + rp.slot0, rp.S, a.K, s_mbuf[warp], 256, s_mtop[warp], false, M, sh, sl);
  const uint64_t k = lane < 8 ? s_mtop[warp][lane] : 0ull;
  if (lane < 8) a.top8[r * 8 + lane] = (lane < a.K && k != 0ull) ? (int32_t)key_id(k) : -1;
}

struct BonusArgs {
  Workspace ws;
  const void* logits;
  int64_t ld;
  int P, V, dtype, S;
  int64_t seg_len;
  uint32_t key0, key1, r0, r1;
  int32_t* bonus;
};

constexpr int kBonusThreads = 256;

// Gumbel-max draw from the final residual: argmax over tokens not rejected at that position of
// x_v - log(-log(u_v)). Grid: B * S CTAs, each a segment of the row.
__global__ void __launch_bounds__(kBonusThreads) verify_bonus_kernel(BonusArgs a) {
  pdl_begin();
  __shared__ unsigned long long s_best;
  __shared__ int32_t s_rej[kMaxP];
  __shared__ int32_t s_last;
  const int b = blockIdx.x / a.S, seg = blockIdx.x % a.S;
  const int tid = threadIdx.x;
  Workspace& ws = a.ws;
  const WalkState* wsb = ws.walk + b;
  const int cur = wsb->cur;
  const int n_rej = wsb->n_rej;
  for (int j = tid; j < n_rej; j += blockDim.x) s_rej[j] = wsb->rej[j];
  if (tid == 0) s_best = 0ull;
  __syncthreads();
  const int64_t r = wsb->row;
  const int64_t v0 = (int64_t)seg * a.seg_len;
  const int64_t v1 = min((int64_t)a.V, v0 + a.seg_len);
  unsigned long long best = 0ull;
  // groups of 4 consecutive tokens share one Philox call
  for (int64_t g = v0 / 4 + tid; g * 4 < v1; g += blockDim.x) {
    const Philox4 w = philox4x32_10(a.r0, a.r1, (uint32_t)(512 * b + cur), (uint32_t)g, a.key0, a.key1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t v = g * 4 + e;
      if (v < v0 || v >= v1) continue;
      const float u = ((float)(w.v[e] >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
      const float gmb = -logf(-logf(u));
      const float y = load_logit(a.logits, a.dtype, r * a.ld + v) + gmb;
      const unsigned long long k = make_key(y, (uint32_t)v);
      if (k > best) {
        bool rej = false;
        for (int j = 0; j < n_rej; ++j) rej |= (s_rej[j] == (int32_t)v);
        if (!rej) best = k;
      }
    }
  }
  atomicMax(&s_best, best);
  __syncthreads();
  if (tid == 0) {
    atomicMax(&ws.bonus_key[b], s_best);
    __threadfence();
    const int prev = atomicAdd(&ws.bonus_counter[b], 1);
    s_last = prev == a.S - 1;
  }
  __syncthreads();
  if (s_last && tid == 0) {
    __threadfence();
    const unsigned long long k = atomicAdd(&ws.bonus_key[b], 0ull);
    a.bonus[b] = k ? (int32_t)key_id(k) : -1;
    ws.bonus_counter[b] = 0;
  }
}

}  // namespace

int stream_grid(const dt_handle* h) { return std::max(1, h->num_sms * kStreamCtasPerSm); }

cudaError_t init_verify_attributes() {
  // the streaming kernels: two CTAs of eight warps with their copy rings per SM
  const cudaFuncAttribute dyn = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const cudaFuncAttribute carve = cudaFuncAttributePreferredSharedMemoryCarveout;
  const int mx = cudaSharedmemCarveoutMaxShared, sb = (int)stream_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel<uint16_t, false>, dyn, sb);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<uint16_t, true>, dyn, sb);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<float, false>, dyn, sb);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<float, true>, dyn, sb);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<uint16_t, false>, carve, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<uint16_t, true>, carve, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<float, false>, carve, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_stream_kernel<float, true>, carve, mx);
  return e;
}

cudaError_t launch_verify_rows(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                               int with_top8, cudaStream_t s) {
  const int packed = (mode & DT_VERIFY_PACKED) ? 1 : 0;
  mode &= ~DT_VERIFY_PACKED;
  StreamArgs ra;
  ra.packed = packed;
  ra.ws = h->ws;
  ra.logits = logits;
  ra.ld = ld;
  ra.B = h->B;
  ra.P = meta->P;
  ra.V = h->cfg.V;
  ra.K = with_top8 ? 8 : 1;
  ra.maxp = stream_max_pieces(ra.K);
  const unsigned grid = (unsigned)stream_grid(h);
  ra.Gtot = (int64_t)grid * kStreamWarps;
  ra.tokens = meta->tokens;
  ra.n_pos = meta->n_pos;
  ra.test_timeout = (h->cfg.flags & DT_FLAG_TEST_TIMEOUT) ? 1 : 0;
#define DT_LAUNCH_ROWS(T, SM) \
  launch_k(verify_stream_kernel<T, SM>, dim3(grid), dim3(kStreamThreads), stream_smem_bytes(), s, ra)
  const bool sm_on = mode == DT_SAMPLE;
  if (h->cfg.dtype == DT_BF16) {
    if (sm_on) DT_LAUNCH_ROWS(uint16_t, true);
    else DT_LAUNCH_ROWS(uint16_t, false);
  } else {
    if (sm_on) DT_LAUNCH_ROWS(float, true);
    else DT_LAUNCH_ROWS(float, false);
  }
#undef DT_LAUNCH_ROWS
  return cudaGetLastError();
}

cudaError_t launch_verify_accept(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld,
                                 int mode, uint64_t seed, uint64_t round, int32_t* accept_len,
                                 int32_t* accept_path, int32_t* bonus, int32_t* top8, cudaStream_t s) {
  const int P = meta->P;
  const int V = h->cfg.V;
  const int esz = h->cfg.dtype == DT_BF16 ? 2 : 4;
  const int packed = (mode & DT_VERIFY_PACKED) ? 1 : 0;
  mode &= ~DT_VERIFY_PACKED;
  cudaError_t e;
  WalkArgs wa;
  wa.packed = packed;
  wa.ws = h->ws;
  wa.meta = *meta;
  wa.logits = logits;
  wa.ld = ld;
  wa.P = P;
  wa.V = V;
  wa.dtype = h->cfg.dtype;
  wa.mode = mode;
  wa.key0 = (uint32_t)seed;
  wa.key1 = (uint32_t)(seed >> 32);
  wa.r0 = (uint32_t)round;
  wa.r1 = (uint32_t)(round >> 32);
  wa.accept_len = accept_len;
  wa.accept_path = accept_path;
  wa.bonus = bonus;
  wa.top8 = top8;
  wa.B = h->B;
  wa.K = top8 ? 8 : 1;
  wa.maxp = stream_max_pieces(wa.K);
  wa.esz = esz;
  wa.vecel = 16 / esz;
  wa.Gtot = (int64_t)stream_grid(h) * kStreamWarps;
  if (top8) {  // the top-8 merges on many CTAs first; the walk then takes each row's argmax alone
    const int64_t rows = (int64_t)h->B * P;
    launch_k(verify_top8_kernel, dim3((unsigned)((rows + kTop8Warps - 1) / kTop8Warps)), dim3(32 * kTop8Warps), 0, s,
             wa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    wa.top8 = nullptr;
  }
  launch_k(verify_walk_kernel, dim3(h->B), dim3(kWalkThreads), 0, s, wa);
  e = cudaGetLastError();
  if (e != cudaSuccess || mode != DT_SAMPLE) return e;

  BonusArgs ba;
  ba.ws = h->ws;
  ba.logits = logits;
  ba.ld = ld;
  ba.P = P;
  ba.V = V;
  ba.dtype = h->cfg.dtype;
  const int64_t target = (int64_t)h->num_sms * 4;
  int Sb = (int)std::max<int64_t>(1, std::min<int64_t>((target + h->B - 1) / h->B, (V + 4095) / 4096));
  ba.S = Sb;
  int64_t Lb = (V + Sb - 1) / Sb;
  ba.seg_len = (Lb + 3) / 4 * 4;
  ba.key0 = wa.key0;
  ba.key1 = wa.key1;
  ba.r0 = wa.r0;
  ba.r1 = wa.r1;
  ba.bonus = bonus;
  launch_k(verify_bonus_kernel, dim3((unsigned)(h->B * Sb)), dim3(kBonusThreads), 0, s, ba);
  return cudaGetLastError();
}

cudaError_t launch_verify(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                          uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* accept_path,
                          int32_t* bonus, int32_t* top8, cudaStream_t s) {
  cudaError_t e = launch_verify_rows(h, meta, logits, ld, mode, top8 != nullptr, s);
  if (e != cudaSuccess) return e;
  return launch_verify_accept(h, meta, logits, ld, mode, seed, round, accept_len, accept_path, bonus, top8, s);
}

}  // namespace dt
