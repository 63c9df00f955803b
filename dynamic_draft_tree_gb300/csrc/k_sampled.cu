// Verify of sampled drafts: recursive rejection against the draft distributions.
//
// EAGLE-2 page §"先把投机解码的账本摆清楚": a drafted token t drawn from q is accepted with
// probability min(1, p(t)/q(t)); after a rejection the next token comes from norm(max(0, p - q)).
// §"无损性为什么没有被动态树破坏": this rule, not the tree, keeps the target distribution. The K
// children of a node were drawn from its draft row q without replacement (Gumbel-top-K at expansion),
// child j from q_j = q without the earlier children, renormalised; it is tested against the current
// residual r_j (r_0 = p): accept with probability min(1, r_j(t)/q_j(t)), else
// r_{j+1} = norm(max(0, r_j - q_j)). When every child of the current node is rejected (or it has none)
// the bonus token is a Gumbel-max draw from the last residual.
#include <algorithm>

#include <cooperative_groups.h>

#include "rowstream.cuh"

namespace dt {
namespace {

constexpr int kSampThreads = 512;
constexpr int kSampWarps = kSampThreads / 32;
// A request's walk runs on a thread-block cluster: every CTA follows the same walk (the decisions are
// computed identically from the same data), each pass over the vocabulary is split across the CTAs,
// and the partial sums and the bonus candidates meet through distributed shared memory.
constexpr int kSampCluster = 8;
constexpr int kMaxKids = kMaxK;  // children of a node <= K <= 32

struct SampledArgs {
  Workspace ws;
  dt_tree_meta meta;
  const void* logits;  // target rows
  int64_t ld;
  const void* draft;   // draft rows: [D_max][B][W][ld_d], layer d's rows at index d - 1
  int64_t ld_d;
  int B, P, V, W, N, dtype, packed;
  int maxp, vecel;     // pieces of the streaming pass (K = 1 keys, softmax statistics)
  int64_t Gtot;
  uint32_t key0, key1, r0, r1;
  int32_t* accept_len;
  int32_t* accept_path;
  int32_t* bonus;
};

__device__ __forceinline__ float load_elt(const void* base, int dtype, int64_t idx) {
  if (dtype == DT_BF16)
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t*>(base) + idx) << 16);
  return __ldg(reinterpret_cast<const float*>(base) + idx);
}

// Residual state of the current node after its first `nrej` children were rejected.
struct Resid {
  float Mp, Mq;          // row maxima
  float invSp, invSq;    // 1 / sum exp(x - max)
  int nrej;
  int32_t tok[kMaxKids];   // rejected children's tokens, in draw order
  float invOneMinusQ[kMaxKids + 1];  // 1 / (1 - Q_i), Q_i = q mass of the first i children
  float invZ[kMaxKids + 1];          // 1 / Z_i (0 when Z_i = 0), Z_i of r_i = norm(max(0, r_{i-1} - q_{i-1}))
};

// r_n(v) for n = s.nrej (r_0 = p) from p(v), q(v) and the token's place among the rejected children.
__device__ __forceinline__ float residual_at(const Resid& s, float p, float q, int32_t v) {
  int l = s.nrej;  // draw index of v among the rejected children (nrej if none)
  for (int i = 0; i < s.nrej; ++i)
    if (s.tok[i] == v) l = min(l, i);
  float r = p;
  for (int i = 0; i < s.nrej; ++i) {
    const float qi = i > l ? 0.0f : q * s.invOneMinusQ[i];  // q_i(v): 0 once v was drawn
    r = fmaxf(0.0f, r - qi) * s.invZ[i + 1];
  }
  return r;
}

// One cluster of kSampCluster CTAs per request.
__global__ void __launch_bounds__(kSampThreads) verify_sampled_kernel(SampledArgs a) {
  pdl_begin();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int ncta = (int)cluster.num_blocks();
  __shared__ double s_zpart[2];               // this CTA's partial Z of a pass (slot = pass parity)
  __shared__ unsigned long long s_bkey;       // this CTA's best bonus key
  __shared__ uint64_t s_mbuf[256];
  __shared__ uint64_t s_mtop[kMaxK];
  __shared__ int32_t s_tok[kMaxP], s_par[kMaxP], s_dep[kMaxP], s_node[kMaxP];
  __shared__ int32_t s_first_child[kMaxP], s_next_sib[kMaxP];
  __shared__ int32_t s_path[kMaxP];
  __shared__ Resid s_res;
  __shared__ double s_red[kSampWarps];
  __shared__ unsigned long long s_best;
  __shared__ int64_t s_A, s_base;
  __shared__ int32_t s_cur, s_len, s_state;
  __shared__ double s_Q;  // q mass of the children tested so far at the current node
  const int b = blockIdx.x / ncta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // this CTA's slice of the vocabulary, in groups of four tokens (one Philox block each)
  const int64_t slice = ((((int64_t)a.V + ncta - 1) / ncta) + 3) / 4 * 4;
  const int64_t v_lo = min((int64_t)a.V, rank * slice), v_hi = min((int64_t)a.V, v_lo + slice);
  int npass = 0;
  Workspace& ws = a.ws;
  const int P = a.P;
  const int Dp = a.meta.D_path;
  const int64_t rb = (int64_t)b * P;
  const int npos = min(max(a.meta.n_pos[b], 0), P);
  auto cnt = [&](int bb) -> int { return min(max(a.meta.n_pos[bb], 0), a.P); };
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
    s_dep[p] = used ? a.meta.depth[rb + p] : -1;
    s_node[p] = used ? a.meta.node_id[rb + p] : -1;
  }
  __syncthreads();
  const int64_t rowA = s_A, rowbase = s_base;
  const PieceMap pm(rowA, a.V, stream_warps(rowA, a.V, a.dtype == DT_BF16 ? 2 : 4, a.Gtot, a.maxp), a.vecel);
  if (rank == 0)
    for (int p = tid; p < npos; p += blockDim.x) ws.row_tau[rowbase + p] = 0ull;  // the pass is over
  if (tid == 0) {
    for (int p = 0; p < P; ++p) {
      s_first_child[p] = -1;
      s_next_sib[p] = -1;
    }
    for (int p = npos - 1; p >= 1; --p) {  // children in increasing position = draw order
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
    const int64_t lrow = a.packed ? rowbase + cur : rb + cur;
    const void* prow = reinterpret_cast<const char*>(a.logits) + lrow * a.ld * (a.dtype == DT_BF16 ? 2 : 4);
    const int node = s_node[cur];
    const bool has_kids = s_first_child[cur] >= 0 && node >= 0 && node < a.N;
    const void* qrow = nullptr;
    if (has_kids) {
      const int d = s_dep[cur];
      const int slot = ws.exp_slot[(int64_t)b * a.N + node];
      qrow = reinterpret_cast<const char*>(a.draft) +
             ((((int64_t)d * a.B + b) * a.W + slot) * a.ld_d) * (a.dtype == DT_BF16 ? 2 : 4);
    }
    // the target row's softmax statistics from its pieces; the draft row's from its expansion
    if (warp == 0) {
      const RowPieces rp = pm.row(rowbase + cur);
      float M = -INFINITY, sh = 0.0f, sl = 0.0f;
      if (s_tok[cur] < 0 || rp.S > a.maxp) {
        if (lane == 0) set_status(ws.status, s_tok[cur] < 0 ? DT_DEV_BAD_TOKEN : DT_DEV_INTERNAL);
      } else {
        warp_merge_row(ws.partials + rp.slot0, rp.S, 1, s_mbuf, 256, s_mtop, true, M, sh, sl);
      }
      if (lane == 0) {
        if (rank == 0 && (sh != sh || !(M > -INFINITY) || M == INFINITY || !(sh > 0.0f) || sh == INFINITY))
          set_status(ws.status, DT_DEV_BAD_LOGITS);
        s_res.Mp = M;
        s_res.invSp = (float)(1.0 / ((double)sh + (double)sl));
        s_res.nrej = 0;
        s_res.invOneMinusQ[0] = 1.0f;
        s_res.invZ[0] = 1.0f;
        s_Q = 0.0;
        if (has_kids) {
          const float4 st = ws.exp_stat[(int64_t)b * a.N + node];
          s_res.Mq = st.x;
          s_res.invSq = (float)(1.0 / ((double)st.y + (double)st.z));
        } else {
          s_res.Mq = 0.0f;
          s_res.invSq = 0.0f;
        }
      }
    }
    __syncthreads();
    int child = s_first_child[cur];
    bool moved = false;
    while (has_kids && child >= 0) {
      // the test of this child (thread 0): r_n(t) < u q_n(t) rejects
      if (tid == 0) {
        const int t = s_tok[child];
        const int n = s_res.nrej;
        s_state = 0;
        if (t < 0 || t >= a.V || n >= kMaxKids) {
          if (rank == 0) set_status(ws.status, t >= a.V || n >= kMaxKids ? DT_DEV_BAD_TOKEN : DT_DEV_BAD_TREE);
          s_state = 2;
        } else {
          const double p_t = exp((double)load_elt(prow, a.dtype, t) - (double)s_res.Mp) * (double)s_res.invSp;
          const double q_t = exp((double)load_elt(qrow, a.dtype, t) - (double)s_res.Mq) * (double)s_res.invSq;
          double r = p_t;
          for (int i = 0; i < n; ++i) {
            const double qi = q_t * (double)s_res.invOneMinusQ[i];
            r = fmax(0.0, r - qi) * (double)s_res.invZ[i + 1];
          }
          const double qn = q_t / (1.0 - s_Q);
          const Philox4 w = philox4x32_10(a.r0, a.r1, (uint32_t)(512 * b + child), 0x80000000u, a.key0, a.key1);
          const double u = (double)(w.v[0] >> 8) * 5.9604644775390625e-08;  // 2^-24
          const bool accept = !(qn > 0.0) || u * qn < r;  // u < min(1, r / q_n)
          if (accept) {
            s_state = 1;
          } else {
            s_res.tok[n] = t;
            s_res.invOneMinusQ[n] = (float)(1.0 / (1.0 - s_Q));
            s_Q += q_t;
            s_res.invOneMinusQ[n + 1] = (float)(1.0 / (1.0 - s_Q));
          }
        }
      }
      __syncthreads();
      const int st = s_state;
      if (st == 1) {
        moved = true;
        break;
      }
      if (st == 0) {
        // rejected: Z_{n+1} = sum_v max(0, r_n(v) - q_n(v)), one pass over both rows, split across the
        // cluster's CTAs
        Resid& R = s_res;
        const int n = R.nrej;  // the rejected child is draw index n
        double part = 0.0;
        for (int64_t v = v_lo + tid; v < v_hi; v += blockDim.x) {
          const float xp = load_elt(prow, a.dtype, v), xq = load_elt(qrow, a.dtype, v);
          const float p = __expf(xp - R.Mp) * R.invSp, q = __expf(xq - R.Mq) * R.invSq;
          const float r = residual_at(R, p, q, (int32_t)v);
          bool drawn = false;  // v among the children rejected before this one: q_n(v) = 0
          for (int i = 0; i < n; ++i) drawn |= R.tok[i] == (int32_t)v;
          const float qn = drawn ? 0.0f : q * R.invOneMinusQ[n];
          part += (double)fmaxf(0.0f, r - qn);
        }
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        if (lane == 0) s_red[warp] = part;
        __syncthreads();
        const int slot = npass & 1;
        if (tid == 0) {
          double z = 0.0;
          for (int w = 0; w < kSampWarps; ++w) z += s_red[w];
          s_zpart[slot] = z;
        }
        // every CTA adds the cluster's partials in rank order (the same Z everywhere); a slot is written
        // again two passes later, after every CTA has passed the next pass's barrier
        cluster.sync();
        if (tid == 0) {
          double Z = 0.0;
          for (int r = 0; r < ncta; ++r) Z += *cluster.map_shared_rank(&s_zpart[slot], r);
          R.invZ[n + 1] = Z > 0.0 ? (float)(1.0 / Z) : 0.0f;
          R.nrej = n + 1;
        }
        ++npass;
        __syncthreads();
      }
      child = s_next_sib[child];
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
    // the bonus: Gumbel-max over log r + G for the tokens with r > 0 (r = p without children)
    if (tid == 0) s_best = 0ull;
    __syncthreads();
    {
      const Resid& R = s_res;
      unsigned long long best = 0ull;
      for (int64_t g4 = v_lo / 4 + tid; g4 * 4 < v_hi; g4 += blockDim.x) {
        const Philox4 w = philox4x32_10(a.r0, a.r1, (uint32_t)(512 * b + cur), (uint32_t)g4, a.key0, a.key1);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t v = g4 * 4 + e;
          if (v >= v_hi) break;
          const float xp = load_elt(prow, a.dtype, v);
          float r;
          if (has_kids) {
            const float q = __expf(load_elt(qrow, a.dtype, v) - R.Mq) * R.invSq;
            r = residual_at(R, __expf(xp - R.Mp) * R.invSp, q, (int32_t)v);
          } else {
            r = __expf(xp - R.Mp) * R.invSp;
          }
          if (!(r > 0.0f)) continue;
          const float u = ((float)(w.v[e] >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
          const float y = logf(r) - logf(-logf(u));
          const unsigned long long k = make_key(y, (uint32_t)v);
          best = k > best ? k : best;
        }
      }
      atomicMax(&s_best, best);
    }
    __syncthreads();
    if (tid == 0) s_bkey = s_best;
    cluster.sync();  // every CTA's best key is in place
    if (rank == 0) {
      if (tid == 0) {
        unsigned long long best = 0ull;
        for (int r = 0; r < ncta; ++r) {
          const unsigned long long k = *cluster.map_shared_rank(&s_bkey, r);
          best = k > best ? k : best;
        }
        // no token with r > 0 (an empty residual): token 0, as an argmax over all -inf
        a.bonus[b] = best ? (int32_t)key_id(best) : 0;
        a.accept_len[b] = s_len;
      }
      for (int j = tid; j < Dp; j += blockDim.x) a.accept_path[(int64_t)b * Dp + j] = j <= s_len ? s_path[j] : -1;
    }
    cluster.sync();  // no CTA leaves while rank 0 may still read its shared memory
    return;
  }
  cluster.sync();  // (never reached in a valid tree) no CTA leaves while another may read its shared memory
  if (rank == 0 && tid == 0) set_status(ws.status, DT_DEV_INTERNAL);
}

}  // namespace

cudaError_t launch_verify_sampled(dt_handle* h, const dt_tree_meta* meta, const void* logits, int64_t ld, int mode,
                                  const void* draft, int64_t ld_d, uint64_t seed, uint64_t round,
                                  int32_t* accept_len, int32_t* accept_path, int32_t* bonus, cudaStream_t s) {
  cudaError_t e = launch_verify_rows(h, meta, logits, ld, DT_SAMPLE | (mode & DT_VERIFY_PACKED), 0, s);
  if (e != cudaSuccess) return e;
  SampledArgs a;
  a.ws = h->ws;
  a.meta = *meta;
  a.logits = logits;
  a.ld = ld;
  a.draft = draft;
  a.ld_d = ld_d;
  a.B = h->B;
  a.P = meta->P;
  a.V = h->cfg.V;
  a.W = h->cfg.W;
  a.N = h->N;
  a.dtype = h->cfg.dtype;
  a.packed = (mode & DT_VERIFY_PACKED) ? 1 : 0;
  a.maxp = stream_max_pieces(1);
  a.vecel = 16 / (h->cfg.dtype == DT_BF16 ? 2 : 4);
  a.Gtot = (int64_t)stream_grid(h) * kStreamWarps;
  a.key0 = (uint32_t)seed;
  a.key1 = (uint32_t)(seed >> 32);
  a.r0 = (uint32_t)round;
  a.r1 = (uint32_t)(round >> 32);
  a.accept_len = accept_len;
  a.accept_path = accept_path;
  a.bonus = bonus;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kSampCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(h->B * kSampCluster));
  cfg.blockDim = dim3(kSampThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, verify_sampled_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dt
