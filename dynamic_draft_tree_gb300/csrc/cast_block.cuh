// CAST width/depth pruning and the Graft checkpoint test as device functions of the pruning kernels.
//
// CAST page §关键设计 2-3: marginal utility (u_k - u_k0)/(c_k - c_k0) against C1 for the width, the
// FIFO gain buffer against C2 for the depth; costs from the S_T/S_D lookup tables.
#pragma once

#include "dt_internal.cuh"

namespace dt {
namespace {

__device__ __forceinline__ int table_row(double c, double L, int M_rows) {
  const double q = floor(c / L);
  return q >= (double)(M_rows - 1) ? M_rows - 1 : (int)q;
}

// GB300 runs fp64 at a small fraction of its fp32 rate, so a dependent chain of fp64 operations is
// slow. The CAST kernels below keep fp64 for every sum and product, but lay the work out so that each
// fp64 instruction serves a whole warp of items, and turn the sequential selection into integer
// comparisons of precomputed fp64 values.

// Ordered 64-bit image of a double: unsigned comparison of images follows the fp64 order (-0 == +0).
__device__ __forceinline__ uint64_t d2ord(double x) {
  uint64_t u = (uint64_t)__double_as_longlong(x == 0.0 ? 0.0 : x);
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

constexpr int kPruneThreads = 1024;  // 32 warps (most threads a prune launch uses)
// Threads of a prune launch: 16 warps while they hold one warp per request plus the helper warps
// (B <= 16; fewer warps make every block barrier shorter), 32 beyond.
inline int prune_threads(int B) { return B <= 16 ? kPruneThreads / 2 : kPruneThreads; }
constexpr int kItemChunk = 64;       // items per pass (two per lane)

// items[s] = (1/B) sum_b vb(b, s) for s < cap, in fp64. Warp w sums requests b = w, w + 32, ... for
// every item (lanes over items), then warps 0 and 1 add the 32 warp partials in warp order.
// `part` is shared scratch of 32 * kItemChunk doubles. All threads call it.
template <typename F>
__device__ void batch_items(double* items, double* part, int cap, int B, F vb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = min(32, B);
  for (int s0 = 0; s0 < cap; s0 += kItemChunk) {
    if (warp < nw) {
      double a0 = 0.0, a1 = 0.0;
      const int sa = s0 + lane, sb = s0 + 32 + lane;
      for (int b = warp; b < B; b += 32) {
        if (sa < cap) a0 += vb(b, sa);
        if (sb < cap) a1 += vb(b, sb);
      }
      part[warp * kItemChunk + lane] = a0;
      part[warp * kItemChunk + 32 + lane] = a1;
    }
    __syncthreads();
    if (warp < 2) {
      const int j = warp * 32 + lane, s2 = s0 + j;
      if (s2 < cap) {
        double acc = 0.0;
        for (int w = 0; w < nw; ++w) acc += part[w * kItemChunk + j];
        // dividing by a power of two is multiplying by its exact inverse (a long fp64 division saved)
        items[s2] = (B & (B - 1)) == 0 ? acc * __hiloint2double((1023 - (31 - __clz(B))) << 20, 0)
                                       : acc / (double)B;
      }
    }
    __syncthreads();
  }
}

// Marginal-utility selection over k = 1..cap (CAST): k0 = 1; for k = 2..cap, k0 = k when
// c_k <= c_k0 or (u_k - u_k0) / (c_k - c_k0) >= thr, with u_k = items[0] + ... + items[k-1]. For
// c_k > c_k0 the second test is u_k - thr c_k >= u_k0 - thr c_k0, so with q_k = u_k - thr c_k both
// tests compare precomputed values. Warp 0 builds u (prefix sums, u[0] = 0), q and the ordered
// images of c and q; thread 0 then walks k while the other warps run during_walk(warp) (work that
// needs u and may overlap the walk). `u`, `cimg`, `qimg` ([cap+1] each) are shared scratch. All threads call
// it; every thread gets k0.
template <class DuringWalk>
__device__ int selection_rule(const double* items, const double* cost, double thr, int cap, double* u,
                              uint64_t* cimg, uint64_t* qimg, int* result, DuringWalk during_walk) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    double carry = 0.0;
    if (lane == 0) u[0] = 0.0;
    for (int c0 = 0; c0 < cap; c0 += 32) {
      const int k = c0 + lane + 1;  // u[k] = carry + inclusive prefix of items[c0..k-1]
      double x = k <= cap ? items[k - 1] : 0.0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      x += carry;
      if (k <= cap) {
        u[k] = x;
        const double q = x - thr * cost[k];
        cimg[k] = d2ord(cost[k]);
        qimg[k] = d2ord(q);
      }
      carry = __shfl_sync(0xFFFFFFFFu, x, 31);
    }
  }
  __syncthreads();
  if (tid == 0) {
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
    *result = k0;
  } else if ((tid >> 5) >= 1) {
    during_walk(tid >> 5);
  }
  __syncthreads();
  return *result;
}

struct PruneArgs {
  Workspace ws;
  dt_prune_params p;
  dt_prune_out out;
  int B, N, LW, D, d, policy;
  int W;          // frontier width limit
  int select;     // width/depth only: also select the next layer's frontier
  int32_t* ftok;  // frontier tokens [B][W] of that selection, or null
  int32_t* sel;   // verify count only: also write the rerank [B][m_cap], or null
};

// CAST width + depth after layer d, by one whole CTA (any multiple of 32 threads up to kPruneThreads;
// every thread calls it). The CAST state is copied to shared memory; every global input is read in
// one round of independent loads.
__device__ __forceinline__ void cast_width_depth_block(const PruneArgs& a) {
  __shared__ double items[kMaxW * kMaxK + 1];
  __shared__ double cost[kMaxW * kMaxK + 2];
  __shared__ double part[32 * kItemChunk];
  __shared__ double u[kMaxW + 2];
  __shared__ uint64_t cimg[kMaxW + 2], qimg[kMaxW + 2];
  __shared__ double ratio_k[kMaxW + 2];
  __shared__ uint8_t grow_k[kMaxW + 2];
  __shared__ double cost_all[kPruneThreads];  // c_k of every table row, when they fit the idle warps
  __shared__ CastState cs;
  __shared__ int s_maxcand, s_grow, s_k0, s_width, s_row;
  const Workspace& ws = a.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = (int)(blockDim.x >> 5);
  // One round of independent loads, no barrier before them: the CAST state (thread 0), each
  // request's candidate nodes for the frontier that follows (warp b), the layer's values (inside
  // batch_items), the layer sizes (warp nwarps - 2) and the cost vector (warp nwarps - 1, which reads
  // the context sum itself rather than waiting for the state).
  if (tid == 0) cs = *ws.cast;
  int f_id = -1, f_tok = -1, f_avail = 0;
  float f_val = -INFINITY;
  const bool f_pref = a.select && a.B <= nwarps;
  if (f_pref && warp < a.B) f_avail = frontier_candidates(ws, warp, a.N, a.W, a.LW, a.D, a.d, f_id, f_tok, f_val);
  const int wcap = min(a.p.width_cap, a.LW);
  // normalised draft cost of k frontier nodes at the current context: c_k = S_D[row][k-1] / S_T[row][0].
  // When the table's rows x wcap entries fit the warps between the request warps and the two helper
  // warps, those compute every row's entries while the last warp finds the row (the row needs the
  // context sum, so this takes the loads off the chain); otherwise the last warp does both in turn.
  const int free0 = a.B * 32, nfree = (nwarps - 2) * 32 - free0;
  const bool par_cost = a.p.M_rows * wcap <= nfree;
  if (par_cost && tid >= free0 && tid < free0 + a.p.M_rows * wcap) {
    const int t = tid - free0, r = t / wcap, k = t - r * wcap + 1;
    cost_all[t] = a.p.S_D[(int64_t)r * a.p.N_cols + (k - 1)] / a.p.S_T[(int64_t)r * a.p.N_cols];
  }
  if (warp == nwarps - 1) {
    const int64_t ctx = ws.cast->ctx_sum;
    const int row = table_row((double)(a.p.n0 + ctx), a.p.L, a.p.M_rows);
    if (par_cost) {
      if (lane == 0) s_row = row;
    } else {
      for (int k = 1 + lane; k <= wcap; k += 32)
        cost[k] = a.p.S_D[(int64_t)row * a.p.N_cols + (k - 1)] / a.p.S_T[(int64_t)row * a.p.N_cols];
    }
  }
  if (warp == nwarps - 2) {
    int mc = 0;
    for (int b = lane; b < a.B; b += 32) mc = max(mc, ws.layer_count[(int64_t)b * (a.D + 1) + a.d]);
    mc = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)max(mc, 0));
    if (lane == 0) s_maxcand = mc;
  }
  // items[s] = (1/B) sum_b exp(value of the s-th node of b's layer), missing nodes count 0 (its first
  // barrier publishes everything above)
  batch_items(items, part, wcap, a.B, [&](int b, int s) {
    const int64_t lb = (int64_t)b * (a.D + 1) + a.d;
    const int cnt = ws.layer_count[lb];
    const float v = ws.layer_val[lb * a.LW + s];  // read with the count: not used past it
    if (s >= cnt) return 0.0;
    return (double)expf(v);
  });
  __syncthreads();
  const int cap = min(a.p.width_cap, s_maxcand);
  const double* costp = par_cost ? cost_all + (int64_t)s_row * wcap - 1 : cost;  // costp[k] = c_k
  // While thread 0 walks the selection, warp 1 evaluates the grow test for every width k the walk may
  // choose, and warp 2 the FIFO entry u_k / u_prev that width would append. The test is
  // alpha u_k / c_k >= C2 with alpha the mean of the FIFO after the append; with S the sum of the
  // entries that stay (the oldest drops out when the FIFO is full) and L its new length it reads
  // (S u_prev + u_k) u_k >= C2 c_k L u_prev for u_prev > 0, and S u_k >= C2 c_k L before the first
  // append, which needs no fp64 division (equal to the quotient form up to rounding).
  auto grow_for_all_widths = [&](int w) {
    const int len = cs.fifo_len;
    const double up = cs.u_prev;
    if (w == 1) {
      const bool app = up >= 0.0;  // this layer appends a ratio
      double kept = 0.0;
      for (int j = app && len >= a.p.R ? 1 : 0; j < len; ++j) kept += cs.fifo[j];
      const int nlen = app ? (len < a.p.R ? len + 1 : len) : len;
      for (int k = 1 + lane; k <= cap; k += 32) {
        const double uk = u[k];
        bool g;
        if (nlen <= 0) {
          g = false;  // the mean of an empty FIFO is NaN
        } else if (app && up > 0.0) {
          g = (kept * up + uk) * uk >= a.p.C2 * costp[k] * (double)nlen * up;
        } else if (app) {  // u_prev = 0: the ratio is not finite; the quotient form as written
          const double alpha = (kept + uk / up) / (double)nlen;
          g = alpha * uk >= a.p.C2 * costp[k];
        } else {
          g = kept * uk >= a.p.C2 * costp[k] * (double)nlen;
        }
        grow_k[k] = (a.d < a.p.D_max) && g;
      }
    } else if (w == 2 && up >= 0.0) {
      for (int k = 1 + lane; k <= cap; k += 32) ratio_k[k] = u[k] / up;
    }
  };
  int n = 0;
  if (cap > 0) n = selection_rule(items, costp, a.p.C1, cap, u, cimg, qimg, &s_k0, grow_for_all_widths);
  if (tid == 0) {
    bool grow = false;
    if (cap > 0) {
      if (cs.u_prev >= 0.0) {
        int len = cs.fifo_len;
        if (len < a.p.R) {
          cs.fifo[len++] = ratio_k[n];
        } else {
          for (int j = 1; j < len; ++j) cs.fifo[j - 1] = cs.fifo[j];
          cs.fifo[len - 1] = ratio_k[n];
        }
        cs.fifo_len = len;
      }
      grow = grow_k[n] != 0;
      cs.u_prev = u[n];
      cs.u_layer = u[n];
      cs.ctx_sum += n;
      *ws.cast = cs;
    }
    a.out.width[0] = n;
    s_grow = grow ? 1 : 0;
    s_width = n;
  }
  __syncthreads();
  for (int b = tid; b < a.B; b += blockDim.x) a.out.stop[b] = s_grow ? 0 : 1;
  if (a.select) {  // the next layer's frontier, as dt_select_frontier(width, stop) would choose it
    const int w_req = s_grow ? s_width : 0;
    if (f_pref) {
      if (warp < a.B)
        select_frontier_write(ws, warp, a.W, max(0, min(min(w_req, a.W), f_avail)), f_id, f_tok, f_val, a.ftok);
    } else {
      for (int b = warp; b < a.B; b += blockDim.x >> 5)
        select_frontier_warp(ws, b, a.N, a.W, a.LW, a.D, a.d, w_req, a.ftok);
    }
  }
}


// Graft page step (1), for request b after layer d: at checkpoint s (layer index d - 1), a request
// whose best path confidence exp(max value) is not above tau[s] stops with stage s and K_draft[s]
// nodes; a request that reaches D_max stops with stage n_ckpt and K_total nodes.
__device__ __forceinline__ void graft_checkpoint_one(const PruneArgs& a, int b) {
  if (a.out.stop[b]) return;
  const Workspace& ws = a.ws;
  const int li = a.d - 1;
  for (int s = 0; s < a.p.n_ckpt; ++s) {
    if (a.p.ckpt_layer[s] != li) continue;
    const int64_t lb = (int64_t)b * (a.D + 1) + a.d;
    double c = 0.0;
    if (ws.layer_count[lb] > 0) c = (double)expf(ws.layer_val[lb * a.LW]);
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

}  // namespace
}  // namespace dt
