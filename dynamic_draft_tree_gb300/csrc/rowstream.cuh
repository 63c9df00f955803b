// Warp-granular streaming row pass of the verify (one read of every used target row).
//
// A launch reads A "active rows" of V elements (request b owns cnt(b) consecutive rows, numbered
// j = 0..A-1 in request order). The rows, laid end to end, form E = A * V elements, which are cut
// into G contiguous, equal ranges of whole 16-byte vectors, one per warp. A warp streams its range
// through its own ring of shared-memory stages filled by cp.async (three 4 KB stages in flight per
// warp), crossing row boundaries without draining; for every row piece it reads, it leaves one
// partial result:
//   * softmax passes: the piece's max m and s = sum exp(x - m) as a double-float,
//   * the piece's top-K keys (logit desc, token id asc), K <= 32.
// Piece (row j, warp g) writes slot j + g: j and g both grow along the concatenation, so distinct
// pieces get distinct slots, and row j's pieces are the warps that own its first and last element
// and those between (at most kMaxPieces).
//
// No warp waits for another and no CTA synchronises: the kernel that consumes the rows (the verify
// walk) merges the pieces after the kernel boundary.
// Warps of different pieces of one row share a filter threshold through a per-row word (the best
// K-th key any of them has seen); the consuming kernel resets it.
#pragma once

#include "rowscan.cuh"

namespace dt {

constexpr int kStreamWarps = 8;                      // warps per CTA of a streaming pass
constexpr int kStreamThreads = 32 * kStreamWarps;
constexpr int kStreamCtasPerSm = 2;                  // one wave of CTAs (registers: <= 128 per thread)
constexpr int kBatchVec = 8;                         // 16-byte vectors per lane per batch
constexpr int64_t kMinPieceBytes = 12288;            // a warp's range is at least this long (one ring of stages)
constexpr int kMaxPieces = 32;                       // pieces per row at most (the merges hold them in smem)

// Dynamic shared memory of a streaming CTA: one WarpStream per warp (declared below).
constexpr size_t stream_smem_bytes();

// Pieces a row may be cut into for top-K lists of K keys: at most 512 keys per row in the merge.
__host__ __device__ __forceinline__ int stream_max_pieces(int K) {
  const int p = 512 / (K < 1 ? 1 : K);
  return p > kMaxPieces ? kMaxPieces : p;  // K <= 32: p >= 16
}

// Division by a per-launch constant d (1 <= d < 2^32) through a 64-bit reciprocal: one real
// division per thread, then a multiply-high and at most two corrections per quotient.
struct DivU64 {
  uint64_t d, inv;
  __device__ __forceinline__ explicit DivU64(uint64_t d_) : d(d_), inv(~0ull / d_) {}
  __device__ __forceinline__ uint64_t div(uint64_t x) const {
    uint64_t q = __umul64hi(x, inv);
    uint64_t r = x - q * d;
    while (r >= d) {
      ++q;
      r -= d;
    }
    return q;
  }
};

// The streaming split: E elements in chunks of `chunk` elements (a whole number of 16-byte vectors,
// chunk >= E / G), warp g reading [g * chunk, min(E, (g + 1) * chunk)). The warp that reads element x
// is x / chunk.
__device__ __forceinline__ int64_t stream_chunk(int64_t E, int64_t G, int vecel) {
  const int64_t c = (E + G - 1) / G;
  return (c + vecel - 1) / vecel * vecel;
}

// Warps of a launch with work: enough that each reads kMinPieceBytes, no more than the grid's warps,
// and few enough that a row has at most `maxp` pieces (maxp >= 4): with G <= (maxp - 3) A every range
// holds at least V / (maxp - 3) - 8 elements, and a row of V elements meets at most
// floor((V - 1) / range) + 2 ranges. Every consumer computes the same G from the same totals.
__device__ __forceinline__ int64_t stream_warps(int64_t A, int64_t V, int esz, int64_t Gtot, int maxp) {
  if (A <= 0) return 0;
  int64_t G = A * V * esz / kMinPieceBytes;
  G = min(G, Gtot);
  G = min(G, (int64_t)(maxp - 3) * A);
  return max(G, (int64_t)1);
}

// Sum of cnt(b) over all requests (every lane gets it). All lanes of the warp call it.
template <class Cnt>
__device__ __forceinline__ int64_t warp_total_rows(int B, Cnt cnt) {
  const int lane = threadIdx.x & 31;
  int64_t A = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int c = (b0 + lane < B) ? cnt(b0 + lane) : 0;
    A += __reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
  }
  return A;
}

// Request b and row i of active row j (warp-uniform result). All lanes call it.
template <class Cnt>
__device__ __forceinline__ void warp_find_row(int B, int64_t j, Cnt cnt, int& b_out, int& i_out) {
  const int lane = threadIdx.x & 31;
  int64_t base = 0;
  b_out = B;
  i_out = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int n = (b0 + lane < B) ? cnt(b0 + lane) : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t lo = base + incl - n;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, n > 0 && lo <= j && j < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      b_out = b0 + src;
      i_out = __shfl_sync(0xFFFFFFFFu, (int)(j - lo), src);
      return;
    }
    base += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
}

// Exclusive prefix of cnt(b) over requests before b (all lanes call it; every lane gets it).
template <class Cnt>
__device__ __forceinline__ int64_t warp_rows_before(int b, Cnt cnt) {
  const int lane = threadIdx.x & 31;
  int64_t s = 0;
  for (int b0 = 0; b0 < b; b0 += 32) {
    const int c = (b0 + lane < b) ? cnt(b0 + lane) : 0;
    s += __reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
  }
  return s;
}

// Result of one row piece, in the lanes of the warp that read it: keys in rg.list[lb][0..nl),
// softmax statistics (every lane), and flags.
struct PieceOut {
  int nl, lb;
  float m, s_hi, s_lo;  // softmax passes: max and sum exp(x - m); otherwise m = the best value
  bool bad;             // a NaN or +inf was seen
  bool internal;        // an overflow refinement bound was hit
};

// ---------------------------------------------------------------- per-warp copy ring ----
// Every lane copies its own 16-byte vectors of a stage into the warp's ring with cp.async (completion
// tracked per thread by commit groups), then reads back only those vectors: no lane reads another
// lane's copies, so the ring needs no barrier. kRingStages stages of 4 KB are in flight per warp.
constexpr int kRingStages = 3;
constexpr int kStageVec = 32 * kBatchVec;  // vectors per stage (4 KB)
constexpr int kMaxSeg = 4;                 // row pieces of a warp described at a time

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One row piece of a warp's range.
struct SegDesc {
  const void* row;  // the row (null: not read, nothing published)
  int64_t s0, s1;   // element range [s0, s1) of the row
  int64_t a0;       // first 16-byte aligned element of the range
  int64_t nvec;     // aligned vectors
  int64_t j;        // active row index
  int32_t b, i;     // request, row of the request
  int32_t st0, nst; // its stages in the warp's stage sequence
};

struct WarpStream {
  WarpRing rg;                            // top-K list and candidate buffer
  SegDesc seg[kMaxSeg];
  uint4 ring[kRingStages][kStageVec];     // the copy ring
};
constexpr size_t stream_smem_bytes() { return sizeof(WarpStream) * kStreamWarps; }

// Pushes into the warp's candidate buffer the elements of this lane's vectors of one stage (ring slot
// sp) whose value is >= tv (and not -inf) and whose key exceeds tk. Vector q of this lane is
// sp[q * 32 + lane] (if q * 32 + lane < nv); its element e has id e0 + (q * 32 + lane) * VEC + e.
// Out of line: one copy of this rarely run code serves every call site.
template <typename T>
static __device__ __noinline__ void push_from_ring(WarpRing& rg, const uint4* sp, int nv, int64_t e0, unsigned qmask,
                                                   float tv, uint64_t tk) {
  constexpr int VEC = Elt<T>::kVec;
  const int lane = threadIdx.x & 31;
  while (qmask) {
    const int q = __ffs(qmask) - 1;
    qmask &= qmask - 1;
    const int vi = q * 32 + lane;
    if (vi >= nv) break;
    const uint4 w = sp[vi];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float x = vec_elt<T>(w, e);
      if (x >= tv && x != -INFINITY) {
        const uint64_t k = make_key(x, (uint32_t)(e0 + (int64_t)vi * VEC + e));
        if (k > tk) {
          const int pos = atomicAdd(&rg.cnt, 1);
          if (pos < kWarpCand) rg.cand[pos] = k;
        }
      }
    }
  }
  __syncwarp();
}

// Issues stage t of the warp's stage sequence (all lanes; a stage past the end issues nothing), then
// commits a group (possibly empty).
template <typename T>
__device__ __forceinline__ void ring_issue(WarpStream& ws_, int nseg, int t) {
  const int lane = threadIdx.x & 31;
  for (int s = 0; s < nseg; ++s) {
    const SegDesc& sd = ws_.seg[s];
    if (t < sd.st0 || t >= sd.st0 + sd.nst) continue;
    const int u = t - sd.st0;
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(sd.row) + sd.a0);
    uint4* dst = ws_.ring[t % kRingStages];
#pragma unroll
    for (int q = 0; q < kBatchVec; ++q) {
      const int64_t vi = (int64_t)u * kStageVec + q * 32 + lane;
      if (vi < sd.nvec) cp_async16(dst + q * 32 + lane, src + vi);
    }
    break;
  }
  cp_async_commit();
}

// The streaming pass of one launch, for warp g of the grid. cnt(b): rows of request b;
// row_of(b, i, j): row i of request b, the j-th row of the pass, or null when it is not to be read
// (no partial is written);
// publish(j, g, b, i, out): called by all lanes after each piece, with rg.list holding its keys.
// The warp's range is described kMaxSeg pieces at a time; the ring runs on across the pieces of a
// description.
template <typename T, bool SOFTMAX, class Cnt, class RowOf, class Publish>
__device__ void stream_rows(int B, int64_t V, int K, int maxp, int64_t Gtot, WarpStream& wsm,
                            unsigned long long* row_tau, Cnt cnt, RowOf row_of, Publish publish) {
  constexpr int VEC = Elt<T>::kVec;
  constexpr int ESZ = (int)sizeof(T);
  constexpr int NV = kBatchVec * VEC;  // values per lane per stage
  const int lane = threadIdx.x & 31;
  WarpRing& rg = wsm.rg;
  const int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t A = warp_total_rows(B, cnt);
  const int64_t G = stream_warps(A, V, ESZ, Gtot, maxp);
  if (g >= G) return;
  const int64_t E = A * V;
  const int64_t chunk = stream_chunk(E, G, VEC);
  const int64_t x0 = g * chunk, x1 = min(E, x0 + chunk);
  if (x0 >= x1) return;
  int64_t j = x0 / V;
  int b, i;
  warp_find_row(B, j, cnt, b, i);
  const uint32_t neg_fill = ESZ == 2 ? 0xFF80FF80u : 0xFF800000u;

  for (int64_t x = x0; x < x1;) {
    // ---- describe up to kMaxSeg pieces (warp-uniform; lane 0 stores them) ----
    int nseg = 0, nst_tot = 0;
    while (nseg < kMaxSeg && x < x1) {
      SegDesc sd;
      sd.s0 = x - j * V;
      sd.s1 = min(V, x1 - j * V);
      sd.j = j;
      sd.b = b;
      sd.i = i;
      const T* row = b < B ? row_of(b, i, j) : nullptr;
      sd.row = row;
      sd.a0 = sd.s0;
      sd.nvec = 0;
      sd.st0 = nst_tot;
      sd.nst = 0;
      if (row) {
        const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + sd.s0);
        sd.a0 = min(sd.s1, sd.s0 + (int64_t)(((16u - (uint32_t)(addr0 & 15u)) & 15u) / ESZ));
        sd.nvec = ((sd.s1 - sd.a0) * ESZ) / 16;
        sd.nst = (int)((sd.nvec + kStageVec - 1) / kStageVec);
      }
      nst_tot += sd.nst;
      if (lane == 0) wsm.seg[nseg] = sd;
      ++nseg;
      x = (j + 1) * V;
      ++j;
      if (x >= x1) break;
      ++i;  // next row: the next request with rows once this one's are done
      while (b < B && i >= cnt(b)) {
        ++b;
        i = 0;
      }
    }
    __syncwarp();
    // ---- the ring: a stage is issued as soon as its slot is free, i.e. once the stage that held it
    // (kRingStages earlier) is released: after its processing, or, for the first stages of a piece
    // (filtered together), after that filter ----
    int next_issue = 0, released = 0;
    auto refill = [&]() {
      const int lim = min(released + kRingStages, nst_tot);
      while (next_issue < lim) ring_issue<T>(wsm, nseg, next_issue++);
    };
    refill();
    for (int si = 0; si < nseg; ++si) {
      const SegDesc sd = wsm.seg[si];
      if (!sd.row) continue;
      unsigned long long* gtau = row_tau ? row_tau + sd.j : nullptr;
      if (lane == 0) rg.cnt = 0;
      __syncwarp();
      float m_t = -INFINITY, s_hi = 0.0f, s_lo = 0.0f;
      float seen_max = -INFINITY;
      int lb = 0, nl = 0;
      uint64_t tau_key = 0ull;
      bool internal = false;
      auto merge = [&](bool dedup) -> bool {
        const ListState o = warp_list_merge(rg, K, nl, lb, dedup);
        nl = o.nl;
        lb = o.lb;
        tau_key = o.tau_key;
        return o.overflow != 0;
      };
      // head + tail elements (< 16 bytes at each end): one per lane, softmax now, keys after the stream
      const T* row = reinterpret_cast<const T*>(sd.row);
      const int64_t a1 = sd.a0 + sd.nvec * VEC;
      const int n_head = (int)(sd.a0 - sd.s0), n_tail = (int)(sd.s1 - a1);
      uint64_t ht_key = 0ull;
      if (lane < n_head + n_tail) {
        const int64_t idx = lane < n_head ? sd.s0 + lane : a1 + (lane - n_head);
        const float xv = Elt<T>::load(row + idx);
        if (SOFTMAX) lane_acc_one(xv, m_t, s_hi, s_lo);
        else seen_max = xv;
        if (!(xv != xv)) ht_key = make_key(xv, (uint32_t)idx);
      }
      uint64_t gt = gtau ? (uint64_t)__ldcg(gtau) : 0ull;
      uint64_t gt_next = gt;
      // the first nb stages (all of a piece that fits the ring; else the first stage) are filtered
      // together once they are all in: against the K-th largest lane maximum over them, one merge
      const int nb = sd.nst <= kRingStages ? sd.nst : 1;  // a longer piece filters its first stage alone
      float bmax = -INFINITY;  // lane maximum over the first nb stages (NaN skipped)
      for (int u = 0; u < sd.nst; ++u) {
        const int t = sd.st0 + u;
        gt = gt_next;  // the row's shared threshold, read one stage ahead
        if (gtau && u + 1 < sd.nst) gt_next = (uint64_t)__ldcg(gtau);
        refill();
        {  // this lane's copies of stage t have landed (at most next_issue - 1 - t later groups pending)
          const int pend = next_issue - 1 - t;
          if (pend >= 2) cp_async_wait<2>();
          else if (pend == 1) cp_async_wait<1>();
          else cp_async_wait<0>();
        }
        const uint4* sp = wsm.ring[t % kRingStages];
        const int nv = (int)min((int64_t)kStageVec, sd.nvec - (int64_t)u * kStageVec);
        uint32_t wv[kBatchVec * 4];
#pragma unroll
        for (int q = 0; q < kBatchVec; ++q) {
          uint4 w = make_uint4(neg_fill, neg_fill, neg_fill, neg_fill);
          if (q * 32 + lane < nv) w = sp[q * 32 + lane];
          wv[4 * q + 0] = w.x;
          wv[4 * q + 1] = w.y;
          wv[4 * q + 2] = w.z;
          wv[4 * q + 3] = w.w;
        }
        // lane max with NaN propagation; its first two levels give each vector's maximum
        float lm;
        float vmax[kBatchVec];
        {
          uint32_t r[kBatchVec * 4];
#pragma unroll
          for (int q = 0; q < kBatchVec * 4; ++q) r[q] = wv[q];
#pragma unroll
          for (int w2 = 1; w2 < kBatchVec * 4; w2 <<= 1) {
#pragma unroll
            for (int q = 0; q + w2 < kBatchVec * 4; q += 2 * w2)
              r[q] = ESZ == 2 ? max_nan_bf16x2(r[q], r[q + w2]) : max_nan_f32u(r[q], r[q + w2]);
            if (w2 == 2) {
#pragma unroll
              for (int q = 0; q < kBatchVec; ++q)
                vmax[q] = ESZ == 2 ? max_nan_f32(bf16_lo(r[4 * q]), bf16_hi(r[4 * q])) : __uint_as_float(r[4 * q]);
            }
          }
          lm = ESZ == 2 ? max_nan_f32(bf16_lo(r[0]), bf16_hi(r[0])) : __uint_as_float(r[0]);
        }
        if (!SOFTMAX) seen_max = max_nan_f32(seen_max, lm);
        if (SOFTMAX) {
          if (lm > m_t) {
            if (m_t != -INFINITY) {
              const float sc = ex2((m_t - lm) * kLog2e);
              s_hi *= sc;
              s_lo *= sc;
            }
            m_t = lm;
          }
          if (lm != lm) {
            s_hi = lm;  // NaN poisons the sum
          } else if (m_t != -INFINITY) {
            float part = 0.0f;
#pragma unroll
            for (int c = 0; c < NV / 16; ++c) {
              float e[16];
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                const int v = c * 16 + q;
                float xv;
                if (ESZ == 2) xv = (v & 1) ? bf16_hi(wv[v >> 1]) : bf16_lo(wv[v >> 1]);
                else xv = __uint_as_float(wv[v]);
                e[q] = ex2((xv - m_t) * kLog2e);
              }
#pragma unroll
              for (int w2 = 1; w2 < 16; w2 <<= 1)
#pragma unroll
                for (int q = 0; q + w2 < 16; q += 2 * w2) e[q] += e[q + w2];
              part += e[0];
            }
            const float y = part - s_lo;
            const float tt = s_hi + y;
            s_lo = (tt - s_hi) - y;
            s_hi = tt;
          }
        }
        const int64_t be0 = sd.a0 + (int64_t)u * kStageVec * VEC;  // id of the stage's first element
        if (u < nb) {
          bmax = fmaxf(bmax, lm);  // (later stages release their slot after processing, below)
          if (u + 1 == nb) {
            // threshold: the K-th largest lane maximum over the nb stages (K lanes hold an element at or
            // above it, so nothing below it is in the top-K), or the row's shared threshold if larger (a
            // key equal to that one is not in this piece: the warp has published nothing yet)
            uint64_t tk = gt;
            float tv = fmaxf(warp_kth_largest(bmax, K), gt ? key_value(gt) : -INFINITY);
            if (__any_sync(0xFFFFFFFFu, bmax >= tv)) {
              auto push_batch = [&](float tv_, uint64_t tk_) {
                const unsigned qm = bmax >= tv_ ? 0xFFu : 0u;
                for (int v = 0; v < nb; ++v) {
                  const int nvv = (int)min((int64_t)kStageVec, sd.nvec - (int64_t)v * kStageVec);
                  push_from_ring<T>(rg, wsm.ring[(sd.st0 + v) % kRingStages], nvv,
                                    sd.a0 + (int64_t)v * kStageVec * VEC, qm, tv_, tk_);
                }
              };
              push_batch(tv, tk);
              bool overflow = merge(false);
              for (int round = 1; overflow; ++round) {
                if (round > nb * NV * 32 / (kWarpCand - kMaxK) + 1) {  // the key rises every round: never hit
                  internal = true;
                  break;
                }
                tk = tau_key;
                tv = key_value(tau_key);
                push_batch(tv, tk);
                overflow = merge(true);
              }
              if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
            }
            __syncwarp();
            released = sd.st0 + nb;  // the batch's slots may be refilled
          }
        } else {
          // later stages: against the larger of the list's K-th key and the row's shared threshold.
          // Ids grow stage by stage within the piece, so a value equal to the warp's own K-th key's
          // value cannot beat it: strict against the own key, not against another warp's. The
          // candidates accumulate in the buffer and are merged at the end of the piece, or as soon as
          // K of them wait (greedy passes) or the buffer is half full (softmax passes); then the
          // threshold rises for the stages that follow, and the stage is filtered again, keys already
          // in the list dropped by the merge. Both limits are the faster one measured for their pass:
          // merging at K keeps a greedy pass's later stages cold; a softmax pass's stages cost more
          // than the extra merges save.
          for (int round = 0;; ++round) {
            uint64_t tk = tau_key;
            bool own = true;
            if (gt > tk) {
              tk = gt;
              own = false;
            }
            const float tv = tk ? key_value(tk) : -INFINITY;
            const bool hot = own ? (lm > tv) : (lm >= tv);
            if (!__any_sync(0xFFFFFFFFu, hot)) break;
            unsigned qm = 0u;
            if (hot) {
#pragma unroll
              for (int q = 0; q < kBatchVec; ++q)
                if (own ? (vmax[q] > tv) : (vmax[q] >= tv)) qm |= 1u << q;
            }
            push_from_ring<T>(rg, sp, nv, be0, qm, tv, tk);
            if (rg.cnt < (SOFTMAX ? kWarpCand / 2 : K)) break;  // deferred: merged later
            // a stage filtered again after an overflow pushes keys the list already holds: every
            // merge of deferred keys drops those first
            const bool overflow = merge(true);
            if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
            if (!overflow) break;
            if (round >= NV * 32 / (kWarpCand - kMaxK) + 1) {
              internal = true;
              break;
            }
          }
          released = t + 1;
        }
      }
      // the deferred candidates and the head/tail elements join after the stream (the buffer holds
      // fewer than kWarpCand / 2 deferred keys, so the at most 32 head/tail keys fit)
      if (ht_key) {
        const int pos = atomicAdd(&rg.cnt, 1);
        if (pos < kWarpCand) rg.cand[pos] = ht_key;
      }
      __syncwarp();
      if (rg.cnt > 0) merge(true);
      PieceOut out;
      out.nl = nl;
      out.lb = lb;
      out.internal = internal;
      out.bad = SOFTMAX ? __any_sync(0xFFFFFFFFu, s_hi != s_hi || m_t == INFINITY)
                        : __any_sync(0xFFFFFFFFu, seen_max != seen_max || seen_max == INFINITY);
      if (SOFTMAX) {
        float wm = m_t;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, o));
        const bool wnan = __any_sync(0xFFFFFFFFu, s_hi != s_hi);
        float ch = 0.0f, cl = 0.0f;
        if (m_t != -INFINITY && !(s_hi != s_hi)) {
          ch = s_hi;
          cl = s_lo;
          if (wm != m_t) ff_scale(ch, cl, ex2((m_t - wm) * kLog2e));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(0xFFFFFFFFu, ch, o);
          const float ol = __shfl_xor_sync(0xFFFFFFFFu, cl, o);
          ff_add(ch, cl, oh, ol);
        }
        out.m = wm;
        out.s_hi = wnan ? __int_as_float(0x7FC00000) : ch;
        out.s_lo = wnan ? 0.0f : cl;
      } else {
        out.m = nl > 0 ? key_value(rg.list[lb][0]) : -INFINITY;
        out.s_hi = out.s_lo = 0.0f;
      }
      publish(sd.j, g, sd.b, sd.i, out);
      __syncwarp();
    }
    cp_async_wait<0>();  // the description's copies are all consumed (only empty groups remain)
    __syncwarp();
  }
}

// Writes one piece's partial: keys (lanes < K), max and sum (lane 0).
__device__ __forceinline__ void publish_partial(Partial* p, const WarpRing& rg, const PieceOut& o, int K) {
  const int lane = threadIdx.x & 31;
  if (lane < K) p->keys[lane] = lane < o.nl ? rg.list[o.lb][lane] : 0ull;
  if (lane == 0) {
    p->m = o.m;
    p->s_hi = o.s_hi;
    p->s_lo = o.s_lo;
  }
}

// ---- consumer side: merging the pieces of one row (one warp) ----

// Row j's pieces: slots j + g for the warps g in [g0, g1] that read its first and last element.
struct RowPieces {
  int64_t slot0;
  int S;
};
struct PieceMap {
  int64_t V;
  DivU64 div;  // by the chunk length
  __device__ __forceinline__ PieceMap(int64_t A, int64_t V_, int64_t G, int vecel)
      : V(V_), div((uint64_t)max(stream_chunk(A * V_, max(G, (int64_t)1), vecel), (int64_t)1)) {}
  __device__ __forceinline__ RowPieces row(int64_t j) const {
    const int64_t g0 = (int64_t)div.div((uint64_t)(j * V)), g1 = (int64_t)div.div((uint64_t)(j * V + V - 1));
    RowPieces r;
    r.slot0 = j + g0;
    r.S = (int)(g1 - g0 + 1);
    return r;
  }
};

// The K-th largest (K <= 32) of the 32 lane keys (distinct, or 0); every lane gets it.
__device__ __forceinline__ uint64_t warp_kth_largest_key(uint64_t v, int K) {
  const int lane = threadIdx.x & 31;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint64_t o = shfl_u64(v, j);
    rank += (o > v) | ((o == v) & (j < lane));
  }
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, rank == K - 1);
  return shfl_u64(v, __ffs(hit) - 1);
}

// Merges the S (<= 32) partials of one row into its top-K keys (top: K keys out, descending,
// 0-padded) and its softmax statistics (every lane gets M and the double-float S; a NaN sum poisons
// it). The S lists (descending, K keys each; at most 256 keys) are staged in the warp's scratch
// `cand` (cap keys) with one round of loads. Every key of the row's top-K is at least T, the K-th largest of the S list
// heads (those are K distinct keys of the row), so only keys >= T are ranked: a key's place is the
// number of staged keys above it. When the lists do not fit the scratch the top-K is taken by K
// rounds of "largest remaining head" instead. All lanes call it.
__device__ __forceinline__ void warp_merge_row(const Partial* __restrict__ parts, int S, int K, uint64_t* cand,
                                               int cap, uint64_t* top, bool softmax, float& M, float& sh,
                                               float& sl) {
  const int lane = threadIdx.x & 31;
  float m0 = -INFINITY, h0 = 0.0f, l0 = 0.0f;
  if (softmax && lane < S) {
    m0 = parts[lane].m;
    h0 = parts[lane].s_hi;
    l0 = parts[lane].s_lo;
  }
  const int n_all = S * K;
  if (n_all <= cap && n_all <= 256) {
    // every key staged with one round of independent loads; the heads are cand[s * K]. idx / K is
    // (idx * ceil(2^16 / K)) >> 16, exact for idx < 512 and K <= 32.
    const uint32_t invK = (65536u + (uint32_t)K - 1u) / (uint32_t)K;
    uint64_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = lane + 32 * u;
      const int sidx = (int)(((uint32_t)t * invK) >> 16);
      v[u] = t < n_all ? parts[sidx].keys[t - sidx * K] : 0ull;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (lane + 32 * u < n_all) cand[lane + 32 * u] = v[u];
    __syncwarp();
    const uint64_t head = lane < S ? cand[lane * K] : 0ull;
    const uint64_t T = S >= K ? warp_kth_largest_key(head, K) : 1ull;
    if (lane < K) top[lane] = 0ull;
    // the candidates (keys >= T), compacted to the front of the scratch from the registers
    int mc = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) mc += (v[u] >= T) & (v[u] != 0ull);
    int off = mc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, off, o);
      if (lane >= o) off += t;
    }
    const int n = __shfl_sync(0xFFFFFFFFu, off, 31);
    off -= mc;
    __syncwarp();  // every lane has read its head from the staged keys
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if ((v[u] >= T) & (v[u] != 0ull)) cand[off++] = v[u];
    __syncwarp();
    for (int t = lane; t < n; t += 32) {
      const uint64_t k = cand[t];
      int rank = 0;  // every key above k is >= T too, so it is a candidate
      for (int q = 0; q < n; ++q) rank += cand[q] > k;
      if (rank < K) top[rank] = k;
    }
  } else {
    // rounds of "take the largest remaining head" (lane s's head is its list's key at pos)
    if (lane < K) top[lane] = 0ull;
    const uint64_t* mine = parts[lane < S ? lane : 0].keys;
    int pos = 0;
    for (int r = 0; r < K; ++r) {
      const uint64_t h = (lane < S && pos < K) ? mine[pos] : 0ull;
      uint64_t best = h;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = shfl_xor_u64(best, o);
        best = x > best ? x : best;
      }
      if (best == 0ull) break;
      if (lane == 0) top[r] = best;
      if (h == best) ++pos;
    }
  }
  M = -INFINITY;
  sh = sl = 0.0f;
  if (softmax) {
    float bm = m0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
    bool nan = h0 != h0;
    float h = 0.0f, l = 0.0f;
    if (!nan && m0 != -INFINITY) {
      ff_scale(h0, l0, ex2((m0 - bm) * kLog2e));
      h = h0;
      l = l0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oh = __shfl_xor_sync(0xFFFFFFFFu, h, o);
      const float ol = __shfl_xor_sync(0xFFFFFFFFu, l, o);
      ff_add(h, l, oh, ol);
    }
    nan = __any_sync(0xFFFFFFFFu, nan);
    M = bm;
    sh = nan ? __int_as_float(0x7FC00000) : h;
    sl = nan ? 0.0f : l;
  }
  __syncwarp();
}

}  // namespace dt
