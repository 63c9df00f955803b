// Warp-granular streaming row pass, shared by the expansion and the verify.
//
// A launch reads A "active rows" of V elements (request b owns cnt(b) consecutive rows, numbered
// j = 0..A-1 in request order). The rows, laid end to end, form E = A * V elements, which are cut
// into G contiguous, equal ranges of whole 16-byte vectors, one per warp. A warp streams its range
// with plain vector loads (8 vectors of 16 bytes per lane in flight, 4 KB per warp), crossing row
// boundaries without stopping; for every row piece it reads, it leaves one partial result:
//   * softmax passes: the piece's max m and s = sum exp(x - m) as a double-float,
//   * the piece's top-K keys (logit desc, token id asc), K <= 32.
// Piece (row j, warp g) writes slot j + g: j and g both grow along the concatenation, so distinct
// pieces get distinct slots, and row j's pieces are the warps that own its first and last element
// and those between (at most kMaxPieces).
//
// No warp waits for another and no CTA synchronises: the kernel that consumes the rows (the
// expansion's finishing kernel, the verify walk) merges the pieces after the kernel boundary.
// Warps of different pieces of one row share a filter threshold through a per-row word (the best
// K-th key any of them has seen); the consuming kernel resets it.
#pragma once

#include "rowscan.cuh"

namespace dt {

constexpr int kStreamWarps = 8;                      // warps per CTA of a streaming pass
constexpr int kStreamThreads = 32 * kStreamWarps;
constexpr int kStreamCtasPerSm = 2;                  // one wave of CTAs (registers: <= 128 per thread)
constexpr int kBatchVec = 8;                         // 16-byte vectors per lane per batch
constexpr int64_t kMinPieceBytes = 16384;            // a warp's range is at least this long when E allows
constexpr int kMaxPieces = 32;                       // pieces per row at most (the merges hold them in smem)

// Pieces a row may be cut into for top-K lists of K keys: at most 512 keys per row in the merge.
__host__ __device__ __forceinline__ int stream_max_pieces(int K) {
  const int p = 512 / (K < 1 ? 1 : K);
  return p > kMaxPieces ? kMaxPieces : p;  // K <= 32: p >= 16
}

// Split of E elements among G warps: warp g reads [wr_start(g), wr_start(g + 1)), boundaries rounded
// down to whole vectors of `vecel` elements (E/G >= vecel holds for every launch).
__device__ __forceinline__ int64_t wr_start(int64_t g, int64_t E, int64_t G, int vecel) {
  if (g <= 0) return 0;
  if (g >= G) return E;
  return range_start(g, E, G) / vecel * vecel;
}
// The warp whose range holds element x.
__device__ __forceinline__ int64_t wr_owner(int64_t x, int64_t E, int64_t G, int vecel) {
  int64_t c = cta_of(x, E, G);
  if (c + 1 < G && wr_start(c + 1, E, G, vecel) <= x) ++c;
  return c;
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

// Pushes into the warp's candidate buffer the elements of this lane's vectors of one batch whose
// value is >= tv (and not -inf) and whose key exceeds tk; the vectors are read again from global
// memory (they were just loaded: a cache hit). Lanes without `scan` push nothing. Vector q of this
// lane is vp[q * 32 + lane] (if q * 32 + lane < nv); its element e has id e0 + (q * 32 + lane) * VEC + e.
// Out of line: one copy of this rarely run code serves every call site.
template <typename T>
static __device__ __noinline__ void push_from_global(WarpRing& rg, const uint4* __restrict__ vp, int64_t nv,
                                                     int64_t e0, unsigned qmask, float tv, uint64_t tk) {
  constexpr int VEC = Elt<T>::kVec;
  const int lane = threadIdx.x & 31;
  while (qmask) {
    const int q = __ffs(qmask) - 1;
    qmask &= qmask - 1;
    const int64_t vi = (int64_t)q * 32 + lane;
    if (vi >= nv) break;
    const uint4 w = __ldg(vp + vi);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float x = vec_elt<T>(w, e);
      if (x >= tv && x != -INFINITY) {
        const uint64_t k = make_key(x, (uint32_t)(e0 + vi * VEC + e));
        if (k > tk) {
          const int pos = atomicAdd(&rg.cnt, 1);
          if (pos < kWarpCand) rg.cand[pos] = k;
        }
      }
    }
  }
  __syncwarp();
}

// One warp reads elements [s0, s1) of `row` (K <= kMaxK). All lanes call it; rg is the warp's own
// list state in shared memory. gtau: the row's shared threshold word, or null.
template <typename T, bool SOFTMAX>
__device__ PieceOut stream_piece(const T* __restrict__ row, int64_t s0, int64_t s1, int K, WarpRing& rg,
                                 unsigned long long* gtau) {
  constexpr int VEC = Elt<T>::kVec;
  constexpr int ESZ = (int)sizeof(T);
  constexpr int NV = kBatchVec * VEC;  // values per lane per batch
  const int lane = threadIdx.x & 31;
  const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + s0);
  int64_t a0 = s0 + (int64_t)(((16u - (uint32_t)(addr0 & 15u)) & 15u) / ESZ);
  if (a0 > s1) a0 = s1;
  const int64_t nvec = ((s1 - a0) * ESZ) / 16;
  const int64_t a1 = a0 + nvec * VEC;
  const uint4* __restrict__ vp = reinterpret_cast<const uint4*>(row + a0);
  if (lane == 0) rg.cnt = 0;
  __syncwarp();

  float m_t = -INFINITY, s_hi = 0.0f, s_lo = 0.0f;
  float seen_max = -INFINITY;
  int lb = 0, nl = 0;
  uint64_t tau_key = 0ull;
  bool internal = false;

  // head + tail elements (< 16 bytes at each end): one per lane, softmax now, keys after the stream
  const int n_head = (int)(a0 - s0), n_tail = (int)(s1 - a1);
  uint64_t ht_key = 0ull;
  if (lane < n_head + n_tail) {
    const int64_t idx = lane < n_head ? s0 + lane : a1 + (lane - n_head);
    const float x = Elt<T>::load(row + idx);
    if (SOFTMAX) lane_acc_one(x, m_t, s_hi, s_lo);
    else seen_max = x;
    if (!(x != x)) ht_key = make_key(x, (uint32_t)idx);
  }

  auto merge = [&](bool dedup) -> bool {
    const ListState o = warp_list_merge(rg, K, nl, lb, dedup);
    nl = o.nl;
    lb = o.lb;
    tau_key = o.tau_key;
    return o.overflow != 0;
  };

  const uint32_t neg_fill = ESZ == 2 ? 0xFF80FF80u : 0xFF800000u;
  uint64_t gt = gtau ? (uint64_t)__ldcg(gtau) : 0ull;
  for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kBatchVec) {
    const int64_t nv = min((int64_t)(32 * kBatchVec), nvec - v0);  // vectors in this batch
    uint32_t wv[kBatchVec * 4];
#pragma unroll
    for (int q = 0; q < kBatchVec; ++q) {
      const int64_t vi = (int64_t)q * 32 + lane;
      uint4 w = make_uint4(neg_fill, neg_fill, neg_fill, neg_fill);
      if (vi < nv) w = __ldg(vp + v0 + vi);
      wv[4 * q + 0] = w.x;
      wv[4 * q + 1] = w.y;
      wv[4 * q + 2] = w.z;
      wv[4 * q + 3] = w.w;
    }
    if (v0 > 0 && gtau) gt = (uint64_t)__ldcg(gtau);

    // lane max with NaN propagation; its first two levels give each vector's maximum
    float lm;
    float vmax[kBatchVec];
    {
      uint32_t r[kBatchVec * 4];
#pragma unroll
      for (int j = 0; j < kBatchVec * 4; ++j) r[j] = wv[j];
#pragma unroll
      for (int w2 = 1; w2 < kBatchVec * 4; w2 <<= 1) {
#pragma unroll
        for (int j = 0; j + w2 < kBatchVec * 4; j += 2 * w2)
          r[j] = ESZ == 2 ? max_nan_bf16x2(r[j], r[j + w2]) : max_nan_f32u(r[j], r[j + w2]);
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
          for (int j = 0; j < 16; ++j) {
            const int v = c * 16 + j;
            float x;
            if (ESZ == 2) x = (v & 1) ? bf16_hi(wv[v >> 1]) : bf16_lo(wv[v >> 1]);
            else x = __uint_as_float(wv[v]);
            e[j] = ex2((x - m_t) * kLog2e);
          }
#pragma unroll
          for (int w2 = 1; w2 < 16; w2 <<= 1)
#pragma unroll
            for (int j = 0; j + w2 < 16; j += 2 * w2) e[j] += e[j + w2];
          part += e[0];
        }
        const float y = part - s_lo;
        const float tt = s_hi + y;
        s_lo = (tt - s_hi) - y;
        s_hi = tt;
      }
    }

    const int64_t be0 = a0 + v0 * VEC;  // id of the batch's first element
    if (v0 == 0) {
      // first batch: threshold = the K-th largest lane maximum (K lanes hold an element at or above
      // it, so nothing below it is in the top-K), or the row's shared threshold if larger (a key equal
      // to that one is not in this piece: the warp has published nothing yet)
      uint64_t tk = gt;
      float tv = fmaxf(warp_kth_largest(lm, K), gt ? key_value(gt) : -INFINITY);
      if (__any_sync(0xFFFFFFFFu, lm >= tv)) {
        unsigned qm = 0u;
#pragma unroll
        for (int q = 0; q < kBatchVec; ++q)
          if (vmax[q] >= tv) qm |= 1u << q;
        if (!(lm >= tv)) qm = 0u;
        push_from_global<T>(rg, vp + v0, nv, be0, qm, tv, tk);
        bool overflow = merge(false);
        for (int round = 1; overflow; ++round) {
          if (round > NV * 32 / (kWarpCand - kMaxK) + 1) {  // the key rises every round: never hit
            internal = true;
            break;
          }
          tk = tau_key;
          tv = key_value(tau_key);
          push_from_global<T>(rg, vp + v0, nv, be0, lm >= tv ? qm : 0u, tv, tk);
          overflow = merge(true);
        }
        if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
      }
    } else {
      // later batches: the larger of the list's K-th key and the row's shared threshold. Ids grow
      // batch by batch within the piece, so a value equal to the warp's own K-th key's value cannot
      // beat it: strict against the own key, not against another warp's.
      bool dedup = false;
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
        push_from_global<T>(rg, vp + v0, nv, be0, qm, tv, tk);
        const bool overflow = merge(dedup);
        dedup = true;
        if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
        if (!overflow) break;
        if (round >= NV * 32 / (kWarpCand - kMaxK) + 1) {
          internal = true;
          break;
        }
      }
    }
  }
  if (__any_sync(0xFFFFFFFFu, ht_key != 0ull)) {  // head/tail elements join after the stream
    if (ht_key) {
      const int pos = atomicAdd(&rg.cnt, 1);
      if (pos < kWarpCand) rg.cand[pos] = ht_key;
    }
    merge(false);
  }

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
  return out;
}

// The streaming pass of one launch, for warp g of the grid. cnt(b): rows of request b;
// row_of(b, i): row i of request b, or null when it is not to be read (no partial is written);
// publish(j, g, b, i, out): called by all lanes after each piece, with rg.list holding its keys.
template <typename T, bool SOFTMAX, class Cnt, class RowOf, class Publish>
__device__ void stream_rows(int B, int64_t V, int K, int maxp, int64_t Gtot, WarpRing& rg,
                            unsigned long long* row_tau, Cnt cnt, RowOf row_of, Publish publish) {
  constexpr int VEC = Elt<T>::kVec;
  const int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t A = warp_total_rows(B, cnt);
  const int64_t G = stream_warps(A, V, (int)sizeof(T), Gtot, maxp);
  if (g >= G) return;
  const int64_t E = A * V;
  const int64_t x0 = wr_start(g, E, G, VEC), x1 = wr_start(g + 1, E, G, VEC);
  if (x0 >= x1) return;
  int64_t j = x0 / V;
  int b, i;
  warp_find_row(B, j, cnt, b, i);
  for (int64_t x = x0; x < x1;) {
    const int64_t e0 = x - j * V, e1 = min(V, x1 - j * V);
    const T* row = b < B ? row_of(b, i) : nullptr;
    if (row) {
      const PieceOut o = stream_piece<T, SOFTMAX>(row, e0, e1, K, rg, row_tau ? row_tau + j : nullptr);
      publish(j, g, b, i, o);
    }
    x = (j + 1) * V;
    ++j;
    if (x >= x1) break;
    ++i;  // next row: the next request with rows once this one's are done
    while (b < B && i >= cnt(b)) {
      ++b;
      i = 0;
    }
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

// Row j's pieces: slots j + g for g in [g0, g1].
struct RowPieces {
  int64_t slot0;
  int S;
};
__device__ __forceinline__ RowPieces row_pieces(int64_t j, int64_t V, int64_t A, int64_t G, int vecel) {
  const int64_t E = A * V;
  const int64_t g0 = wr_owner(j * V, E, G, vecel), g1 = wr_owner(j * V + V - 1, E, G, vecel);
  RowPieces r;
  r.slot0 = j + g0;
  r.S = (int)(g1 - g0 + 1);
  return r;
}

// Merges the S (<= 32) partials of one row into its top-K keys (buf: the warp's scratch of S * K keys,
// top: K keys out, descending, 0-padded) and its softmax statistics (every lane gets M and the
// double-float S; a NaN sum poisons it). Keys are distinct, so a key's place is the number of larger
// keys over all lists. All lanes call it.
__device__ __forceinline__ void warp_merge_row(const Partial* __restrict__ parts, int S, int K, uint64_t* buf,
                                               uint64_t* top, bool softmax, float& M, float& sh, float& sl) {
  const int lane = threadIdx.x & 31;
  const int n = S * K;
  for (int t = lane; t < n; t += 32) {
    const int s = t / K;
    buf[t] = parts[s].keys[t - s * K];
  }
  if (lane < K) top[lane] = 0ull;
  float m0 = -INFINITY, h0 = 0.0f, l0 = 0.0f;
  if (softmax && lane < S) {
    m0 = parts[lane].m;
    h0 = parts[lane].s_hi;
    l0 = parts[lane].s_lo;
  }
  __syncwarp();
  for (int t = lane; t < n; t += 32) {
    const uint64_t k = buf[t];
    if (k == 0ull) continue;
    int rank = 0;
    for (int s = 0; s < S && rank < K; ++s) {
      const uint64_t* L = buf + s * K;
      int lo = 0, hi = K;  // keys of list s above k (lists are descending, 0-padded)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (L[mid] > k) lo = mid + 1;
        else hi = mid;
      }
      rank += lo;
    }
    if (rank < K) top[rank] = k;
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
