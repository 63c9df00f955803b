// Row-segment scan shared by the expand and verify row passes.
//
// A CTA of kScanWarps warps reduces one contiguous segment of one logits row to
//   * the segment max m and s = sum exp(x - m), and
//   * the segment top-K under the total order (logit desc, token id asc).
// The segment's 16-byte-aligned middle is split into one contiguous chunk per warp. Each warp
// streams its chunk through a private ring of shared-memory stages filled by 1-D TMA bulk copies
// (cp.async.bulk, completion counted on one mbarrier per stage), so warps never wait on each
// other while streaming; the CTA synchronises once, at the end of the segment.
//   * softmax: every lane keeps a running max and a compensated sum, rescaled when its max grows;
//   * top-K: every warp keeps a sorted list of its K best keys in shared memory. A chunk that fits
//     the warp's ring is filtered in one pass once all of it has arrived, against the K-th largest
//     lane maximum; a longer chunk filters its first stage that way and every later stage against
//     the list's K-th key. Candidates go to a small per-warp buffer and are merged into the list by
//     rank counting.
// Unaligned heads/tails (< 16 bytes at each end) are read with plain loads by warp 0.
#pragma once

#include "dt_internal.cuh"

namespace dt {

template <typename T>
struct Elt;
template <>
struct Elt<uint16_t> {  // bf16 bit patterns
  static constexpr int kVec = 8;
  static __device__ __forceinline__ float load(const uint16_t* p) {
    return __uint_as_float((uint32_t)__ldg(p) << 16);
  }
};
template <>
struct Elt<float> {
  static constexpr int kVec = 4;
  static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
};

// ---------------------------------------------------------------- PTX: mbarrier + bulk copy ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// NaN-propagating maxima (max.NaN): a NaN operand gives NaN.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float max_nan_f32(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_nan_f32u(uint32_t a, uint32_t b) {
  return __float_as_uint(max_nan_f32(__uint_as_float(a), __uint_as_float(b)));
}

// Waits at most `cap` polls; returns false when the bound ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t cap) {
  for (uint32_t it = 0; it < cap; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

constexpr uint32_t kSpinCap = 1u << 22;

// ---------------------------------------------------------------- shared state ----
struct WarpRing {
  uint64_t bar[kWarpStages];
  uint64_t cand[kWarpCand];
  uint64_t list[2][kMaxK];  // the warp's top-K list (descending), double-buffered for merges
  int32_t cnt;
  int32_t ovf;
};

struct ScanSmem {
  WarpRing ring[kScanWarps];
  uint64_t topk[kMaxK];
  uint64_t wl[kScanWarps][kMaxK];  // the warps' final lists (not aliased with the stages)
  float red_m[kScanWarps];
  float red_sh[kScanWarps], red_sl[kScanWarps];
  int32_t flags[kScanWarps];
  int32_t last;
  // Merge / sort buffer of kCandCap keys. It aliases the dynamic stage memory, which is free once
  // every warp has finished streaming (after the block barrier that ends the scan).
  uint64_t* cand;
};

// Top-K of S descending lists of K keys each, list s at src[s * stride ..] (empty = 0), into
// sm.topk[0..K). Keys are distinct, so the place of a key is the number of larger keys over all
// lists. Up to kLinearMerge keys that number is counted directly (independent loads, issued in
// groups of eight); above it by a binary search in each list. All threads call it. The reads of a
// group may run up to 7 keys past a list's end; the callers' buffers extend past it.
constexpr int kLinearMerge = 256;
__device__ __forceinline__ void merge_sorted_lists(ScanSmem& sm, const uint64_t* src, int S, int K, int stride) {
  const int n = S * K;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int s0 = i / K;
    const uint64_t k = src[s0 * stride + (i - s0 * K)];
    if (k == 0ull) continue;
    int rank = 0;
    if (n <= kLinearMerge) {
      for (int s = 0; s < S; ++s) {
        const uint64_t* L = src + s * stride;
        for (int j0 = 0; j0 < K; j0 += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint64_t v = L[j0 + u];
            rank += (j0 + u < K) & (v > k);
          }
        }
      }
    } else {
      for (int s = 0; s < S && rank < K; ++s) {
        const uint64_t* L = src + s * stride;
        int lo = 0, hi = K;  // first index whose key is <= k
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (L[mid] > k) lo = mid + 1;
          else hi = mid;
        }
        rank += lo;
      }
    }
    if (rank < K) sm.topk[rank] = k;
  }
  __syncthreads();
}

// Softmax statistics of a row or segment: max m and S = sum exp(x - m) = s_hi + s_lo.
struct SoftmaxStat {
  float m, s_hi, s_lo;
  bool nan;  // the sum was poisoned by a NaN
};

// log softmax(x) = (x - M) - log S of a row with statistics st, as a double-float (dh, dl).
// log S: S = mant * 2^e with mant in [1, 2) (exact scaling), log S = e * ln2 (Cody-Waite split:
// e * LN2_HI is exact for |e| < 2^9) + log(mant_hi) + mant_lo / mant_hi.
__device__ __forceinline__ void log_softmax_dd(const SoftmaxStat& st, float x, float& dh, float& dl) {
  constexpr float LN2_HI = 0.693145751953125f, LN2_LO = 1.4286068203094173e-06f;
  float lh, ll;
  const float sh = st.s_hi, sl = st.s_lo;
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
  two_sum(x, -st.m, dh, dl);
  ff_add(dh, dl, -lh, -ll);
}

// (h, l) * f for a float factor f, renormalised (the product's rounding error is kept by an fma).
__device__ __forceinline__ void ff_scale(float& h, float& l, float f) {
  const float p = __fmul_rn(h, f);
  const float pe = fmaf(h, f, -p);
  const float t = fmaf(l, f, pe);
  h = __fadd_rn(p, t);
  l = __fsub_rn(t, __fsub_rn(h, p));
}

// Warp 0: combines up to 64 (m, s_hi, s_lo) partials held two per lane into M = max m and
// S = sum s * exp(m - M) (double-float); lane 0 leaves the result in sm.red_*[0]. A NaN sum poisons
// the result.
__device__ __forceinline__ void combine_partial_sums(ScanSmem& sm, float m0, float h0, float l0, float m1, float h1,
                                                     float l1) {
  float bm = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
  bool nan = (h0 != h0) || (h1 != h1);
  float h = 0.0f, l = 0.0f;
  if (!nan) {
    if (m0 != -INFINITY) {
      ff_scale(h0, l0, ex2((m0 - bm) * kLog2e));
      ff_add(h, l, h0, l0);
    }
    if (m1 != -INFINITY) {
      ff_scale(h1, l1, ex2((m1 - bm) * kLog2e));
      ff_add(h, l, h1, l1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, h, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, l, o);
    ff_add(h, l, oh, ol);
  }
  nan = __any_sync(0xFFFFFFFFu, nan);
  if ((threadIdx.x & 31) == 0) {
    sm.red_m[0] = bm;
    sm.red_sh[0] = nan ? __int_as_float(0x7FC00000) : h;
    sm.red_sl[0] = nan ? 0.0f : l;
  }
}

// ---------------------------------------------------------------- warp top-K list ----
// Result of a segment scan; the segment's top-K keys are left in sm.topk (descending, 0-padded).
struct SegOut {
  float m;            // softmax scans: thread 0 holds the max; otherwise every thread: the best key's value
  float s_hi, s_lo;   // softmax scans, thread 0: sum exp(x - m)
  bool timed_out;     // a bounded copy wait ran out
  bool internal;      // the overflow refinement bound was hit
  bool bad;           // non-softmax scans: a NaN or +inf was seen
};

// Per-lane softmax accumulation of one value (head/tail elements).
__device__ __forceinline__ void lane_acc_one(float x, float& m_t, float& s_hi, float& s_lo) {
  if (x != x) {
    s_hi = x;  // NaN poisons the sum
    return;
  }
  if (x == -INFINITY) return;
  if (x > m_t) {
    if (m_t != -INFINITY) {
      const float sc = ex2((m_t - x) * kLog2e);
      s_hi *= sc;
      s_lo *= sc;
    }
    m_t = x;
  }
  const float y = ex2((x - m_t) * kLog2e) - s_lo;
  const float t = s_hi + y;
  s_lo = (t - s_hi) - y;
  s_hi = t;
}

// The warp's list after a merge.
struct ListState {
  int nl, lb;        // keys in the list, current list buffer
  uint64_t tau_key;  // K-th key of the list (0 while it has fewer than K keys)
  int overflow;      // the candidate buffer had overflowed (candidates beyond it were not stored)
};

// Merges the warp's candidate buffer rg.cand[0..min(cnt, kWarpCand)) into its top-K list. Keys are
// distinct elements, so a key's place in the merged list is its rank among list + candidates; with
// `dedup` a candidate already in the list is dropped first. Out of line: one copy serves every call
// site, which keeps the scan's code small enough for the instruction cache.
static __device__ __noinline__ ListState warp_list_merge(WarpRing& rg, int K, int nl, int lb, bool dedup) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const int cnt = rg.cnt;
  ListState out;
  out.overflow = cnt > kWarpCand;
  if (cnt == 0) {
    out.nl = nl;
    out.lb = lb;
    out.tau_key = nl == K ? rg.list[lb][K - 1] : 0ull;
    return out;
  }
  const int n = min(cnt, kWarpCand);
  const uint64_t* cur = rg.list[lb];
  uint64_t* nxt = rg.list[lb ^ 1];
  if (dedup) {
    for (int q = lane; q < n; q += 32) {
      const uint64_t k = rg.cand[q];
      bool dup = false;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        const uint64_t v = cur[j];  // read unconditionally (in bounds), masked after
        dup |= (j < nl) & (v == k);
      }
      if (dup) rg.cand[q] = 0ull;
    }
    __syncwarp();
  }
  int valid = 0;
  for (int q = lane; q < n; q += 32) {
    const uint64_t k = rg.cand[q];
    if (k == 0ull) continue;
    ++valid;
    int r = 0;
    // loads are unconditional (every index is inside the arrays) and masked after, so that the eight
    // of a group issue back to back
    for (int j0 = 0; j0 < nl; j0 += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t v = cur[j0 + u];
        r += (j0 + u < nl) & (v > k);
      }
    }
    for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t v = rg.cand[j0 + u];
        r += (j0 + u < n) & (v > k);
      }
    }
    if (r < K) nxt[r] = k;
  }
  if (lane < nl) {
    const uint64_t l = cur[lane];
    int r = lane;
    for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t v = rg.cand[j0 + u];
        r += (j0 + u < n) & (v > l);
      }
    }
    if (r < K) nxt[r] = l;
  }
  valid = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)valid);
  __syncwarp();
  out.nl = min(K, nl + valid);
  out.lb = lb ^ 1;
  out.tau_key = out.nl == K ? rg.list[out.lb][K - 1] : 0ull;
  if (lane == 0) rg.cnt = 0;
  __syncwarp();
  return out;
}

// Element e of a 16-byte vector of T.
template <typename T>
__device__ __forceinline__ float vec_elt(const uint4& w, int e) {
  if (sizeof(T) == 2) {
    const int wi = e >> 1;
    const uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
    return (e & 1) ? bf16_hi(word) : bf16_lo(word);
  }
  const uint32_t word = e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w;
  return __uint_as_float(word);
}

// The K-th largest (K <= 32) of the 32 lane values v, -inf standing for NaN; every lane gets it.
// A lane's rank is the number of lanes with a larger value, or an equal one at a lower lane, so the
// ranks are 0..31 and exactly one lane has rank K - 1.
__device__ __forceinline__ float warp_kth_largest(float v, int K) {
  const int lane = threadIdx.x & 31;
  if (!(v > -INFINITY)) v = -INFINITY;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float o = __shfl_sync(0xFFFFFFFFu, v, j);
    rank += (o > v) | ((o == v) & (j < lane));
  }
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, rank == K - 1);
  return __shfl_sync(0xFFFFFFFFu, v, __ffs(hit) - 1);
}

// Pushes into the warp's candidate buffer the elements of the warp's first nb chunk stages (resident
// in its ring, stage u in buffer u) whose value is >= tv and not -inf and whose key exceeds tk.
// Draw noise of sampled drafts (children drawn without replacement by Gumbel-top-K): token v of the
// row of node n of request b gets G_v = -log(-log u_v), u_v = (k + 1/2) 2^-23 with k the top 23 bits
// of word v & 3 of Philox4x32-10(key = seed; counter = (round_lo, round_hi, c2, v >> 2)),
// c2 = 0x40000000 + 4096 b + n. The row's keys are then x_v + G_v instead of x_v.
struct GumbelCtx {
  uint32_t k0, k1, r0, r1, c2;
};

__device__ __forceinline__ float gumbel_of_word(uint32_t w) {
  const float u = ((float)(w >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
  return -logf(-logf(u));
}

// G of the four tokens of one Philox block. Out of line: one copy serves every call site.
static __device__ __noinline__ float4 gumbel_group4(GumbelCtx g, uint32_t group) {
  const Philox4 w = philox4x32_10(g.r0, g.r1, g.c2, group, g.k0, g.k1);
  return make_float4(gumbel_of_word(w.v[0]), gumbel_of_word(w.v[1]), gumbel_of_word(w.v[2]), gumbel_of_word(w.v[3]));
}

// G of token id, reusing the block of the previous call when id is in the same group of four (the
// four values are kept in registers: no indexed array).
struct GumbelCursor {
  uint32_t group = 0xFFFFFFFFu;
  float g0 = 0.0f, g1 = 0.0f, g2 = 0.0f, g3 = 0.0f;
  __device__ __forceinline__ float at(const GumbelCtx& g, uint32_t id) {
    if ((id >> 2) != group) {
      group = id >> 2;
      const float4 v = gumbel_group4(g, group);
      g0 = v.x;
      g1 = v.y;
      g2 = v.z;
      g3 = v.w;
    }
    const uint32_t s = id & 3u;
    return s == 0u ? g0 : (s == 1u ? g1 : (s == 2u ? g2 : g3));
  }
};

// Lanes without `scan` push nothing. Out of line: one copy serves every call site. With GUMBEL the
// tested value of token id is x + G(id).
template <typename T, bool GUMBEL>
static __device__ __noinline__ void push_batch_candidates(WarpRing& rg, const uint8_t* my_stages, int nb,
                                                          int64_t wbytes, int64_t we0, float tv, uint64_t tk,
                                                          bool scan, GumbelCtx gc) {
  constexpr int VEC = Elt<T>::kVec;
  constexpr int ESZ = (int)sizeof(T);
  constexpr int QV = kStageBytes / 16 / 32;
  const int lane = threadIdx.x & 31;
  if (scan) {
    for (int u = 0; u < nb; ++u) {
      const uint8_t* sp = my_stages + (size_t)u * kStageBytes;
      const int st_bytes = (int)min((int64_t)kStageBytes, wbytes - (int64_t)u * kStageBytes);
      const int64_t st_e0 = we0 + (int64_t)u * (kStageBytes / ESZ);
      for (int q = 0; q < QV; ++q) {
        const int vi = q * 32 + lane;
        if (vi * 16 >= st_bytes) break;
        const uint4 w = *reinterpret_cast<const uint4*>(sp + (size_t)vi * 16);
        if (!GUMBEL) {  // a vector whose maximum is below the threshold holds no candidate
          const uint32_t m2 = ESZ == 2 ? max_nan_bf16x2(max_nan_bf16x2(w.x, w.y), max_nan_bf16x2(w.z, w.w))
                                       : max_nan_f32u(max_nan_f32u(w.x, w.y), max_nan_f32u(w.z, w.w));
          const float vm = ESZ == 2 ? max_nan_f32(bf16_lo(m2), bf16_hi(m2)) : __uint_as_float(m2);
          if (vm < tv) continue;  // (a NaN maximum is not below it: its elements are looked at)
        }
        GumbelCursor gcur;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const uint32_t id = (uint32_t)(st_e0 + (int64_t)(vi * VEC + e));
          const float x = vec_elt<T>(w, e);
          const float y = GUMBEL ? x + gcur.at(gc, id) : x;
          if (y >= tv && x != -INFINITY) {
            const uint64_t k = make_key(y, id);
            if (k > tk) {
              const int pos = atomicAdd(&rg.cnt, 1);
              if (pos < kWarpCand) rg.cand[pos] = k;
            }
          }
        }
      }
    }
  }
  __syncwarp();
}

// Scans elements [s0, s1) of `row`. K <= kMaxK. `stages` is kScanWarps * kWarpStages * kStageBytes of
// shared memory (dynamic). All threads of the CTA call it. With GUMBEL the keys (top-K, thresholds)
// are x + G of the draw noise gc; the softmax statistics stay those of x.
template <typename T, bool SOFTMAX, bool GUMBEL = false>
__device__ SegOut scan_segment(const T* __restrict__ row, int64_t s0, int64_t s1, int K, ScanSmem& sm,
                               uint8_t* stages, uint32_t first_wait_cap, unsigned long long* gtau,
                               GumbelCtx gc = GumbelCtx{}) {
  constexpr int VEC = Elt<T>::kVec;
  constexpr int ESZ = (int)sizeof(T);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  WarpRing& rg = sm.ring[warp];
  uint8_t* my_stages = stages + (size_t)warp * kWarpStages * kStageBytes;

  // aligned middle [a0, a1) split into kScanWarps contiguous chunks of whole vectors
  const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + s0);
  int64_t a0 = s0 + (int64_t)(((16u - (uint32_t)(addr0 & 15u)) & 15u) / ESZ);
  if (a0 > s1) a0 = s1;
  const int64_t nvec = ((s1 - a0) * ESZ) / 16;
  const int64_t a1 = a0 + nvec * (16 / ESZ);
  const int64_t per = (nvec + kScanWarps - 1) / kScanWarps;
  const int64_t wv0 = min(nvec, per * warp), wv1 = min(nvec, per * (warp + 1));
  const int64_t wbytes = (wv1 - wv0) * 16;
  const char* wsrc = reinterpret_cast<const char*>(row + a0) + wv0 * 16;
  const int64_t we0 = a0 + wv0 * VEC;                       // first element of my chunk
  const int n_st = (int)((wbytes + kStageBytes - 1) / kStageBytes);

  if (tid == 0) sm.cand = reinterpret_cast<uint64_t*>(stages);  // used only after the closing barrier
  if (tid < kMaxK) sm.topk[tid] = 0ull;                          // filled by the closing merge
  if (lane == 0) {
    for (int st = 0; st < kWarpStages; ++st) mbar_init(&rg.bar[st], 1);
    fence_mbar_init();
    rg.cnt = 0;
    rg.ovf = 0;
    sm.flags[warp] = 0;
    for (int t = 0; t < n_st && t < kWarpStages; ++t) {
      const int64_t off = (int64_t)t * kStageBytes;
      const uint32_t bytes = (uint32_t)min((int64_t)kStageBytes, wbytes - off);
      mbar_arrive_expect_tx(&rg.bar[t], bytes);
      bulk_g2s(my_stages + (size_t)t * kStageBytes, wsrc + off, bytes, &rg.bar[t]);
    }
  }
  __syncwarp();

  float m_t = -INFINITY, s_hi = 0.0f, s_lo = 0.0f;
  float seen_max = -INFINITY;
  int lb = 0, nl = 0;           // current list buffer, keys in the list
  uint64_t tau_key = 0ull;      // K-th key of the list (0 while it has fewer than K keys)
  float tau_val = -INFINITY;
  bool timed_out = false;

  // head + tail elements (warp 0): softmax, and always candidates
  const int n_head = (int)(a0 - s0), n_tail = (int)(s1 - a1);
  uint64_t ht_key = 0ull;
  if (warp == 0 && lane < n_head + n_tail) {
    const int64_t idx = lane < n_head ? s0 + lane : a1 + (lane - n_head);
    const float x = Elt<T>::load(row + idx);
    if (SOFTMAX) {
      lane_acc_one(x, m_t, s_hi, s_lo);
    } else {
      seen_max = x;
    }
    // its key joins the warp list only after streaming: the strict tie test of later stages relies on
    // the list holding earlier (smaller) ids of this warp's own chunk
    if (!(x != x)) {
      GumbelCursor gcur;
      ht_key = make_key(GUMBEL ? x + gcur.at(gc, (uint32_t)idx) : x, (uint32_t)idx);
    }
  }
  __syncwarp();

  // Merges the candidate buffer rg.cand[0..min(cnt, kWarpCand)) into the list. Keys are distinct
  // elements, so a key's place in the merged list is its rank among list + candidates; with `dedup` a
  // candidate already in the list is dropped first. Returns true if the buffer had overflowed (the
  // candidates beyond its capacity were not stored).
  auto merge = [&](bool dedup) -> bool {
    const ListState o = warp_list_merge(rg, K, nl, lb, dedup);
    nl = o.nl;
    lb = o.lb;
    tau_key = o.tau_key;
    tau_val = tau_key ? key_value(tau_key) : -INFINITY;
    return o.overflow != 0;
  };
  auto push = [&](uint64_t k) {
    const int pos = atomicAdd(&rg.cnt, 1);
    if (pos < kWarpCand) rg.cand[pos] = k;
  };

  constexpr int QV = kStageBytes / 16 / 32;   // vectors per lane per stage (8)
  constexpr int NV = QV * VEC;                 // values per lane per stage
  const uint32_t neg_fill = ESZ == 2 ? 0xFF80FF80u : 0xFF800000u;  // -inf in every element
  // The first nb stages are filtered together once all of them are in (the whole chunk, when it
  // fits the ring; else the first stage): against the K-th largest lane maximum over them, with one
  // merge. Later stages stream against the list's K-th key.
  const int nb = n_st <= kWarpStages ? n_st : 1;
  float bmax = -INFINITY;  // lane maximum over the batch stages (a stage's NaN maximum is skipped)
  // the row's shared threshold (read early: used after the stage's data has arrived)
  uint64_t gt = gtau ? (uint64_t)__ldcg(gtau) : 0ull;
  for (int t = 0; t < n_st; ++t) {
    const int st = t % kWarpStages;
    const uint32_t parity = (uint32_t)((t / kWarpStages) & 1);
    if (t >= nb && gtau) gt = (uint64_t)__ldcg(gtau);
    const bool ok = mbar_wait_bounded(&rg.bar[st], parity, t == 0 ? first_wait_cap : kSpinCap);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      timed_out = true;
      const int issued = min(n_st, t + kWarpStages);  // drain: wait (bounded) for every issued copy
      for (int u = t; u < issued; ++u)
        mbar_wait_bounded(&rg.bar[u % kWarpStages], (uint32_t)((u / kWarpStages) & 1), kSpinCap);
      break;
    }
    const int64_t st_off = (int64_t)t * kStageBytes;
    const int st_bytes = (int)min((int64_t)kStageBytes, wbytes - st_off);
    const int64_t st_e0 = we0 + st_off / ESZ;
    const uint8_t* sp = my_stages + (size_t)st * kStageBytes;

    // the whole stage in registers: vector q of this lane is stage vector q*32 + lane
    uint32_t wv[QV * 4];
#pragma unroll
    for (int q = 0; q < QV; ++q) {
      const int vi = q * 32 + lane;
      uint4 w = make_uint4(neg_fill, neg_fill, neg_fill, neg_fill);
      if (vi * 16 < st_bytes) w = *reinterpret_cast<const uint4*>(sp + (size_t)vi * 16);
      wv[4 * q + 0] = w.x;
      wv[4 * q + 1] = w.y;
      wv[4 * q + 2] = w.z;
      wv[4 * q + 3] = w.w;
    }

    // lane max with NaN propagation (a NaN makes it NaN): packed bf16x2 or fp32 tree. Its first two
    // levels give the maximum of each of the lane's vectors (vmax), kept for the rare paths below.
    float lm;
    float vmax[QV];
    {
      uint32_t r[QV * 4];
#pragma unroll
      for (int j = 0; j < QV * 4; ++j) r[j] = wv[j];
#pragma unroll
      for (int w2 = 1; w2 < QV * 4; w2 <<= 1) {
#pragma unroll
        for (int j = 0; j + w2 < QV * 4; j += 2 * w2) r[j] = ESZ == 2 ? max_nan_bf16x2(r[j], r[j + w2])
                                                                       : max_nan_f32u(r[j], r[j + w2]);
        if (w2 == 2) {
#pragma unroll
          for (int q = 0; q < QV; ++q)
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
        // sum of exp(x - m) over the stage: four 16-value trees (bf16) / 2 x 16 (fp32)
        float part = 0.0f;
#pragma unroll
        for (int c = 0; c < NV / 16; ++c) {
          float e[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int v = c * 16 + j;  // value index within the lane's stage values
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

    // the filter's maxima: of x, or with GUMBEL of x + G (every element's noise, lane by lane)
    float flm = lm;
    if (GUMBEL) {
      flm = -INFINITY;
      GumbelCursor gcur;
#pragma unroll
      for (int q = 0; q < QV; ++q) {
        float vm = -INFINITY;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int v = q * VEC + e;  // value index within the lane's stage values
          float x;
          if (ESZ == 2) x = (v & 1) ? bf16_hi(wv[v >> 1]) : bf16_lo(wv[v >> 1]);
          else x = __uint_as_float(wv[v]);
          const uint32_t id = (uint32_t)(st_e0 + (int64_t)((q * 32 + lane) * VEC + e));
          if (x != -INFINITY) vm = fmaxf(vm, x + gcur.at(gc, id));
        }
        vmax[q] = vm;
        flm = fmaxf(flm, vm);
      }
    }

    // The rarely taken candidate paths below read the stage from shared memory with rolled loops:
    // straight-line code over all NV register values would be large and, being rarely executed,
    // always cold in the instruction cache. Vector q of this lane is stage vector q * 32 + lane; its
    // element e has token id st_e0 + (q * 32 + lane) * VEC + e.
    auto vec_at = [&](int q, uint4& w) -> bool {
      const int vi = q * 32 + lane;
      if (vi * 16 >= st_bytes) return false;
      w = *reinterpret_cast<const uint4*>(sp + (size_t)vi * 16);
      return true;
    };
    auto id_of = [&](int q, int e) -> uint32_t {
      return (uint32_t)(st_e0 + (int64_t)((q * 32 + lane) * VEC + e));
    };

    if (t < nb) {
      bmax = fmaxf(bmax, flm);
      if (t + 1 < nb) continue;  // the next batch stage
      // Threshold: the K-th largest lane maximum (K lanes hold an element at or above it, so no
      // element below it is in the top-K), or the row's shared threshold if larger. The warp has
      // published nothing to the shared threshold yet, so a key equal to it is not in this chunk.
      uint64_t tk = gt;
      float tv = fmaxf(warp_kth_largest(bmax, K), gt ? key_value(gt) : -INFINITY);
      if (__any_sync(0xFFFFFFFFu, bmax >= tv)) {
        push_batch_candidates<T, GUMBEL>(rg, my_stages, nb, wbytes, we0, tv, tk, bmax >= tv, gc);
        bool overflow = merge(false);
        // An overflowed buffer still raised the list's K-th key: filter again above it (keys already
        // in the list are dropped by the merge). The key rises every round.
        for (int round = 1; overflow; ++round) {
          if (round > nb * NV * 32 / (kWarpCand - kMaxK) + 1) {  // never hit
            if (lane == 0) sm.flags[warp] |= 2;
            break;
          }
          tk = tau_key;
          tv = tau_val;
          push_batch_candidates<T, GUMBEL>(rg, my_stages, nb, wbytes, we0, tv, tk, bmax >= tv, gc);
          overflow = merge(true);
        }
        if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
      }
    } else {
      // Filter against the larger of the list's K-th key and the row's shared threshold (the best K-th
      // key any warp of any piece of the row has published: that warp holds K keys at or above it, so
      // no element below it can be in the row's top-K). Within a warp's chunk token ids grow stage by
      // stage, so after the first stage a value equal to the warp's own K-th key's value has a larger
      // id and cannot beat it: the test is strict there (not against another warp's key). Lanes whose
      // maximum clears the threshold push their candidates, which are then merged into the list. If the
      // buffer overflowed, the merge still raised the threshold: the stage is filtered again against it
      // (keys already in the list are dropped by the merge).
      bool dedup = false;
      for (int round = 0;; ++round) {
        uint64_t tk = tau_key;
        bool own = true;
        if (gt > tk) {
          tk = gt;
          own = false;
        }
        const float tv = tk ? key_value(tk) : -INFINITY;
        const bool strict = t > 0 && own;
        const bool hot = strict ? (flm > tv) : (flm >= tv);
        if (!__any_sync(0xFFFFFFFFu, hot)) break;
        if (hot) {
          unsigned vm = 0u;  // vectors that may hold candidates
#pragma unroll
          for (int q = 0; q < QV; ++q)
            if (strict ? (vmax[q] > tv) : (vmax[q] >= tv)) vm |= 1u << q;
          while (vm) {
            const int q = __ffs(vm) - 1;
            vm &= vm - 1;
            uint4 w;
            if (!vec_at(q, w)) break;
            GumbelCursor gcur;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const float x = vec_elt<T>(w, e);
              const float y = GUMBEL ? x + gcur.at(gc, id_of(q, e)) : x;
              if (y >= tv && x != -INFINITY) {
                const uint64_t k = make_key(y, id_of(q, e));
                if (k > tk) push(k);
              }
            }
          }
        }
        const bool overflow = merge(dedup);
        dedup = true;
        if (gtau && lane == 0 && nl == K) atomicMax(gtau, (unsigned long long)tau_key);
        if (!overflow) break;
        if (round >= NV * 32 / (kWarpCand - kMaxK) + 1) {  // the threshold rises every round: never hit
          if (lane == 0) sm.flags[warp] |= 2;
          break;
        }
      }
    }

    // the stage has been read for the last time: refill its buffer with stage t + kWarpStages
    __syncwarp();
    if (lane == 0 && t + kWarpStages < n_st) {
      fence_proxy_async_smem();
      const int64_t off = (int64_t)(t + kWarpStages) * kStageBytes;
      const uint32_t bytes = (uint32_t)min((int64_t)kStageBytes, wbytes - off);
      mbar_arrive_expect_tx(&rg.bar[st], bytes);
      bulk_g2s(my_stages + (size_t)st * kStageBytes, wsrc + off, bytes, &rg.bar[st]);
    }
  }
  if (__any_sync(0xFFFFFFFFu, ht_key != 0ull)) {  // head/tail elements (warp 0)
    if (ht_key) push(ht_key);
    merge(false);
  }
  // every copy has landed: retire the barriers so that a later scan in this CTA can initialise them
  // again (after a timeout a copy may still be in flight, and the barriers are left alone)
  if (lane == 0 && !timed_out)
    for (int st = 0; st < kWarpStages; ++st) mbar_inval(&rg.bar[st]);

  // ---- warp results -> CTA: one barrier, then the merge of the warp lists ----
  // (the stage memory, which sm.cand aliases, may still be in use by other warps here)
  if (lane < K) sm.wl[warp][lane] = lane < nl ? rg.list[lb][lane] : 0ull;
  float wm = m_t;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, o));
  float ch = 0.0f, cl = 0.0f;
  bool wnan = false;
  if (SOFTMAX) {
    wnan = __any_sync(0xFFFFFFFFu, s_hi != s_hi);
    if (m_t != -INFINITY && !(s_hi != s_hi)) {
      ch = s_hi;
      cl = s_lo;
      if (wm != m_t) ff_scale(ch, cl, ex2((m_t - wm) * kLog2e));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {  // double-float warp sum
      const float oh = __shfl_xor_sync(0xFFFFFFFFu, ch, o);
      const float ol = __shfl_xor_sync(0xFFFFFFFFu, cl, o);
      ff_add(ch, cl, oh, ol);
    }
  }
  const bool wbad = !SOFTMAX && __any_sync(0xFFFFFFFFu, seen_max != seen_max || seen_max == INFINITY);
  if (lane == 0) {
    sm.red_m[warp] = wm;
    sm.red_sh[warp] = wnan ? __int_as_float(0x7FC00000) : ch;
    sm.red_sl[warp] = wnan ? 0.0f : cl;
    sm.flags[warp] |= (timed_out ? 4 : 0) | (wbad ? 8 : 0);
  }
  __syncthreads();
  int fl = 0;
#pragma unroll
  for (int w = 0; w < kScanWarps; ++w) fl |= sm.flags[w];
  SegOut out;
  out.timed_out = (fl & 4) != 0;
  out.bad = (fl & 8) != 0;
  out.internal = (fl & 2) != 0;
  merge_sorted_lists(sm, &sm.wl[0][0], kScanWarps, K, kMaxK);  // sm.topk was cleared at the start
  out.m = -INFINITY;
  out.s_hi = 0.0f;
  out.s_lo = 0.0f;
  if (SOFTMAX) {
    if (tid == 0) {
      float M = -INFINITY;
      for (int w = 0; w < kScanWarps; ++w) M = fmaxf(M, sm.red_m[w]);
      float h = 0.0f, l = 0.0f;
      bool nan = false;
      for (int w = 0; w < kScanWarps; ++w) {
        float hh = sm.red_sh[w], ll = sm.red_sl[w];
        if (hh != hh) nan = true;
        else if (sm.red_m[w] != -INFINITY) {
          ff_scale(hh, ll, ex2((sm.red_m[w] - M) * kLog2e));
          ff_add(h, l, hh, ll);
        }
      }
      out.m = M;
      out.s_hi = nan ? __int_as_float(0x7FC00000) : h;
      out.s_lo = nan ? 0.0f : l;
    }
  } else {
    out.m = sm.topk[0] ? key_value(sm.topk[0]) : -INFINITY;
  }
  return out;
}

// ---------------------------------------------------------------- balanced row pass ----
// The rows a launch reads ("active rows") are numbered j = 0..A-1 in request order: request b owns
// cnt(b) consecutive numbers, its rows i = 0..cnt(b)-1. The work is laid out in one of two ways:
//  * few rows (A <= gridDim): every row is cut into S_row equal segments, one per CTA (CTA c takes
//    segment c % S_row of row c / S_row); a row's pieces are CTAs j S_row .. j S_row + S_row - 1 and
//    piece c leaves its partial at slot c;
//  * many rows: the rows' E = A * V elements, concatenated, are cut into G equal ranges, one per CTA
//    (CTA c takes [floor(c E / G), floor((c + 1) E / G))), so that every SM gets the same bytes. The
//    part of row j inside CTA c's range is the piece (j, c), with its partial at slot j + c (distinct
//    for distinct pieces, since j and c both grow along the concatenation); a row's pieces are CTAs
//    cta_of(j V) .. cta_of(j V + V - 1).
// The CTA whose arrival completes a row's count merges the row's partials.
struct RowPlan {
  int64_t A, E;    // active rows, A * V
  int G;           // CTAs with work (the others exit)
  int S_row;       // segments per row (few-rows layout), 0 for the concatenated layout
  int64_t j0;      // first row of this CTA
  int64_t x0, x1;  // this CTA's element range in the concatenation (x0 == x1: an empty segment)
  int b, i;        // request and row of active row j0
};

__device__ __forceinline__ int64_t range_start(int64_t c, int64_t E, int64_t G) {
  return (E / G) * c + ((E % G) * c) / G;  // floor(c E / G) without overflow
}
// CTA whose range holds element x (E * G < 2^63: E <= 2^52, G <= 4096)
__device__ __forceinline__ int cta_of(int64_t x, int64_t E, int64_t G) {
  return (int)(((uint64_t)(x + 1) * (uint64_t)G - 1ull) / (uint64_t)E);
}

// Warp 0 of every CTA: the layout, this CTA's range and the (b, i) of its first row. A piece holds at
// least r_min elements: min_stages stages per warp (two for the streaming passes, whose time is the
// chain of dependent steps; one for compute-heavy passes such as the draw noise of sampled drafts;
// either way every lane of a warp sees data and the top-K list starts full), and
// r_min >= (V - 1) / (Smax - 2), so that a row has at most Smax pieces. The first 32 counts are read
// once and kept in a register.
template <class Cnt>
__device__ void plan_rows(RowPlan& p, int B, int64_t V, int Smax, int esz, Cnt cnt, int min_stages = 2) {
  const int lane = threadIdx.x & 31;
  const int head = lane < B ? cnt(lane) : 0;
  int64_t A = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    int c = b0 == 0 ? head : ((b0 + lane < B) ? cnt(b0 + lane) : 0);
    A += __reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
  }
  p.A = A;
  p.E = A * V;
  p.G = 0;
  p.S_row = 0;
  p.j0 = p.x0 = p.x1 = 0;
  p.b = p.i = 0;
  if (p.E == 0) return;
  // 32-bit unsigned arithmetic where it suffices (V < 2^31, A and the grid <= 4096): the divisions
  // here are on the launch's critical path
  const uint32_t Vu = (uint32_t)V;
  const uint32_t r_min = max((uint32_t)(kScanWarps * min_stages * kStageBytes / esz),
                             (Vu - 1u + (uint32_t)(Smax - 3)) / (uint32_t)(Smax - 2));
  const int64_t c = blockIdx.x;
  if (A <= (int64_t)gridDim.x) {
    const uint32_t Au = (uint32_t)A, cu = (uint32_t)c;
    uint32_t S = min(gridDim.x / Au, (Vu - 1u) / r_min + 1u);  // ceil(V / r_min) for V >= 1
    S = max(1u, min(S, (uint32_t)Smax));
    p.S_row = (int)S;
    p.G = (int)(Au * S);
    if (c >= p.G) return;
    const uint32_t j0 = cu / S, seg = cu - j0 * S;
    uint32_t L = (Vu - 1u) / S + 1u;  // ceil(V / S)
    L = (L + 7u) / 8u * 8u;
    p.j0 = j0;
    const int64_t e0 = min(V, (int64_t)seg * L), e1 = min(V, e0 + L);
    p.x0 = p.j0 * V + e0;
    p.x1 = p.j0 * V + e1;
  } else {
    int64_t G = p.E / (int64_t)r_min;
    G = max(G, (int64_t)1);
    G = min(G, (int64_t)gridDim.x);
    p.G = (int)G;
    if (c >= G) return;
    p.x0 = range_start(c, p.E, G);
    p.x1 = range_start(c + 1, p.E, G);
    p.j0 = p.x0 / V;
  }
  const int64_t j = p.j0;
  int64_t base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int n = b0 == 0 ? head : ((b0 + lane < B) ? cnt(b0 + lane) : 0);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t lo = base + incl - n;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, n > 0 && lo <= j && j < base + incl);
    const int off = (int)(j - lo);
    if (hit) {  // warp-uniform
      const int src = __ffs(hit) - 1;
      p.b = b0 + src;
      p.i = __shfl_sync(0xFFFFFFFFu, off, src);
      break;
    }
    base += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
}

// Scans this CTA's pieces in order (all threads). row_of(b, i) gives row i of request b, or nullptr
// when that row is not to be read (its pieces leave empty partials); it is called when a piece
// starts, so it may also start loads the row's finish will need. When a piece completes its row,
// noise(b, i) gives the draw noise of row (b, i) when GUMBEL (called after row_of(b, i)).
// finish(b, i, st) runs on all threads with the row's merged top-K in sm.topk and its softmax
// statistics st (max and sum for softmax passes; the best key's value otherwise). After a timed-out copy wait the CTA reads nothing more (empty partials), so
// that every row still completes its count.
template <typename T, bool SOFTMAX, bool GUMBEL = false, class RowOf, class Cnt, class Finish, class Noise>
__device__ void scan_pieces(const RowPlan& p, int64_t V, int K, int B, Partial* partials, int32_t* counter,
                            unsigned long long* row_tau, ScanSmem& sm, uint8_t* stages, uint32_t first_wait_cap,
                            int32_t* status, RowOf row_of, Cnt cnt, Finish finish, Noise noise) {
  const int tid = threadIdx.x;
  const int64_t c = blockIdx.x;
  if (tid == 0) sm.cand = reinterpret_cast<uint64_t*>(stages);
  __syncthreads();
  int64_t x = p.x0, j = p.j0;
  int b = p.b, i = p.i;
  bool halted = false;
  while (true) {
    const int64_t e0 = x - j * V;
    const int64_t e1 = min(V, p.x1 - j * V);
    int c_first, c_last;
    int64_t slot, row_slot0;
    if (p.S_row > 0) {
      c_first = (int)(j * p.S_row);
      c_last = c_first + p.S_row - 1;
      slot = c;
      row_slot0 = c_first;
    } else {
      c_first = cta_of(j * V, p.E, p.G);
      c_last = cta_of(j * V + V - 1, p.E, p.G);
      slot = j + c;
      row_slot0 = j + c_first;
    }
    Partial* part = partials + slot;
    const T* row = row_of(b, i);
    const bool scan = row != nullptr && !halted && e1 > e0;
    SegOut so;
    if (scan) {
      so = scan_segment<T, SOFTMAX, GUMBEL>(row, e0, e1, K, sm, stages, first_wait_cap,
                                            row_tau ? row_tau + j : nullptr, GUMBEL ? noise(b, i) : GumbelCtx{});
    } else {
      so.m = -INFINITY;
      so.s_hi = so.s_lo = 0.0f;
      so.timed_out = so.internal = so.bad = false;
    }
    // warp 0 publishes the piece: its keys and sums, then (after a fence) its arrival
    if (tid < 32) {
      if (tid < K) part->keys[tid] = scan ? sm.topk[tid] : 0ull;
      if (tid == 0) {
        part->m = so.m;
        part->s_hi = so.s_hi;
        part->s_lo = so.s_lo;
        if (so.timed_out) set_status(status, DT_DEV_TIMEOUT);
        if (so.internal) set_status(status, DT_DEV_INTERNAL);
        if (so.bad) set_status(status, DT_DEV_BAD_LOGITS);
      }
      __threadfence();
      __syncwarp();
      if (tid == 0) {
        const int prev = atomicAdd(&counter[j], 1);
        sm.last = (prev == c_last - c_first);
      }
    }
    halted = halted || so.timed_out;
    __syncthreads();
    if (sm.last) {  // block-uniform: merge the row's partials (read from L2, which the fenced
                    // publications of every piece reached before their arrivals)
      if (tid == 0) {
        counter[j] = 0;
        if (row_tau) row_tau[j] = 0ull;  // every piece of the row has finished with it
      }
      const int S = c_last - c_first + 1;
      const Partial* rp = partials + row_slot0;
      for (int k = tid; k < S * K; k += blockDim.x) sm.cand[k] = __ldcg(&rp[k / K].keys[k % K]);
      // warp 0 loads the partial sums alongside (two per lane, S <= 64)
      float m0 = -INFINITY, h0 = 0.0f, l0 = 0.0f, m1 = -INFINITY, h1 = 0.0f, l1 = 0.0f;
      if (SOFTMAX && tid < 32) {
        if (tid < S) {
          m0 = __ldcg(&rp[tid].m);
          h0 = __ldcg(&rp[tid].s_hi);
          l0 = __ldcg(&rp[tid].s_lo);
        }
        if (tid + 32 < S) {
          m1 = __ldcg(&rp[tid + 32].m);
          h1 = __ldcg(&rp[tid + 32].s_hi);
          l1 = __ldcg(&rp[tid + 32].s_lo);
        }
      }
      if (tid < kMaxK) sm.topk[tid] = 0ull;
      __syncthreads();
      if (SOFTMAX && tid < 32) combine_partial_sums(sm, m0, h0, l0, m1, h1, l1);
      merge_sorted_lists(sm, sm.cand, S, K, K);  // ends with a barrier, after which sm.red_*[0] is visible
      SoftmaxStat st;
      st.m = SOFTMAX ? sm.red_m[0] : (sm.topk[0] ? key_value(sm.topk[0]) : -INFINITY);
      st.s_hi = SOFTMAX ? sm.red_sh[0] : 0.0f;
      st.s_lo = SOFTMAX ? sm.red_sl[0] : 0.0f;
      st.nan = st.s_hi != st.s_hi;
      finish(b, i, st);
    }
    x = (j + 1) * V;
    ++j;
    if (x >= p.x1) break;
    // next row; the stage memory is handed back to the async proxy
    ++i;
    while (b < B && i >= cnt(b)) {
      ++b;
      i = 0;
    }
    fence_proxy_async_smem();
    __syncthreads();
  }
}

}  // namespace dt
