// Row-segment scan shared by the expand and verify row passes.
//
// One CTA streams a contiguous segment of one logits row through a ring of
// shared-memory tiles filled by 1-D TMA bulk copies (cp.async.bulk, completion
// counted on an mbarrier per stage), and reduces it to
//   * the segment max m and s = sum exp(x - m) (online: per-thread running max,
//     rescaled when it grows; per-tile sums added with a compensation term), and
//   * the segment top-K under the total order (logit desc, token id asc),
//     found by filtering against a running threshold key: the first tile sets
//     it to the K-th largest per-thread maximum, later compactions raise it to
//     the K-th best candidate so far; only elements at or above it are kept in
//     a small shared-memory candidate buffer.
// Unaligned row heads/tails (rows whose start is not 16-byte aligned, or
// segments whose length is not a whole number of 16-byte vectors) are read
// with plain loads and always kept as candidates.
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

// Waits at most `cap` polls; returns false when the bound ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t cap) {
  for (uint32_t it = 0; it < cap; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

constexpr uint32_t kSpinCap = 1u << 22;

// ---------------------------------------------------------------- shared state ----
struct ScanSmem {
  uint64_t bar[kStages];
  uint64_t cand[kCandCap];
  uint64_t topk[kMaxK];
  unsigned long long tau;   // threshold key (CTA-uniform between syncs)
  int32_t cnt;
  int32_t flag;
  int32_t last;
  int32_t pad;
  float red_m[kRowThreads / 32];
  double red_s[kRowThreads / 32];
};

// Top-K (descending) of cand[0..cnt) into sm.topk[0..n), n = min(cnt, K); cand is not modified.
// Keys are distinct (one per element). All threads must call it.
__device__ __forceinline__ int select_topk(ScanSmem& sm, int cnt, int K) {
  const int tid = threadIdx.x;
  for (int i = tid; i < cnt; i += blockDim.x) {
    const uint64_t k = sm.cand[i];
    int rank = 0;
    for (int j = 0; j < cnt; ++j) rank += (sm.cand[j] > k);
    if (rank < K) sm.topk[rank] = k;
  }
  __syncthreads();
  return cnt < K ? cnt : K;
}

// Replaces cand[0..cnt) by its top-K; returns the new count.
__device__ __forceinline__ int compact_topk(ScanSmem& sm, int cnt, int K) {
  const int n = select_topk(sm, cnt, K);
  for (int i = threadIdx.x; i < n; i += blockDim.x) sm.cand[i] = sm.topk[i];
  __syncthreads();
  return n;
}

// Merge of the S (<= blockDim) segment partials of a row by the whole CTA:
// M = max_s m_s, S = sum_s s_s * exp(m_s - M). Every thread gets the results; `nan` reports a
// poisoned (NaN) segment sum. All threads must call it.
__device__ __forceinline__ void merge_softmax(const Partial* part, int S, ScanSmem& sm, float& M, double& Sum,
                                              bool& nan) {
  // warp 0 merges (S <= 64: two segments per lane)
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float m0 = -INFINITY, m1 = -INFINITY;
    double s0 = 0.0, s1 = 0.0;
    if (lane < S) {
      m0 = __ldcg(&part[lane].m);
      s0 = __ldcg(&part[lane].s);
    }
    if (lane + 32 < S) {
      m1 = __ldcg(&part[lane + 32].m);
      s1 = __ldcg(&part[lane + 32].s);
    }
    float bm = fmaxf(m0, m1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
    double c = 0.0;
    if (s0 != s0) c += s0;
    else if (m0 != -INFINITY) c += s0 * (double)ex2((m0 - bm) * kLog2e);
    if (s1 != s1) c += s1;
    else if (m1 != -INFINITY) c += s1 * (double)ex2((m1 - bm) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) {
      sm.red_m[0] = bm;
      sm.red_s[0] = c;
    }
  }
  __syncthreads();
  M = sm.red_m[0];
  Sum = sm.red_s[0];
  nan = Sum != Sum;
  __syncthreads();
}

struct SegOut {
  float m;        // thread 0 only (softmax scans); all threads: best key value otherwise
  double s;       // thread 0 only
  int nkeys;      // all threads: keys in sm.cand[0..nkeys), descending
  bool timed_out; // a bounded copy wait ran out
  bool internal;  // the overflow refinement bound was hit
  bool bad;       // non-softmax scans: a NaN or +inf was seen
};

// Scans elements [s0, s1) of `row`. K <= kMaxK. `tiles` is kStages * kTileBytes of shared memory.
template <typename T, bool SOFTMAX>
__device__ SegOut scan_segment(const T* __restrict__ row, int64_t s0, int64_t s1, int K, ScanSmem& sm,
                               uint8_t* tiles, uint32_t first_wait_cap) {
  constexpr int VEC = Elt<T>::kVec;
  constexpr int ESZ = (int)sizeof(T);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // aligned middle [a0, a1) moved by bulk copies; head [s0, a0) and tail [a1, s1) by plain loads
  const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + s0);
  int64_t head = (int64_t)(((16u - (uint32_t)(addr0 & 15u)) & 15u) / ESZ);
  int64_t a0 = s0 + head;
  if (a0 > s1) a0 = s1;
  const int64_t nvec = ((s1 - a0) * ESZ) / 16;
  const int64_t a1 = a0 + nvec * (16 / ESZ);
  const int64_t mid_bytes = nvec * 16;
  const int n_tiles = (int)((mid_bytes + kTileBytes - 1) / kTileBytes);

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&sm.bar[st], 1);
    fence_mbar_init();
    sm.cnt = 0;
    sm.flag = 0;
    sm.tau = 0ull;
    const char* src = reinterpret_cast<const char*>(row + a0);
    for (int t = 0; t < n_tiles && t < kStages; ++t) {
      const int64_t off = (int64_t)t * kTileBytes;
      const uint32_t bytes = (uint32_t)min((int64_t)kTileBytes, mid_bytes - off);
      mbar_arrive_expect_tx(&sm.bar[t], bytes);
      bulk_g2s(tiles + (size_t)t * kTileBytes, src + off, bytes, &sm.bar[t]);
    }
  }
  __syncthreads();

  float m_t = -INFINITY;
  float s_hi = 0.0f, s_lo = 0.0f;

  // head + tail elements: plain loads, always candidates
  const int n_head = (int)(a0 - s0), n_tail = (int)(s1 - a1);
  uint32_t bad_bits = 0u;  // non-softmax scans: largest |x| bit pattern (NaN above 0x7F800000)
  float seen_max = -INFINITY;
  if (tid < n_head + n_tail) {
    const int64_t idx = tid < n_head ? s0 + tid : a1 + (tid - n_head);
    const float x = Elt<T>::load(row + idx);
    if (SOFTMAX) {
      // m = x, s = exp(0) = 1; a -inf element contributes nothing; NaN/+inf poison s
      m_t = x;
      s_hi = (x == -INFINITY) ? 0.0f : ex2((x - x) * kLog2e);
    } else {
      bad_bits = __float_as_uint(x) & 0x7FFFFFFFu;
      seen_max = x;
    }
    if (!(x != x)) {
      const int pos = atomicAdd(&sm.cnt, 1);
      sm.cand[pos] = make_key(x, (uint32_t)idx);
    }
  }
  __syncthreads();

  float tau_val = -INFINITY;
  uint64_t tau_key = 0ull;
  bool timed_out = false;
  int overflow_rounds = 0;

  for (int t = 0; t < n_tiles; ++t) {
    const int st = t % kStages;
    const uint32_t parity = (uint32_t)((t / kStages) & 1);
    // every thread polls the barrier; a run-out is reported once per CTA
    const uint32_t cap = (t == 0) ? first_wait_cap : kSpinCap;
    bool ok = mbar_wait_bounded(&sm.bar[st], parity, cap);
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      // drain: wait (bounded) for every copy that was issued, then leave
      const int issued = min(n_tiles, t + kStages);
      for (int u = t; u < issued; ++u)
        mbar_wait_bounded(&sm.bar[u % kStages], (uint32_t)((u / kStages) & 1), kSpinCap);
      __syncthreads();
      break;
    }
    const int64_t tile_off = (int64_t)t * kTileBytes;
    const int tile_bytes = (int)min((int64_t)kTileBytes, mid_bytes - tile_off);
    const int64_t tile_e0 = a0 + tile_off / ESZ;
    const uint8_t* tile = tiles + (size_t)st * kTileBytes;

    // my vectors: q*256 + tid, q = 0..3
    constexpr int QV = kTileBytes / 16 / kRowThreads;  // vectors per thread per tile (4)
    float x[QV * VEC];
    bool have[QV];
#pragma unroll
    for (int q = 0; q < QV; ++q) {
      const int vi = q * kRowThreads + tid;
      have[q] = vi * 16 < tile_bytes;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (have[q]) w = *reinterpret_cast<const uint4*>(tile + (size_t)vi * 16);
      if (ESZ == 2) {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[q * VEC + 2 * e] = have[q] ? bf16_lo(ww[e]) : -INFINITY;
          x[q * VEC + 2 * e + 1] = have[q] ? bf16_hi(ww[e]) : -INFINITY;
        }
      } else {
        x[q * VEC + 0] = have[q] ? __uint_as_float(w.x) : -INFINITY;
        x[q * VEC + 1] = have[q] ? __uint_as_float(w.y) : -INFINITY;
        x[q * VEC + 2] = have[q] ? __uint_as_float(w.z) : -INFINITY;
        x[q * VEC + 3] = have[q] ? __uint_as_float(w.w) : -INFINITY;
      }
    }

    // ---- online softmax over my values ----
    float lm = -INFINITY;
#pragma unroll
    for (int j = 0; j < QV * VEC; ++j) lm = fmaxf(lm, x[j]);
    if (!SOFTMAX) {
#pragma unroll
      for (int j = 0; j < QV * VEC; ++j) bad_bits = max(bad_bits, __float_as_uint(x[j]) & 0x7FFFFFFFu);
      seen_max = fmaxf(seen_max, lm);
    }
    if (SOFTMAX) {
      // NaN inputs are ignored by fmaxf but poison the sum below (detected by the caller)
      if (lm > m_t) {
        if (m_t != -INFINITY) {
          const float sc = ex2((m_t - lm) * kLog2e);
          s_hi *= sc;
          s_lo *= sc;
        }
        m_t = lm;
      }
      if (m_t != -INFINITY) {
        float e[QV * VEC];
#pragma unroll
        for (int j = 0; j < QV * VEC; ++j) e[j] = ex2((x[j] - m_t) * kLog2e);
#pragma unroll
        for (int w = 1; w < QV * VEC; w <<= 1)
#pragma unroll
          for (int j = 0; j + w < QV * VEC; j += 2 * w) e[j] += e[j + w];
        const float part = e[0];
        // compensated accumulation of the per-tile sums
        const float y = part - s_lo;
        const float tt = s_hi + y;
        s_lo = (tt - s_hi) - y;
        s_hi = tt;
      } else {
        // all my values so far are -inf (or NaN): a NaN must still poison the sum
#pragma unroll
        for (int j = 0; j < QV * VEC; ++j)
          if (x[j] != x[j]) s_hi = x[j];
      }
    }

    // ---- first tile: threshold from the K-th largest per-thread maximum key ----
    if (tau_key == 0ull) {
      uint64_t best = 0ull;
#pragma unroll
      for (int q = 0; q < QV; ++q)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float v = x[q * VEC + e];
          if (have[q] && !(v != v)) {
            const uint64_t k = make_key(v, (uint32_t)(tile_e0 + (int64_t)(q * kRowThreads + tid) * VEC + e));
            best = k > best ? k : best;
          }
        }
      const uint64_t srt = warp_sort_desc(best);
      const uint64_t kth = shfl_u64(srt, K - 1);
      if (lane == 0) atomicMax(&sm.tau, (unsigned long long)kth);
      __syncthreads();
      tau_key = sm.tau;
      tau_val = tau_key ? key_value(tau_key) : -INFINITY;
    }

    // ---- filter into the candidate buffer (re-run with a higher threshold on overflow) ----
    const int base_cnt = sm.cnt;  // entries of earlier tiles; at most kCandCap / 2
    for (;;) {
      if (lm >= tau_val) {
#pragma unroll
        for (int q = 0; q < QV; ++q)
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float v = x[q * VEC + e];
            if (have[q] && v >= tau_val) {
              const uint64_t k =
                  make_key(v, (uint32_t)(tile_e0 + (int64_t)(q * kRowThreads + tid) * VEC + e));
              if (k >= tau_key) {
                const int pos = atomicAdd(&sm.cnt, 1);
                if (pos < kCandCap) sm.cand[pos] = k;
              }
            }
          }
      }
      __syncthreads();
      if (sm.cnt <= kCandCap) break;
      // Overflow: the K-th best of the full buffer is a valid, strictly higher threshold. Drop this
      // tile's entries (earlier tiles' entries in [0, base_cnt) stay) and filter the tile again.
      select_topk(sm, kCandCap, K);
      if (tid == 0) {
        sm.tau = sm.topk[K - 1];
        sm.cnt = base_cnt;
      }
      __syncthreads();
      tau_key = sm.tau;
      tau_val = key_value(tau_key);
      if (++overflow_rounds > 64) {
        if (tid == 0) {
          sm.flag |= 2;
          sm.cnt = min(sm.cnt, kCandCap);
        }
        __syncthreads();
        break;
      }
    }

    // ---- release the stage and refill it ----
    if (tid == 0 && t + kStages < n_tiles) {
      fence_proxy_async_smem();
      const int64_t off = (int64_t)(t + kStages) * kTileBytes;
      const uint32_t bytes = (uint32_t)min((int64_t)kTileBytes, mid_bytes - off);
      mbar_arrive_expect_tx(&sm.bar[st], bytes);
      bulk_g2s(tiles + (size_t)st * kTileBytes, reinterpret_cast<const char*>(row + a0) + off, bytes,
               &sm.bar[st]);
    }

    // ---- compaction: after the first tile, and whenever the buffer is half full ----
    const int cnt = sm.cnt;
    if (t == 0 || cnt > kCandCap / 2) {
      const int n = compact_topk(sm, cnt, K);
      if (tid == 0) {
        sm.cnt = n;
        if (n == K) sm.tau = sm.cand[K - 1];
      }
      __syncthreads();
      tau_key = sm.tau;
      tau_val = tau_key ? key_value(tau_key) : -INFINITY;
    }
  }

  SegOut out;
  out.timed_out = timed_out;
  out.internal = (sm.flag & 2) != 0;
  out.bad = false;
  if (!SOFTMAX) out.bad = __syncthreads_or(bad_bits > 0x7F800000u || seen_max == INFINITY) != 0;
  // ---- final top-K ----
  {
    __syncthreads();
    const int cnt = min(sm.cnt, kCandCap);
    out.nkeys = compact_topk(sm, cnt, K);
  }
  // ---- block reduction of (m, s) ----
  out.m = -INFINITY;
  out.s = 0.0;
  if (SOFTMAX) {
    float bm = m_t;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
    if (lane == 0) sm.red_m[warp] = bm;
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < kRowThreads / 32; ++w) M = fmaxf(M, sm.red_m[w]);
    // NaN in a thread's sum propagates; a thread with m_t = +inf makes M = +inf (caller flags it).
    // Warp sums are double-float (hi, lo) pairs combined with TwoSum: no fp64 in the hot kernel.
    float ch = 0.0f, cl = 0.0f;
    if (m_t != -INFINITY || s_hi != s_hi) {
      const float sc = (M == m_t) ? 1.0f : ex2((m_t - M) * kLog2e);
      ch = s_hi * sc;
      cl = s_lo * sc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oh = __shfl_xor_sync(0xFFFFFFFFu, ch, o);
      const float ol = __shfl_xor_sync(0xFFFFFFFFu, cl, o);
      const float sum = ch + oh;
      const float bp = sum - ch;
      const float err = (ch - (sum - bp)) + (oh - bp);
      ch = sum;
      cl = cl + ol + err;
    }
    if (lane == 0) sm.red_s[warp] = (double)ch + (double)cl;
    __syncthreads();
    if (tid == 0) {
      double S = 0.0;
      for (int w = 0; w < kRowThreads / 32; ++w) S += sm.red_s[w];
      out.m = M;
      out.s = S;
    }
  } else {
    out.m = out.nkeys > 0 ? key_value(sm.cand[0]) : -INFINITY;
  }
  return out;
}

}  // namespace dt
