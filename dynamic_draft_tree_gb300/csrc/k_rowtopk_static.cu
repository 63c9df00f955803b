// Row log-softmax top-K on a fixed static scratch: nothing on this path allocates.
//
// EAGLE-2 page, §"置信度为什么可以近似接受率" and §"扩展阶段": the confidence of a candidate
// token is its draft probability, and an expanded node's children are the top-K entries of
// softmax(row). This is the row pass of the layer expansion as a standalone op over plain rows.
// Its cross-CTA scratch (one partial result per row segment and one arrival counter per row)
// lives in file-scope device arrays of fixed size instead of a handle's workspace, so a caller
// needs no handle and no device allocation.
#include <algorithm>
#include <mutex>

#include "rowscan.cuh"

namespace dt {

namespace {

// Scratch shared by every call on a device (one copy per device context).
// g_static_partials: fully written by every call before it is read; no initial value needed.
// g_static_counter: MUST be zero when a call's kernel starts. It is zero at module load, and the
// last CTA of each row puts that row's counter back to zero, so every complete call leaves it zero.
static __device__ __align__(256) Partial g_static_partials[kStaticPartials];
static __device__ __align__(256) int32_t g_static_counter[kStaticRows];

struct StaticArgs {
  const void* logits;
  int64_t ld;
  int rows, S, K, V;
  int64_t seg_len;
  Partial* partials;
  int32_t* counter;
  float* logp;
  int32_t* ids;
  int32_t* status;
};

__device__ __forceinline__ void or_status(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// rows * S CTAs; CTA (r, seg) scans segment seg of row r, the last CTA of the row merges.
template <typename T>
__global__ void __launch_bounds__(kRowThreads, 3) row_topk_static_kernel(StaticArgs a) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ ScanSmem sm;
  const int r = blockIdx.x / a.S;
  const int seg = blockIdx.x % a.S;
  const int tid = threadIdx.x;

  const T* row = reinterpret_cast<const T*>(a.logits) + (int64_t)r * a.ld;
  const int64_t s0 = (int64_t)seg * a.seg_len;
  const int64_t s1 = min((int64_t)a.V, s0 + a.seg_len);
  SegOut so = scan_segment<T, true>(row, s0, s1, a.K, sm, dyn_smem, kSpinCap, nullptr);

  Partial* part = a.partials + (int64_t)r * a.S;
  if (tid < 32) {  // warp 0 publishes the segment, then (after a fence) its arrival
    if (tid < a.K) part[seg].keys[tid] = sm.topk[tid];
    if (tid == 0) {
      part[seg].m = so.m;
      part[seg].s_hi = so.s_hi;
      part[seg].s_lo = so.s_lo;
      if (so.timed_out) or_status(a.status, DT_DEV_TIMEOUT);
      if (so.internal) or_status(a.status, DT_DEV_INTERNAL);
    }
    __threadfence();
    __syncwarp();
    if (tid == 0) {
      const int prev = atomicAdd(&a.counter[r], 1);
      sm.last = (prev == a.S - 1);
    }
  }
  __syncthreads();
  if (!sm.last) return;

  // ---- last segment of the row: merge the partials, write K (log p, id) pairs ----
  __threadfence();
  if (tid == 0) a.counter[r] = 0;  // back to zero for the next call
  const int nk = a.S * a.K;
  for (int i = tid; i < nk; i += blockDim.x) sm.cand[i] = __ldcg(&part[i / a.K].keys[i % a.K]);
  float m0 = -INFINITY, h0 = 0.0f, l0 = 0.0f, m1 = -INFINITY, h1 = 0.0f, l1 = 0.0f;
  if (tid < 32) {
    if (tid < a.S) {
      m0 = __ldcg(&part[tid].m);
      h0 = __ldcg(&part[tid].s_hi);
      l0 = __ldcg(&part[tid].s_lo);
    }
    if (tid + 32 < a.S) {
      m1 = __ldcg(&part[tid + 32].m);
      h1 = __ldcg(&part[tid + 32].s_hi);
      l1 = __ldcg(&part[tid + 32].s_lo);
    }
  }
  if (tid < kMaxK) sm.topk[tid] = 0ull;
  __syncthreads();
  if (tid < 32) combine_partial_sums(sm, m0, h0, l0, m1, h1, l1);
  merge_sorted_lists(sm, sm.cand, a.S, a.K, a.K);
  const float M = sm.red_m[0];
  const double Ssum = (double)sm.red_sh[0] + (double)sm.red_sl[0];
  const bool nan = Ssum != Ssum;
  if (tid == 0 && (nan || !(M > -INFINITY) || M == INFINITY || !(Ssum > 0.0)))
    or_status(a.status, DT_DEV_BAD_LOGITS);
  // log S from the exponent (exact) plus the fp32 log of the mantissa in [1, 2)
  double logS;
  {
    const unsigned long long bits = (unsigned long long)__double_as_longlong(Ssum);
    const int e = (int)((bits >> 52) & 0x7FF) - 1023;
    const double mant = __longlong_as_double((long long)((bits & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull));
    logS = (double)e * 0.6931471805599453 + (double)logf((float)mant);
    if (!(Ssum > 0.0) || Ssum != Ssum || e == 1024) logS = log(Ssum);
  }
  if (tid < a.K) {
    const uint64_t k = sm.topk[tid];
    const int64_t o = (int64_t)r * a.K + tid;
    a.logp[o] = (float)(((double)key_value(k) - (double)M) - logS);
    a.ids[o] = (int32_t)key_id(k);
  }
}

struct StaticDevice {
  bool ready = false;
  Partial* partials = nullptr;
  int32_t* counter = nullptr;
  int num_sms = 0;
};

constexpr int kMaxDevices = 64;
StaticDevice g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device set-up, once: the scratch addresses, the SM count and the kernels' shared-memory limit.
cudaError_t static_setup(int dev, StaticDevice* out) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  StaticDevice& d = g_dev[dev];
  if (!d.ready) {
    cudaError_t e = cudaGetSymbolAddress((void**)&d.partials, g_static_partials);
    if (e == cudaSuccess) e = cudaGetSymbolAddress((void**)&d.counter, g_static_counter);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(row_topk_static_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kScanSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(row_topk_static_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kScanSmemBytes);
    if (e != cudaSuccess) return e;
    d.ready = true;
  }
  *out = d;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_row_topk_static(const void* logits, int64_t ld, int rows, int V, int K, int dtype, float* logp,
                                   int32_t* ids, int32_t* status, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  StaticDevice d;
  e = static_setup(dev, &d);
  if (e != cudaSuccess) return e;

  // segments: one wave of CTAs (3 per SM), at least 8 KB per segment, within the scratch
  const int64_t row_bytes = (int64_t)V * (dtype == DT_BF16 ? 2 : 4);
  int64_t S = ((int64_t)d.num_sms * 3 + rows - 1) / rows;
  S = std::min<int64_t>(S, (row_bytes + 8191) / 8192);
  S = std::min<int64_t>(S, kCandCap / K);
  S = std::min<int64_t>(S, 64);
  S = std::min<int64_t>(S, kStaticPartials / rows);
  if (S < 1) S = 1;
  int64_t L = ((int64_t)V + S - 1) / S;
  L = (L + 7) / 8 * 8;

  StaticArgs a;
  a.logits = logits;
  a.ld = ld;
  a.rows = rows;
  a.S = (int)S;
  a.K = K;
  a.V = V;
  a.seg_len = L;
  a.partials = d.partials;
  a.counter = d.counter;
  a.logp = logp;
  a.ids = ids;
  a.status = status;
  const unsigned grid = (unsigned)(rows * S);
  if (dtype == DT_BF16)
    row_topk_static_kernel<uint16_t><<<grid, kRowThreads, kScanSmemBytes, s>>>(a);
  else
    row_topk_static_kernel<float><<<grid, kRowThreads, kScanSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dt
