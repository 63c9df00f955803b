// Seeded synthetic logits rows, device implementation (the draft/target model
// forwards are replaced by this generator; it is not part of the draft-tree
// path and is never timed as part of it).
//
// Same definition as synth_cpu.c, written for the device: integer hashing,
// then fp32 steps with explicit round-to-nearest intrinsics so that nothing is
// fused and every step rounds once, exactly as on the host. The test suite
// checks host and device rows for bitwise equality.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;
constexpr uint64_t PEAK_SALT = 0xA5A5A5A5C3C3C3C3ULL;
constexpr uint64_t HEIGHT_SALT = 0x3C3C3C3C5A5A5A5AULL;
constexpr uint64_t ZIPF_A_SALT = 0x1234567890ABCDEFULL;
constexpr uint64_t ZIPF_C_SALT = 0x0FEDCBA987654321ULL;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

__host__ __device__ __forceinline__ uint64_t hk(uint64_t a, uint64_t x) {
  return mix64(a ^ mix64(x + GOLDEN));
}

__device__ __forceinline__ uint64_t gcd64(uint64_t a, uint64_t b) {
  while (b) {
    uint64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

__device__ __forceinline__ int32_t ih12(uint64_t r, uint64_t v, uint64_t lane) {
  int64_t s = 0;
#pragma unroll
  for (uint64_t j = 0; j < 3; ++j) {
    uint64_t w = mix64(r ^ ((v << 3) | (lane << 2) | j));
#pragma unroll
    for (int q = 0; q < 4; ++q) s += (int64_t)((w >> (16 * q)) & 0xFFFFu);
  }
  return (int32_t)(s - 393210);
}

__device__ __forceinline__ uint16_t bf16_rne(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

struct RowParams {
  uint64_t r;
  int64_t peak;
  float h;
  uint64_t za, zc;
  int valid;
};

}  // namespace

extern "C" {

struct synth_spec {
  int32_t kind;
  int32_t V;
  int32_t dtype;
  int32_t height_per_request;
  float sigma;
  float zipf_s;
  const float* peak_lo;   // [B] device
  const float* peak_hi;   // [B] device
  const float* ln_table;  // [V] device
  const uint64_t* salts;  // [B] device per-request salt, or null for the call's salt
};

}

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;

__global__ void __launch_bounds__(kThreads) gen_rows_kernel(
    synth_spec sp, uint64_t seed, uint64_t salt, int32_t stream, const int32_t* __restrict__ ctx,
    const int32_t* __restrict__ depth, int32_t depth_add, int32_t rows_per_b, const int32_t* __restrict__ row_req,
    void* out, int64_t ld) {
  const int rr = blockIdx.y;
  __shared__ RowParams rp;
  if (threadIdx.x == 0) {
    const int32_t c = ctx[rr];
    rp.valid = c >= 0;
    if (rp.valid) {
      const int64_t b = row_req ? row_req[rr] : rr / rows_per_b;
      if (sp.salts) salt = sp.salts[b];
      const int64_t dk = (int64_t)(depth ? depth[rr] : 0) + depth_add;
      const uint64_t r = hk(hk(hk(hk(seed, salt), (uint64_t)b), (uint64_t)dk), (uint64_t)c);
      rp.r = r;
      rp.peak = -1;
      rp.h = 0.0f;
      rp.za = rp.zc = 0;
      if (sp.kind != 1) {
        rp.peak = (int64_t)(mix64(r ^ PEAK_SALT) % (uint64_t)sp.V);
        uint64_t hsrc = sp.height_per_request ? hk(hk(seed, salt), (uint64_t)b) : r;
        uint32_t u24 = (uint32_t)(mix64(hsrc ^ HEIGHT_SALT) >> 40);
        float uf = __fmul_rn((float)u24, 1.0f / 16777216.0f);
        float lo = sp.peak_lo[b];
        float range = __fsub_rn(sp.peak_hi[b], lo);
        rp.h = __fadd_rn(lo, __fmul_rn(range, uf));
      }
      if (sp.kind != 0) {
        uint64_t a = mix64(r ^ ZIPF_A_SALT) % (uint64_t)(sp.V - 1) + 1;
        while (gcd64(a, (uint64_t)sp.V) != 1) a = a % (uint64_t)(sp.V - 1) + 1;
        rp.za = a;
        rp.zc = mix64(r ^ ZIPF_C_SALT) % (uint64_t)sp.V;
        // kind 2: shift the permutation so that the peak token holds rank 0 (the Zipf mode)
        if (sp.kind == 2) rp.zc = ((uint64_t)sp.V - (a * (uint64_t)rp.peak) % (uint64_t)sp.V) % (uint64_t)sp.V;
      }
    }
  }
  __syncthreads();
  if (!rp.valid) return;
  const float sA = (float)((double)sp.sigma / 65536.0);
  const float sT = (float)((double)sp.sigma / (5.0 * 65536.0));
  const int64_t v0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * kPerThread;
  for (int k = 0; k < kPerThread; ++k) {
    const int64_t v = v0 + k;
    if (v >= sp.V) break;
    const int32_t ia = ih12(rp.r, (uint64_t)v, 0);
    float noise;
    if (stream == 0) {
      noise = __fmul_rn((float)ia, sA);
    } else {
      const int32_t ib = ih12(rp.r, (uint64_t)v, 1);
      noise = __fmul_rn((float)(4 * ia + 3 * ib), sT);
    }
    float x = noise;
    if (sp.kind != 0) {
      const uint64_t rank = (rp.za * (uint64_t)v + rp.zc) % (uint64_t)sp.V;
      x = __fadd_rn(__fmul_rn(-sp.zipf_s, sp.ln_table[rank]), noise);
    }
    if (v == rp.peak) x = __fadd_rn(x, rp.h);
    if (sp.dtype == 0)
      reinterpret_cast<uint16_t*>(out)[(int64_t)rr * ld + v] = bf16_rne(x);
    else
      reinterpret_cast<float*>(out)[(int64_t)rr * ld + v] = x;
  }
}

}  // namespace

extern "C" int synth_gen_rows_gpu(const synth_spec* sp, uint64_t seed, uint64_t salt, int32_t stream,
                                  const int32_t* ctx, const int32_t* depth, int32_t depth_add,
                                  int32_t rows_per_b, const int32_t* row_req, void* out, int64_t ld,
                                  int32_t R, cudaStream_t cs) {
  if (R <= 0) return 0;
  if (sp == nullptr || ctx == nullptr || out == nullptr || rows_per_b <= 0 || sp->V < 2 || ld < sp->V)
    return -1;
  if (R > 65535) return -1;
  dim3 grid((unsigned)((sp->V + kThreads * kPerThread - 1) / (kThreads * kPerThread)), (unsigned)R);
  gen_rows_kernel<<<grid, kThreads, 0, cs>>>(*sp, seed, salt, stream, ctx, depth, depth_add, rows_per_b,
                                              row_req, out, ld);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// ---- host rows into device buffers by a kernel (end-to-end timing) ----
// A span moves `bytes` from src (pinned host memory, through its device mapping) to dst (device
// memory). The SMs read the host memory directly over the host link, many loads in flight, instead of
// one DMA copy per span.
extern "C" {
struct synth_span {
  const void* src;
  void* dst;
  int64_t bytes;
};
}

namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherMaxSpans = 512;
constexpr int64_t kGatherUnit = (int64_t)kGatherThreads * 16 * 16;  // bytes of one work item (64 KB)

__global__ void __launch_bounds__(kGatherThreads) gather_spans_kernel(const synth_span* __restrict__ spans, int n) {
  __shared__ int64_t first[kGatherMaxSpans + 1];  // first work item of each span
  __shared__ synth_span sp[kGatherMaxSpans];
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    for (int i = 0; i < n; ++i) {
      sp[i] = spans[i];
      first[i] = acc;
      acc += (sp[i].bytes + kGatherUnit - 1) / kGatherUnit;
    }
    first[n] = acc;
  }
  __syncthreads();
  const int64_t items = first[n];
  int span = 0;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    while (span + 1 < n && first[span + 1] <= it) ++span;  // items grow, so the span only moves forward
    const synth_span s = sp[span];
    const int64_t lo = (it - first[span]) * kGatherUnit;
    const int64_t hi = lo + kGatherUnit < s.bytes ? lo + kGatherUnit : s.bytes;
    const char* src = static_cast<const char*>(s.src) + lo;
    char* dst = static_cast<char*>(s.dst) + lo;
    const int64_t nb = hi - lo;
    if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)nb) & 15u) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      const int n4 = (int)(nb / 16);
      uint4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int q = threadIdx.x + u * kGatherThreads;
        if (q < n4) v[u] = s4[q];
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int q = threadIdx.x + u * kGatherThreads;
        if (q < n4) d4[q] = v[u];
      }
    } else {
      for (int64_t q = threadIdx.x; q < nb; q += kGatherThreads) dst[q] = src[q];
    }
  }
}

}  // namespace

// Device address of pinned host memory (0 on success).
extern "C" int synth_host_device_ptr(void* host, void** dev) {
  return cudaHostGetDevicePointer(dev, host, 0) == cudaSuccess ? 0 : -1;
}

// Moves every span (descriptors in device memory) with `blocks` CTAs on stream cs.
extern "C" int synth_gather_spans_gpu(const synth_span* spans_dev, int32_t n, int32_t blocks, cudaStream_t cs) {
  if (n <= 0) return 0;
  if (spans_dev == nullptr || n > kGatherMaxSpans || blocks <= 0) return -1;
  gather_spans_kernel<<<blocks, kGatherThreads, 0, cs>>>(spans_dev, n);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
