// Accepted-path KV compaction.
//
// EAGLE-2 page §"一段更贴近实现的流程": after verification the accepted tokens and their KV are
// committed to the cache and the rejected candidates' temporary KV is discarded (§"工程实现里的几个难点":
// the tree's KV lives in a temporary area while it is verified). Each request commits accept_len + 1
// rows: the root (the token committed last round, whose KV the verify forward computed at position 0)
// and the accepted positions, in path order, appended after its cache_len committed rows. A row is
// an opaque run of bytes (all layers' keys and values of one token); the copy is a bandwidth-bound
// gather of 16-byte vectors.
#include <algorithm>

#include "dt_internal.cuh"

namespace dt {
namespace {

struct KvArgs {
  Workspace ws;
  const uint4* tmp;
  int64_t tmp_pos, tmp_req;      // 16-byte vectors between positions / requests
  int32_t P;
  uint4* cache;
  int64_t cache_pos, cache_req;  // 16-byte vectors between cache rows / requests
  int32_t L_max;
  int64_t nv;                    // 16-byte vectors per row
  int32_t D_path, chunks;
  const int32_t* cache_len;
  const int32_t* accept_len;
  const int32_t* accept_path;
  const int32_t* tmp_row_off;    // [B+1] packed temporary rows (row_off[b] + i), or null: [B][P]
  int32_t* len_out;              // cache_len updated by the second kernel
};

constexpr int kKvThreads = 256;
constexpr int kKvPer = 8;                         // 16-byte vectors per thread
constexpr int kKvChunk = kKvThreads * kKvPer;     // vectors per CTA (32 KB)

// Request b commits n = accept_len[b] + 1 rows when they fit (len0 + n <= L_max) and its path is valid.
__device__ __forceinline__ bool kv_commit_ok(const KvArgs& a, int b, int& n, int& len0) {
  n = a.accept_len[b] + 1;
  len0 = a.cache_len[b];
  return n >= 1 && n <= a.D_path && len0 >= 0 && (int64_t)len0 + n <= a.L_max;
}

// Grid: B * D_path * chunks CTAs; CTA (b, j, c) copies chunk c (32 KB) of the j-th committed row of b.
__global__ void __launch_bounds__(kKvThreads) kv_commit_kernel(KvArgs a) {
  pdl_begin();
  const int c = (int)(blockIdx.x % a.chunks);
  const int bj = (int)(blockIdx.x / a.chunks);
  const int b = bj / a.D_path, j = bj - b * a.D_path;
  int n, len0;
  const bool ok = kv_commit_ok(a, b, n, len0);
  if (!ok) {
    if (j == 0 && c == 0 && threadIdx.x == 0) set_status(a.ws.status, DT_DEV_KV_FULL);
    return;
  }
  if (j >= n) return;
  const int pos = a.accept_path[(int64_t)b * a.D_path + j];
  const int rows_b = a.tmp_row_off ? a.tmp_row_off[b + 1] - a.tmp_row_off[b] : a.P;
  if (pos < 0 || pos >= a.P || pos >= rows_b) {
    if (c == 0 && threadIdx.x == 0) set_status(a.ws.status, DT_DEV_BAD_TREE);
    return;
  }
  const uint4* src = a.tmp_row_off ? a.tmp + ((int64_t)a.tmp_row_off[b] + pos) * a.tmp_pos
                                   : a.tmp + b * a.tmp_req + pos * a.tmp_pos;
  uint4* dst = a.cache + b * a.cache_req + (int64_t)(len0 + j) * a.cache_pos;
  // chunk c: vectors [c * kKvChunk, (c + 1) * kKvChunk); each thread loads its eight vectors before it
  // stores any (independent loads in flight, not a load-store chain)
  const int64_t v0 = (int64_t)c * kKvChunk + threadIdx.x;
  uint4 r[kKvPer];
#pragma unroll
  for (int u = 0; u < kKvPer; ++u) {
    const int64_t v = v0 + (int64_t)u * kKvThreads;
    if (v < a.nv) r[u] = __ldcs(src + v);
  }
#pragma unroll
  for (int u = 0; u < kKvPer; ++u) {
    const int64_t v = v0 + (int64_t)u * kKvThreads;
    if (v < a.nv) __stcs(dst + v, r[u]);
  }
}

// cache_len[b] += accept_len[b] + 1 for every request whose rows were committed.
__global__ void kv_len_kernel(KvArgs a, int B) {
  pdl_begin();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int n, len0;
  if (kv_commit_ok(a, b, n, len0)) a.len_out[b] = len0 + n;
}

}  // namespace

cudaError_t launch_commit_kv(dt_handle* h, const void* tmp_kv, int64_t tmp_pos_stride, int64_t tmp_req_stride, int P,
                             void* cache, int64_t cache_pos_stride, int64_t cache_req_stride, int L_max,
                             int64_t row_bytes, int32_t* cache_len, const int32_t* accept_len,
                             const int32_t* accept_path, int D_path, const int32_t* tmp_row_off,
                             cudaStream_t s) {
  KvArgs a;
  a.ws = h->ws;
  a.tmp = reinterpret_cast<const uint4*>(tmp_kv);
  a.tmp_pos = tmp_pos_stride / 16;
  a.tmp_req = tmp_req_stride / 16;
  a.P = P;
  a.cache = reinterpret_cast<uint4*>(cache);
  a.cache_pos = cache_pos_stride / 16;
  a.cache_req = cache_req_stride / 16;
  a.L_max = L_max;
  a.nv = row_bytes / 16;
  a.D_path = D_path;
  const int64_t chunks = std::max<int64_t>(1, (a.nv + kKvChunk - 1) / kKvChunk);
  if (chunks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  a.chunks = (int)chunks;
  a.cache_len = cache_len;
  a.accept_len = accept_len;
  a.accept_path = accept_path;
  a.tmp_row_off = tmp_row_off;
  a.len_out = cache_len;
  const int64_t grid = (int64_t)h->B * D_path * a.chunks;
  if (grid > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;  // rows of more than ~2^31 / (B D_path) x 32 KB
  launch_k(kv_commit_kernel, dim3((unsigned)grid), dim3(kKvThreads), 0, s, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_k(kv_len_kernel, dim3((h->B + 127) / 128), dim3(128), 0, s, a, h->B);
  return cudaGetLastError();
}

}  // namespace dt
