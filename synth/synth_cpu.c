/* Seeded synthetic logits rows, host implementation.
 *
 * Holds none of the draft-tree arithmetic: it only produces the inputs that
 * the oracle and the GPU path both consume. The device twin (synth_gpu.cu)
 * implements the same definition and must agree bit for bit; the test suite
 * checks that. The definition (integer core, explicit fp32 rounding steps) is
 * spelled out in synth/__init__.py.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared (no fused multiply-add, so
 * every fp32 product and sum is rounded exactly once, as on the device).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define PEAK_SALT 0xA5A5A5A5C3C3C3C3ULL
#define HEIGHT_SALT 0x3C3C3C3C5A5A5A5AULL
#define ZIPF_A_SALT 0x1234567890ABCDEFULL
#define ZIPF_C_SALT 0x0FEDCBA987654321ULL
#define ROOT_SALT 0x7777777711111111ULL

/* SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014). */
static uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static uint64_t hk(uint64_t a, uint64_t x) { return mix64(a ^ mix64(x + GOLDEN)); }

static uint64_t gcd64(uint64_t a, uint64_t b) {
  while (b) {
    uint64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

static uint16_t f32_to_bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

typedef struct {
  int32_t kind;        /* 0 = normal noise + one peak, 1 = Zipf over a permutation + noise,
                          2 = Zipf + noise + one peak */
  int32_t V;
  int32_t dtype;       /* 0 = bf16, 1 = fp32 */
  int32_t height_per_request;
  float sigma;         /* noise standard deviation */
  float zipf_s;        /* Zipf exponent (kind 1) */
  const float* peak_lo;  /* [B] */
  const float* peak_hi;  /* [B] */
  const float* ln_table; /* [V], kind 1: ln(rank + 1) rounded to fp32 */
  const uint64_t* salts; /* [B] per-request salt, or NULL for the call's salt */
} synth_spec;

/* Integer Irwin-Hall sum of 12 16-bit uniforms, centred: in [-393210, 393210]. */
static int32_t ih12(uint64_t r, uint64_t v, uint64_t lane) {
  int64_t s = 0;
  for (uint64_t j = 0; j < 3; ++j) {
    uint64_t w = mix64(r ^ ((v << 3) | (lane << 2) | j));
    for (int q = 0; q < 4; ++q) s += (int64_t)((w >> (16 * q)) & 0xFFFFu);
  }
  return (int32_t)(s - 393210);
}

uint64_t synth_row_key(uint64_t seed, uint64_t salt, int64_t b, int64_t depthkey, int64_t ctx) {
  return hk(hk(hk(hk(seed, salt), (uint64_t)b), (uint64_t)depthkey), (uint64_t)ctx);
}

int32_t synth_root_token(uint64_t seed, uint64_t salt, int64_t b, int32_t V) {
  return (int32_t)(hk(hk(seed, salt), (uint64_t)b ^ ROOT_SALT) % (uint64_t)V);
}

void synth_zipf_table(int32_t V, float* out) {
  for (int32_t k = 0; k < V; ++k) out[k] = (float)log((double)k + 1.0);
}

/* One row. stream 0 = draft, 1 = target. */
static void gen_row(const synth_spec* sp, uint64_t seed, uint64_t salt, int stream, int64_t b,
                    int64_t depthkey, int64_t ctx, void* out) {
  const int32_t V = sp->V;
  if (sp->salts) salt = sp->salts[b];
  const uint64_t r = synth_row_key(seed, salt, b, depthkey, ctx);
  const float sA = (float)((double)sp->sigma / 65536.0);
  const float sT = (float)((double)sp->sigma / (5.0 * 65536.0));
  int64_t peak = -1;
  float h = 0.0f;
  uint64_t za = 0, zc = 0;
  if (sp->kind != 1) {
    peak = (int64_t)(mix64(r ^ PEAK_SALT) % (uint64_t)V);
    uint64_t hsrc = sp->height_per_request ? hk(hk(seed, salt), (uint64_t)b) : r;
    uint32_t u24 = (uint32_t)(mix64(hsrc ^ HEIGHT_SALT) >> 40);
    float uf = (float)u24 * (1.0f / 16777216.0f);
    float lo = sp->peak_lo[b], range = sp->peak_hi[b] - sp->peak_lo[b];
    float t = range * uf;
    h = lo + t;
  }
  if (sp->kind != 0) {
    za = mix64(r ^ ZIPF_A_SALT) % (uint64_t)(V - 1) + 1;
    while (gcd64(za, (uint64_t)V) != 1) za = za % (uint64_t)(V - 1) + 1;
    zc = mix64(r ^ ZIPF_C_SALT) % (uint64_t)V;
    /* kind 2: shift the permutation so that the peak token holds rank 0 (the Zipf mode) */
    if (sp->kind == 2) zc = ((uint64_t)V - (za * (uint64_t)peak) % (uint64_t)V) % (uint64_t)V;
  }
  for (int32_t v = 0; v < V; ++v) {
    int32_t ia = ih12(r, (uint64_t)v, 0);
    float noise;
    if (stream == 0) {
      noise = (float)ia * sA;
    } else {
      int32_t ib = ih12(r, (uint64_t)v, 1);
      noise = (float)(4 * ia + 3 * ib) * sT;
    }
    float x = noise;
    if (sp->kind != 0) {
      uint64_t rank = (za * (uint64_t)v + zc) % (uint64_t)V;
      float base = (-sp->zipf_s) * sp->ln_table[rank];
      x = base + noise;
    }
    if (v == peak) x = x + h;
    if (sp->dtype == 0)
      ((uint16_t*)out)[v] = f32_to_bf16_rne(x);
    else
      ((float*)out)[v] = x;
  }
}

/* R rows. Row rr uses request b = b0 + rr / rows_per_b, context token ctx[rr]
 * (rows with ctx < 0 are left untouched) and depth key
 * (depth ? depth[rr] : 0) + depth_add. Row rr starts at element rr * ld. */
void synth_gen_rows(const synth_spec* sp, uint64_t seed, uint64_t salt, int32_t stream,
                    const int32_t* ctx, const int32_t* depth, int32_t depth_add, int32_t rows_per_b,
                    int32_t b0, void* out, int64_t ld, int32_t R) {
  const size_t esz = sp->dtype == 0 ? 2 : 4;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t rr = 0; rr < R; ++rr) {
    if (ctx[rr] < 0) continue;
    int64_t b = b0 + rr / rows_per_b;
    int64_t dk = (int64_t)(depth ? depth[rr] : 0) + depth_add;
    gen_row(sp, seed, salt, stream, b, dk, ctx[rr], (char*)out + (size_t)rr * (size_t)ld * esz);
  }
}
