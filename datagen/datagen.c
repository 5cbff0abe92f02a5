/*
 * Seeded synthetic input generator shared by the tests, the benchmark and the
 * oracle harness.  It produces input data only: it holds none of the MoE
 * layer's arithmetic (no router, no softmax, no expert math, no dequantiser).
 *
 * Random numbers are counter based so that any slice of any tensor can be
 * regenerated on its own:
 *
 *   key(seed, stream) = mix64(mix64(seed) ^ (stream * 0xD1B54A32D192ED03))
 *   r(c)              = mix64(key + c * 0x9E3779B97F4A7C15)
 *
 * where mix64 is the splitmix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).  Normal
 * deviates use the Box-Muller transform (Box and Muller, 1958) on the pair
 * j = i / 2 of element i:
 *
 *   u1 = ((r(2j) >> 11) + 1) * 2^-53      in (0, 1]
 *   u2 =  (r(2j+1) >> 11) * 2^-53         in [0, 1)
 *   z  = sqrt(-2 ln u1) * (i even ? cos(2 pi u2) : sin(2 pi u2))
 *
 * evaluated in double, scaled by the standard deviation, rounded to fp32 and,
 * for bf16 tensors, rounded again to bf16 with round-to-nearest-even.
 *
 * The 4-bit encoder writes the block format of the decode 4-bit layer: blocks
 * of 32 consecutive elements along a row (the reduction dimension), one fp16
 * scale d = fp16(max|w| / 7) per block, q = clamp(round(w / d), -8, 7) with
 * rounding half away from zero, stored as q + 8, two values per byte with the
 * even element in the low nibble.  Each row is stored as its C/2 nibble bytes
 * followed by its C/32 fp16 scales (little endian), so a row is 9C/16 bytes.
 * Encoding the weights is input preparation (the layer only ever reads the
 * encoded form); decoding belongs to the layer and is not here.
 *
 * The int8 encoder writes one fp32 scale per row, s = fp32(max|w|) / 127 in
 * fp32, and q = clamp(round(w / s), -127, 127) (division in fp32, rounding
 * half away from zero; an all-zero row gets s = 0 and q = 0); a row is its C
 * signed bytes, then s (little endian), then 12 zero bytes, C + 16 bytes.
 *
 * Portable C11, no intrinsics: identical integer streams on x86-64 and
 * aarch64.  Built with -ffp-contract=off so the double arithmetic is not
 * fused differently on the two machines.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DG_GAMMA 0x9E3779B97F4A7C15ULL
#define DG_STREAM_MUL 0xD1B54A32D192ED03ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t dg_mix64(uint64_t z) { return mix64(z); }

uint64_t dg_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed) ^ (stream * DG_STREAM_MUL));
}

uint64_t dg_raw(uint64_t seed, uint64_t stream, uint64_t counter) {
  return mix64(dg_key(seed, stream) + counter * DG_GAMMA);
}

static double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t j = i >> 1;
  uint64_t a = mix64(key + (2 * j) * DG_GAMMA);
  uint64_t b = mix64(key + (2 * j + 1) * DG_GAMMA);
  double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
  double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
  double rad = sqrt(-2.0 * log(u1));
  return (i & 1) ? rad * sin(two_pi * u2) : rad * cos(two_pi * u2);
}

/* fp32 -> bf16 bits, round to nearest even; NaN kept quiet. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> IEEE binary16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t absu = u & 0x7FFFFFFFu;
  if (absu >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (absu > 0x7F800000u ? 0x200u : 0));
  if (absu >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to >= 65520: inf */
  if (absu < 0x38800000u) {                                   /* below 2^-14: subnormal half */
    if (absu < 0x33000000u) return (uint16_t)sign;            /* below 2^-25: rounds to 0 */
    uint32_t mant = (absu & 0x007FFFFFu) | 0x00800000u;
    int e = (int)(absu >> 23);                                 /* 102 .. 112 */
    int shift = 126 - e;                                       /* 14 .. 24 */
    uint32_t half = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u);
    uint32_t mid = 1u << (shift - 1);
    if (rem > mid || (rem == mid && (half & 1u))) half++;
    return (uint16_t)(sign | half);
  }
  uint32_t e = (absu >> 23) - 112u;
  uint32_t mant = absu & 0x007FFFFFu;
  uint32_t half = (e << 10) | (mant >> 13);
  uint32_t rem = mant & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (half & 1u))) half++;
  return (uint16_t)(sign | half);
}

static float f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1Fu;
  uint32_t m = h & 0x3FFu;
  uint32_t u;
  if (e == 0) {
    if (m == 0) {
      u = sign;
    } else { /* subnormal: m * 2^-24 */
      float f = (float)m * (1.0f / 16777216.0f);
      memcpy(&u, &f, 4);
      u |= sign;
    }
  } else if (e == 31) {
    u = sign | 0x7F800000u | (m << 13);
  } else {
    u = sign | ((e + 112u) << 23) | (m << 13);
  }
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t dg_f32_to_bf16(float f) { return f32_to_bf16(f); }
float dg_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }
uint16_t dg_f32_to_f16(float f) { return f32_to_f16(f); }
float dg_f16_to_f32(uint16_t h) { return f16_to_f32(h); }

/* ------------------------------------------------------------------ */
/* Threaded fill helpers                                               */

typedef struct {
  uint64_t key, offset;
  int64_t begin, end;
  double std;
  void* out;
  int kind; /* 0: f32, 1: bf16 */
} fill_job;

static void store_at(const fill_job* j, int64_t i, double z) {
  float v = (float)(z * j->std);
  if (j->kind == 0)
    ((float*)j->out)[i] = v;
  else
    ((uint16_t*)j->out)[i] = f32_to_bf16(v);
}

/* Elements of one Box-Muller pair share u1, u2 and the radius: both are
 * formed from one evaluation of them (the same expressions as normal_at,
 * so the same bits). */
static void* fill_worker(void* arg) {
  const double two_pi = 6.283185307179586476925286766559;
  fill_job* j = (fill_job*)arg;
  int64_t i = j->begin;
  while (i < j->end) {
    const uint64_t c = j->offset + (uint64_t)i;
    if ((c & 1) || i + 1 == j->end) {
      store_at(j, i, normal_at(j->key, c));
      ++i;
      continue;
    }
    const uint64_t a = mix64(j->key + c * DG_GAMMA);
    const uint64_t b = mix64(j->key + (c + 1) * DG_GAMMA);
    const double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
    const double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
    const double rad = sqrt(-2.0 * log(u1));
    store_at(j, i, rad * cos(two_pi * u2));
    store_at(j, i + 1, rad * sin(two_pi * u2));
    i += 2;
  }
  return NULL;
}

static void run_fill(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double std, void* out,
                     int kind, int nthreads) {
  if (n <= 0) return;
  uint64_t key = dg_key(seed, stream);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < (int64_t)1 << 16) nthreads = 1;
  fill_job jobs[256];
  pthread_t th[256];
  int created[256];
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int njobs = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[njobs++] = (fill_job){key, offset, b, e, std, out, kind};
  }
  for (int t = 1; t < njobs; ++t) created[t] = pthread_create(&th[t], NULL, fill_worker, &jobs[t]) == 0;
  fill_worker(&jobs[0]);
  for (int t = 1; t < njobs; ++t) {
    if (created[t])
      pthread_join(th[t], NULL);
    else
      fill_worker(&jobs[t]);
  }
}

/* Elements [offset, offset + n) of stream (seed, stream), N(0, std^2), as fp32. */
void dg_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double std, float* out,
                   int nthreads) {
  run_fill(seed, stream, offset, n, std, out, 0, nthreads);
}

/* Same values as dg_normal_f32, rounded to bf16 (round to nearest even). */
void dg_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double std, uint16_t* out,
                    int nthreads) {
  run_fill(seed, stream, offset, n, std, out, 1, nthreads);
}

void dg_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------ */
/* 4-bit block encoder (input preparation for the 4-bit weight format) */

/* Encode one row of `cols` bf16 values (cols % 32 == 0) into 9*cols/16 bytes. */
static void encode_row(const uint16_t* w, int64_t cols, uint8_t* dst) {
  uint8_t* nib = dst;
  uint8_t* sc = dst + cols / 2;
  for (int64_t b = 0; b < cols / 32; ++b) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
      float v = fabsf(bf16_to_f32(w[b * 32 + j]));
      if (v > amax) amax = v;
    }
    float d32 = amax / 7.0f;
    uint16_t dh = f32_to_f16(d32);
    float d = f16_to_f32(dh);
    sc[2 * b] = (uint8_t)(dh & 0xFF);
    sc[2 * b + 1] = (uint8_t)(dh >> 8);
    for (int j = 0; j < 32; j += 2) {
      int q[2];
      for (int h = 0; h < 2; ++h) {
        int qq = 0;
        if (d != 0.0f) {
          float r = roundf(bf16_to_f32(w[b * 32 + j + h]) / d);
          qq = (int)r;
          if (qq < -8) qq = -8;
          if (qq > 7) qq = 7;
        }
        q[h] = qq + 8;
      }
      nib[b * 16 + j / 2] = (uint8_t)(q[0] | (q[1] << 4));
    }
  }
}

typedef struct {
  const uint16_t* w;
  int64_t cols, r0, r1;
  uint8_t* out;
} enc_job;

static void* enc_worker(void* arg) {
  enc_job* j = (enc_job*)arg;
  int64_t rb = j->cols * 9 / 16;
  for (int64_t r = j->r0; r < j->r1; ++r) encode_row(j->w + r * j->cols, j->cols, j->out + r * rb);
  return NULL;
}

/* Encode a row-major [rows, cols] bf16 matrix.  Returns 0, or -1 when cols % 32 != 0. */
int dg_encode_q4b32(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* out, int nthreads) {
  if (cols % 32 != 0 || rows < 0) return -1;
  if (rows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (rows * cols < (int64_t)1 << 16) nthreads = 1;
  enc_job jobs[256];
  pthread_t th[256];
  int created[256];
  int njobs = 0;
  int64_t chunk = (rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= rows) break;
    if (e > rows) e = rows;
    jobs[njobs++] = (enc_job){w, cols, b, e, out};
  }
  for (int t = 1; t < njobs; ++t) created[t] = pthread_create(&th[t], NULL, enc_worker, &jobs[t]) == 0;
  enc_worker(&jobs[0]);
  for (int t = 1; t < njobs; ++t) {
    if (created[t])
      pthread_join(th[t], NULL);
    else
      enc_worker(&jobs[t]);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* int8 row encoder (input preparation for the int8 weight format)     */

/* Encode a row-major [rows, cols] bf16 matrix into rows of cols int8 values
 * followed by the row's fp32 scale and 12 bytes of padding.  Returns 0, or -1
 * when cols % 16 != 0. */
int dg_encode_i8(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* out) {
  if (cols % 16 != 0 || rows < 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* src = w + r * cols;
    uint8_t* dst = out + r * (cols + 16);
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) {
      float v = fabsf(bf16_to_f32(src[c]));
      if (v > amax) amax = v;
    }
    float s = amax / 127.0f;
    for (int64_t c = 0; c < cols; ++c) {
      int q = 0;
      if (s != 0.0f) {
        q = (int)roundf(bf16_to_f32(src[c]) / s);
        if (q > 127) q = 127;
        if (q < -127) q = -127;
      }
      dst[c] = (uint8_t)(int8_t)q;
    }
    memcpy(dst + cols, &s, 4);
    memset(dst + cols + 4, 0, 12);
  }
  return 0;
}
