/*
 * Seeded synthetic inputs for the quantized MoE layer: Gaussian weights and
 * activations from a counter-based generator, and the checkpoint encoders
 * that turn FP32 weights into the published block-quantized formats.
 *
 * This file is input synthesis only.  It produces what a checkpoint and a
 * batch of activations would contain; it holds none of the layer's own
 * arithmetic (no decoding, routing, GEMV or combine).  Both the CUDA path and
 * the oracle consume what it writes.
 *
 * Random numbers: a SplitMix64-style counter generator.  Element i of a
 * stream keyed by (seed, kind, expert, projection) is the SplitMix64 output
 * function applied to key + (i + 1) * 0x9E3779B97F4A7C15 (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Normals use the Box-Muller transform on element pairs (2j, 2j+1).  Any
 * expert of any tensor can be regenerated alone, in any order, on any thread.
 *
 * Encoders (the DGPP pages serve NVFP4, MXFP4, int4/int8 group-64 and FP8
 * block-128 checkpoints but do not say how they were produced; the rules
 * below are the plain readings of the public format definitions):
 *   NVFP4  tensor scale ts = fl32(amax / (6 * 448)); per 16-element block
 *          s = e4m3_rne_sat(amax_blk / (6 * ts)); code = e2m1_rne_sat(x / (s * ts)).
 *   MXFP4  per 32-element block e = smallest integer with 6 * 2^e >= amax_blk
 *          (stored as e + 127, clamped to [0, 254]); code = e2m1_rne_sat(x / 2^e).
 *   INT4   per 64-element group s = bf16_rne(amax / 7), q = clamp(rne(x / s), -8, 7).
 *   INT8   per 64-element group s = bf16_rne(amax / 127), q = clamp(rne(x / s), -127, 127).
 *   FP8    per 128x128 block s = fl32(amax / 448), q = e4m3_rne_sat(x / s).
 * E2M1 rounding is round-to-nearest with ties to the even code; a zero scale
 * gives all-zero codes.
 *
 * Built with -ffp-contract=off so results do not depend on FMA contraction.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define QS_GOLDEN 0x9E3779B97F4A7C15ull

enum { QS_NVFP4 = 1, QS_MXFP4 = 2, QS_INT4_G64 = 3, QS_INT8_G64 = 4, QS_FP8_B128 = 5, QS_INT4_G128 = 6 };

static inline uint64_t qs_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t qs_stream_key(uint64_t seed, uint32_t kind, uint32_t expert, uint32_t proj) {
  uint64_t k = qs_mix(seed + QS_GOLDEN);
  k = qs_mix(k ^ (((uint64_t)kind << 48) | ((uint64_t)proj << 40) | (uint64_t)expert));
  return k;
}

uint64_t qs_draw_u64(uint64_t key, uint64_t i) { return qs_mix(key + (i + 1) * QS_GOLDEN); }

static inline double qs_normal_at(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  uint64_t a = qs_draw_u64(key, 2 * j), b = qs_draw_u64(key, 2 * j + 1);
  double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
  double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);         /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* Both members of Box-Muller pair j: element 2j takes the cosine, 2j+1 the sine. */
static inline void qs_normal_pair(uint64_t key, uint64_t j, double* c, double* s) {
  uint64_t a = qs_draw_u64(key, 2 * j), b = qs_draw_u64(key, 2 * j + 1);
  double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0);
  double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  *c = r * cos(t);
  *s = r * sin(t);
}

void qs_normal_f32(uint64_t key, uint64_t start, uint64_t n, double sigma, float* out) {
  uint64_t i = 0;
  if ((start & 1) && n) { out[0] = (float)(sigma * qs_normal_at(key, start)); i = 1; }
  for (; i + 1 < n; i += 2) {
    double c, s;
    qs_normal_pair(key, (start + i) >> 1, &c, &s);
    out[i] = (float)(sigma * c);
    out[i + 1] = (float)(sigma * s);
  }
  if (i < n) out[i] = (float)(sigma * qs_normal_at(key, start + i));
}

/* float -> bf16 bits, round to nearest even (NaN kept quiet). */
static inline uint16_t qs_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* double -> bf16 bits with a single round-to-nearest-even (finite inputs). */
static inline uint16_t qs_f64_to_bf16(double d) {
  if (d == 0.0) return signbit(d) ? 0x8000 : 0;
  int e;
  double m = frexp(fabs(d), &e); /* |d| = m * 2^e, m in [0.5, 1) */
  /* bf16 normal: 8 significant bits; subnormal below 2^-126 */
  int q = e - 8; /* spacing exponent for 8 significant bits */
  if (e - 1 < -126) q = -133;
  double scaled = ldexp(fabs(d), -q);
  double r = nearbyint(scaled); /* default rounding mode: ties to even */
  double v = ldexp(r, q);
  float f = (float)v; /* exact: v has <= 8 significant bits, within float range */
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t bits = (uint16_t)(u >> 16);
  if (signbit(d)) bits |= 0x8000;
  return bits;
}

void qs_normal_bf16(uint64_t key, uint64_t start, uint64_t n, double sigma, uint16_t* out) {
  float buf[256];
  for (uint64_t i = 0; i < n; i += 256) {
    uint64_t m = (n - i < 256) ? n - i : 256;
    qs_normal_f32(key, start + i, m, sigma, buf);
    for (uint64_t j = 0; j < m; ++j) out[i + j] = qs_f32_to_bf16(buf[j]);
  }
}

/* ---- minifloat encoders (round to nearest, ties to even code, saturating) ---- */

/* Magnitude grid of E2M1 indexed by the 3-bit code. */
static const double kE2m1Grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static inline uint8_t qs_e2m1_encode(double y) {
  uint8_t sign = (y < 0.0) ? 8 : 0;
  double a = fabs(y);
  if (a >= 6.0) return sign | 7;
  int lo = 0;
  while (lo < 7 && kE2m1Grid[lo + 1] <= a) ++lo;
  if (kE2m1Grid[lo] == a) return sign | (uint8_t)lo;
  double dlo = a - kE2m1Grid[lo], dhi = kE2m1Grid[lo + 1] - a;
  int code;
  if (dlo < dhi) code = lo;
  else if (dhi < dlo) code = lo + 1;
  else code = (lo & 1) ? lo + 1 : lo; /* tie: even code */
  return sign | (uint8_t)code;
}

/* Non-negative value -> E4M3 code (sign bit 0), RNE, saturate at 448. */
static inline uint8_t qs_e4m3_encode_mag(double a) {
  if (!(a > 0.0)) return 0;
  if (a >= 448.0) return 0x7E;
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int ue = e - 1;  /* unbiased exponent of the leading bit */
  if (ue < -6) ue = -6; /* subnormal binade shares spacing 2^-9 */
  double spacing = ldexp(1.0, ue - 3);
  double r = nearbyint(a / spacing); /* exact division by a power of two */
  double v = r * spacing;
  if (v >= 448.0) return 0x7E;
  if (v == 0.0) return 0;
  frexp(v, &e);
  int ve = e - 1;
  if (ve < -6) { /* subnormal: mantissa = v / 2^-9 */
    return (uint8_t)(int)(v / ldexp(1.0, -9));
  }
  int mant = (int)(v / ldexp(1.0, ve - 3)) - 8;
  return (uint8_t)(((ve + 7) << 3) | mant);
}

static inline uint8_t qs_e4m3_encode(double y) {
  uint8_t m = qs_e4m3_encode_mag(fabs(y));
  if (y < 0.0 && m != 0) m |= 0x80;
  return m;
}

static inline double qs_e4m3_value_mag(uint8_t c) {
  int e = (c >> 3) & 15, m = c & 7;
  if (e == 0) return ldexp((double)m, -9);
  return ldexp(1.0 + m / 8.0, e - 7);
}

/* ---- per-format matrix encoders: W[N, K] row-major, K innermost ---- */

static void qs_quant_nvfp4(const float* W, int N, int K, uint8_t* data, uint8_t* sc, float* ts_out) {
  float amax = 0.0f;
  for (size_t i = 0; i < (size_t)N * K; ++i) { float a = fabsf(W[i]); if (a > amax) amax = a; }
  float ts = amax / 2688.0f; /* 6 * 448, fl32 division */
  *ts_out = ts;
  for (int n = 0; n < N; ++n) {
    const float* row = W + (size_t)n * K;
    for (int b = 0; b < K / 16; ++b) {
      double ablk = 0.0;
      for (int i = 0; i < 16; ++i) { double a = fabs((double)row[b * 16 + i]); if (a > ablk) ablk = a; }
      uint8_t s = (ts > 0.0f) ? qs_e4m3_encode_mag(ablk / (6.0 * (double)ts)) : 0;
      sc[(size_t)n * (K / 16) + b] = s;
      double step = qs_e4m3_value_mag(s) * (double)ts;
      for (int i = 0; i < 16; i += 2) {
        uint8_t c0 = 0, c1 = 0;
        if (s != 0) {
          c0 = qs_e2m1_encode((double)row[b * 16 + i] / step);
          c1 = qs_e2m1_encode((double)row[b * 16 + i + 1] / step);
        }
        data[(size_t)n * (K / 2) + (b * 16 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

static void qs_quant_mxfp4(const float* W, int N, int K, uint8_t* data, uint8_t* sc) {
  for (int n = 0; n < N; ++n) {
    const float* row = W + (size_t)n * K;
    for (int b = 0; b < K / 32; ++b) {
      double ablk = 0.0;
      for (int i = 0; i < 32; ++i) { double a = fabs((double)row[b * 32 + i]); if (a > ablk) ablk = a; }
      int e = 0;
      if (ablk > 0.0) {
        int q;
        frexp(ablk, &q);
        e = q - 3;
        while (6.0 * ldexp(1.0, e) < ablk) ++e;
        while (6.0 * ldexp(1.0, e - 1) >= ablk) --e;
      }
      int code = e + 127;
      if (code < 0) code = 0;
      if (code > 254) code = 254;
      sc[(size_t)n * (K / 32) + b] = (uint8_t)code;
      double step = ldexp(1.0, code - 127);
      for (int i = 0; i < 32; i += 2) {
        uint8_t c0 = qs_e2m1_encode((double)row[b * 32 + i] / step);
        uint8_t c1 = qs_e2m1_encode((double)row[b * 32 + i + 1] / step);
        data[(size_t)n * (K / 2) + (b * 32 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

static double qs_f16_value(uint16_t b) {
  const int e = (b >> 10) & 0x1F, m = b & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x400), e - 25);
  return (b & 0x8000) ? -v : v;
}

static inline double qs_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static void qs_quant_int_g64(const float* W, int N, int K, int bits, uint8_t* data, uint16_t* sc) {
  const double qmax = (bits == 4) ? 7.0 : 127.0;
  const double qmin = (bits == 4) ? -8.0 : -127.0;
  for (int n = 0; n < N; ++n) {
    const float* row = W + (size_t)n * K;
    for (int g = 0; g < K / 64; ++g) {
      double agrp = 0.0;
      for (int i = 0; i < 64; ++i) { double a = fabs((double)row[g * 64 + i]); if (a > agrp) agrp = a; }
      uint16_t sb = qs_f64_to_bf16(agrp / qmax);
      sc[(size_t)n * (K / 64) + g] = sb;
      double s = qs_bf16_value(sb);
      for (int i = 0; i < 64; ++i) {
        double q = 0.0;
        if (s != 0.0) {
          q = nearbyint((double)row[g * 64 + i] / s);
          if (q > qmax) q = qmax;
          if (q < qmin) q = qmin;
        }
        int qi = (int)q;
        size_t k = (size_t)g * 64 + i;
        if (bits == 4) {
          uint8_t nib = (uint8_t)(qi & 15);
          uint8_t* p = data + (size_t)n * (K / 2) + k / 2;
          if (k & 1) *p = (uint8_t)((*p & 0x0F) | (nib << 4));
          else *p = (uint8_t)((*p & 0xF0) | nib);
        } else {
          data[(size_t)n * K + k] = (uint8_t)(int8_t)qi;
        }
      }
    }
  }
}

/* Nearest binary16 of a double (ties to even), as bits; overflow to infinity. */
static uint16_t qs_f64_to_f16(double v) {
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double a = fabs(v);
  if (isnan(v)) return 0x7E00;
  if (a == 0.0) return sign;
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00);
  int ex;
  frexp(a, &ex);
  int E = ex - 1;                             /* 2^E <= a < 2^(E+1) */
  if (E < -14) {                              /* subnormal: quantum 2^-24 */
    const double q = nearbyint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)q);    /* q == 1024 is the smallest normal, 0x0400 */
  }
  double q = nearbyint(ldexp(a, 10 - E));     /* 1024 .. 2048 */
  if (q >= 2048.0) { q = 1024.0; ++E; }
  if (E > 15) return (uint16_t)(sign | 0x7C00);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* AutoRound / GPTQ-style int4 with group 128: s = f16(amax / 7) per 128
 * columns, q = clamp(rne(x / s), -8, 7) stored as the unsigned nibble q + 8
 * (zero point 8), low nibble = even k. */
static void qs_quant_int4_g128(const float* W, int N, int K, uint8_t* data, uint16_t* sc) {
  for (int n = 0; n < N; ++n) {
    const float* row = W + (size_t)n * K;
    for (int g = 0; g < K / 128; ++g) {
      double agrp = 0.0;
      for (int i = 0; i < 128; ++i) { double a = fabs((double)row[g * 128 + i]); if (a > agrp) agrp = a; }
      const uint16_t sb = qs_f64_to_f16(agrp / 7.0);
      sc[(size_t)n * (K / 128) + g] = sb;
      const double s = qs_f16_value(sb);
      for (int i = 0; i < 128; ++i) {
        double q = 0.0;
        if (s != 0.0) {
          q = nearbyint((double)row[g * 128 + i] / s);
          if (q > 7.0) q = 7.0;
          if (q < -8.0) q = -8.0;
        }
        const uint8_t nib = (uint8_t)((int)q + 8);
        const size_t k = (size_t)g * 128 + i;
        uint8_t* p = data + (size_t)n * (K / 2) + k / 2;
        if (k & 1) *p = (uint8_t)((*p & 0x0F) | (nib << 4));
        else *p = (uint8_t)((*p & 0xF0) | nib);
      }
    }
  }
}

static void qs_quant_fp8_b128(const float* W, int N, int K, uint8_t* data, float* sc) {
  for (int bn = 0; bn < N / 128; ++bn)
    for (int bk = 0; bk < K / 128; ++bk) {
      float amax = 0.0f;
      for (int r = 0; r < 128; ++r)
        for (int c = 0; c < 128; ++c) {
          float a = fabsf(W[(size_t)(bn * 128 + r) * K + bk * 128 + c]);
          if (a > amax) amax = a;
        }
      float s = amax / 448.0f;
      sc[(size_t)bn * (K / 128) + bk] = s;
      for (int r = 0; r < 128; ++r)
        for (int c = 0; c < 128; ++c) {
          size_t i = (size_t)(bn * 128 + r) * K + bk * 128 + c;
          data[i] = (s > 0.0f) ? qs_e4m3_encode((double)W[i] / (double)s) : 0;
        }
    }
}

/* Public single-matrix encoders (used by tests and by the stack builder). */
int qs_quantize(int fmt, const float* W, int N, int K, void* data, void* scales, float* ts) {
  switch (fmt) {
    case QS_NVFP4: if (K % 16) return -1; qs_quant_nvfp4(W, N, K, (uint8_t*)data, (uint8_t*)scales, ts); return 0;
    case QS_MXFP4: if (K % 32) return -1; qs_quant_mxfp4(W, N, K, (uint8_t*)data, (uint8_t*)scales); *ts = 1.0f; return 0;
    case QS_INT4_G64: if (K % 64) return -1; qs_quant_int_g64(W, N, K, 4, (uint8_t*)data, (uint16_t*)scales); *ts = 1.0f; return 0;
    case QS_INT8_G64: if (K % 64) return -1; qs_quant_int_g64(W, N, K, 8, (uint8_t*)data, (uint16_t*)scales); *ts = 1.0f; return 0;
    case QS_FP8_B128: if (K % 128 || N % 128) return -1; qs_quant_fp8_b128(W, N, K, (uint8_t*)data, (float*)scales); *ts = 1.0f; return 0;
    case QS_INT4_G128: if (K % 128) return -1; qs_quant_int4_g128(W, N, K, (uint8_t*)data, (uint16_t*)scales); *ts = 1.0f; return 0;
    default: return -1;
  }
}

size_t qs_data_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case QS_NVFP4: case QS_MXFP4: case QS_INT4_G64: case QS_INT4_G128: return (size_t)N * K / 2;
    case QS_INT8_G64: case QS_FP8_B128: return (size_t)N * K;
    default: return 0;
  }
}

size_t qs_scale_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case QS_NVFP4: return (size_t)N * (K / 16);
    case QS_MXFP4: return (size_t)N * (K / 32);
    case QS_INT4_G64: case QS_INT8_G64: return (size_t)N * (K / 64) * 2;
    case QS_FP8_B128: return (size_t)(N / 128) * (K / 128) * 4;
    case QS_INT4_G128: return (size_t)N * (K / 128) * 2;
    default: return 0;
  }
}

/* ---- stacked experts, generated in parallel ---- */

typedef struct {
  int fmt, N, K, E, next;
  uint64_t seed;
  uint32_t kind, proj, expert0;
  double sigma;
  uint8_t* data;
  uint8_t* scales;
  float* ts;
  pthread_mutex_t mu;
  int err;
} qs_job;

static void* qs_worker(void* arg) {
  qs_job* j = (qs_job*)arg;
  size_t nel = (size_t)j->N * j->K;
  float* W = (float*)malloc(nel * sizeof(float));
  if (!W) { pthread_mutex_lock(&j->mu); j->err = -2; pthread_mutex_unlock(&j->mu); return NULL; }
  size_t db = qs_data_bytes(j->fmt, j->N, j->K), sb = qs_scale_bytes(j->fmt, j->N, j->K);
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int e = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (e >= j->E) break;
    uint64_t key = qs_stream_key(j->seed, j->kind, j->expert0 + (uint32_t)e, j->proj);
    qs_normal_f32(key, 0, nel, j->sigma, W);
    float ts = 1.0f;
    int rc = qs_quantize(j->fmt, W, j->N, j->K, j->data + (size_t)e * db, j->scales + (size_t)e * sb, &ts);
    if (j->ts) j->ts[e] = ts;
    if (rc) { pthread_mutex_lock(&j->mu); j->err = rc; pthread_mutex_unlock(&j->mu); }
  }
  free(W);
  return NULL;
}

int qs_num_threads(void) {
  cpu_set_t set;
  if (sched_getaffinity(0, sizeof(set), &set) == 0) {
    int c = CPU_COUNT(&set);
    if (c > 0) return c;
  }
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Generate experts [expert0, expert0 + E) of one projection: N(0, sigma) FP32
 * weights from stream (seed, kind, expert, proj), encoded in format fmt.
 * data/scales/ts are stacked per expert (ts may be NULL).
 */
int qs_make_stack(int fmt, uint64_t seed, uint32_t kind, uint32_t proj, uint32_t expert0, int E, int N, int K,
                  double sigma, void* data, void* scales, float* ts, int nthreads) {
  qs_job j;
  memset(&j, 0, sizeof(j));
  j.fmt = fmt; j.N = N; j.K = K; j.E = E; j.seed = seed; j.kind = kind; j.proj = proj; j.expert0 = expert0;
  j.sigma = sigma; j.data = (uint8_t*)data; j.scales = (uint8_t*)scales; j.ts = ts;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads <= 0) nthreads = qs_num_threads();
  if (nthreads > E) nthreads = E;
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, qs_worker, &j);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&j.mu);
  return j.err;
}

/* Seeded permutation of [0, n) by Fisher-Yates driven by the counter stream. */
void qs_permutation(uint64_t key, int n, int32_t* out) {
  for (int i = 0; i < n; ++i) out[i] = i;
  for (int i = n - 1; i > 0; --i) {
    uint64_t r = qs_draw_u64(key, (uint64_t)(n - 1 - i));
    int j = (int)(r % (uint64_t)(i + 1));
    int32_t t = out[i]; out[i] = out[j]; out[j] = t;
  }
}
