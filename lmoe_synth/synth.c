/*
 * Seeded synthetic inputs for the latent MoE layer (Edge0-145B launch blog,
 * "Under the Hood of Edge0: Architecture" -- 512 experts, groups of 64 sharing
 * two large matrices, small per-expert parameters; byteiota "SSD expert
 * streaming" and "Recover-LoRA" -- int4 frozen base plus a bf16 LoRA branch).
 *
 * This file only DRAWS inputs: random numbers, their bf16 rounding, the int4
 * symmetric per-32 quantisation that turns drawn fp32 weights into the frozen
 * 4-bit base, the Zipf router bias and synthetic routing tables. It holds none
 * of the layer's arithmetic (no router, top-k, permutation, projection, SwiGLU
 * or combine). Both the oracle and the CUDA library consume its outputs as
 * plain bytes.
 *
 * Random numbers: a counter-based generator. Element i of a tensor drawn with
 * (seed, stream) uses splitmix64 (Steele, Lea, Flood 2014, "Fast splittable
 * pseudorandom number generators") applied to key(seed, stream) + i, so the
 * values do not depend on thread count or call order. Normals come from the
 * Box-Muller transform (Box & Muller 1958) on two such uniforms; element 2p
 * takes the cosine branch and 2p+1 the sine branch of pair p.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static inline uint64_t sm64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return sm64(sm64(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* uniform in (0, 1]: 53 random bits */
static inline double u01(uint64_t key, uint64_t ctr) {
  return ((double)(sm64(key + ctr) >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  double u1 = u01(key, 2 * p), u2 = u01(key, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925 * u2;
  return (i & 1) ? r * sin(th) : r * cos(th);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ---------------------------------------------------------------------------
 * a tiny parallel-for on pthreads (no OpenMP: avoids a second libgomp next to
 * the one PyTorch ships)
 */
typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void* ctx; int64_t lo, hi; } pf_job;
static int g_threads = 0;

void synth_set_threads(int n) { g_threads = n; }

static void* pf_run(void* a) {
  pf_job* j = (pf_job*)a;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, int64_t min_chunk, range_fn fn, void* ctx) {
  int nt = g_threads;
  if (nt <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nt = c > 0 ? (int)c : 1;
    if (nt > 64) nt = 64;
  }
  if (n < 2 * min_chunk || nt == 1) {
    fn(ctx, 0, n);
    return;
  }
  int64_t chunks = n / min_chunk;
  if (chunks < nt) nt = (int)chunks;
  pthread_t th[64];
  pf_job jobs[64];
  for (int i = 0; i < nt; i++) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].lo = n * i / nt;
    jobs[i].hi = n * (i + 1) / nt;
  }
  for (int i = 1; i < nt; i++) pthread_create(&th[i], NULL, pf_run, &jobs[i]);
  pf_run(&jobs[0]);
  for (int i = 1; i < nt; i++) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------- */
typedef struct { uint64_t key; double sigma; float* out; uint16_t* out16; } nctx;

static void normal_f32_rng(void* c, int64_t lo, int64_t hi) {
  nctx* x = (nctx*)c;
  for (int64_t i = lo; i < hi; i++) x->out[i] = (float)(x->sigma * normal_at(x->key, (uint64_t)i));
}
static void normal_bf16_rng(void* c, int64_t lo, int64_t hi) {
  nctx* x = (nctx*)c;
  for (int64_t i = lo; i < hi; i++)
    x->out16[i] = f32_to_bf16_rne((float)(x->sigma * normal_at(x->key, (uint64_t)i)));
}

/* n fp32 values sigma * N(0,1) */
void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double sigma, float* out) {
  nctx c = {stream_key(seed, stream), sigma, out, NULL};
  parallel_for(n, 1 << 16, normal_f32_rng, &c);
}

/* n bf16 values (bit patterns), RNE of fp32(sigma * N(0,1)) */
void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, double sigma, uint16_t* out) {
  nctx c = {stream_key(seed, stream), sigma, NULL, out};
  parallel_for(n, 1 << 16, normal_bf16_rng, &c);
}

/* ---------------------------------------------------------------------------
 * int4 weights: a [rows][K] matrix of fp32 sigma*N(0,1) draws, quantised
 * symmetrically in groups of 32 consecutive elements along K:
 *   s = bf16_rne(amax / 7), q = clamp(round_half_even(w / s), -7, 7),
 *   amax == 0 -> s = 0, q = 0.
 * Packed row-major, K contiguous: byte j of a row holds element 2j in its low
 * nibble and 2j+1 in its high nibble, two's complement. scales: [rows][K/32].
 */
typedef struct { uint64_t key; double sigma; int K; uint8_t* q; uint16_t* s; } qctx;

static void quant_rows(void* c, int64_t lo, int64_t hi) {
  qctx* x = (qctx*)c;
  const int K = x->K, ng = K / 32;
  float w[32];
  for (int64_t r = lo; r < hi; r++) {
    for (int g = 0; g < ng; g++) {
      float amax = 0.f;
      for (int i = 0; i < 32; i++) {
        uint64_t idx = (uint64_t)r * (uint64_t)K + (uint64_t)(g * 32 + i);
        w[i] = (float)(x->sigma * normal_at(x->key, idx));
        float a = fabsf(w[i]);
        if (a > amax) amax = a;
      }
      uint16_t sb = f32_to_bf16_rne(amax / 7.0f);
      float s = bf16_to_f32(sb);
      x->s[r * ng + g] = sb;
      uint8_t* qb = x->q + r * (K / 2) + g * 16;
      for (int i = 0; i < 32; i += 2) {
        int q0 = 0, q1 = 0;
        if (s != 0.f) {
          float a0 = nearbyintf(w[i] / s), a1 = nearbyintf(w[i + 1] / s);
          q0 = a0 > 7.f ? 7 : (a0 < -7.f ? -7 : (int)a0);
          q1 = a1 > 7.f ? 7 : (a1 < -7.f ? -7 : (int)a1);
        }
        qb[i / 2] = (uint8_t)((q0 & 15) | ((q1 & 15) << 4));
      }
    }
  }
}

int synth_int4_matrix(uint64_t seed, uint64_t stream, int64_t rows, int K, double sigma, uint8_t* q,
                      uint16_t* scales) {
  if (K % 32 != 0 || rows < 0) return -1;
  qctx c = {stream_key(seed, stream), sigma, K, q, scales};
  parallel_for(rows, 64, quant_rows, &c);
  return 0;
}

/* ---------------------------------------------------------------------------
 * NVFP4 weights (NVIDIA's FP4 format): the same fp32 draws as
 * synth_int4_matrix, quantised per tensor of rows_per_tensor rows:
 *   gs = amax(tensor) / (6 * 448)                        (fp32; 0 if amax == 0)
 *   per block of 16 consecutive elements along K:
 *     sb = e4m3_rne(amax(block) / 6 / gs), saturated at 448 (0 if gs == 0)
 *     code_i = e2m1_rne(w_i / (e4m3(sb) * gs)), saturated at 6 (0 if sb == 0)
 * E2M1 codes are packed two per byte like the int4 format (element 2j in the
 * low nibble; bit 3 = sign); block scales [rows][K/16] bytes; gs [tensors].
 * Ties go to the even code (mantissa bit 0) in both roundings.
 */
static const float E2M1_MAG[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};

static int e2m1_rne(float v) {
  const float a = fabsf(v);
  int best = 7;
  if (a < 6.f) {
    float bd = INFINITY;
    for (int c = 0; c < 8; c++) {
      const float dd = fabsf(a - E2M1_MAG[c]);
      if (dd < bd || (dd == bd && (c & 1) == 0)) {
        bd = dd;
        best = c;
      }
    }
  }
  return (v < 0.f ? 8 : 0) | best;
}

static float e4m3_val(uint8_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  return e == 0 ? ldexpf((float)m / 8.f, -6) : ldexpf(1.f + (float)m / 8.f, e - 7);
}

/* x >= 0 -> the nearest E4M3 byte (ties to even mantissa), saturated at 448 */
uint8_t synth_e4m3_rne(float x) {
  if (!(x > 0.f)) return 0;
  if (x >= 448.f) return 0x7E;
  if (x < ldexpf(1.f, -6)) {
    const int m = (int)nearbyintf(x / ldexpf(1.f, -9)); /* 0 .. 8; 8 is the smallest normal */
    return (uint8_t)m;
  }
  int ex;
  const float fr = frexpf(x, &ex); /* x = fr * 2^ex, fr in [0.5, 1) */
  int e = ex - 1;
  int m = (int)nearbyintf((fr * 2.f - 1.f) * 8.f);
  if (m == 8) {
    m = 0;
    e += 1;
  }
  if (e + 7 > 15 || (e + 7 == 15 && m == 7)) return 0x7E;
  return (uint8_t)(((e + 7) << 3) | m);
}

typedef struct { uint64_t key; double sigma; int K; int64_t rpt; uint8_t* q; uint8_t* s; float* gs; } nvctx;

static void nvfp4_tensors(void* c, int64_t lo, int64_t hi) {
  nvctx* x = (nvctx*)c;
  const int K = x->K;
  float w[16];
  for (int64_t t = lo; t < hi; t++) {
    float amax = 0.f;
    for (int64_t r = t * x->rpt; r < (t + 1) * x->rpt; r++)
      for (int c2 = 0; c2 < K; c2++) {
        const float a = fabsf((float)(x->sigma * normal_at(x->key, (uint64_t)r * (uint64_t)K + (uint64_t)c2)));
        if (a > amax) amax = a;
      }
    const float gs = amax / (6.f * 448.f);
    x->gs[t] = gs;
    for (int64_t r = t * x->rpt; r < (t + 1) * x->rpt; r++)
      for (int b = 0; b < K / 16; b++) {
        float ab = 0.f;
        for (int i = 0; i < 16; i++) {
          w[i] = (float)(x->sigma * normal_at(x->key, (uint64_t)r * (uint64_t)K + (uint64_t)(b * 16 + i)));
          if (fabsf(w[i]) > ab) ab = fabsf(w[i]);
        }
        const uint8_t sb = gs > 0.f ? synth_e4m3_rne(ab / 6.f / gs) : 0;
        x->s[r * (K / 16) + b] = sb;
        const float denom = e4m3_val(sb) * gs;
        uint8_t* qb = x->q + r * (K / 2) + b * 8;
        for (int i = 0; i < 16; i += 2) {
          const int c0 = denom > 0.f ? e2m1_rne(w[i] / denom) : 0;
          const int c1 = denom > 0.f ? e2m1_rne(w[i + 1] / denom) : 0;
          qb[i / 2] = (uint8_t)(c0 | (c1 << 4));
        }
      }
  }
}

int synth_nvfp4_matrix(uint64_t seed, uint64_t stream, int64_t rows, int K, double sigma, int64_t rows_per_tensor,
                       uint8_t* q, uint8_t* scales, float* gs) {
  if (K % 16 != 0 || rows < 0 || rows_per_tensor <= 0 || rows % rows_per_tensor != 0) return -1;
  nvctx c = {stream_key(seed, stream), sigma, K, rows_per_tensor, q, scales, gs};
  parallel_for(rows / rows_per_tensor, 1, nvfp4_tensors, &c);
  return 0;
}

/* the same fp32 draws synth_int4_matrix quantises (for tests of the quantiser) */
void synth_int4_source(uint64_t seed, uint64_t stream, int64_t rows, int K, double sigma, float* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < rows * (int64_t)K; i++) out[i] = (float)(sigma * normal_at(key, (uint64_t)i));
}

/* ---------------------------------------------------------------------------
 * Zipf(s) router bias: expert popularity p_r ∝ r^-s over ranks r = 1..E, ranks
 * assigned to experts by a seeded Fisher-Yates shuffle; bias_e = ln p_rank(e).
 */
void synth_zipf_bias(uint64_t seed, int E, double s, float* bias) {
  uint64_t key = stream_key(seed, 0x5a495046ull);
  int* perm = (int*)malloc(sizeof(int) * (size_t)E);
  for (int i = 0; i < E; i++) perm[i] = i;
  for (int i = E - 1; i > 0; i--) {
    int j = (int)(u01(key, (uint64_t)i) * (double)(i + 1));
    if (j > i) j = i;
    int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  double z = 0.0;
  for (int r = 1; r <= E; r++) z += pow((double)r, -s);
  for (int i = 0; i < E; i++) {
    int rank = i + 1; /* perm[i] is the expert holding rank i+1 */
    bias[perm[i]] = (float)log(pow((double)rank, -s) / z);
  }
  free(perm);
}

/* ---------------------------------------------------------------------------
 * Synthetic routing tables (for exercising the permutation and expert steps in
 * isolation): per token k distinct experts drawn uniformly (or, if skew > 0,
 * from a Zipf(skew) popularity), weights positive, descending, summing to 1.
 */
void synth_routing(uint64_t seed, int T, int E, int k, double skew, int32_t* idx, float* w) {
  uint64_t key = stream_key(seed, 0x524f555445ull);
  double* cdf = NULL;
  if (skew > 0) {
    cdf = (double*)malloc(sizeof(double) * (size_t)E);
    double z = 0;
    for (int e = 0; e < E; e++) z += pow((double)(e + 1), -skew);
    double acc = 0;
    for (int e = 0; e < E; e++) {
      acc += pow((double)(e + 1), -skew) / z;
      cdf[e] = acc;
    }
  }
  uint64_t ctr = 0;
  for (int t = 0; t < T; t++) {
    int32_t* it = idx + (int64_t)t * k;
    for (int j = 0; j < k; j++) {
      for (;;) {
        double u = u01(key, ctr++);
        int e;
        if (cdf) {
          int lo = 0, hi = E - 1;
          while (lo < hi) {
            int mid = (lo + hi) / 2;
            if (cdf[mid] >= u) hi = mid; else lo = mid + 1;
          }
          e = lo;
        } else {
          e = (int)(u * E);
          if (e >= E) e = E - 1;
        }
        int dup = 0;
        for (int i = 0; i < j; i++) dup |= (it[i] == e);
        if (!dup) { it[j] = e; break; }
      }
    }
    float* wt = w + (int64_t)t * k;
    double sum = 0;
    double v[64];
    for (int j = 0; j < k; j++) { v[j] = u01(key, ctr++) + 0.05; sum += v[j]; }
    /* descending order of weights */
    for (int a = 0; a < k; a++)
      for (int b = a + 1; b < k; b++)
        if (v[b] > v[a]) { double tmp = v[a]; v[a] = v[b]; v[b] = tmp; }
    for (int j = 0; j < k; j++) wt[j] = (float)(v[j] / sum);
  }
  free(cdf);
}
