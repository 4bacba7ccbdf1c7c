/*
 * TEST INFRASTRUCTURE -- the CPU oracle for the latent MoE layer.
 *
 * A plain, slow, single-threaded implementation of what the layer computes,
 * in fp64, written to be checked by eye against its definition. Only the
 * test suite, the package's smoke check and the benchmark's CPU-baseline leg
 * use it; the CUDA library never links, loads or calls it, and it shares no
 * code with the CUDA library (the two see the same input bytes and nothing
 * else).
 *
 * What the pages fix (cited by page title and section):
 *  - "Edge0-145B: Frontier AI Capabilities on Your Own Computer", section
 *    "Under the Hood of Edge0", paragraph "Architecture: share large matrices
 *    across sparse experts": each group of 64 experts shares two large
 *    matrices; each expert keeps a small set of its own parameters.
 *  - "Edge0-145B: Run a 145B Open-Source Model on Your Laptop", section "Not
 *    Compression -- Architecture": 512 experts, 10 active per token; section
 *    "The Three Pillars That Make It Fast": int4 expert tensors (SSD expert
 *    streaming) and a Recover-LoRA branch running in parallel with the frozen
 *    4-bit base.
 *  - The Chinese explainer of the release (section on why 145B need not sit in
 *    GPU memory at once): 512 experts, 10 activated per token, groups of 64
 *    sharing two large matrices.
 *
 * The concrete operator form is this library's stated assumption (the pages
 * only sketch it): per group g a shared int4 down-projection W_in[g] (d -> L)
 * and up-projection W_out[g] (L -> d); per expert an int4 SwiGLU in the
 * latent space (gate/up L -> f, down f -> L); int4 symmetric per 32 elements
 * along the reduction dimension with bf16 scales; optional bf16 LoRA
 * (rank r, scale 1) on each shared projection; fp32 router weights with an
 * optional bias; top-k by descending logit with ties to the lower expert
 * index; softmax renormalised over the selected k.
 *
 * Every function's pins (what checks it against something other than itself)
 * live in the CPU test suite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int d, E, G, k, L, f, r; /* r: LoRA rank, 0 = no LoRA branch */
  const float* W_r;        /* [E][d] */
  const float* b_r;        /* [E] or NULL */
  const uint8_t* W_in_q;   /* [G][L][d/2] */
  const uint16_t* W_in_s;  /* [G][L][d/32] bf16 bits */
  const uint8_t* W_out_q;  /* [G][d][L/2] */
  const uint16_t* W_out_s; /* [G][d][L/32] */
  const uint8_t* gate_q;   /* [E][f][L/2] */
  const uint16_t* gate_s;  /* [E][f][L/32] */
  const uint8_t* up_q;     /* [E][f][L/2] */
  const uint16_t* up_s;
  const uint8_t* down_q;   /* [E][L][f/2] */
  const uint16_t* down_s;  /* [E][L][f/32] */
  const uint16_t* A_in;    /* [G][d][r] bf16 */
  const uint16_t* B_in;    /* [G][r][L] */
  const uint16_t* A_out;   /* [G][L][r] */
  const uint16_t* B_out;   /* [G][r][d] */
  /* Weight format: 0 = int4 as above; 1 = NVFP4: every *_q holds E2M1 codes
   * (same nibble order), every *_s points at E4M3 block scales, one byte per
   * 16 elements along K ([rows][K/16]), and each weight tensor (one group's
   * W_in or W_out, one expert's gate, up or Down) has an fp32 scale in the
   * matching *_gs array ([G] or [E]). */
  int wfmt;
  const float* W_in_gs;
  const float* W_out_gs;
  const float* gate_gs;
  const float* up_gs;
  const float* down_gs;
} oracle_layer;

/* ------------------------------------------------------------------ formats */

double oracle_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* bf16 round-to-nearest-even of a double, rounded once (no detour through
 * fp32). Finite inputs; values beyond bf16's range saturate to +-inf. */
uint16_t oracle_bf16_round(double v) {
  if (v == 0.0 || !isfinite(v)) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
  }
  int e;
  double m = frexp(v, &e); /* v = m * 2^e, 0.5 <= |m| < 1 */
  double r;
  if (e - 1 < -126) {
    /* bf16 subnormal: fixed quantum 2^-133 */
    r = ldexp(nearbyint(ldexp(v, 133)), -133);
  } else {
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* 8 significant bits */
  }
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

void oracle_bf16_round_array(int64_t n, const double* v, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_bf16_round(v[i]);
}

/* element k of a packed int4 row: byte k/2, low nibble for even k, high for
 * odd k, two's complement */
int oracle_int4_at(const uint8_t* row, int k) {
  int byte = row[k >> 1];
  int v = (k & 1) ? (byte >> 4) : (byte & 15);
  return v >= 8 ? v - 16 : v;
}

/* dequantised rows: out[i][c] = q(row0+i, c) * s(row0+i, c/32) */
void oracle_dequant_rows(const uint8_t* q, const uint16_t* s, int K, int64_t row0, int nrows, double* out) {
  for (int i = 0; i < nrows; i++) {
    const uint8_t* qr = q + (row0 + i) * (int64_t)(K / 2);
    const uint16_t* sr = s + (row0 + i) * (int64_t)(K / 32);
    for (int c = 0; c < K; c++) out[(int64_t)i * K + c] = oracle_int4_at(qr, c) * oracle_bf16_value(sr[c / 32]);
  }
}

/* NVFP4 ("Edge0-145B: Run a 145B Open-Source Model on Your Laptop", section
 * "What You Need to Run It": a checkpoint in NVIDIA's FP4 format). The
 * elements are FP4 E2M1 -- sign, 2 exponent bits (bias 1), 1 mantissa bit,
 * exponent 0 subnormal, no infinities or NaN -- so a code is
 * (-1)^s * (e == 0 ? m/2 : (1 + m/2) * 2^(e-1)). */
double oracle_e2m1_value(int code) {
  const int sgn = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
  return sgn ? -mag : mag;
}

/* The block scales are FP8 E4M3 (finite-only): sign, 4 exponent bits (bias
 * 7), 3 mantissa bits, exponent 0 subnormal; exponent 15 with mantissa 7 is
 * NaN and there are no infinities. */
double oracle_e4m3_value(uint8_t b) {
  const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? (m / 8.0) * ldexp(1.0, -6) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return sgn ? -mag : mag;
}

/* NVFP4 rows: out[i][c] = e2m1(q(row0+i, c)) * e4m3(s(row0+i, c/16)) * gs, the
 * codes packed two per byte like the int4 format (element 2j in the low
 * nibble), gs the fp32 scale of the tensor the rows belong to. */
void oracle_nvfp4_dequant_rows(const uint8_t* q, const uint8_t* s, double gs, int K, int64_t row0, int nrows,
                               double* out) {
  for (int i = 0; i < nrows; i++) {
    const uint8_t* qr = q + (row0 + i) * (int64_t)(K / 2);
    const uint8_t* sr = s + (row0 + i) * (int64_t)(K / 16);
    for (int c = 0; c < K; c++) {
      const int code = (c & 1) ? (qr[c >> 1] >> 4) : (qr[c >> 1] & 15);
      out[(int64_t)i * K + c] = oracle_e2m1_value(code) * oracle_e4m3_value(sr[c / 16]) * gs;
    }
  }
}

/* y[o] = sum_c What[row0+o][c] * v[c] for o < nrows, What the dequantised
 * weights of the layer's format; rows row0 .. row0+nrows-1 lie in tensor
 * row0 / rows_per_tensor (whose NVFP4 scale is gs[that tensor]). */
static void w_matvec(const oracle_layer* Ly, const uint8_t* q, const uint16_t* s, const float* gs,
                     int rows_per_tensor, int K, int64_t row0, int nrows, const double* v, double* y,
                     double* rowbuf) {
  for (int o = 0; o < nrows; o++) {
    if (Ly->wfmt == 1)
      oracle_nvfp4_dequant_rows(q, (const uint8_t*)s, gs[(row0 + o) / rows_per_tensor], K, row0 + o, 1, rowbuf);
    else
      oracle_dequant_rows(q, s, K, row0 + o, 1, rowbuf);
    double acc = 0.0;
    for (int c = 0; c < K; c++) acc += rowbuf[c] * v[c];
    y[o] = acc;
  }
}

/* ------------------------------------------------------------------- router */

/* Router logits (Architecture: a router picks experts among 512): l_e =
 * sum_i x_i W_r[e][i] (+ b_e), x the bf16 token. */
void oracle_router_logits(const oracle_layer* Ly, int n, const uint16_t* x, double* logits) {
  const int d = Ly->d, E = Ly->E;
  for (int t = 0; t < n; t++) {
    for (int e = 0; e < E; e++) {
      double acc = 0.0;
      for (int i = 0; i < d; i++) acc += oracle_bf16_value(x[(int64_t)t * d + i]) * (double)Ly->W_r[(int64_t)e * d + i];
      if (Ly->b_r) acc += (double)Ly->b_r[e];
      logits[(int64_t)t * E + e] = acc;
    }
  }
}

typedef struct { double key; int e; } kv;

static int kv_cmp(const void* a, const void* b) {
  const kv* x = (const kv*)a;
  const kv* y = (const kv*)b;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return x->e < y->e ? -1 : (x->e > y->e);
}

/* Top-k with softmax renormalisation ("10 of 512 experts activated per
 * token"): full sort of all E experts by (logit descending, index ascending);
 * the selection is decided on the logits rounded to fp32 (the precision the
 * GPU router decides in); w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over
 * the selected k, in fp64 from the unrounded logits. */
void oracle_topk(int n, int E, int k, const double* logits, int32_t* idx, double* w) {
  kv* a = (kv*)malloc(sizeof(kv) * (size_t)E);
  for (int t = 0; t < n; t++) {
    const double* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; e++) {
      a[e].key = (double)(float)l[e];
      a[e].e = e;
    }
    qsort(a, (size_t)E, sizeof(kv), kv_cmp);
    double l0 = l[a[0].e], z = 0.0;
    for (int j = 0; j < k; j++) z += exp(l[a[j].e] - l0);
    for (int j = 0; j < k; j++) {
      idx[(int64_t)t * k + j] = a[j].e;
      w[(int64_t)t * k + j] = exp(l[a[j].e] - l0) / z;
    }
  }
  free(a);
}

/* -------------------------------------------------------------- permutation */

typedef struct { int32_t e, a; } ea;

static int ea_cmp(const void* x, const void* y) {
  const ea* p = (const ea*)x;
  const ea* q = (const ea*)y;
  if (p->e != q->e) return p->e < q->e ? -1 : 1;
  return p->a < q->a ? -1 : (p->a > q->a);
}

/* Token permutation by group then expert (experts are numbered so that group
 * g = e / (E/G) holds a contiguous range, so sorting by expert also sorts by
 * group). Assignment a = t*k + j.
 *   expert_offsets[E+1]   exclusive prefix sum of per-expert counts
 *   sorted_assign[T*k]    assignments sorted by (expert, a)  -- stable
 *   inv[T*k]              inv[sorted_assign[p]] = p
 *   group_offsets[G+1]    expert_offsets[g * E/G]
 *   group_tok_offsets[G+1], group_tokens[]: per group, the distinct tokens
 *                         routed into it, ascending
 *   assign_row[T*k]       row of (t, group of idx[a]) in group_tokens
 * Returns sum_g n_g (the number of (group, token) rows). */
int oracle_permute(int T, int E, int G, int k, const int32_t* idx, int32_t* expert_offsets, int32_t* sorted_assign,
                   int32_t* inv, int32_t* group_offsets, int32_t* group_tok_offsets, int32_t* group_tokens,
                   int32_t* assign_row) {
  const int n = T * k, epg = E / G;
  ea* a = (ea*)malloc(sizeof(ea) * (size_t)(n > 0 ? n : 1));
  for (int i = 0; i < n; i++) {
    a[i].e = idx[i];
    a[i].a = i;
  }
  qsort(a, (size_t)n, sizeof(ea), ea_cmp);
  for (int e = 0; e <= E; e++) expert_offsets[e] = 0;
  for (int i = 0; i < n; i++) expert_offsets[idx[i] + 1]++;
  for (int e = 0; e < E; e++) expert_offsets[e + 1] += expert_offsets[e];
  for (int p = 0; p < n; p++) {
    sorted_assign[p] = a[p].a;
    inv[a[p].a] = p;
  }
  for (int g = 0; g <= G; g++) group_offsets[g] = expert_offsets[g * epg];
  int rows = 0;
  for (int g = 0; g < G; g++) {
    group_tok_offsets[g] = rows;
    for (int t = 0; t < T; t++) {
      int hit = 0;
      for (int j = 0; j < k; j++) hit |= (idx[t * k + j] / epg == g);
      if (hit) {
        for (int j = 0; j < k; j++)
          if (idx[t * k + j] / epg == g) assign_row[t * k + j] = rows;
        group_tokens[rows++] = t;
      }
    }
  }
  group_tok_offsets[G] = rows;
  free(a);
  return rows;
}

/* ------------------------------------------------------------ expert pieces */

static double bf(uint16_t b) { return oracle_bf16_value(b); }

/* h = What_in[g] x (+ B_in[g]^T (A_in[g]^T x) when the LoRA branch is on).
 * "Each group of 64 experts shares two large matrices" -- the first one. */
void oracle_shared_in(const oracle_layer* Ly, int g, const double* x, double* h) {
  const int d = Ly->d, L = Ly->L, r = Ly->r;
  double* row = (double*)malloc(sizeof(double) * (size_t)d);
  w_matvec(Ly, Ly->W_in_q, Ly->W_in_s, Ly->W_in_gs, L, d, (int64_t)g * L, L, x, h, row);
  if (r > 0) {
    /* Recover-LoRA: a bf16 low-rank branch in parallel with the int4 base */
    double* p = (double*)calloc((size_t)r, sizeof(double));
    const uint16_t* A = Ly->A_in + (int64_t)g * d * r;
    const uint16_t* B = Ly->B_in + (int64_t)g * r * L;
    for (int i = 0; i < d; i++)
      for (int c = 0; c < r; c++) p[c] += x[i] * bf(A[(int64_t)i * r + c]);
    for (int l = 0; l < L; l++) {
      double acc = 0.0;
      for (int c = 0; c < r; c++) acc += p[c] * bf(B[(int64_t)c * L + l]);
      h[l] += acc;
    }
    free(p);
  }
  free(row);
}

/* o = What_out[g] u (+ B_out[g]^T (A_out[g]^T u)) -- the second shared matrix */
void oracle_shared_out(const oracle_layer* Ly, int g, const double* u, double* o) {
  const int d = Ly->d, L = Ly->L, r = Ly->r;
  double* row = (double*)malloc(sizeof(double) * (size_t)L);
  w_matvec(Ly, Ly->W_out_q, Ly->W_out_s, Ly->W_out_gs, d, L, (int64_t)g * d, d, u, o, row);
  if (r > 0) {
    double* p = (double*)calloc((size_t)r, sizeof(double));
    const uint16_t* A = Ly->A_out + (int64_t)g * L * r;
    const uint16_t* B = Ly->B_out + (int64_t)g * r * d;
    for (int l = 0; l < L; l++)
      for (int c = 0; c < r; c++) p[c] += u[l] * bf(A[(int64_t)l * r + c]);
    for (int i = 0; i < d; i++) {
      double acc = 0.0;
      for (int c = 0; c < r; c++) acc += p[c] * bf(B[(int64_t)c * d + i]);
      o[i] += acc;
    }
    free(p);
  }
  free(row);
}

/* The expert's own small parameters ("each expert retains a small set of
 * parameters that captures its differences"): a latent SwiGLU
 *   a = Gate_e h, b = Up_e h, v = silu(a) * b = a / (1 + exp(-a)) * b,
 *   u = Down_e v. */
void oracle_expert_latent(const oracle_layer* Ly, int e, const double* h, double* u) {
  const int L = Ly->L, f = Ly->f;
  double* a = (double*)malloc(sizeof(double) * (size_t)f);
  double* b = (double*)malloc(sizeof(double) * (size_t)f);
  double* row = (double*)malloc(sizeof(double) * (size_t)(L > f ? L : f));
  w_matvec(Ly, Ly->gate_q, Ly->gate_s, Ly->gate_gs, f, L, (int64_t)e * f, f, h, a, row);
  w_matvec(Ly, Ly->up_q, Ly->up_s, Ly->up_gs, f, L, (int64_t)e * f, f, h, b, row);
  for (int i = 0; i < f; i++) a[i] = a[i] / (1.0 + exp(-a[i])) * b[i];
  w_matvec(Ly, Ly->down_q, Ly->down_s, Ly->down_gs, L, f, (int64_t)e * L, L, a, u, row);
  free(a);
  free(b);
  free(row);
}

/* ------------------------------------------------------------- layer forward */

/* One token through the layer, literal per-assignment form, given its routing:
 *   y = sum_j w_j * Wout[g_j] ( Expert_{e_j} ( Win[g_j] x ) ),  g_j = e_j / (E/G)
 * (each assignment recomputes its own shared projections). */
void oracle_token_routed(const oracle_layer* Ly, const uint16_t* x_bf16, const int32_t* idx, const double* w,
                         double* y) {
  const int d = Ly->d, L = Ly->L, k = Ly->k, epg = Ly->E / Ly->G;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* h = (double*)malloc(sizeof(double) * (size_t)L);
  double* u = (double*)malloc(sizeof(double) * (size_t)L);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; i++) {
    x[i] = bf(x_bf16[i]);
    y[i] = 0.0;
  }
  for (int j = 0; j < k; j++) {
    int e = idx[j], g = e / epg;
    oracle_shared_in(Ly, g, x, h);
    oracle_expert_latent(Ly, e, h, u);
    oracle_shared_out(Ly, g, u, o);
    for (int i = 0; i < d; i++) y[i] += w[j] * o[i];
  }
  free(x);
  free(h);
  free(u);
  free(o);
}

/* n tokens, routing given (idx [n][k], w [n][k]) -> y [n][d] */
void oracle_forward_routed(const oracle_layer* Ly, int n, const uint16_t* x, const int32_t* idx, const double* w,
                           double* y) {
  for (int t = 0; t < n; t++)
    oracle_token_routed(Ly, x + (int64_t)t * Ly->d, idx + (int64_t)t * Ly->k, w + (int64_t)t * Ly->k,
                        y + (int64_t)t * Ly->d);
}

/* The whole layer for n tokens: router, top-k, latent experts, weighted
 * combine. logits may be NULL. */
void oracle_layer_forward(const oracle_layer* Ly, int n, const uint16_t* x, double* y, int32_t* idx, double* w,
                          double* logits) {
  double* l = logits ? logits : (double*)malloc(sizeof(double) * (size_t)n * Ly->E);
  oracle_router_logits(Ly, n, x, l);
  oracle_topk(n, Ly->E, Ly->k, l, idx, w);
  oracle_forward_routed(Ly, n, x, idx, w, y);
  if (!logits) free(l);
}

/* The group-factored form of the same layer (used to pin the literal form by
 * linearity of Wout and of Win's reuse): for each group g that token t routes
 * into, in ascending g,
 *   h = Win[g] x;  z = sum_{j: g_j = g} w_j Expert_{e_j}(h);  y += Wout[g] z. */
void oracle_forward_routed_factored(const oracle_layer* Ly, int n, const uint16_t* xb, const int32_t* idxs,
                                    const double* ws, double* ys) {
  const int d = Ly->d, L = Ly->L, k = Ly->k, G = Ly->G, epg = Ly->E / Ly->G;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* h = (double*)malloc(sizeof(double) * (size_t)L);
  double* u = (double*)malloc(sizeof(double) * (size_t)L);
  double* z = (double*)malloc(sizeof(double) * (size_t)L);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int t = 0; t < n; t++) {
    const int32_t* idx = idxs + (int64_t)t * k;
    const double* w = ws + (int64_t)t * k;
    double* y = ys + (int64_t)t * d;
    for (int i = 0; i < d; i++) {
      x[i] = bf(xb[(int64_t)t * d + i]);
      y[i] = 0.0;
    }
    for (int g = 0; g < G; g++) {
      int hit = 0;
      for (int j = 0; j < k; j++) hit |= (idx[j] / epg == g);
      if (!hit) continue;
      oracle_shared_in(Ly, g, x, h);
      for (int l = 0; l < L; l++) z[l] = 0.0;
      for (int j = 0; j < k; j++) {
        if (idx[j] / epg != g) continue;
        oracle_expert_latent(Ly, idx[j], h, u);
        for (int l = 0; l < L; l++) z[l] += w[j] * u[l];
      }
      oracle_shared_out(Ly, g, z, o);
      for (int i = 0; i < d; i++) y[i] += o[i];
    }
  }
  free(x);
  free(h);
  free(u);
  free(z);
  free(o);
}

/* One (group, token) row of the group-factored form: Y[g,t] = Wout[g] z with
 * z = sum_{j: g_j = g} w_j Expert_{e_j}(Win[g] x_t). Rows of tokens that do
 * not route into g are all zero. */
void oracle_group_row(const oracle_layer* Ly, int g, const uint16_t* x_bf16, const int32_t* idx, const double* w,
                      double* yrow) {
  const int d = Ly->d, L = Ly->L, k = Ly->k, epg = Ly->E / Ly->G;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* h = (double*)malloc(sizeof(double) * (size_t)L);
  double* u = (double*)malloc(sizeof(double) * (size_t)L);
  double* z = (double*)calloc((size_t)L, sizeof(double));
  for (int i = 0; i < d; i++) x[i] = bf(x_bf16[i]);
  int hit = 0;
  for (int j = 0; j < k; j++) hit |= (idx[j] / epg == g);
  if (!hit) {
    for (int i = 0; i < d; i++) yrow[i] = 0.0;
  } else {
    oracle_shared_in(Ly, g, x, h);
    for (int j = 0; j < k; j++) {
      if (idx[j] / epg != g) continue;
      oracle_expert_latent(Ly, idx[j], h, u);
      for (int l = 0; l < L; l++) z[l] += w[j] * u[l];
    }
    oracle_shared_out(Ly, g, z, yrow);
  }
  free(x);
  free(h);
  free(u);
  free(z);
}

/* Residual step between stacked layers (48 layers, "512 expert networks
 * across 48 layers"): x_next = bf16(x + bf16(y)), each rounding once. */
void oracle_residual(int64_t n, const uint16_t* x, const double* y, uint16_t* x_next) {
  for (int64_t i = 0; i < n; i++) {
    double yb = oracle_bf16_value(oracle_bf16_round(y[i]));
    x_next[i] = oracle_bf16_round(oracle_bf16_value(x[i]) + yb);
  }
}

/* The weighted un-permute and combine on its own: y_t = sum over the
 * distinct groups g of token t's experts, in ascending g, of Y[row(g, t)]
 * (+ residual_t), where row(g, t) = assign_row[t*k + j] for any j with
 * g(idx[t][j]) = g. Y holds one fp32 row of width d per (group, token). */
void oracle_combine(int T, int d, int k, int G, int epg, const float* Y, const int32_t* idx,
                    const int32_t* assign_row, const uint16_t* residual, double* y) {
  for (int t = 0; t < T; t++) {
    double* yt = y + (int64_t)t * d;
    for (int i = 0; i < d; i++) yt[i] = residual ? oracle_bf16_value(residual[(int64_t)t * d + i]) : 0.0;
    for (int g = 0; g < G; g++) {
      int row = -1;
      for (int j = 0; j < k; j++)
        if (idx[t * k + j] / epg == g) row = assign_row[t * k + j];
      if (row < 0) continue;
      for (int i = 0; i < d; i++) yt[i] += (double)Y[(int64_t)row * d + i];
    }
  }
}
