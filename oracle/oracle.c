/*
 * oracle.c -- plain, slow CPU reference of the fused small-batch MoE decode layer.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg may call this file's library; the product path never does.  It shares no
 * code with the CUDA kernels.  Each function names the passage it follows; where the
 * pages name a stage without a formula, the reading used is stated beside it.
 *
 * Pages: "Mono decode layer for DeepSeek-V4.1-Flash on MI355X" (vllm PR #60397),
 * "Mono decode for the DSpark draft layers" (vllm PR #62131), "DecodeSpec /
 * SpecializedDecode" (vllm PR #61311).
 *
 * Build with -ffp-contract=off: the f32 decisions (KV codes, router logits) must not be
 * fused into FMAs differently on different hosts.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int orc_get_threads(void) { return g_threads; }

/* ======================================================================================
 * Number formats.  The pages name MXFP8 (e4m3) and MXFP4 (e2m1) with E8M0 block scales
 * ("Design": MXFP8 32x32 E8M0 scales, MXFP4 routed experts); the bit layouts are those of
 * the OCP Microscaling Formats specification v1.0.
 * ==================================================================================== */

/* E8M0: an unsigned biased exponent, value 2^(e-127); 0xFF is NaN. */
double orc_e8m0(uint8_t e) {
  if (e == 0xFF) return NAN;
  return ldexp(1.0, (int)e - 127);
}

/* e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN, no infinity.
 * Normal (1 + m/8) * 2^(e-7); subnormal (m/8) * 2^-6. */
double orc_e4m3(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp(m / 8.0, -6);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* e2m1: sign, 2 exponent bits (bias 1), 1 mantissa bit.
 * Normal (1 + m/2) * 2^(e-1); subnormal m * 0.5. */
double orc_e2m1(uint8_t nib) {
  int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double v;
  if (e == 0)
    v = m * 0.5;
  else
    v = ldexp(1.0 + m / 2.0, e - 1);
  return s ? -v : v;
}

/* Round to the nearest e4m3 value, ties to even, saturating at +-448 (the largest finite
 * e4m3 value); NaN maps to the NaN code.  Used by the KV insert (reading: "fp8 KV cache
 * with per-token f32 scale", codes round to nearest even and saturate). */
uint8_t orc_encode_e4m3(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);              /* a = f * 2^e with f in [0.5, 1): leading bit is 2^(e-1) */
  int q = (e - 1) - 3;       /* weight of the last of 3 mantissa bits */
  if (q < -9) q = -9;        /* subnormal spacing 2^-9 */
  double r = ldexp(rint(ldexp(a, -q)), q); /* rint: round half to even */
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  int er;
  frexp(r, &er);
  int E = er - 1;            /* r = 1.m * 2^E */
  if (E < -6) return sign | (uint8_t)(int)ldexp(r, 9);
  int m = (int)ldexp(r, 3 - E) - 8;
  return sign | (uint8_t)(((E + 7) << 3) | m);
}

/* bf16: 8 significant bits, 8 exponent bits.  Round a double to the nearest bf16 value,
 * ties to even (the layer's activations are bf16; see the rounding points in orc_layer). */
double orc_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e);
  int q = e - 8;             /* keep 8 significant bits */
  if (q < -133) q = -133;    /* bf16 subnormal spacing */
  double r = ldexp(rint(ldexp(v, -q)), q);
  const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (fabs(r) > bf16_max) r = copysign(INFINITY, v);
  return r;
}

uint16_t orc_bf16_bits(double v) {
  float f = (float)orc_round_bf16(v); /* exact: the value already has 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return 0x7FC0;
  return (uint16_t)(u >> 16);
}

void orc_bf16_bits_array(const double *v, size_t n, uint16_t *out) {
  for (size_t i = 0; i < n; i++) out[i] = orc_bf16_bits(v[i]);
}

double orc_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double *bf16_rows(const uint16_t *x, size_t n) {
  double *d = (double *)malloc(n * sizeof(double));
  for (size_t i = 0; i < n; i++) d[i] = orc_bf16_value(x[i]);
  return d;
}

/* ======================================================================================
 * Stages
 * ==================================================================================== */

/* RMSNorm, the attention-front norm, the q/kv norms and the FFN-seam norm (launch table:
 * K1 "q/kv norms", K2 "the FFN seam").  Reading: y = x / sqrt(mean(x^2) + eps) * gamma,
 * rounded to bf16. */
void orc_rmsnorm(const uint16_t *x, const uint16_t *gamma, int rows, int dim, float eps,
                 uint16_t *out) {
  for (int r = 0; r < rows; r++) {
    double ss = 0.0;
    for (int i = 0; i < dim; i++) {
      double v = orc_bf16_value(x[(size_t)r * dim + i]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / dim + (double)eps);
    for (int i = 0; i < dim; i++) {
      double v = orc_bf16_value(x[(size_t)r * dim + i]) * inv * orc_bf16_value(gamma[i]);
      out[(size_t)r * dim + i] = orc_bf16_bits(v);
    }
  }
}

/* y[r, j] = sum_k x[r, k] * W[j, k] with W an MXFP8 matrix: e4m3 code (j, k) times the E8M0
 * scale of its 32x32 block, scale[j/32][k/32] ("Design": row-major MXFP8, 32x32 E8M0
 * scales, read in place).  Activations are bf16 and products are formed exactly; the
 * result is returned unrounded. */
void orc_gemv_mxfp8(const uint16_t *x, int rows, const uint8_t *w, const uint8_t *s, int n,
                    int k, double *y) {
  double *xd = bf16_rows(x, (size_t)rows * k);
  int kb = k / 32;
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int j = 0; j < n; j++) {
    double *wd = (double *)malloc((size_t)k * sizeof(double));
    for (int i = 0; i < k; i++)
      wd[i] = orc_e4m3(w[(size_t)j * k + i]) * orc_e8m0(s[(size_t)(j / 32) * kb + i / 32]);
    for (int r = 0; r < rows; r++) {
      double acc = 0.0;
      const double *xr = xd + (size_t)r * k;
      for (int i = 0; i < k; i++) acc += xr[i] * wd[i];
      y[(size_t)r * n + j] = acc;
    }
    free(wd);
  }
  free(xd);
}

/* As orc_gemv_mxfp8 for an MXFP4 matrix: byte (j, i/2) holds element i in its low nibble
 * when i is even and in its high nibble when i is odd; one E8M0 scale per row and per 32
 * consecutive k, scale[j][k/32] ("Design": MXFP4 routed experts; 1x32 scales). */
void orc_gemv_mxfp4(const uint16_t *x, int rows, const uint8_t *w, const uint8_t *s, int n,
                    int k, double *y) {
  double *xd = bf16_rows(x, (size_t)rows * k);
  int kb = k / 32;
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int j = 0; j < n; j++) {
    double *wd = (double *)malloc((size_t)k * sizeof(double));
    for (int i = 0; i < k; i++) {
      uint8_t byte = w[(size_t)j * (k / 2) + i / 2];
      uint8_t nib = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
      wd[i] = orc_e2m1(nib) * orc_e8m0(s[(size_t)j * kb + i / 32]);
    }
    for (int r = 0; r < rows; r++) {
      double acc = 0.0;
      const double *xr = xd + (size_t)r * k;
      for (int i = 0; i < k; i++) acc += xr[i] * wd[i];
      y[(size_t)r * n + j] = acc;
    }
    free(wd);
  }
  free(xd);
}

/* One token's KV record (launch table: K1 "the KV insert"; scope: "fp8_ds_mla KV records";
 * workload: fp8-e4m3 cache with a per-token f32 scale).  Reading: s = amax / 448 in f32
 * (s = 1 when amax = 0), code_i = e4m3(kv_i / s) computed in f32, round half to even,
 * saturating. */
void orc_kv_quant(const uint16_t *kv, int dim, uint8_t *codes, float *scale) {
  float amax = 0.0f;
  for (int i = 0; i < dim; i++) {
    float a = fabsf((float)orc_bf16_value(kv[i]));
    if (a > amax) amax = a;
  }
  float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int i = 0; i < dim; i++) codes[i] = orc_encode_e4m3((float)orc_bf16_value(kv[i]) / s);
  *scale = s;
}

/* Address of the cache record of token t of request q through the block table; NULL when
 * the table does not map it.  Record layout: kv_dim e4m3 codes, then the f32 scale.  The
 * record view is [blocks, block, record] and consecutive pages are stride_block apart
 * ("DecodeSpec / SpecializedDecode", review: the block stride must be >= block * record). */
static uint8_t *record_of(const orc_spec *sp, const orc_step *st, int q, int t) {
  int lb = t / sp->block_size;
  if (t < 0 || lb >= st->max_blocks) return NULL;
  int pb = st->block_table[(size_t)q * st->max_blocks + lb];
  if (pb < 0 || pb >= st->num_blocks) return NULL;
  return st->cache + (size_t)pb * st->stride_block + (size_t)(t % sp->block_size) * st->stride_tok;
}

static int check_cache_view(const orc_spec *sp, const orc_step *st) {
  if (sp->kv_record_bytes < sp->kv_dim + 4) return -1;
  if (st->stride_tok < sp->kv_record_bytes) return -1;
  if (st->stride_block < (int64_t)sp->block_size * sp->kv_record_bytes) return -1;
  return 0;
}

/* KV insert for every non-pad row at its own position ("Test Plan": pad rows have slot -1
 * and are skipped).  Returns -1 on a bad cache view or an unmapped slot. */
int orc_kv_insert(const orc_spec *sp, const orc_step *st, const uint16_t *kvn) {
  if (check_cache_view(sp, st)) return -1;
  int bad = 0;
  for (int r = 0; r < st->rows; r++) {
    int p = st->positions[r];
    if (p < 0) continue;
    uint8_t *rec = record_of(sp, st, st->row_req[r], p);
    if (!rec) { bad = 1; continue; }
    float s;
    orc_kv_quant(kvn + (size_t)r * sp->kv_dim, sp->kv_dim, rec, &s);
    memcpy(rec + sp->kv_dim, &s, 4);
  }
  return bad ? -1 : 0;
}

/* Softmax attention of one query over n_keys keys: out = sum_t p_t v_t with
 * p = softmax(scale * q.k_t). */
void orc_attend(const double *q, const double *keys, const double *vals, int n_keys, int dim,
                double scale, double *out) {
  double *sc = (double *)malloc((size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
  double mx = -INFINITY;
  for (int t = 0; t < n_keys; t++) {
    double d = 0.0;
    for (int i = 0; i < dim; i++) d += q[i] * keys[(size_t)t * dim + i];
    sc[t] = d * scale;
    if (sc[t] > mx) mx = sc[t];
  }
  double l = 0.0;
  for (int t = 0; t < n_keys; t++) {
    sc[t] = exp(sc[t] - mx);
    l += sc[t];
  }
  for (int i = 0; i < dim; i++) out[i] = 0.0;
  for (int t = 0; t < n_keys; t++)
    for (int i = 0; i < dim; i++) out[i] += sc[t] * vals[(size_t)t * dim + i];
  for (int i = 0; i < dim; i++) out[i] = n_keys > 0 ? out[i] / l : 0.0;
  free(sc);
}

/* Keys a row attends ("Scope": causal sliding windows; "Details" of the draft layers:
 * non-causal rows swa_width = 192 wide).  Reading: a causal row at position p attends
 * positions (p - window, p]; a non-causal row attends (e - swa_width, e] where e is the last
 * position any row of its request holds in this step.  Returns 0 for a pad row. */
int orc_key_range(const orc_spec *sp, const orc_step *st, int row, int *lo, int *hi) {
  int p = st->positions[row];
  if (p < 0) return 0;
  if (sp->causal) {
    *hi = p;
    *lo = p - sp->window + 1;
  } else {
    int e = p;
    for (int r = 0; r < st->rows; r++)
      if (st->row_req[r] == st->row_req[row] && st->positions[r] > e) e = st->positions[r];
    *hi = e;
    *lo = e - sp->swa_width + 1;
  }
  if (*lo < 0) *lo = 0;
  return 1;
}

/* Sliding-window attention over the fp8 cache (launch table: K2 "split attention,
 * combine").  Reading: the single cached kv_dim latent is both key and value; it is viewed
 * as kv_dim/head_dim groups of head_dim and q head h reads group h / (n_q_heads / groups);
 * scores are scaled by 1/sqrt(head_dim); softmax in full precision; no sink, no bias.  The
 * split over the window and the log-sum-exp combine are an evaluation order of the same
 * softmax, so the reference takes the softmax whole.  Output rounded to bf16; pad rows
 * give zero.  Returns -1 if a key's page is unmapped. */
int orc_attention(const orc_spec *sp, const orc_step *st, const uint16_t *q, uint16_t *o) {
  int nq = sp->n_q_heads, dh = sp->head_dim, G = sp->kv_dim / sp->head_dim;
  int hpg = nq / G, width = nq * dh, bad = 0;
  double scale = 1.0 / sqrt((double)dh);
  for (int r = 0; r < st->rows; r++) {
    int lo, hi;
    if (!orc_key_range(sp, st, r, &lo, &hi)) {
      for (int i = 0; i < width; i++) o[(size_t)r * width + i] = 0;
      continue;
    }
    int T = hi - lo + 1;
    double *K = (double *)malloc((size_t)T * dh * sizeof(double));
    double *qh = (double *)malloc((size_t)dh * sizeof(double));
    double *oh = (double *)malloc((size_t)dh * sizeof(double));
    for (int g = 0; g < G; g++) {
      for (int t = 0; t < T; t++) {
        const uint8_t *rec = record_of(sp, st, st->row_req[r], lo + t);
        if (!rec) { bad = 1; for (int i = 0; i < dh; i++) K[(size_t)t * dh + i] = 0.0; continue; }
        float s;
        memcpy(&s, rec + sp->kv_dim, 4);
        for (int i = 0; i < dh; i++) K[(size_t)t * dh + i] = orc_e4m3(rec[g * dh + i]) * (double)s;
      }
      for (int h = g * hpg; h < (g + 1) * hpg; h++) {
        for (int i = 0; i < dh; i++) qh[i] = orc_bf16_value(q[(size_t)r * width + h * dh + i]);
        orc_attend(qh, K, K, T, dh, scale, oh);
        for (int i = 0; i < dh; i++) o[(size_t)r * width + h * dh + i] = orc_bf16_bits(oh[i]);
      }
    }
    free(K), free(qh), free(oh);
  }
  return bad ? -1 : 0;
}

/* Router and top-k (launch table: K2 "router, top-6"; ATOM changes: "f32 router logits";
 * draft layers: top-3).  Reading: logits z = u . W_r^T rounded to f32; p = softmax(z) over
 * all experts; the k experts with the largest z (equivalently p), ties to the lower index;
 * weights w_j = p_j / sum of the selected p, times routed_scale.  Pad rows route nowhere
 * (index -1, weight 0).  force_idx, when given, replaces the selection. */
void orc_router(const uint16_t *u, const float *wr, int rows, int n_experts, int hidden,
                int topk, float routed_scale, const int32_t *positions,
                const int32_t *force_idx, float *logits, double *probs, int32_t *idx,
                double *w) {
  double *p = (double *)malloc((size_t)n_experts * sizeof(double));
  char *taken = (char *)malloc((size_t)n_experts);
  for (int r = 0; r < rows; r++) {
    float *z = logits + (size_t)r * n_experts;
    for (int e = 0; e < n_experts; e++) {
      double acc = 0.0;
      for (int i = 0; i < hidden; i++)
        acc += orc_bf16_value(u[(size_t)r * hidden + i]) * (double)wr[(size_t)e * hidden + i];
      z[e] = (float)acc;
    }
    double zmax = -INFINITY, l = 0.0;
    for (int e = 0; e < n_experts; e++) if (z[e] > zmax) zmax = z[e];
    for (int e = 0; e < n_experts; e++) { p[e] = exp((double)z[e] - zmax); l += p[e]; }
    for (int e = 0; e < n_experts; e++) p[e] /= l;
    if (probs) memcpy(probs + (size_t)r * n_experts, p, (size_t)n_experts * sizeof(double));
    int32_t *sel = idx + (size_t)r * topk;
    double *ws = w + (size_t)r * topk;
    if (positions && positions[r] < 0) {
      for (int j = 0; j < topk; j++) sel[j] = -1, ws[j] = 0.0;
      continue;
    }
    if (force_idx) {
      for (int j = 0; j < topk; j++) sel[j] = force_idx[(size_t)r * topk + j];
    } else {
      memset(taken, 0, (size_t)n_experts);
      for (int j = 0; j < topk; j++) {
        int best = -1;
        for (int e = 0; e < n_experts; e++)
          if (!taken[e] && (best < 0 || z[e] > z[best])) best = e;
        taken[best] = 1;
        sel[j] = best;
      }
    }
    double sum = 0.0;
    for (int j = 0; j < topk; j++) sum += p[sel[j]];
    for (int j = 0; j < topk; j++) ws[j] = p[sel[j]] / sum * (double)routed_scale;
  }
  free(p), free(taken);
}

/* SwiGLU with clamp (ATOM changes: vLLM's silu_and_mul_with_clamp; workloads: clamp +-7).
 * Reading: both halves clamped to [-c, c], then silu(g) * u. */
double orc_swiglu(double g, double u, double clamp) {
  if (g > clamp) g = clamp;
  if (g < -clamp) g = -clamp;
  if (u > clamp) u = clamp;
  if (u < -clamp) u = -clamp;
  return g / (1.0 + exp(-g)) * u;
}

/* One expert MLP on `rows` rows (launch table: K2 "shared expert, MXFP4 experts").
 * gate_up is [2*inter, hidden] with gate rows first, then up rows; down is
 * [hidden, inter].  t = bf16(swiglu(gate, up)); y = t . down^T, unrounded.  fmt4 selects
 * MXFP4 (routed experts) over MXFP8 (shared expert). */
void orc_ffn(const uint16_t *x, int rows, int fmt4, const uint8_t *gu, const uint8_t *gu_s,
             const uint8_t *d, const uint8_t *d_s, int inter, int hidden, double clamp,
             uint16_t *t, double *y) {
  double *a = (double *)malloc((size_t)rows * 2 * inter * sizeof(double));
  if (fmt4)
    orc_gemv_mxfp4(x, rows, gu, gu_s, 2 * inter, hidden, a);
  else
    orc_gemv_mxfp8(x, rows, gu, gu_s, 2 * inter, hidden, a);
  for (int r = 0; r < rows; r++)
    for (int i = 0; i < inter; i++)
      t[(size_t)r * inter + i] = orc_bf16_bits(
          orc_swiglu(a[(size_t)r * 2 * inter + i], a[(size_t)r * 2 * inter + inter + i], clamp));
  if (fmt4)
    orc_gemv_mxfp4(t, rows, d, d_s, hidden, inter, y);
  else
    orc_gemv_mxfp8(t, rows, d, d_s, hidden, inter, y);
  free(a);
}

static void round_rows(const double *v, size_t n, uint16_t *out) {
  for (size_t i = 0; i < n; i++) out[i] = orc_bf16_bits(v[i]);
}

/* The FFN seam and the MoE of one step (launch table, row K2 from "the FFN seam" on; the
 * same half is the whole of the row FFN), given the residual h after attention:
 *   B5 u = rmsnorm(h, ffn_norm)                             -> bf16
 *   B6 router + top-k on u
 *   B8 shared expert on u;  B9 routed experts on u, weighted
 *   B10 out = h + y_shared + sum_j w_j y_j                  -> bf16; pad rows: out = x
 * Writes out[rows, H] and the trace fields u .. y_r. */
static void moe_half(const orc_spec *sp, const orc_weights *w, const uint16_t *x,
                     const int32_t *positions, const int32_t *force_idx, int R,
                     const uint16_t *h, uint16_t *out, orc_trace *tr) {
  int H = sp->hidden, E = sp->n_experts, K = sp->topk, I = sp->moe_inter, Is = sp->shared_inter;
  uint16_t *u = malloc((size_t)R * H * 2), *ts = malloc((size_t)R * Is * 2);
  double *ys = malloc((size_t)R * H * sizeof(double));
  double *yr = calloc((size_t)R * H, sizeof(double));
  float *logits = malloc((size_t)R * E * sizeof(float));
  double *probs = malloc((size_t)R * E * sizeof(double));
  int32_t *idx = malloc((size_t)R * K * sizeof(int32_t));
  double *wt = malloc((size_t)R * K * sizeof(double));

  orc_rmsnorm(h, w->ffn_norm, R, H, sp->eps, u);                               /* B5 */
  orc_router(u, w->router, R, E, H, K, sp->routed_scale, positions, force_idx, logits, probs,
             idx, wt);                                                         /* B6 */
  orc_ffn(u, R, 0, w->sh_gu, w->sh_gu_s, w->sh_d, w->sh_d_s, Is, H, sp->swiglu_clamp, ts,
          ys);                                                                 /* B8 */
  /* B9: each expert once, on the rows routed to it; the weighted outputs are added per row
   * in slot order j = 0..k-1. */
  double *yslot = calloc((size_t)R * K * H, sizeof(double));
  /* a forced routing may repeat an expert within a row, so allow R * K rows per expert */
  uint16_t *xe = malloc((size_t)R * K * H * 2), *te = malloc((size_t)R * K * I * 2);
  double *yo = malloc((size_t)R * K * H * sizeof(double));
  int *who = malloc((size_t)R * K * sizeof(int));
  size_t gu_w = (size_t)2 * I * H / 2, gu_s = (size_t)2 * I * (H / 32);
  size_t d_w = (size_t)H * I / 2, d_s = (size_t)H * (I / 32);
  for (int e = 0; e < E; e++) {
    int n = 0;
    for (int r = 0; r < R; r++)
      for (int j = 0; j < K; j++)
        if (idx[(size_t)r * K + j] == e) {
          memcpy(xe + (size_t)n * H, u + (size_t)r * H, (size_t)H * 2);
          who[n++] = r * K + j;
        }
    if (!n) continue;
    orc_ffn(xe, n, 1, w->ex_gu + e * gu_w, w->ex_gu_s + e * gu_s, w->ex_d + e * d_w,
            w->ex_d_s + e * d_s, I, H, sp->swiglu_clamp, te, yo);
    for (int i = 0; i < n; i++) {
      memcpy(yslot + (size_t)who[i] * H, yo + (size_t)i * H, (size_t)H * sizeof(double));
      if (tr && tr->t_r) memcpy(tr->t_r + (size_t)who[i] * I, te + (size_t)i * I, (size_t)I * 2);
    }
  }
  for (int r = 0; r < R; r++)
    for (int j = 0; j < K; j++) {
      if (idx[(size_t)r * K + j] < 0) continue;
      for (int i = 0; i < H; i++)
        yr[(size_t)r * H + i] += wt[(size_t)r * K + j] * yslot[((size_t)r * K + j) * H + i];
    }
  /* B10 */
  for (int r = 0; r < R; r++)
    for (int i = 0; i < H; i++) {
      size_t a = (size_t)r * H + i;
      out[a] = positions[r] < 0 ? x[a] : orc_bf16_bits(orc_bf16_value(h[a]) + ys[a] + yr[a]);
    }

  if (tr) {
#define KEEP(dst, src, n) if (tr->dst) memcpy(tr->dst, src, n)
    KEEP(u, u, (size_t)R * H * 2);
    KEEP(logits, logits, (size_t)R * E * sizeof(float));
    KEEP(probs, probs, (size_t)R * E * sizeof(double));
    KEEP(topk_idx, idx, (size_t)R * K * sizeof(int32_t));
    KEEP(topk_w, wt, (size_t)R * K * sizeof(double));
    KEEP(t_s, ts, (size_t)R * Is * 2);
    KEEP(y_s, ys, (size_t)R * H * sizeof(double));
    KEEP(y_r, yr, (size_t)R * H * sizeof(double));
#undef KEEP
  }
  free(u), free(ts), free(ys), free(yr), free(logits), free(probs), free(idx), free(wt);
  free(yslot), free(xe), free(te), free(yo), free(who);
}

/* The whole layer step, stage by stage in launch order (launch table, rows K1 and K2):
 *   A1 xn = rmsnorm(x, attn_norm)                          -> bf16
 *   A2 qkv = xn . wqkv^T  (q latent of q_rank, then kv of kv_dim) -> bf16
 *   A3 q_latn = rmsnorm(q latent, q_norm); kvn = rmsnorm(kv, kv_norm) -> bf16
 *   A4 KV insert of kvn at each row's position
 *   A5 q = q_latn . wq_b^T                                  -> bf16 [rows, n_q * head_dim]
 *   B1-B2 o = windowed attention over the cache            -> bf16
 *   B3 oa = o . wo_a^T                                      -> bf16
 *   B4 h = x + oa . wo_b^T                                  -> bf16
 *   B5-B10 the FFN seam and the MoE (moe_half)
 * Rounding to bf16 happens exactly at the arrows; everything between is unrounded.
 * Returns 0, or -1 on a bad cache view / unmapped page. */
int orc_layer(const orc_spec *sp, const orc_weights *w, const orc_step *st, orc_trace *tr) {
  int R = st->rows, H = sp->hidden, qr = sp->q_rank, kvd = sp->kv_dim, orank = sp->o_rank;
  int QW = sp->n_q_heads * sp->head_dim, A = qr + kvd;
  int rc = 0;
  if (check_cache_view(sp, st)) return -1;

  uint16_t *xn = malloc((size_t)R * H * 2), *qkv = malloc((size_t)R * A * 2);
  uint16_t *qlat = malloc((size_t)R * qr * 2), *kv = malloc((size_t)R * kvd * 2);
  uint16_t *qlatn = malloc((size_t)R * qr * 2), *kvn = malloc((size_t)R * kvd * 2);
  uint16_t *q = malloc((size_t)R * QW * 2), *o = malloc((size_t)R * QW * 2);
  uint16_t *oa = malloc((size_t)R * orank * 2), *h = malloc((size_t)R * H * 2);
  int maxw = A;
  if (QW > maxw) maxw = QW;
  if (H > maxw) maxw = H;
  if (orank > maxw) maxw = orank;
  double *f = malloc((size_t)R * maxw * sizeof(double));

  /* K1: attention front */
  orc_rmsnorm(st->x, w->attn_norm, R, H, sp->eps, xn);                         /* A1 */
  orc_gemv_mxfp8(xn, R, w->wqkv, w->wqkv_s, A, H, f);                          /* A2 */
  round_rows(f, (size_t)R * A, qkv);
  for (int r = 0; r < R; r++) {
    memcpy(qlat + (size_t)r * qr, qkv + (size_t)r * A, (size_t)qr * 2);
    memcpy(kv + (size_t)r * kvd, qkv + (size_t)r * A + qr, (size_t)kvd * 2);
  }
  orc_rmsnorm(qlat, w->q_norm, R, qr, sp->eps, qlatn);                         /* A3 */
  orc_rmsnorm(kv, w->kv_norm, R, kvd, sp->eps, kvn);
  if (orc_kv_insert(sp, st, kvn)) rc = -1;                                     /* A4 */
  orc_gemv_mxfp8(qlatn, R, w->wq_b, w->wq_b_s, QW, qr, f);                     /* A5 */
  round_rows(f, (size_t)R * QW, q);

  /* K2: attention back, FFN seam, MoE */
  if (orc_attention(sp, st, q, o)) rc = -1;                                    /* B1-B2 */
  orc_gemv_mxfp8(o, R, w->wo_a, w->wo_a_s, orank, QW, f);                      /* B3 */
  round_rows(f, (size_t)R * orank, oa);
  orc_gemv_mxfp8(oa, R, w->wo_b, w->wo_b_s, H, orank, f);                      /* B4 */
  for (size_t i = 0; i < (size_t)R * H; i++) h[i] = orc_bf16_bits(orc_bf16_value(st->x[i]) + f[i]);
  uint16_t *out = tr && tr->out ? tr->out : malloc((size_t)R * H * 2);
  moe_half(sp, w, st->x, st->positions, st->force_idx, R, h, out, tr);         /* B5-B10 */

  if (tr) {
#define KEEP(dst, src, n) if (tr->dst) memcpy(tr->dst, src, n)
    KEEP(xn, xn, (size_t)R * H * 2);
    KEEP(qkv, qkv, (size_t)R * A * 2);
    KEEP(q_latn, qlatn, (size_t)R * qr * 2);
    KEEP(kvn, kvn, (size_t)R * kvd * 2);
    KEEP(q, q, (size_t)R * QW * 2);
    KEEP(o, o, (size_t)R * QW * 2);
    KEEP(oa, oa, (size_t)R * orank * 2);
    KEEP(h, h, (size_t)R * H * 2);
#undef KEEP
  }
  if (!(tr && tr->out)) free(out);
  free(xn), free(qkv), free(qlat), free(kv), free(qlatn), free(kvn), free(q), free(o), free(oa);
  free(h), free(f);
  return rc;
}

/* The FFN launch of one step (launch table, row FFN: for the layers whose attention runs
 * elsewhere, "the attention TP all-reduce ... then K2's FFN seam and MoE").  `a` is the
 * attention block's output for each row, bf16 [rows, H] (wo_b's output; on one GPU the
 * all-reduce of the tensor-parallel partials is the identity, so `a` is already the sum).
 * Reading: the residual is h = bf16(x + a), formed in unrounded arithmetic from the two
 * bf16 inputs, as B4 forms it from x and wo_b's unrounded output; then B5-B10 exactly as in
 * orc_layer.  Pad rows (positions < 0) output x.  No cache is touched; only the FFN fields
 * of `w` (ffn_norm, router, sh_*, ex_*) are read, and the attention fields of `sp` are not. */
void orc_ffn_layer(const orc_spec *sp, const orc_weights *w, const uint16_t *x, const uint16_t *a,
                   const int32_t *positions, const int32_t *force_idx, int rows,
                   orc_trace *tr) {
  size_t n = (size_t)rows * sp->hidden;
  uint16_t *h = malloc(n * 2);
  for (size_t i = 0; i < n; i++) h[i] = orc_bf16_bits(orc_bf16_value(x[i]) + orc_bf16_value(a[i]));
  uint16_t *out = tr && tr->out ? tr->out : malloc(n * 2);
  moe_half(sp, w, x, positions, force_idx, rows, h, out, tr);
  if (tr && tr->h) memcpy(tr->h, h, n * 2);
  if (!(tr && tr->out)) free(out);
  free(h);
}
