/*
 * oracle.h -- plain, slow CPU reference of the fused small-batch MoE decode layer.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg may call this library.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Source passages (vllm PR #60397 "Mono decode layer for DeepSeek-V4.1-Flash on MI355X",
 * section Purpose, launch table; section Design; vllm PR #62131 "Mono decode for the
 * DSpark draft layers", section Details; vllm PR #61311 "DecodeSpec / SpecializedDecode",
 * review comment on the KV-cache record view).  The pages name the stages and number
 * formats but print no per-element formulas; every formula below is the plainest reading,
 * and each reading is stated at the function that takes it.
 *
 * Arithmetic: doubles throughout, with bf16 round-to-nearest-even applied exactly at the
 * layer's rounding points.  Where floating point decides an integer -- the e4m3 codes of
 * the KV insert and the router's top-k -- the decision is taken in f32, the precision the
 * pages give for the router logits and the precision of the CUDA kernels.
 */
#ifndef MONO_ORACLE_H
#define MONO_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t hidden, n_q_heads, head_dim, kv_dim, q_rank, o_rank;
  int32_t n_experts, topk, moe_inter, shared_inter;
  int32_t window, swa_width, causal, block_size, kv_record_bytes;
  float eps, swiglu_clamp, routed_scale;
} orc_spec;

/* host pointers; matrices row-major [out, in] */
typedef struct {
  const uint16_t *attn_norm, *q_norm, *kv_norm, *ffn_norm;        /* bf16 gammas */
  const uint8_t *wqkv, *wqkv_s, *wq_b, *wq_b_s, *wo_a, *wo_a_s, *wo_b, *wo_b_s; /* e4m3 + E8M0 32x32 */
  const float *router;                                            /* f32 [E, H] */
  const uint8_t *sh_gu, *sh_gu_s, *sh_d, *sh_d_s;                 /* e4m3 + E8M0 32x32 */
  const uint8_t *ex_gu, *ex_gu_s, *ex_d, *ex_d_s;                 /* e2m1 pairs + E8M0 1x32, [E, ...] */
} orc_weights;

typedef struct {
  int32_t rows;
  const uint16_t *x;                 /* bf16 [rows, H] */
  const int32_t *positions;          /* [rows]; < 0 marks a pad row */
  const int32_t *row_req;            /* [rows] request of each row */
  const int32_t *block_table;        /* [n_req, max_blocks] physical page of each logical page */
  int32_t max_blocks;
  uint8_t *cache;                    /* [num_blocks, block_size, record] bytes, updated in place */
  int64_t stride_block, stride_tok, num_blocks;
  const int32_t *force_idx;          /* optional [rows, topk]: route to these experts */
} orc_step;

/* optional outputs of every stage; any pointer may be NULL */
typedef struct {
  uint16_t *xn, *qkv, *q_latn, *kvn, *q, *o, *oa, *h, *u;  /* bf16 */
  float *logits;                     /* [rows, E] f32 */
  double *probs;                     /* [rows, E] */
  int32_t *topk_idx;                 /* [rows, k] (-1 on pad rows) */
  double *topk_w;                    /* [rows, k] */
  uint16_t *t_s;                     /* [rows, I_s] bf16 shared SwiGLU output */
  double *y_s;                       /* [rows, H] shared expert output */
  uint16_t *t_r;                     /* [rows, k, I] bf16 routed SwiGLU outputs */
  double *y_r;                       /* [rows, H] weighted routed sum */
  uint16_t *out;                     /* [rows, H] bf16 layer output */
} orc_trace;

/* number formats */
double orc_e8m0(uint8_t e);
double orc_e4m3(uint8_t code);
double orc_e2m1(uint8_t nibble);
uint8_t orc_encode_e4m3(float v);
double orc_round_bf16(double v);
uint16_t orc_bf16_bits(double v);
void orc_bf16_bits_array(const double *v, size_t n, uint16_t *out);
double orc_bf16_value(uint16_t bits);

/* stages */
void orc_rmsnorm(const uint16_t *x, const uint16_t *gamma, int rows, int dim, float eps,
                 uint16_t *out);
void orc_gemv_mxfp8(const uint16_t *x, int rows, const uint8_t *w, const uint8_t *s, int n,
                    int k, double *y);
void orc_gemv_mxfp4(const uint16_t *x, int rows, const uint8_t *w, const uint8_t *s, int n,
                    int k, double *y);
void orc_kv_quant(const uint16_t *kv, int dim, uint8_t *codes, float *scale);
int orc_kv_insert(const orc_spec *sp, const orc_step *st, const uint16_t *kvn);
void orc_attend(const double *q, const double *keys, const double *vals, int n_keys, int dim,
                double scale, double *out);
int orc_key_range(const orc_spec *sp, const orc_step *st, int row, int *lo, int *hi);
int orc_attention(const orc_spec *sp, const orc_step *st, const uint16_t *q, uint16_t *o);
void orc_router(const uint16_t *u, const float *wr, int rows, int n_experts, int hidden,
                int topk, float routed_scale, const int32_t *positions,
                const int32_t *force_idx, float *logits, double *probs, int32_t *idx,
                double *w);
double orc_swiglu(double g, double u, double clamp);
void orc_ffn(const uint16_t *x, int rows, int fmt4, const uint8_t *gu, const uint8_t *gu_s,
             const uint8_t *d, const uint8_t *d_s, int inter, int hidden, double clamp,
             uint16_t *t, double *y);
int orc_layer(const orc_spec *sp, const orc_weights *w, const orc_step *st, orc_trace *tr);
void orc_ffn_layer(const orc_spec *sp, const orc_weights *w, const uint16_t *x, const uint16_t *a,
                   const int32_t *positions, const int32_t *force_idx, int rows,
                   orc_trace *tr);

void orc_set_threads(int n);
int orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
