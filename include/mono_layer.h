/*
 * mono_layer.h -- C ABI of the fused small-batch MoE decode layer for one GB300 (sm_103a).
 *
 * One layer step of a DeepSeek-style MoE decoder for at most 48 rows (8 requests x 1 + 5
 * speculative drafts), as described in "Mono decode layer for DeepSeek-V4.1-Flash on
 * MI355X" (vllm PR #60397), section Purpose, launch table: an attention front (RMSNorm,
 * the MXFP8 wqkv / wq_b GEMVs, the q/kv norms, the fp8 KV-cache insert) followed by the
 * attention back and the MoE (split sliding-window attention with a log-sum-exp combine,
 * wo_a / wo_b, the residual and FFN-seam norm, an f32 router with top-k, an MXFP8 shared
 * expert and MXFP4 routed experts with clamped SwiGLU).  The pages' tensor-parallel
 * all-reduces do not exist here: one GPU holds the whole layer.  The draft-layer variant
 * ("Mono decode for the DSpark draft layers", vllm PR #62131, section Details: top-3,
 * non-causal rows 192 wide) is the same library with other spec integers.
 *
 * Conventions
 *  - Every pointer in mono_layer_weights and mono_step_args is a DEVICE pointer.  The
 *    library borrows them: weights are read in place ("Design": no second copy) and must
 *    stay valid and unchanged for the handle's lifetime; step buffers for the step's
 *    duration on the stream.
 *  - The library owns a scratch arena and a device status word, both sized at build.
 *  - Functions return MONO_OK (0) or a negative MONO_ERR_* code and never abort.
 *  - mono_layer_step enqueues kernels on the given stream and returns without waiting;
 *    it allocates nothing and does no host synchronisation, so a step can be captured in
 *    a CUDA graph.
 *  - Matrices are row-major [out, in].  bf16 values are IEEE bfloat16 bit patterns.
 */
#ifndef MONO_LAYER_H
#define MONO_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mono_layer mono_layer_t; /* opaque handle */

enum {
  MONO_OK = 0,
  MONO_ERR_INVALID_ARG = -1,      /* null pointer, rows out of range, bad enum */
  MONO_ERR_UNSUPPORTED_DIMS = -2, /* dims not multiples of 32, head/latent mismatch, ... */
  MONO_ERR_TOO_MANY_ROWS = -3,    /* rows > max_rows, or max_rows > 48 */
  MONO_ERR_BAD_ALIGNMENT = -4,    /* a pointer or stride not 16-byte aligned */
  MONO_ERR_BAD_KV_VIEW = -5,      /* cache strides smaller than the record / page */
  MONO_ERR_UNSUPPORTED_DEVICE = -6, /* not an sm_103 GPU */
  MONO_ERR_CUDA = -7,             /* a CUDA runtime call failed */
  MONO_ERR_OUT_OF_MEMORY = -8,    /* the scratch arena could not be allocated */
  MONO_ERR_DEVICE_STATUS = -9     /* a previous step raised the device status word */
};

/* Device status bits (mono_layer_status). */
enum {
  MONO_STATUS_UNMAPPED_PAGE = 1, /* a block-table entry was outside [0, kv_num_blocks) */
  MONO_STATUS_WAIT_TIMEOUT = 2,  /* a pipeline wait ran past its time budget */
  MONO_STATUS_BAD_ROUTE = 4,     /* routing metadata out of range */
  MONO_STATUS_F16_RANGE = 8      /* an activation copied to f16 for the tensor cores was
                                    beyond +-65504 and was saturated there (the step's
                                    result then differs from the unsaturated layer) */
};

/*
 * Layer dimensions and constants (the pages' build integers, "MonoBuild / MoeBuild").
 * Constraints checked by mono_layer_build: every reduction length (hidden, q_rank, o_rank,
 * n_q_heads*head_dim, moe_inter, shared_inter) a multiple of 128; kv_dim a multiple of 32
 * and <= 1024; head_dim 64 or 128; kv_dim a multiple of head_dim, n_q_heads a multiple of
 * kv_dim/head_dim with at most 16 heads per latent slice; 1 <= topk <= 8, topk <=
 * n_experts <= 256; 1 <= max_rows <= 48; window, swa_width in 1..1024; kv_record_bytes >=
 * kv_dim + 4 and a multiple of 16.
 */
typedef struct {
  int32_t hidden;          /* H, model width */
  int32_t n_q_heads;       /* query heads */
  int32_t head_dim;        /* per-head width */
  int32_t kv_dim;          /* width of the one cached latent, used as both key and value;
                              head h reads slice h / (n_q_heads / (kv_dim/head_dim)) */
  int32_t q_rank;          /* q latent width: first q_rank outputs of wqkv, input of wq_b */
  int32_t o_rank;          /* output of wo_a, input of wo_b */
  int32_t n_experts;       /* routed experts */
  int32_t topk;            /* experts per row */
  int32_t moe_inter;       /* routed expert intermediate width I */
  int32_t shared_inter;    /* shared expert intermediate width */
  int32_t window;          /* causal rows: a row at position p attends (p - window, p] */
  int32_t swa_width;       /* non-causal rows attend (e - swa_width, e], e = last position
                              of the row's request in this step */
  int32_t causal;          /* 1 causal, 0 non-causal (draft layers) */
  int32_t block_size;      /* tokens per KV page */
  int32_t kv_record_bytes; /* bytes per cached token: kv_dim e4m3 codes, f32 scale, pad */
  int32_t max_rows;        /* largest step this handle accepts (<= 48) */
  float eps;               /* RMSNorm epsilon */
  float swiglu_clamp;      /* gate and up are clamped to [-c, c] before silu(gate) * up */
  float routed_scale;      /* multiplies the renormalised top-k weights */
} mono_layer_spec;

/*
 * Weights, read in place.  MXFP8 = e4m3 codes [N, K] with E8M0 scales [N/32, K/32] (one
 * per 32x32 block); MXFP4 = e2m1 codes packed two per byte (element 2i in the low nibble)
 * [.., N, K/2] with E8M0 scales [.., N, K/32].  All pointers 16-byte aligned.
 */
typedef struct {
  const void *attn_norm, *q_norm, *kv_norm, *ffn_norm; /* bf16 [H], [q_rank], [kv_dim], [H] */
  const uint8_t *wqkv, *wqkv_s;   /* MXFP8 [q_rank + kv_dim, H]: q latent rows, then kv rows */
  const uint8_t *wq_b, *wq_b_s;   /* MXFP8 [n_q_heads * head_dim, q_rank] */
  const uint8_t *wo_a, *wo_a_s;   /* MXFP8 [o_rank, n_q_heads * head_dim] */
  const uint8_t *wo_b, *wo_b_s;   /* MXFP8 [H, o_rank] */
  const float *router;            /* f32 [n_experts, H] */
  const uint8_t *sh_gu, *sh_gu_s; /* MXFP8 [2 * shared_inter, H]: gate rows, then up rows */
  const uint8_t *sh_d, *sh_d_s;   /* MXFP8 [H, shared_inter] */
  const uint8_t *ex_gu, *ex_gu_s; /* MXFP4 [n_experts, 2 * moe_inter, H]: gate, then up */
  const uint8_t *ex_d, *ex_d_s;   /* MXFP4 [n_experts, H, moe_inter] */
} mono_layer_weights;

/*
 * One step.  Rows with positions[r] < 0 are pad rows ("Test Plan": pad rows have slot -1):
 * no KV insert, no attention, no routing, and x_out[r] = x_in[r].
 * The KV cache is a [blocks, block_size, record] byte view; the step writes each valid
 * row's record at (block_table[row_req[r]][p / block_size], p % block_size).  Its strides
 * must satisfy kv_stride_tok >= kv_record_bytes and kv_stride_block >= block_size *
 * kv_stride_tok, so no page overlaps the next (the record-view check asked for in the
 * review of "DecodeSpec / SpecializedDecode", vllm PR #61311: block stride >= block *
 * record), both multiples of 16; the base 16-byte aligned.
 */
typedef struct {
  const void *x_in;        /* bf16 [rows, H] */
  void *x_out;             /* bf16 [rows, H]; may equal x_in */
  const int32_t *positions;   /* [rows] token position, < 0 for a pad row */
  const int32_t *row_req;     /* [rows] request index of each row */
  const int32_t *block_table; /* [n_req, max_blocks] physical page of each logical page */
  int32_t max_blocks;      /* columns of block_table */
  int32_t n_req;           /* rows of block_table; row_req values outside [0, n_req) are errors */
  int32_t rows;            /* 1 <= rows <= max_rows */
  uint8_t *kv_cache;       /* base of the [blocks, block_size, record] view */
  int64_t kv_stride_block; /* bytes between pages */
  int64_t kv_stride_tok;   /* bytes between tokens of a page */
  int64_t kv_num_blocks;   /* pages in the view; table entries outside are errors */
  int32_t *topk_idx_out;   /* optional [rows, topk] chosen experts (-1 on pad rows) */
  float *topk_w_out;       /* optional [rows, topk] their weights */
} mono_step_args;

/* Validates spec and weights on the current CUDA device, allocates the scratch arena and
 * status word, and returns a handle.  Fails with MONO_ERR_UNSUPPORTED_DEVICE on a GPU
 * other than compute capability 10.3.
 * The attention weights (attn_norm, q_norm, kv_norm, wqkv, wq_b, wo_a, wo_b and their
 * scales) are all given or all NULL.  All NULL builds an FFN-only handle for the layers whose
 * attention runs elsewhere: it accepts mono_ffn_step only, reads only the FFN fields of the
 * spec (hidden, n_experts, topk, moe_inter, shared_inter, max_rows, eps, swiglu_clamp,
 * routed_scale) and allocates no attention scratch.  Some but not all of them NULL is
 * MONO_ERR_INVALID_ARG. */
int mono_layer_build(const mono_layer_spec *spec, const mono_layer_weights *weights,
                     mono_layer_t **out);

/* Enqueues one layer step on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * Validates the arguments on the host and returns an error before enqueuing anything if
 * they are wrong.  Device-side faults (an unmapped page) set the status word instead.
 * MONO_ERR_INVALID_ARG on an FFN-only handle. */
int mono_layer_step(mono_layer_t *h, const mono_step_args *args, void *stream);

/*
 * The FFN launch ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", section Purpose,
 * launch table, row FFN; section Scope): for a layer whose attention runs elsewhere, the
 * residual after attention and then K2's FFN seam and MoE -- the second half of
 * mono_layer_step, with the same kernels.  Per row: h = bf16(x_in + attn_in), u =
 * RMSNorm(h, ffn_norm), the f32 router and top-k, the MXFP8 shared expert and the MXFP4
 * routed experts on u, x_out = bf16(h + shared + weighted routed sum); pad rows (positions
 * < 0) are not routed and x_out = x_in.  The pages' attention all-reduce of wo_b's
 * tensor-parallel partials is the identity on one GPU: attn_in is the whole attention output.
 * Every pointer is a DEVICE pointer, 16-byte aligned; bf16 rows are [rows, H] row-major.
 * Works on full and on FFN-only handles; validates on the host before enqueuing anything;
 * allocates nothing and does no host synchronisation (graph-capturable), like a step.
 * MONO_BUF_H then holds h and MONO_BUF_U .. MONO_BUF_YR this step's values; the attention
 * buffers are untouched.  With profiling events set, it records events[7 + i] before its
 * i-th launch (launch names 7..14 of the step list) and events[15] after the last.
 */
typedef struct {
  const void *x_in;          /* bf16 [rows, H] residual stream entering the layer */
  const void *attn_in;       /* bf16 [rows, H] attention output (wo_b's, all-reduced) */
  void *x_out;               /* bf16 [rows, H]; may equal x_in or attn_in */
  const int32_t *positions;  /* [rows] token position, < 0 for a pad row */
  int32_t rows;              /* 1 <= rows <= max_rows */
  int32_t *topk_idx_out;     /* optional [rows, topk] chosen experts (-1 on pad rows) */
  float *topk_w_out;         /* optional [rows, topk] their weights */
} mono_ffn_args;

int mono_ffn_step(mono_layer_t *h, const mono_ffn_args *args, void *stream);

/* Reads the device status word (synchronously; call after the step's stream has
 * finished).  Returns the MONO_STATUS_* bits (>= 0) or a negative error code; clears the
 * word when `clear` is non-zero. */
int mono_layer_status(mono_layer_t *h, int clear);

/* Failure-path check: enqueues one thread that waits, through the same bounded mbarrier wait
 * the pipelines use, on a barrier that nothing completes.  After budget_ns (1 us .. 1 s) the
 * wait gives up, raises MONO_STATUS_WAIT_TIMEOUT in the handle's status word and the kernel
 * returns normally, so the context stays usable.  MONO_ERR_INVALID_ARG for a budget out of
 * range. */
int mono_layer_selftest_wait_timeout(mono_layer_t *h, int64_t budget_ns, void *stream);

/* Releases the handle's scratch arena and status word.  NULL is accepted. */
void mono_layer_free(mono_layer_t *h);

/* Static text for a MONO_OK / MONO_ERR_* code. */
const char *mono_layer_strerror(int code);

/* Intermediate buffers inside the scratch arena, for stage-by-stage testing.  They hold
 * the last step's values until the next step overwrites them. */
enum {
  MONO_BUF_XN = 0,      /* f16 [max_rows, H]          attention-norm output */
  MONO_BUF_QKV = 1,     /* bf16 [max_rows, q_rank + kv_dim] wqkv output */
  MONO_BUF_QLATN = 2,   /* f16 [max_rows, q_rank]     q-norm output */
  MONO_BUF_KVN = 3,     /* bf16 [max_rows, kv_dim]    kv-norm output (what the insert quantises) */
  MONO_BUF_Q = 4,       /* bf16 [max_rows, n_q_heads * head_dim] wq_b output */
  MONO_BUF_O = 5,       /* f16 [max_rows, n_q_heads * head_dim] attention output */
  MONO_BUF_OA = 6,      /* f16 [max_rows, o_rank]     wo_a output */
  MONO_BUF_H = 7,       /* bf16 [max_rows, H]         residual after attention */
  MONO_BUF_U = 8,       /* f16 [max_rows, H]          FFN-seam norm output */
  MONO_BUF_LOGITS = 9,  /* f32 [max_rows, n_experts]  router logits */
  MONO_BUF_TOPK_IDX = 10, /* i32 [max_rows, topk] */
  MONO_BUF_TOPK_W = 11, /* f32 [max_rows, topk] */
  MONO_BUF_SLOT_POS = 12, /* i32 [max_rows, topk] expert-sorted position of (row, slot) */
  MONO_BUF_TS = 13,     /* f16 [max_rows, shared_inter] shared SwiGLU output */
  MONO_BUF_YS = 14,     /* f32 [max_rows, H]          shared expert output */
  MONO_BUF_TR = 15,     /* f16 [max_rows * topk, moe_inter] routed SwiGLU outputs, sorted */
  MONO_BUF_YR = 16,     /* f32 [max_rows * topk, H]   routed expert outputs, sorted, unweighted */
  MONO_BUF_COUNT = 17
};

/* Device address and size in bytes of an intermediate buffer. */
int mono_layer_buffer(mono_layer_t *h, int which, void **dev_ptr, size_t *bytes);

/* Copies an intermediate buffer to host memory (synchronously, after all queued work on the
 * device has finished).  `bytes` may be smaller than the buffer. */
int mono_layer_read_buffer(mono_layer_t *h, int which, void *host_dst, size_t bytes);

/* Number of launch slots of a step: the profiling events below bracket each slot.  A slot
 * that the step's size does not use launches nothing (mono_layer_kernels_last_step counts the
 * kernels actually enqueued). */
int mono_layer_launches_per_step(mono_layer_t *h);

/* Number of kernels the last mono_layer_step or mono_ffn_step call on this handle enqueued
 * (0 before the first call). */
int mono_layer_kernels_last_step(mono_layer_t *h);

/* Short name of the i-th launch of a step ("attn_norm", "wqkv", ...), or NULL. */
const char *mono_layer_launch_name(int i);

/* Profiling support.  With `events` non-NULL (an array of launches_per_step + 1
 * cudaEvent_t), every later mono_layer_step records events[i] just before its i-th launch
 * and events[launches_per_step] after the last one, and launches without programmatic
 * overlap, so that consecutive events bracket exactly one kernel.  The array is borrowed
 * until profiling is turned off again with events = NULL. */
int mono_layer_set_profile_events(mono_layer_t *h, void *const *events, int n_events);

/*
 * Window attention without any allocation, for callers that cannot call cudaMalloc (for
 * example code that runs while a CUDA graph is being captured, or a runtime without a
 * device allocator).  The pages have no counterpart: this is a packaging of the layer's own
 * split-window attention (launch 5 of a step) whose scratch -- per-split partials, the
 * combine counters and a status word -- lives in one array compiled into the library,
 * MONO_NOALLOC_SCRATCH_BYTES on every device that loads it, held until the process exits.
 *
 * q: bf16 [rows, n_q_heads * head_dim] (device); o: f16 [rows, n_q_heads * head_dim]
 * (device, written: each value is the bf16-rounded attention output); both 16-byte
 * aligned; the cache view, positions, row_req and block table as in mono_step_args; only
 * the attention fields of `spec` are read.  The caller owns every buffer.
 * The window is split into S = ceil(max(causal ? window : swa_width, window) / 128) parts,
 * as in a step.  Errors: MONO_ERR_TOO_MANY_ROWS when rows > 48, or when S > 1 and the split
 * partials, rows * n_q_heads * S * (head_dim + 4) * 4 bytes, exceed the scratch less its
 * 8 KB header; MONO_ERR_BAD_ALIGNMENT for q, o or the cache view not 16-byte aligned; the
 * other codes as for a step, all returned before anything is enqueued.  The first call on
 * each device looks the array's device address up (with that device current) and raises
 * two kernels' shared-memory limits; make that first call before any stream capture.  Every call shares the one array and clears its counters
 * and status word on `stream` first: calls whose work overlaps on the GPU (other streams,
 * other threads) race on it and must be serialised by the caller.  Unmapped pages are
 * skipped and their status bit is not reported by this entry point, so a caller must
 * check its block table before the call.
 */
#define MONO_NOALLOC_SCRATCH_BYTES (4u << 20)
int mono_attention_noalloc(const mono_layer_spec *spec, const void *q, void *o,
                           const int32_t *positions, const int32_t *row_req,
                           const int32_t *block_table, int32_t max_blocks, int32_t n_req,
                           int32_t rows, const uint8_t *kv_cache, int64_t kv_stride_block,
                           int64_t kv_stride_tok, int64_t kv_num_blocks, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MONO_LAYER_H */
