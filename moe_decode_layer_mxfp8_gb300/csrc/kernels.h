// Internal launch interface between the host API (mono_layer.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "mx_gemm.cuh"

namespace mono {

// Launch helper: every kernel of the step is launched with programmatic stream
// serialisation so that it may be scheduled while its predecessor drains; each kernel
// calls griddepcontrol.wait before it touches anything the predecessor wrote.
struct Launch {
  cudaStream_t stream;
  bool pdl;
};

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(const Launch& L, dim3 grid, dim3 block, size_t smem,
                             void (*kern)(KArgs...), Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct NormArgs {
  const __nv_bfloat16* in;
  int in_ld;
  const __nv_bfloat16* gamma;
  int dim;
  float eps;
  __half* out;
  int out_ld;
  // optional residual: when resid is set, the kernel normalises h = bf16(in + resid) and
  // also stores h to sum_out
  const __nv_bfloat16* resid = nullptr;
  int resid_ld = 0;
  __nv_bfloat16* sum_out = nullptr;
  int sum_ld = 0;
  int* status = nullptr;  // f16 range bit of the normed output
  // optional e2m1 term split of the normed row (the FP4 tensor-core experts' input; dim a
  // multiple of 256): terms [rows][dim / 256][ACT_TERMS][128 B], each 128-byte term row
  // stored with its 16-byte piece j at piece j ^ t (the 128-byte swizzle of shared-memory
  // row t mod 8); term_scales [rows][dim / 256][ACT_TERMS][8 blocks]
  uint8_t* terms = nullptr;
  uint8_t* term_scales = nullptr;
  // optional e4m3 hi/lo split of the normed rows for the dense tensor-core GEMMs (the layout
  // in common.cuh; rows <= 48)
  uint8_t* e4_data = nullptr;
  uint8_t* e4_img = nullptr;
  // 1: the launch follows a kernel of the same step that is still running, so the kernel runs
  // its output code once on no data (storing nothing) before griddepcontrol.wait, to have it
  // in the instruction caches when the row arrives; 0 for a step's first launch
  int warm = 0;
};

struct QkvNormInsertArgs {
  const __nv_bfloat16* qkv;  // [rows, q_rank + kv_dim]
  int q_rank, kv_dim;
  const __nv_bfloat16 *gq, *gkv;
  float eps;
  __half* qlatn;             // [rows, q_rank]
  __nv_bfloat16* kvn;        // [rows, kv_dim]
  const int *positions, *row_req, *block_table;
  int max_blocks, n_req, block_size;
  uint8_t* cache;
  long long stride_block, stride_tok, num_blocks;
  int* status;
  uint8_t* e4_data = nullptr;  // optional e4m3 split of qlatn (as NormArgs)
  uint8_t* e4_img = nullptr;
};

struct AttnArgs {
  const __nv_bfloat16* q;  // [rows, n_q * head_dim]
  __half* o;               // [rows, n_q * head_dim]
  const int *positions, *row_req, *block_table;
  int rows, max_blocks, n_req, block_size;
  int n_q, kv_dim, window, swa_width, causal;
  const uint8_t* cache;
  long long stride_block, stride_tok, num_blocks;
  int splits;
  float* part;   // [rows, n_q, splits, head_dim + 2]
  int* counters; // [rows, kv_dim / head_dim], left at zero
  int* status;
  uint8_t* e4_data = nullptr;  // optional e4m3 split of o (as NormArgs)
  uint8_t* e4_img = nullptr;
};

constexpr int ROUTER_KSLICE = 1024;  // K per router CTA (the router sums partial logits)
constexpr int ROUTER_MAX_KSLICES = 8;  // hidden <= 8192
constexpr int ATTN_MAX_SPLITS = 8;   // window splits of the attention at most
constexpr int ATTN_PART_HEAD = 4;    // f32 words before a split's partial output: m, l, padding

struct RouterArgs {
  const __half* u;  // [rows, H]
  const float* wr;  // [E, H]
  int rows, E, H;
  float* partial;   // [ceil(H / ROUTER_KSLICE), rows, E]
};

struct TopkArgs {
  const float* partial;  // router partials, summed in slice order
  int kslices;
  float* logits;         // [rows, E] (for tests)
  const int* positions;
  int rows, E, k;
  float routed_scale;
  int* topk_idx;
  float* topk_w;
  int* slot_pos;  // [rows, k] expert-sorted position of (row, slot)
  int* perm;      // [rows * k] sorted position -> row
  RouteInfo* route;
  int* user_idx;
  float* user_w;
  int* status;
  int lpt;  // 1: also write the hit experts in decreasing row count (RouteInfo::lpt_*)
};

struct FinalArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* h;
  const float* ys;
  const float* yr;
  const int* slot_pos;
  const float* topk_w;
  const int* positions;
  int rows, H, k;
  __nv_bfloat16* out;
};

cudaError_t launch_rmsnorm(const Launch&, const NormArgs&, int rows);
cudaError_t launch_qkv_norm_insert(const Launch&, const QkvNormInsertArgs&, int rows);
cudaError_t launch_attention(const Launch&, const AttnArgs&, int head_dim, int groups);
cudaError_t attention_prepare(int head_dim);  // raises the dynamic shared-memory limit
cudaError_t launch_router(const Launch&, const RouterArgs&);
cudaError_t router_prepare();  // raises the dynamic shared-memory limit
cudaError_t launch_topk(const Launch&, const TopkArgs&);
cudaError_t launch_final(const Launch&, const FinalArgs&);
// A bounded wait that runs out (see mono_layer_selftest_wait_timeout).
cudaError_t launch_wait_timeout(cudaStream_t stream, int* status, unsigned long long budget_ns);

// The routed-expert GEMMs of large steps on the FP4 tensor cores (k_expert_tc.cu).  Weight
// maps (packed e2m1, 128-byte swizzle, 128-byte boxes along K): gate_up 4D [experts][2 halves]
// [I rows][H / 2 bytes] with {128 B, 64 rows, 2 halves, 1} boxes (a tile's gate rows, then the
// up rows they pair with); down 2D [experts * H rows][I / 2 bytes] with {128 B, 128 rows}
// boxes.  Scale maps (E8M0, K / 32 bytes a row): the same shapes with 16-byte boxes along K.
// The activations arrive as e2m1 term splits (ACT_TERMS terms, see common.cuh).
struct ExpertTcParams {
  int K;             // reduction length, a multiple of 256
  int rows_per_mat;  // weight rows per expert: 2 I (gate_up) or H (down)
  int I;             // gate_up: the intermediate width (tile t = gate rows 64t.., up rows I + 64t..)
  int n_tiles;       // weight tiles per expert: I / 64 (gate_up) or H / 128 (down)
  int n_experts;
  int n_slots;       // routed (row, slot) pairs of the step
  int act_rows;      // gate_up: rows of the activation split (the step's rows)
  const int* rowmap; // gate_up: expert-sorted slot -> activation row
  const RouteInfo* route;
  int* item_next;    // the launch's work counter, zero at entry
  // activation terms and their scales: gate_up [rows][K / 256][ACT_TERMS][128 B] and
  // [rows][K / 256][ACT_TERMS][8]; down [K / 256][n_slots][ACT_TERMS][128 B] and
  // [K / 256][n_slots][ACT_TERMS][8] (an item's consecutive slots are one run per stage)
  const uint8_t* bterms;
  const uint8_t* bscales;
  __half* t16;             // gate_up: SwiGLU outputs, f16 [slots, I]
  uint8_t* tterms;         // gate_up: their term split, in down's layout
  uint8_t* tscales;
  float* y;                // down: outputs f32 [slots, rows_per_mat]
  // down: the shared expert's down GEMM as extra items (sh_tiles = H / 128, 0: none): its
  // weights by the launch's third map (e4m3 [H][Is], {128 B, 128 rows} boxes), E8M0 scales
  // [H / 32][sh_scale_ld = Is / 32], t_s's split (common.cuh), rows sh_rows in sh_halves
  // halves of at most 24, output y_s f32 [sh_rows, H]
  int sh_tiles, sh_halves, sh_nck, sh_rows;
  const uint8_t* sh_scales;
  int sh_scale_ld;
  const uint8_t* sh_bsplit;
  const uint8_t* sh_bimg;
  float* ys;
  float clamp;
  int* status;
};
// raises the dynamic shared-memory limit; *ctas_per_sm = co-resident CTAs (the grid is that
// times the SM count)
cudaError_t expert_tc_prepare(int* ctas_per_sm);
cudaError_t launch_expert_tc(const Launch&, bool gate_up, const CUtensorMap& wmap,
                             const CUtensorMap& smap, const CUtensorMap& shmap,
                             const ExpertTcParams& p, int grid);

// The dense MXFP8 GEMMs of many-row steps on the tensor cores (k_dense_tc.cu).  Weight map:
// e4m3 [N rows][K bytes], 128-byte swizzle, {128 B, 128 rows} boxes; SwiGLU matrices (gate
// rows, then the up rows I on) 3D [2][I][K] with {128 B, 64 rows, 2} boxes.  Grid: n_tiles x
// ksplit CTAs in clusters of ksplit along K (1, 2, 4, 8 or 16; K / (ksplit 128) <= 8 stages).
// The activations come as their e4m3 split (common.cuh); an F16 or SwiGLU output can be
// split in turn for the next GEMM.
struct DenseTcParams {
  int K, N;
  int swiglu_I;            // > 0: tile t = gate rows 64t.. and up rows I + 64t..
  int n_tiles, ksplit;
  const uint8_t* scales;   // E8M0 [N / 32][K / 32]
  int scale_ld;            // K / 32
  const uint8_t* bsplit;   // the activations' split data [K / 128][SPLIT_STAGE_BYTES]
  const uint8_t* bimg;     // and scale images [K / 128][SPLIT_IMG_BYTES]
  int rows;                // <= 48
  int epi;                 // EPI_* as for the MMA-sync GEMM
  void* out;
  int out_ld;
  const __nv_bfloat16* resid;
  int resid_ld;
  uint8_t* osplit;         // optional split of the output (EPI_F16, EPI_SWIGLU_F16)
  uint8_t* oimg;
  float clamp;
  int* status;
};
cudaError_t dense_tc_prepare();
int dense_tc_max_clusters(int ksplit);  // co-resident clusters of that size on the GPU
cudaError_t launch_dense_tc(const Launch&, const CUtensorMap& wmap, const DenseTcParams& p);

// MX GEMM variants: fmt 8 (MXFP8) with nt in {1, 2, 4, 6}; fmt 4 (MXFP4) with nt 1.
struct GemmVariant {
  int fmt, nt;
  int ks = 0;  // K-share warps per M-tile; 0: the format's default (dense 2, experts 1)
};
int gemm_smem_bytes(GemmVariant v);
cudaError_t gemm_prepare(GemmVariant v);  // raises the dynamic shared-memory limit
int gemm_ctas_per_sm(GemmVariant v);
int gemm_max_clusters(GemmVariant v, int cluster);  // co-resident clusters of that size
// grid must be a multiple of cluster; cluster = p.ksplit for dense matrices, 1 for experts.
// smap: the scale tensor map of an fmt-4 launch with p.sc_tma (else null).
cudaError_t launch_gemm(const Launch&, GemmVariant v, const CUtensorMap& map,
                        const CUtensorMap* smap, const GemmParams& p, int grid, int cluster);

}  // namespace mono
