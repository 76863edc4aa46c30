// Host side of the C ABI (include/mono_layer.h): validation, tensor maps, the scratch arena
// and the launch schedule of one layer step.
//
// Schedule (stream order, each launch programmatically serialised on its predecessor):
//   K1  rmsnorm(x) -> wqkv -> q/kv norm + KV insert -> wq_b
//   K2  split-window attention (+ combine) -> wo_a -> wo_b + residual -> rmsnorm(h)
//       -> router -> top-k + grouping -> shared gate_up/SwiGLU -> shared down
//       -> routed gate_up/SwiGLU -> routed down -> final combine
// ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", launch table K1 and K2; the
// pages' in-kernel tensor-parallel all-reduces have no counterpart on one GPU.)
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>

#include "../../include/mono_layer.h"
#include "kernels.h"

using namespace mono;

namespace {

constexpr int kLaunchesPerStep = 15;
constexpr int kFfnFirstLaunch = 7;  // the FFN launch runs launches 7..14 of the list
const char* const kLaunchNames[kLaunchesPerStep] = {
    "attn_norm", "wqkv", "qkv_norm_insert", "wq_b", "attention", "wo_a", "wo_b", "ffn_norm",
    "router", "topk_group", "shared_gate_up", "shared_down", "expert_gate_up", "expert_down",
    "final"};

enum DenseId { D_WQKV = 0, D_WQB, D_WOA, D_WOB, D_SHGU, D_SHD, D_COUNT };

// The e4m3 split of an activation (layout in common.cuh) for the dense tensor-core GEMMs.
struct SplitBuf {
  uint8_t* data = nullptr;
  uint8_t* img = nullptr;
};
// The split activations: the inputs of wqkv, wq_b, wo_a, wo_b, the shared gate_up and down
// (split i feeds dense GEMM i).
enum SplitId { S_XN = 0, S_QLATN, S_O, S_OA, S_U, S_TS, S_COUNT };
static_assert((int)S_COUNT == (int)D_COUNT && (int)S_OA == (int)D_WOB && (int)S_TS == (int)D_SHD,
              "split i is the input of dense GEMM i");

struct DensePlan {
  CUtensorMap map;
  const uint8_t* scales;
  int N, K, n_tiles, ksplit, swiglu_I;
  int max_clusters[7];  // co-resident clusters of size ksplit, by activation-tile count nt
  // the tensor-core version for many-row steps: its map, tiles and cluster size (0: none)
  CUtensorMap tc_map;
  int tc_tiles = 0, tc_ks = 0;
};

// Steps with more rows than this run the dense GEMMs on the tensor cores.
constexpr int kDenseTcMinRows = 8;

}  // namespace

struct mono_layer {
  mono_layer_spec spec;
  mono_layer_weights w;
  bool ffn_only = false;  // built without attention weights: FFN launches only
  int device = 0, num_sms = 0;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  size_t buf_off[MONO_BUF_COUNT] = {};
  size_t buf_bytes[MONO_BUF_COUNT] = {};
  int* attn_counters = nullptr;
  float* attn_part = nullptr;
  float* router_part = nullptr;
  int router_kslices = 1;
  // the shared expert runs on a second stream, concurrently with the router and top-k
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  int kernels_last = 0;  // kernels the last step call enqueued
  int* status = nullptr;
  RouteInfo* route = nullptr;
  int* perm = nullptr;
  DensePlan dense[D_COUNT];
  CUtensorMap map_ex_gu, map_ex_d;
  // the expert scale matrices as TMA maps when their rows are whole 16-byte runs
  CUtensorMap map_ex_gu_s, map_ex_d_s;
  bool sc_tma_gu = false, sc_tma_d = false;
  // large steps: the routed experts on the FP4 tensor cores (64-row boxes), with the e2m1
  // term splits of u and t in the arena
  bool expert_tc = false;
  int tc_ctas = 0;  // its grid: co-resident CTAs on every SM
  CUtensorMap map_tc_gu, map_tc_d, map_tc_gu_s, map_tc_d_s;
  uint8_t *u_terms = nullptr, *u_tscales = nullptr, *t_terms = nullptr, *t_tscales = nullptr;
  // many-row steps: the dense GEMMs on the tensor cores, each fed by its activation's split
  bool dense_tc[D_COUNT] = {};
  SplitBuf split[S_COUNT];
  int ctas_gemm8[7] = {};  // by nt
  int ex_ctas = 0;      // persistent CTAs of the expert GEMM (large steps)
  int ex_clusters = 0;  // clusters of EXPERT_CLUSTER CTAs of the K-splitting expert GEMM
  int attn_min_splits = 1;
  cudaEvent_t prof[kLaunchesPerStep + 1] = {};
  bool profiling = false;
  template <class T>
  T* buf(int which) const {
    return reinterpret_cast<T*>(arena + buf_off[which]);
  }
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2D byte tensor [rows, row_bytes] with box_rows x 128-byte boxes and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long row_bytes,
              int box_rows = BOX_ROWS) {
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {BOX_BYTES, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Byte tensor of the given rank (dims innermost first, strides in bytes of dims 1..) with the
// given box; false (and no map) on a misaligned base or stride.
bool make_map_nd(CUtensorMap* m, const void* base, int rank, const long long* dims,
                 const long long* strides, const int* box, bool swizzle128) {
  if (!aligned16(base)) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    b[i] = (cuuint32_t)box[i];
    es[i] = 1;
    if (i > 0) {
      if (strides[i - 1] % 16) return false;
      st[i - 1] = (cuuint64_t)strides[i - 1];
    }
  }
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), d, st, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core expert path's maps (shapes in kernels.h, above ExpertTcParams).
bool make_expert_tc_maps(mono_layer* h) {
  const mono_layer_spec& s = h->spec;
  const long long E = s.n_experts, H = s.hidden, I = s.moe_inter;
  const long long gw[4] = {H / 2, I, 2, E}, gws[3] = {H / 2, I * H / 2, 2 * I * H / 2};
  const long long gs[4] = {H / 32, I, 2, E}, gss[3] = {H / 32, I * H / 32, 2 * I * H / 32};
  const int gwb[4] = {128, 64, 2, 1}, gsb[4] = {16, 64, 2, 1};
  const long long dw[2] = {I / 2, E * H}, dws[1] = {I / 2};
  const long long ds[2] = {I / 32, E * H}, dss[1] = {I / 32};
  const int dwb[2] = {128, 128}, dsb[2] = {16, 128};
  return make_map_nd(&h->map_tc_gu, h->w.ex_gu, 4, gw, gws, gwb, true) &&
         make_map_nd(&h->map_tc_gu_s, h->w.ex_gu_s, 4, gs, gss, gsb, false) &&
         make_map_nd(&h->map_tc_d, h->w.ex_d, 2, dw, dws, dwb, true) &&
         make_map_nd(&h->map_tc_d_s, h->w.ex_d_s, 2, ds, dss, dsb, false);
}

// 2D byte tensor [rows, row_bytes] of E8M0 scales with 16-byte x box_rows boxes, no swizzle;
// false (and no map) unless the rows are whole 16-byte runs at a 16-byte aligned base.
bool make_scale_map(CUtensorMap* m, const void* base, long long rows, long long row_bytes,
                    int box_rows = BOX_ROWS) {
  if (row_bytes % 16 || !aligned16(base)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {16, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FFN fields: hidden, the experts, the intermediates, max_rows.  Attention fields only when
// the handle holds attention weights.
int check_spec(const mono_layer_spec& s, bool ffn_only) {
  if (s.hidden <= 0 || s.moe_inter <= 0 || s.shared_inter <= 0 || s.n_experts <= 0)
    return MONO_ERR_UNSUPPORTED_DIMS;
  // reduction lengths are whole 128-element stages
  if (s.hidden % 128 || s.moe_inter % 128 || s.shared_inter % 128) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.hidden > 8192) return MONO_ERR_UNSUPPORTED_DIMS;  // row kernels
  if (s.topk < 1 || s.topk > 8 || s.topk > s.n_experts || s.n_experts > MAX_EXPERTS)
    return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.max_rows < 1 || s.max_rows > 48) return MONO_ERR_TOO_MANY_ROWS;
  if (ffn_only) return MONO_OK;
  const int qw = s.n_q_heads * s.head_dim;
  if (s.n_q_heads <= 0 || s.q_rank <= 0 || s.o_rank <= 0 || s.kv_dim <= 0 || s.block_size <= 0)
    return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.q_rank % 128 || s.o_rank % 128 || qw % 128) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.kv_dim % 32 || s.kv_dim > 1024) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.q_rank > 4096) return MONO_ERR_UNSUPPORTED_DIMS;  // row kernels
  if (s.head_dim != 64 && s.head_dim != 128) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.kv_dim % s.head_dim) return MONO_ERR_UNSUPPORTED_DIMS;
  const int G = s.kv_dim / s.head_dim;
  if (s.n_q_heads % G || s.n_q_heads / G > 16) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.window < 1 || s.window > 1024 || s.swa_width < 1 || s.swa_width > 1024)
    return MONO_ERR_UNSUPPORTED_DIMS;
  if (s.kv_record_bytes < s.kv_dim + 4 || s.kv_record_bytes % 16) return MONO_ERR_UNSUPPORTED_DIMS;
  return MONO_OK;
}

int nt_bucket(int rows) {
  const int t = (rows + 7) / 8;
  return t <= 1 ? 1 : t <= 2 ? 2 : t <= 4 ? 4 : 6;
}

int cuda_fail(cudaError_t e) {
  (void)cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? MONO_ERR_OUT_OF_MEMORY : MONO_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* mono_layer_strerror(int code) {
  switch (code) {
    case MONO_OK: return "ok";
    case MONO_ERR_INVALID_ARG: return "invalid argument";
    case MONO_ERR_UNSUPPORTED_DIMS: return "unsupported layer dimensions";
    case MONO_ERR_TOO_MANY_ROWS: return "too many rows";
    case MONO_ERR_BAD_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case MONO_ERR_BAD_KV_VIEW: return "KV-cache view strides overlap records or pages";
    case MONO_ERR_UNSUPPORTED_DEVICE: return "not an sm_103 (GB300) device";
    case MONO_ERR_CUDA: return "CUDA runtime error";
    case MONO_ERR_OUT_OF_MEMORY: return "out of device memory";
    case MONO_ERR_DEVICE_STATUS: return "device status word raised";
    default: return "unknown error";
  }
}

int mono_layer_build(const mono_layer_spec* spec, const mono_layer_weights* wt, mono_layer_t** out) {
  if (!spec || !wt || !out) return MONO_ERR_INVALID_ARG;
  *out = nullptr;
  const void* attn_ptrs[] = {wt->attn_norm, wt->q_norm, wt->kv_norm, wt->wqkv, wt->wqkv_s,
                             wt->wq_b,      wt->wq_b_s, wt->wo_a,    wt->wo_a_s, wt->wo_b,
                             wt->wo_b_s};
  const void* ffn_ptrs[] = {wt->ffn_norm, wt->router, wt->sh_gu, wt->sh_gu_s, wt->sh_d,
                            wt->sh_d_s,   wt->ex_gu,  wt->ex_gu_s, wt->ex_d,  wt->ex_d_s};
  int n_attn = 0;
  for (const void* p : attn_ptrs) n_attn += p != nullptr;
  if (n_attn != 0 && n_attn != (int)(sizeof(attn_ptrs) / sizeof(attn_ptrs[0])))
    return MONO_ERR_INVALID_ARG;  // attention weights: all or none
  const bool ffn_only = n_attn == 0;
  int rc = check_spec(*spec, ffn_only);
  if (rc) return rc;
  for (const void* p : attn_ptrs)
    if (p && !aligned16(p)) return MONO_ERR_BAD_ALIGNMENT;
  for (const void* p : ffn_ptrs) {
    if (!p) return MONO_ERR_INVALID_ARG;
    if (!aligned16(p)) return MONO_ERR_BAD_ALIGNMENT;
  }
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MONO_ERR_CUDA;
  }
  if (prop.major != 10 || prop.minor != 3) return MONO_ERR_UNSUPPORTED_DEVICE;
  if (!get_encoder()) return MONO_ERR_CUDA;

  mono_layer* h = new (std::nothrow) mono_layer();
  if (!h) return MONO_ERR_OUT_OF_MEMORY;
  h->spec = *spec;
  h->w = *wt;
  h->ffn_only = ffn_only;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  const mono_layer_spec& s = h->spec;
  const int R = s.max_rows, H = s.hidden, E = s.n_experts, K = s.topk;
  // an FFN-only handle leaves the attention fields unread and sizes no attention buffers
  const int QW = ffn_only ? 0 : s.n_q_heads * s.head_dim;
  const int A = ffn_only ? 0 : s.q_rank + s.kv_dim;
  const int G = ffn_only ? 0 : s.kv_dim / s.head_dim;
  const int q_rank = ffn_only ? 0 : s.q_rank, kv_dim = ffn_only ? 0 : s.kv_dim;
  const int o_rank = ffn_only ? 0 : s.o_rank, n_q = ffn_only ? 0 : s.n_q_heads;
  const int head_dim = ffn_only ? 0 : s.head_dim;

  // dense GEMV plans: K split until the tiles cover the SMs
  struct Def {
    const uint8_t *w, *sc;
    int N, K, swiglu;
  } defs[D_COUNT] = {{wt->wqkv, wt->wqkv_s, A, H, 0},
                     {wt->wq_b, wt->wq_b_s, QW, s.q_rank, 0},
                     {wt->wo_a, wt->wo_a_s, s.o_rank, QW, 0},
                     {wt->wo_b, wt->wo_b_s, H, s.o_rank, 0},
                     {wt->sh_gu, wt->sh_gu_s, 2 * s.shared_inter, H, s.shared_inter},
                     {wt->sh_d, wt->sh_d_s, H, s.shared_inter, 0}};
  for (int i = ffn_only ? D_SHGU : 0; i < D_COUNT; ++i) {
    DensePlan& d = h->dense[i];
    d.scales = defs[i].sc;
    d.N = defs[i].N;
    d.K = defs[i].K;
    d.swiglu_I = defs[i].swiglu;
    d.n_tiles = d.swiglu_I ? d.swiglu_I / BOX_ROWS : (d.N + TILE_M - 1) / TILE_M;
    const int chunks = d.K / 128;
    d.ksplit = 1;  // = cluster size: split K until the tiles cover the SMs
    while (d.n_tiles * d.ksplit < h->num_sms && d.ksplit * 2 <= chunks &&
           d.ksplit * 2 <= MAX_CLUSTER)
      d.ksplit *= 2;
    if (!make_map(&d.map, defs[i].w, d.N, d.K)) {
      delete h;
      return MONO_ERR_CUDA;
    }
    // tensor-core map: {128 B, 128 rows} boxes, SwiGLU matrices as [2][I][K] with 64-row boxes
    bool tc_ok;
    if (d.swiglu_I) {
      const long long dims[3] = {d.K, d.swiglu_I, 2}, st[2] = {d.K, (long long)d.swiglu_I * d.K};
      const int box[3] = {128, 64, 2};
      tc_ok = d.swiglu_I % 64 == 0 && make_map_nd(&d.tc_map, defs[i].w, 3, dims, st, box, true);
      d.tc_tiles = d.swiglu_I / 64;
    } else {
      const long long dims[2] = {d.K, d.N}, st[1] = {d.K};
      const int box[2] = {128, 128};
      tc_ok = make_map_nd(&d.tc_map, defs[i].w, 2, dims, st, box, true);
      d.tc_tiles = (d.N + 127) / 128;
    }
    d.tc_ks = tc_ok ? -1 : 0;  // K split chosen once the kernel's occupancy is known
  }
  if (!make_map(&h->map_ex_gu, wt->ex_gu, (long long)E * 2 * s.moe_inter, H / 2) ||
      !make_map(&h->map_ex_d, wt->ex_d, (long long)E * H, s.moe_inter / 2)) {
    delete h;
    return MONO_ERR_CUDA;
  }
  h->sc_tma_gu =
      make_scale_map(&h->map_ex_gu_s, wt->ex_gu_s, (long long)E * 2 * s.moe_inter, H / 32);
  h->sc_tma_d = make_scale_map(&h->map_ex_d_s, wt->ex_d_s, (long long)E * H, s.moe_inter / 32);
  // the tensor-core expert path wants whole 256-element stages and 16-byte scale boxes
  h->expert_tc = H % 512 == 0 && s.moe_inter % 512 == 0 && make_expert_tc_maps(h);
  const int width = std::max(s.causal ? s.window : s.swa_width, s.window);
  h->attn_min_splits = ffn_only ? 0 : (width + 127) / 128;
  const int attn_splits_max = ffn_only ? 0 : ATTN_MAX_SPLITS;

  // scratch arena
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t sizes[MONO_BUF_COUNT] = {
      (size_t)R * (ffn_only ? 0 : H) * 2, (size_t)R * A * 2, (size_t)R * q_rank * 2,
      (size_t)R * kv_dim * 2, (size_t)R * QW * 2, (size_t)R * QW * 2, (size_t)R * o_rank * 2,
      (size_t)R * H * 2,
      (size_t)R * H * 2,  (size_t)R * E * 4,      (size_t)R * K * 4,        (size_t)R * K * 4,
      (size_t)R * K * 4,  (size_t)R * s.shared_inter * 2, (size_t)R * H * 4,
      (size_t)R * K * s.moe_inter * 2, (size_t)R * K * H * 4};
  for (int b = 0; b < MONO_BUF_COUNT; ++b) {
    h->buf_bytes[b] = sizes[b];
    h->buf_off[b] = take(sizes[b]);
  }
  const size_t o_ctr = take((size_t)R * G * 4);
  const size_t o_part = take((size_t)R * n_q * attn_splits_max * (head_dim + ATTN_PART_HEAD) * 4);
  const size_t o_status = take(16);
  const size_t o_route = take(sizeof(RouteInfo));
  const size_t o_perm = take((size_t)R * K * 4);
  h->router_kslices = (H + ROUTER_KSLICE - 1) / ROUTER_KSLICE;
  const size_t o_rpart = take((size_t)h->router_kslices * R * E * 4);
  // the activation splits of many-row steps (used by the GEMMs that get a tensor-core plan)
  const bool many_rows = R > kDenseTcMinRows;
  const int split_k[S_COUNT] = {ffn_only ? 0 : H, q_rank, QW, o_rank, H, s.shared_inter};
  size_t o_split[S_COUNT][2];
  for (int i = 0; i < S_COUNT; ++i) {
    const size_t stages = many_rows ? (size_t)split_k[i] / 128 : 0;
    o_split[i][0] = take(stages * SPLIT_STAGE_BYTES);
    o_split[i][1] = take(stages * SPLIT_IMG_BYTES);
  }
  const int tc_slots = h->expert_tc ? R * K : 0;
  const size_t o_ut = take((size_t)(h->expert_tc ? R : 0) * (H / 256) * ACT_TERMS * 128);
  const size_t o_us = take((size_t)(h->expert_tc ? R : 0) * (H / 256) * ACT_TERMS * 8);
  const size_t o_tt = take((size_t)tc_slots * (s.moe_inter / 256) * ACT_TERMS * 128);
  const size_t o_ts = take((size_t)tc_slots * (s.moe_inter / 256) * ACT_TERMS * 8);
  h->arena_bytes = off;
  cudaError_t e = cudaMalloc(&h->arena, h->arena_bytes);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e);
  }
  e = cudaMemset(h->arena, 0, h->arena_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->arena);
    delete h;
    return cuda_fail(e);
  }
  h->attn_counters = reinterpret_cast<int*>(h->arena + o_ctr);
  h->attn_part = reinterpret_cast<float*>(h->arena + o_part);
  h->status = reinterpret_cast<int*>(h->arena + o_status);
  h->route = reinterpret_cast<RouteInfo*>(h->arena + o_route);
  h->perm = reinterpret_cast<int*>(h->arena + o_perm);
  h->router_part = reinterpret_cast<float*>(h->arena + o_rpart);
  if (many_rows)
    for (int i = 0; i < S_COUNT; ++i)
      if (split_k[i] > 0) {
        h->split[i].data = h->arena + o_split[i][0];
        h->split[i].img = h->arena + o_split[i][1];
      }
  if (h->expert_tc) {
    h->u_terms = h->arena + o_ut;
    h->u_tscales = h->arena + o_us;
    h->t_terms = h->arena + o_tt;
    h->t_tscales = h->arena + o_ts;
  }

  // kernel attributes and occupancy
  for (int nt : {1, 2, 4, 6}) {
    if (gemm_prepare({8, nt}) != cudaSuccess) rc = MONO_ERR_CUDA;
    h->ctas_gemm8[nt] = std::max(1, gemm_ctas_per_sm({8, nt}));
    for (int i = 0; i < D_COUNT; ++i) {
      DensePlan& d = h->dense[i];
      d.max_clusters[nt] = d.ksplit > 1 ? gemm_max_clusters({8, nt}, d.ksplit)
                                        : h->num_sms * h->ctas_gemm8[nt];
      if (d.max_clusters[nt] < 1) rc = MONO_ERR_CUDA;
    }
  }
  if (gemm_prepare({4, 1, 1}) != cudaSuccess || gemm_prepare({4, 1, 2}) != cudaSuccess)
    rc = MONO_ERR_CUDA;
  h->ex_ctas = h->num_sms * std::max(1, gemm_ctas_per_sm({4, 1, 1}));
  // a margin of clusters below the empty-GPU maximum, so that every cluster is resident at
  // once even while the previous kernels' last CTAs drain (items are assigned statically)
  h->ex_clusters = gemm_max_clusters({4, 1, 2}, EXPERT_CLUSTER) * 7 / 8;
  if (h->ex_clusters < 1) rc = MONO_ERR_CUDA;
  if (!ffn_only && attention_prepare(s.head_dim) != cudaSuccess) rc = MONO_ERR_CUDA;
  if (router_prepare() != cudaSuccess) rc = MONO_ERR_CUDA;
  if (dense_tc_prepare() != cudaSuccess) rc = MONO_ERR_CUDA;
  for (int i = ffn_only ? D_SHGU : 0; i < D_COUNT && !rc && many_rows; ++i) {
    // K split: the largest power of two up to 16 that keeps one CTA per SM, whole stages
    // (at most 8 a CTA), every cluster of the launch resident at once and an owner's receive
    // slots within its rings; else the plain GEMM
    DensePlan& d = h->dense[i];
    if (!d.tc_ks) continue;
    d.tc_ks = 0;
    int ks = 1;
    while (d.tc_tiles * ks * 2 <= h->num_sms && (d.K / 128) % (ks * 2) == 0 && ks * 2 <= 16)
      ks *= 2;
    const int nb = d.swiglu_I ? 2 : 4, brows = d.swiglu_I ? 64 : 32;
    for (; ks >= 1; ks /= 2) {
      const bool fits = d.K / (ks * 128) <= 8 &&
                        (ks == 1 || (nb + ks - 1) / ks * ks * brows * 49 * 4 <= 128 * 1024);
      if (fits && (ks == 1 || dense_tc_max_clusters(ks) >= d.tc_tiles)) {
        d.tc_ks = ks;
        break;
      }
    }
  }
  // a GEMM whose input is another GEMM's output needs that one on the tensor cores too (its
  // epilogue writes the split)
  for (int i = 0; i < D_COUNT; ++i) h->dense_tc[i] = many_rows && h->dense[i].tc_ks > 0;
  h->dense_tc[D_WOB] = h->dense_tc[D_WOB] && h->dense_tc[D_WOA];
  h->dense_tc[D_SHD] = h->dense_tc[D_SHD] && h->dense_tc[D_SHGU];
  if (h->expert_tc) {
    int per_sm = 0;
    if (expert_tc_prepare(&per_sm) != cudaSuccess || per_sm < 1) rc = MONO_ERR_CUDA;
    h->tc_ctas = h->num_sms * per_sm;
  }
  if (!rc && (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
              cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
              cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess))
    rc = MONO_ERR_CUDA;
  if (rc) {
    (void)cudaGetLastError();
    mono_layer_free(h);
    return rc;
  }
  *out = h;
  return MONO_OK;
}

void mono_layer_free(mono_layer_t* h) {
  if (!h) return;
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->arena) cudaFree(h->arena);
  delete h;
}

int mono_layer_status(mono_layer_t* h, int clear) {
  if (!h) return MONO_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(h->status, 0, sizeof(int));
  if (e == cudaSuccess && clear) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  return v;
}

int mono_layer_selftest_wait_timeout(mono_layer_t* h, int64_t budget_ns, void* stream) {
  if (!h || budget_ns < 1000 || budget_ns > 1000000000) return MONO_ERR_INVALID_ARG;
  const cudaError_t e = launch_wait_timeout(reinterpret_cast<cudaStream_t>(stream), h->status,
                                            (unsigned long long)budget_ns);
  return e == cudaSuccess ? MONO_OK : cuda_fail(e);
}

int mono_layer_buffer(mono_layer_t* h, int which, void** dev_ptr, size_t* bytes) {
  if (!h || which < 0 || which >= MONO_BUF_COUNT) return MONO_ERR_INVALID_ARG;
  if (dev_ptr) *dev_ptr = h->arena + h->buf_off[which];
  if (bytes) *bytes = h->buf_bytes[which];
  return MONO_OK;
}

int mono_layer_read_buffer(mono_layer_t* h, int which, void* host_dst, size_t bytes) {
  if (!h || which < 0 || which >= MONO_BUF_COUNT || !host_dst) return MONO_ERR_INVALID_ARG;
  if (bytes > h->buf_bytes[which]) return MONO_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(host_dst, h->arena + h->buf_off[which], bytes, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MONO_OK : cuda_fail(e);
}

int mono_layer_launches_per_step(mono_layer_t* h) { return h ? kLaunchesPerStep : MONO_ERR_INVALID_ARG; }

int mono_layer_kernels_last_step(mono_layer_t* h) { return h ? h->kernels_last : MONO_ERR_INVALID_ARG; }

const char* mono_layer_launch_name(int i) {
  return (i >= 0 && i < kLaunchesPerStep) ? kLaunchNames[i] : nullptr;
}

int mono_layer_set_profile_events(mono_layer_t* h, void* const* events, int n_events) {
  if (!h) return MONO_ERR_INVALID_ARG;
  if (!events) {
    h->profiling = false;
    return MONO_OK;
  }
  if (n_events != kLaunchesPerStep + 1) return MONO_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return MONO_ERR_INVALID_ARG;
    h->prof[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  }
  h->profiling = true;
  return MONO_OK;
}

}  // extern "C"

namespace {

// Enqueues the launches of a step in order, recording the profiling event of each launch
// index before it when profiling is on.
struct Enqueue {
  mono_layer* h;
  cudaStream_t stream;
  int next;      // launch index (into the layer's launch-name list) of the next launch
  int kernels = 0;  // kernels enqueued so far
  template <class F>
  int operator()(F&& launch) {
    const int rc = skip();
    if (rc != MONO_OK) return rc;
    ++kernels;
    const cudaError_t e = launch();
    return e == cudaSuccess ? MONO_OK : cuda_fail(e);
  }
  // a slot this step leaves empty (its profiling event is still recorded)
  int skip() {
    if (h->profiling) {
      const cudaError_t e = cudaEventRecord(h->prof[next], stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    ++next;
    return MONO_OK;
  }
};

#define TRY(x)                          \
  do {                                  \
    const int rc_ = (x);                \
    if (rc_ != MONO_OK) return rc_;     \
  } while (0)
#define TRY_CUDA(x)                                 \
  do {                                              \
    const cudaError_t e_ = (x);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_);    \
  } while (0)

// One MXFP8 dense GEMV of the layer over R rows.
// Dense GEMM id runs on the tensor cores in this step, fed by split id (which its producer
// then writes).
bool use_dense_tc(const mono_layer* h, int R, int id) {
  return h->dense_tc[id] && R > kDenseTcMinRows;
}
const SplitBuf* split_of(const mono_layer* h, int R, int id) {
  return use_dense_tc(h, R, id) ? &h->split[id] : nullptr;
}

cudaError_t dense_launch(const mono_layer* h, int id, int R, const __half* act, int act_ld,
                         int epi, void* outp, int out_ld, const __nv_bfloat16* resid,
                         const Launch& L, const SplitBuf* in = nullptr,
                         const SplitBuf* out = nullptr) {
  const DensePlan& d = h->dense[id];
  if (in && use_dense_tc(h, R, id)) {
    DenseTcParams q = {};
    q.K = d.K;
    q.N = d.N;
    q.swiglu_I = d.swiglu_I;
    q.n_tiles = d.tc_tiles;
    q.ksplit = d.tc_ks;
    q.scales = d.scales;
    q.scale_ld = d.K / 32;
    q.bsplit = in->data;
    q.bimg = in->img;
    q.rows = R;
    q.osplit = out ? out->data : nullptr;
    q.oimg = out ? out->img : nullptr;
    q.epi = epi;
    q.out = outp;
    q.out_ld = out_ld;
    q.resid = resid;
    q.resid_ld = h->spec.hidden;
    q.clamp = h->spec.swiglu_clamp;
    q.status = h->status;
    return launch_dense_tc(L, d.tc_map, q);
  }
  const int nt = nt_bucket(R);
  GemmParams p = {};
  p.scales = d.scales;
  p.scale_ld = d.K / 32;
  p.K = d.K;
  p.N = d.N;
  p.swiglu_I = d.swiglu_I;
  p.act = act;
  p.act_ld = act_ld;
  p.dense_rows = R;
  p.n_tiles = d.n_tiles;
  p.ksplit = d.ksplit;
  p.epi = epi;
  p.out = outp;
  p.out_ld = out_ld;
  p.resid = resid;
  p.resid_ld = h->spec.hidden;
  p.clamp = h->spec.swiglu_clamp;
  p.status = h->status;
  const int clusters = std::min(d.n_tiles, d.max_clusters[nt]);
  return launch_gemm(L, {8, nt}, d.map, nullptr, p, clusters * d.ksplit, d.ksplit);
}

// One MXFP4 routed-expert GEMM over the R * topk (row, slot) pairs grouped by expert.
cudaError_t expert_launch(const mono_layer* h, int R, const CUtensorMap& map,
                          const CUtensorMap* smap, const uint8_t* sc,
                          int Kdim, int rows_per_mat, int swiglu, int n_tiles, const __half* act,
                          int act_ld, const int* rowmap, int epi, void* outp, int out_ld,
                          const Launch& L) {
  const int K = h->spec.topk;
  GemmParams p = {};
  p.scales = sc;
  p.scale_ld = Kdim / 32;
  p.K = Kdim;
  p.N = rows_per_mat;
  p.rows_per_mat = rows_per_mat;
  p.swiglu_I = swiglu;
  p.act = act;
  p.act_ld = act_ld;
  p.act_rowmap = rowmap;
  p.n_tiles = n_tiles;
  // small steps: clusters that split the K of each item when the items are few
  const bool small = R * K <= EXPERT_SMALL_SLOTS;
  p.ksplit = small ? EXPERT_CLUSTER : 1;
  p.n_slots = R * K;
  p.route = h->route;
  p.epi = epi;
  p.out = outp;
  p.out_ld = out_ld;
  p.clamp = h->spec.swiglu_clamp;
  p.status = h->status;
  p.sc_tma = smap != nullptr;
  // large steps schedule items dynamically over the counter the top-k zeroes each step
  p.item_next = small ? nullptr : h->route->item_next + (swiglu > 0 ? 0 : 1);
  if (small)
    return launch_gemm(L, {4, 1, 2}, map, smap, p, h->ex_clusters * EXPERT_CLUSTER,
                       EXPERT_CLUSTER);
  return launch_gemm(L, {4, 1, 1}, map, smap, p, h->ex_ctas, 1);
}

// Inputs of the FFN half of a step (shared by the whole-layer step and the FFN launch).
struct MoeIn {
  NormArgs seam;              // the FFN-seam norm; it writes u (and h, when it forms the residual)
  const __nv_bfloat16* x;     // the layer input, returned unchanged on pad rows
  const int32_t* positions;
  int R;
  int32_t* topk_idx_out;
  float* topk_w_out;
  void* x_out;
};

// K2's FFN half: FFN-seam norm -> router -> top-k + grouping, the shared expert on the side
// stream, routed gate_up / down -> final combine.  Launch indices 7..14 of the layer's list.
int enqueue_moe(mono_layer* h, const MoeIn& m, Enqueue& run) {
  const mono_layer_spec& s = h->spec;
  const cudaStream_t stream = run.stream;
  const Launch L{stream, !h->profiling};
  const int R = m.R, H = s.hidden, E = s.n_experts, K = s.topk;
  // large steps run the routed experts on the FP4 tensor cores; the seam norm then also
  // writes u's e2m1 term split
  const bool tc = h->expert_tc && R * K > EXPERT_SMALL_SLOTS;
  NormArgs seam = m.seam;
  if (tc) {
    seam.terms = h->u_terms;
    seam.term_scales = h->u_tscales;
  }
  if (const SplitBuf* sp = split_of(h, R, S_U)) seam.e4_data = sp->data, seam.e4_img = sp->img;
  TRY(run([&] { return launch_rmsnorm(L, seam, R); }));
  // The shared expert depends only on u: it runs on the side stream, forked right after the
  // seam norm, so that it overlaps the router and the top-k and is done (or nearly) before
  // the routed experts' persistent CTAs take every SM -- forked later, its down GEMM found no
  // SM free until the routed gate_up drained and then held up the routed down.  While
  // profiling, everything stays on one stream in launch-name order.
  const bool fork = !h->profiling;
  const Launch Ls{fork ? h->side : stream, !h->profiling};
  if (fork) TRY_CUDA(cudaEventRecord(h->ev_fork, stream));
  TRY(run([&] {
    return launch_router(L, {h->buf<__half>(MONO_BUF_U), h->w.router, R, E, H, h->router_part});
  }));
  {
    TopkArgs t = {};
    t.partial = h->router_part;
    t.kslices = h->router_kslices;
    t.logits = h->buf<float>(MONO_BUF_LOGITS);
    t.positions = m.positions;
    t.rows = R;
    t.E = E;
    t.k = K;
    t.routed_scale = s.routed_scale;
    t.topk_idx = h->buf<int>(MONO_BUF_TOPK_IDX);
    t.topk_w = h->buf<float>(MONO_BUF_TOPK_W);
    t.slot_pos = h->buf<int>(MONO_BUF_SLOT_POS);
    t.perm = h->perm;
    t.route = h->route;
    t.user_idx = m.topk_idx_out;
    t.user_w = m.topk_w_out;
    t.status = h->status;
    t.lpt = tc ? 1 : 0;  // the tensor-core expert launches hand out items in that order
    TRY(run([&] { return launch_topk(L, t); }));
  }
  if (fork) TRY_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
  TRY(run([&] {
    return dense_launch(h, D_SHGU, R, h->buf<__half>(MONO_BUF_U), H, EPI_SWIGLU_F16,
                        h->buf<void>(MONO_BUF_TS), s.shared_inter, nullptr, Ls,
                        split_of(h, R, S_U), split_of(h, R, S_TS));
  }));
  // Large steps with the shared expert on the tensor cores: its down GEMM runs inside the
  // routed down launch (items ahead of the routed ones) instead of as its own launch -- on
  // its own, its CTAs found no SM until the routed gate_up's persistent CTAs drained and then
  // held up the routed down.  Its launch slot then stays empty (for the profiling events).
  const bool sh_fused = tc && use_dense_tc(h, R, D_SHGU) && use_dense_tc(h, R, D_SHD) &&
                        s.shared_inter % 512 == 0 && H % 128 == 0;
  if (sh_fused) {
    TRY(run.skip());
  } else {
    TRY(run([&] {
      return dense_launch(h, D_SHD, R, h->buf<__half>(MONO_BUF_TS), s.shared_inter, EPI_F32,
                          h->buf<void>(MONO_BUF_YS), H, nullptr, Ls, split_of(h, R, S_TS));
    }));
  }
  if (fork) TRY_CUDA(cudaEventRecord(h->ev_join, h->side));
  // The routed experts start right after the top-k and the shared expert joins before the
  // final combine.  (Small steps' routed clusters take their items statically; those placed
  // on SMs the shared expert still holds start a little later, which costs less than
  // waiting for the whole shared expert: 1 row 81.3 -> 75.0 us, 6 draft rows 82.5 -> 77.6.)
  if (tc) {
    ExpertTcParams p = {};
    p.n_experts = E;
    p.n_slots = R * K;
    p.route = h->route;
    p.clamp = s.swiglu_clamp;
    p.status = h->status;
    p.K = H;
    p.rows_per_mat = 2 * s.moe_inter;
    p.I = s.moe_inter;
    p.n_tiles = s.moe_inter / 64;
    p.act_rows = R;
    p.rowmap = h->perm;
    p.item_next = h->route->item_next;
    p.bterms = h->u_terms;
    p.bscales = h->u_tscales;
    p.t16 = h->buf<__half>(MONO_BUF_TR);
    p.tterms = h->t_terms;
    p.tscales = h->t_tscales;
    TRY(run([&] {
      return launch_expert_tc(L, true, h->map_tc_gu, h->map_tc_gu_s, h->map_tc_gu, p,
                              h->tc_ctas);
    }));
    p.K = s.moe_inter;
    p.rows_per_mat = H;
    p.n_tiles = H / 128;
    p.rowmap = nullptr;
    p.item_next = h->route->item_next + 1;
    p.bterms = h->t_terms;
    p.bscales = h->t_tscales;
    p.y = h->buf<float>(MONO_BUF_YR);
    if (sh_fused) {
      p.sh_tiles = H / 128;
      p.sh_rows = R;
      p.sh_halves = (R + 23) / 24;
      p.sh_nck = s.shared_inter / 128;
      p.sh_scales = h->dense[D_SHD].scales;
      p.sh_scale_ld = s.shared_inter / 32;
      p.sh_bsplit = h->split[S_TS].data;
      p.sh_bimg = h->split[S_TS].img;
      p.ys = h->buf<float>(MONO_BUF_YS);
      // its input, t_s's split, comes from the shared gate_up on the side stream
      if (fork) TRY_CUDA(cudaStreamWaitEvent(stream, h->ev_join, 0));
    }
    TRY(run([&] {
      return launch_expert_tc(L, false, h->map_tc_d, h->map_tc_d_s, h->dense[D_SHD].tc_map, p,
                              h->tc_ctas);
    }));
  } else {
    TRY(run([&] {
      return expert_launch(h, R, h->map_ex_gu, h->sc_tma_gu ? &h->map_ex_gu_s : nullptr,
                           h->w.ex_gu_s, H, 2 * s.moe_inter, s.moe_inter,
                           s.moe_inter / BOX_ROWS, h->buf<__half>(MONO_BUF_U), H, h->perm,
                           EPI_SWIGLU_F16, h->buf<void>(MONO_BUF_TR), s.moe_inter, L);
    }));
    TRY(run([&] {
      return expert_launch(h, R, h->map_ex_d, h->sc_tma_d ? &h->map_ex_d_s : nullptr,
                           h->w.ex_d_s, s.moe_inter, H, 0, H / TILE_M,
                           h->buf<__half>(MONO_BUF_TR), s.moe_inter, nullptr, EPI_F32,
                           h->buf<void>(MONO_BUF_YR), H, L);
    }));
  }
  // (with the shared down inside the routed down, that launch has already joined the side
  // stream; a second join here would only keep the final combine from launching early)
  if (fork && !sh_fused) TRY_CUDA(cudaStreamWaitEvent(stream, h->ev_join, 0));
  {
    FinalArgs f = {};
    f.x = m.x;
    f.h = h->buf<__nv_bfloat16>(MONO_BUF_H);
    f.ys = h->buf<float>(MONO_BUF_YS);
    f.yr = h->buf<float>(MONO_BUF_YR);
    f.slot_pos = h->buf<int>(MONO_BUF_SLOT_POS);
    f.topk_w = h->buf<float>(MONO_BUF_TOPK_W);
    f.positions = m.positions;
    f.rows = R;
    f.H = H;
    f.k = K;
    f.out = reinterpret_cast<__nv_bfloat16*>(m.x_out);
    TRY(run([&] { return launch_final(L, f); }));
  }
  if (h->profiling) TRY_CUDA(cudaEventRecord(h->prof[kLaunchesPerStep], stream));
  h->kernels_last = run.kernels;
  return MONO_OK;
}

}  // namespace

extern "C" {

int mono_layer_step(mono_layer_t* h, const mono_step_args* a, void* stream_ptr) {
  if (!h || !a) return MONO_ERR_INVALID_ARG;
  if (h->ffn_only) return MONO_ERR_INVALID_ARG;
  const mono_layer_spec& s = h->spec;
  const int R = a->rows;
  if (R < 1) return MONO_ERR_INVALID_ARG;
  if (R > s.max_rows) return MONO_ERR_TOO_MANY_ROWS;
  if (!a->x_in || !a->x_out || !a->positions || !a->row_req || !a->block_table || !a->kv_cache)
    return MONO_ERR_INVALID_ARG;
  if (a->max_blocks < 1 || a->n_req < 1 || a->kv_num_blocks < 1) return MONO_ERR_INVALID_ARG;
  if (!aligned16(a->x_in) || !aligned16(a->x_out) || !aligned16(a->kv_cache) ||
      a->kv_stride_tok % 16 || a->kv_stride_block % 16)
    return MONO_ERR_BAD_ALIGNMENT;
  if (a->kv_stride_tok < s.kv_record_bytes ||
      a->kv_stride_block < (int64_t)s.block_size * a->kv_stride_tok)
    return MONO_ERR_BAD_KV_VIEW;

  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  const Launch L{stream, !h->profiling};
  Enqueue run{h, stream, 0};
  const int H = s.hidden, QW = s.n_q_heads * s.head_dim;
  const int A = s.q_rank + s.kv_dim, G = s.kv_dim / s.head_dim;
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a->x_in);

  // ---------------------------------------------------------------- K1: attention front
  TRY(run([&] {
    NormArgs n = {x, H, (const __nv_bfloat16*)h->w.attn_norm, H, s.eps,
                  h->buf<__half>(MONO_BUF_XN), H};
    n.status = h->status;
    if (const SplitBuf* sp = split_of(h, R, S_XN)) n.e4_data = sp->data, n.e4_img = sp->img;
    return launch_rmsnorm(L, n, R);
  }));
  TRY(run([&] {
    return dense_launch(h, D_WQKV, R, h->buf<__half>(MONO_BUF_XN), H, EPI_BF16,
                        h->buf<void>(MONO_BUF_QKV), A, nullptr, L, split_of(h, R, S_XN));
  }));
  {
    QkvNormInsertArgs q = {};
    q.qkv = h->buf<__nv_bfloat16>(MONO_BUF_QKV);
    q.q_rank = s.q_rank;
    q.kv_dim = s.kv_dim;
    q.gq = (const __nv_bfloat16*)h->w.q_norm;
    q.gkv = (const __nv_bfloat16*)h->w.kv_norm;
    q.eps = s.eps;
    q.qlatn = h->buf<__half>(MONO_BUF_QLATN);
    q.kvn = h->buf<__nv_bfloat16>(MONO_BUF_KVN);
    q.positions = a->positions;
    q.row_req = a->row_req;
    q.block_table = a->block_table;
    q.max_blocks = a->max_blocks;
    q.n_req = a->n_req;
    q.block_size = s.block_size;
    q.cache = a->kv_cache;
    q.stride_block = a->kv_stride_block;
    q.stride_tok = a->kv_stride_tok;
    q.num_blocks = a->kv_num_blocks;
    q.status = h->status;
    if (const SplitBuf* sp = split_of(h, R, S_QLATN)) q.e4_data = sp->data, q.e4_img = sp->img;
    TRY(run([&] { return launch_qkv_norm_insert(L, q, R); }));
  }
  TRY(run([&] {
    return dense_launch(h, D_WQB, R, h->buf<__half>(MONO_BUF_QLATN), s.q_rank, EPI_BF16,
                        h->buf<void>(MONO_BUF_Q), QW, nullptr, L, split_of(h, R, S_QLATN));
  }));

  // ---------------------------------------------------------------- K2: attention back
  {
    AttnArgs t = {};
    t.q = h->buf<__nv_bfloat16>(MONO_BUF_Q);
    t.o = h->buf<__half>(MONO_BUF_O);
    t.positions = a->positions;
    t.row_req = a->row_req;
    t.block_table = a->block_table;
    t.rows = R;
    t.max_blocks = a->max_blocks;
    t.n_req = a->n_req;
    t.block_size = s.block_size;
    t.n_q = s.n_q_heads;
    t.kv_dim = s.kv_dim;
    t.window = s.window;
    t.swa_width = s.swa_width;
    t.causal = s.causal;
    t.cache = a->kv_cache;
    t.stride_block = a->kv_stride_block;
    t.stride_tok = a->kv_stride_tok;
    t.num_blocks = a->kv_num_blocks;
    // one split per 128 window keys: a single CTA reads a 128-key window faster than
    // several CTAs read it and combine
    t.splits = h->attn_min_splits;
    t.part = h->attn_part;
    t.counters = h->attn_counters;
    t.status = h->status;
    if (const SplitBuf* sp = split_of(h, R, S_O)) t.e4_data = sp->data, t.e4_img = sp->img;
    TRY(run([&] { return launch_attention(L, t, s.head_dim, G); }));
  }
  TRY(run([&] {
    return dense_launch(h, D_WOA, R, h->buf<__half>(MONO_BUF_O), QW, EPI_F16,
                        h->buf<void>(MONO_BUF_OA), s.o_rank, nullptr, L, split_of(h, R, S_O),
                        split_of(h, R, S_OA));
  }));
  TRY(run([&] {
    return dense_launch(h, D_WOB, R, h->buf<__half>(MONO_BUF_OA), s.o_rank, EPI_RESID_BF16,
                        h->buf<void>(MONO_BUF_H), H, x, L, split_of(h, R, S_OA));
  }));

  // ---------------------------------------------------------------- K2: FFN seam and MoE
  MoeIn m = {};
  m.seam = {h->buf<__nv_bfloat16>(MONO_BUF_H), H, (const __nv_bfloat16*)h->w.ffn_norm, H, s.eps,
            h->buf<__half>(MONO_BUF_U), H};
  m.seam.status = h->status;
  m.seam.warm = 1;  // wo_b is still running when its CTAs become resident
  m.x = x;
  m.positions = a->positions;
  m.R = R;
  m.topk_idx_out = a->topk_idx_out;
  m.topk_w_out = a->topk_w_out;
  m.x_out = a->x_out;
  return enqueue_moe(h, m, run);
}

int mono_ffn_step(mono_layer_t* h, const mono_ffn_args* a, void* stream_ptr) {
  if (!h || !a) return MONO_ERR_INVALID_ARG;
  const mono_layer_spec& s = h->spec;
  const int R = a->rows;
  if (R < 1) return MONO_ERR_INVALID_ARG;
  if (R > s.max_rows) return MONO_ERR_TOO_MANY_ROWS;
  if (!a->x_in || !a->attn_in || !a->x_out || !a->positions) return MONO_ERR_INVALID_ARG;
  if (!aligned16(a->x_in) || !aligned16(a->attn_in) || !aligned16(a->x_out))
    return MONO_ERR_BAD_ALIGNMENT;
  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  Enqueue run{h, stream, kFfnFirstLaunch};
  const int H = s.hidden;
  MoeIn m = {};
  m.seam = {reinterpret_cast<const __nv_bfloat16*>(a->x_in), H,
            (const __nv_bfloat16*)h->w.ffn_norm, H, s.eps, h->buf<__half>(MONO_BUF_U), H,
            reinterpret_cast<const __nv_bfloat16*>(a->attn_in), H,
            h->buf<__nv_bfloat16>(MONO_BUF_H), H};
  m.seam.status = h->status;
  m.x = reinterpret_cast<const __nv_bfloat16*>(a->x_in);
  m.positions = a->positions;
  m.R = R;
  m.topk_idx_out = a->topk_idx_out;
  m.topk_w_out = a->topk_w_out;
  m.x_out = a->x_out;
  return enqueue_moe(h, m, run);
}

#undef TRY
#undef TRY_CUDA

}  // extern "C"
