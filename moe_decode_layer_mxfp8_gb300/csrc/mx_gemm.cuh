// MX block-scaled skinny GEMM: y[rows, N] = x[rows, K] . W[N, K]^T with W in MXFP8 (e4m3,
// 32x32 E8M0 blocks) or MXFP4 (e2m1, 1x32 E8M0 blocks), x bf16 (fed to the tensor cores as
// exact f16 copies), f32 accumulation.  Used for every weight contraction of the layer:
// wqkv, wq_b, wo_a, wo_b, the shared expert and the routed experts ("Mono decode layer for
// DeepSeek-V4.1-Flash on MI355X", launch table rows K1 and K2; section Design: weights read
// in place, MXFP8 row-major with 32x32 E8M0 scales, MXFP4 experts).
//
// Work item = 64 weight rows (two 32-row TMA boxes) x a K range x up to NT*8 activation
// rows.  Dense matrices split K over the CTAs of a thread-block cluster: every CTA leaves
// its partial tile in shared memory, signals its peers through remote mbarriers, and each
// CTA sums one slice of rows across the cluster's tiles through distributed shared memory
// in a fixed order -- deterministic and without a global round trip.  Routed experts take
// one item per (expert, 64 rows, up to 8 routed rows) and the full K; the routing metadata
// is staged in shared memory once per CTA.
//
// CTA = 1 producer warp + 4*KS consumer warps (4 M-tiles x KS K-shares), persistent over
// items: a fixed share per CTA, except in the large-step routed-expert kernel, whose producer
// takes items from a per-launch counter and passes each one to the consumers in the ring
// slot of its first stage.  The producer streams weight tiles with cp.async.bulk.tensor
// (128-byte swizzle), the routed experts' E8M0 scales as 16-byte x 32-row TMA boxes, and
// the activation rows (bulk copies, or 16-byte cp.async for dense matrices) into an NSTAGE
// ring guarded by mbarriers; for dense matrices it issues the first stages' weights before
// waiting on the previous kernel, so that weight streaming overlaps it.  A consumer warp
// owns 16 tile rows (16mt..16mt+15, or in the large-step SwiGLU tiles 8 gate rows with
// their up rows): it decodes its weight fragment in registers (cvt e2m1x2 / e4m3x2 ->
// f16x2), runs m16n8k16 MMAs per 32-wide K block against every 8-row activation tile, and
// applies the block's E8M0 scale to the block's f32 result (or, for MXFP8 with many
// activation tiles, to the decoded weights while that is exact in f16).  Within a 32-wide
// block the MMA's 16 K slots are a fixed permutation of the block's K positions, applied to
// both operands, which leaves the dot product unchanged.
#pragma once

#include "common.cuh"

namespace mono {

constexpr int MAX_EXPERTS = 256;
constexpr int MAX_SLOTS = 48 * 8;  // routed (row, slot) pairs of one step at most
constexpr int EXPERT_ROWS = 8;     // routed rows per expert work item
constexpr int TILE_M = 64;         // weight rows per work item
constexpr int BOX_ROWS = 32;       // rows per TMA box; two boxes per stage
constexpr int BOX_BYTES = 128;     // bytes per row per box = the 128-byte swizzle span
constexpr int W_STAGE_BYTES = TILE_M * BOX_BYTES;
// Threads of a CTA whose consumers are 4 M-tile warps times KS K-shares (the KS warps of an
// M-tile each take 1/KS of every stage's K blocks), plus the producer warp.
__host__ __device__ constexpr int gemm_threads(int ks) { return (4 * ks + 1) * 32; }
constexpr int MAX_CLUSTER = 8;
constexpr int EXPERT_CLUSTER = 4;       // CTAs per cluster of the K-splitting expert GEMM
constexpr int EXPERT_SMALL_SLOTS = 24;  // routed (row, slot) pairs of a step that uses it

// Routing metadata written by the top-k kernel and read by the expert GEMMs.
struct RouteInfo {
  int n_hit;                       // experts with at least one routed row
  int hit_e[MAX_EXPERTS];          // expert id of the d-th hit expert (increasing)
  int hit_off[MAX_EXPERTS];        // first expert-sorted position of its rows
  int hit_cnt[MAX_EXPERTS];        // number of rows routed to it
  int rg_prefix[MAX_EXPERTS + 1];  // prefix sum of ceil(hit_cnt / EXPERT_ROWS)
  int item_next[2];                // work counters of the large-step gate_up / down launches
  // The same hit experts in decreasing row count (ties in expert order): the order in which
  // the large-step launches hand out their items, largest groups first.
  int lpt_e[MAX_EXPERTS], lpt_off[MAX_EXPERTS], lpt_cnt[MAX_EXPERTS];
  int lpt_gpre[MAX_EXPERTS + 1];   // prefix sum of ceil(lpt_cnt / EXPERT_ROWS)
};

// Shared-memory copy of the routing metadata plus the activation row map, and the hit
// expert of every row group (expert d owns row groups [rg_prefix[d], rg_prefix[d + 1]) and
// items [rg_prefix[d] * n_tiles, rg_prefix[d + 1] * n_tiles), so item q belongs to the
// expert of row group q / n_tiles).
struct RouteSmem {
  int n_hit;
  int tile_shift;  // log2(n_tiles) when n_tiles is a power of two, else -1
  int hit_e[MAX_EXPERTS], hit_off[MAX_EXPERTS], hit_cnt[MAX_EXPERTS];
  int rg_prefix[MAX_EXPERTS + 1];
  int rowmap[MAX_SLOTS];
  uint8_t rg_expert[MAX_SLOTS];  // row groups <= routed slots <= MAX_SLOTS
};
static_assert(MAX_EXPERTS <= 256, "rg_expert holds hit-expert indices in a byte");

enum : int { EPI_BF16 = 0, EPI_F16 = 1, EPI_RESID_BF16 = 2, EPI_SWIGLU_F16 = 3, EPI_F32 = 4 };

struct GemmParams {
  const uint8_t* scales;  // E8M0 scales (fmt 8: [N/32, K/32]; fmt 4: [E*N, K/32])
  long long scale_ld;     // bytes per scale row (K/32)
  int K;                  // reduction length in elements (multiple of 128)
  int N;                  // weight rows per matrix
  int rows_per_mat;       // tensor-map rows per expert matrix (expert mode)
  int swiglu_I;           // > 0: tile t = gate rows [32t, 32t+32) and up rows I + [32t, 32t+32)
  const __half* act;      // activations, f16 [*, act_ld]
  int act_ld;
  const int* act_rowmap;  // expert mode: sorted position -> activation row (or null)
  int n_slots;            // expert mode: entries of act_rowmap
  int dense_rows;         // dense mode: activation rows
  int n_tiles;            // work tiles per matrix
  int ksplit;             // dense mode: K splits per tile = cluster size
  int sc_tma;             // fmt 4: scales by TMA (16-byte x 32-row boxes of the scale tensor map)
  int* item_next;         // large-step routed experts: the launch's work counter, zero at entry
  const RouteInfo* route; // non-null selects expert mode
  int epi;
  void* out;
  int out_ld;
  const __nv_bfloat16* resid;  // EPI_RESID_BF16: added before rounding
  int resid_ld;
  float clamp;                 // EPI_SWIGLU_F16
  int* status;
};

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<8> {
  static constexpr int KC = 128;                   // K elements per stage (128 bytes per row)
  static constexpr int ACT_STRIDE = 128 * 2 + 32;  // bytes per activation row (bank spread)
  static constexpr int SC_BYTES = 8;               // 2 block rows x 4 K blocks
};
template <>
struct FmtTraits<4> {
  static constexpr int KC = 256;
  static constexpr int ACT_STRIDE = 256 * 2 + 64;
  // 64 weight rows x 16 bytes: the 16-byte aligned run of scale bytes that holds the
  // stage's 8 K blocks (at byte (k0 / 32) & 8 of the run)
  static constexpr int SC_ROW = 16;
  static constexpr int SC_BYTES = TILE_M * SC_ROW;
};

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

template <int FMT, int NT, int NSTAGE, int KS>
struct GemmLayout {
  static constexpr bool EXPERT = FMT == 4;
  static constexpr int ROWS = NT * 8;
  static constexpr int ACT_BYTES = ROWS * FmtTraits<FMT>::ACT_STRIDE;
  static constexpr int SC_BYTES = FmtTraits<FMT>::SC_BYTES;
  static constexpr int EP_LD = ROWS + 1;  // odd stride: conflict-free column reads
  static constexpr int W_OFF = 0;         // 1024-aligned (128-byte swizzle)
  static constexpr int ACT_OFF = NSTAGE * W_STAGE_BYTES;
  static constexpr int SC_OFF = ACT_OFF + NSTAGE * ACT_BYTES;
  static constexpr int EP_OFF = align_up(SC_OFF + NSTAGE * SC_BYTES, 16);
  // one partial tile per K share, then the K-split receive tile
  static constexpr int EP_TILE = TILE_M * EP_LD;  // floats
  static constexpr int EP_BYTES = (KS + 1) * EP_TILE * 4;
  static constexpr int ROUTE_OFF = align_up(EP_OFF + EP_BYTES, 16);
  static constexpr int ROUTE_BYTES = EXPERT ? (int)sizeof(RouteSmem) : 0;
  static constexpr int BAR_OFF = align_up(ROUTE_OFF + ROUTE_BYTES, 16);
  // full[NSTAGE], empty[NSTAGE], red_full, red_done
  static constexpr int MISC_OFF = BAR_OFF + (2 * NSTAGE + 2) * 8;
  // per ring slot: the work item whose first stage it holds (dynamically scheduled launches)
  static constexpr int SLOTQ_OFF = MISC_OFF + 16;
  static constexpr int BYTES = SLOTQ_OFF + align_up(4 * NSTAGE, 16) + 1024;  // + alignment slack
};

struct Item {
  int wrow_a, wrow_b;  // tensor-map rows of the two boxes
  int sc_a, sc_b;      // scale rows of the two boxes
  bool a_ok, b_ok;     // boxes start inside the matrix
  int k0, nck;         // first K element, number of stages
  int n;               // activation rows
  int row0;            // first output row (expert mode: sorted position)
  int tile, split;
  int col0;            // first output column
};

// Work items of a launch: with ks > 1 every (tile or expert item) is split over the ks CTAs
// of a cluster along K, virtual item q = item * ks + split.
__device__ __forceinline__ int expert_items(const GemmParams& p, const RouteSmem* rs) {
  return rs->rg_prefix[rs->n_hit] * p.n_tiles;
}
// Routed experts split K across the cluster only when there are too few items to fill the
// grid's clusters twice (one-token and draft steps); dense matrices always do.
__device__ __forceinline__ int split_of(const GemmParams& p, const RouteSmem* rs) {
  if (p.ksplit <= 1) return 1;
  if (!rs) return p.ksplit;
  return expert_items(p, rs) <= 2 * (int)(gridDim.x / p.ksplit) ? p.ksplit : 1;
}

template <int FMT>
__device__ __forceinline__ void decode_item(const GemmParams& p, const RouteSmem* rs, int q,
                                            int ks, Item& it) {
  constexpr int KC = FmtTraits<FMT>::KC;
  int base = 0;
  // every CTA's producer and consumer warps decode each of its items: the common cases (no K
  // split, an expert with one row group) take no integer division
  it.split = 0;
  if (ks > 1) {
    it.split = q % ks;
    q /= ks;
  }
  const int nck_all = (p.K + KC - 1) / KC;
  const int cps = ks > 1 ? (nck_all + ks - 1) / ks : nck_all;
  const int c0 = it.split * cps;
  it.nck = max(0, min(cps, nck_all - c0));
  it.k0 = c0 * KC;
  if (rs) {
    const int d = rs->rg_expert[rs->tile_shift >= 0 ? q >> rs->tile_shift : q / p.n_tiles];
    const int rgc = rs->rg_prefix[d + 1] - rs->rg_prefix[d];
    const int local = q - rs->rg_prefix[d] * p.n_tiles;
    it.tile = rgc == 1 ? local : local / rgc;
    const int rg = local - it.tile * rgc;
    base = rs->hit_e[d] * p.rows_per_mat;
    it.n = min(EXPERT_ROWS, rs->hit_cnt[d] - rg * EXPERT_ROWS);
    it.row0 = rs->hit_off[d] + rg * EXPERT_ROWS;
  } else {
    it.tile = q;
    it.n = p.dense_rows;
    it.row0 = 0;
  }
  int ra, rb;
  if (p.swiglu_I > 0) {
    ra = BOX_ROWS * it.tile;
    rb = p.swiglu_I + BOX_ROWS * it.tile;
    it.col0 = BOX_ROWS * it.tile;
  } else {
    ra = TILE_M * it.tile;
    rb = ra + BOX_ROWS;
    it.col0 = ra;
  }
  it.a_ok = ra < p.N;
  it.b_ok = rb < p.N;
  it.wrow_a = base + ra;
  it.wrow_b = base + rb;
  if (FMT == 8) {
    it.sc_a = ra / 32;
    it.sc_b = rb / 32;
  } else {
    it.sc_a = base + ra;
    it.sc_b = base + rb;
  }
}

__device__ __forceinline__ int total_items(const GemmParams& p, const RouteSmem* rs, int ks) {
  return (rs ? expert_items(p, rs) : p.n_tiles) * ks;
}

template <int NTHR>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHR) : "memory");
}

// Waits on an mbarrier phase; gives up when another warp of the CTA has aborted or the
// time budget runs out (then raises the status bit and the CTA's abort flag).
template <bool CLUSTER_ACQUIRE = false>
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort) {
  auto probe = [&]() {
    return CLUSTER_ACQUIRE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (probe()) return true;
    if ((spin & 31) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WAIT_BUDGET_NS) {
        atomicOr(status, ST_WAIT_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// The large-step routed-expert kernel (one K share, never a cluster) schedules its work items
// dynamically; every other variant takes a fixed share.
template <int FMT, int KS>
constexpr bool DYNAMIC_ITEMS = FMT == 4 && KS == 1;

// ------------------------------------------------------------------------------ producer
// A stage has two independent halves: the weight tile with its scales (constant data, safe
// to fetch before the previous kernel has finished) and the activation rows (written by
// it).  The stage's full barrier counts the TMA bytes, one arrival from lane 0 and one
// cp.async arrival per lane issued after the activation copies.
template <int FMT, int NT, int NSTAGE, int KS>
__device__ __forceinline__ void issue_weights(const GemmParams& p, const CUtensorMap* map,
                                              const CUtensorMap* smap,
                                              uint8_t* smem, uint64_t* full, const Item& it,
                                              int c, int s, int lane) {
  using L = GemmLayout<FMT, NT, NSTAGE, KS>;
  constexpr int KC = FmtTraits<FMT>::KC;
  const int k0 = it.k0 + c * KC;
  const int kvalid = min(KC, p.K - k0);
  uint8_t* sst = smem + L::SC_OFF + s * L::SC_BYTES;
  const int kb0 = k0 / 32, nkb = kvalid / 32;
  if (FMT == 8) {
    if (lane < 2) {
      const bool ok = lane == 0 ? it.a_ok : it.b_ok;
      const int row = lane == 0 ? it.sc_a : it.sc_b;
      const uint8_t* src = p.scales + row * p.scale_ld + kb0;
      cp_async4(sst + lane * 4, ok ? (const void*)src : (const void*)p.scales,
                ok ? (uint32_t)min(4, nkb) : 0u);
    }
  } else if (!p.sc_tma) {
    // scale rows that are not whole 16-byte runs: two 4-byte copies per weight row, placed
    // where the TMA path puts them
    constexpr int SC_ROW = FmtTraits<4>::SC_ROW;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool ok = half == 0 ? it.a_ok : it.b_ok;
      const long long row = (long long)(half == 0 ? it.sc_a : it.sc_b) + lane;
      const uint8_t* src = p.scales + row * p.scale_ld + kb0;
      uint8_t* dst = sst + (half * BOX_ROWS + lane) * SC_ROW + (kb0 & 8);
      const int n0 = ok ? min(4, nkb) : 0, n1 = ok ? max(0, min(4, nkb - 4)) : 0;
      cp_async4(dst, n0 ? (const void*)src : (const void*)p.scales, (uint32_t)n0);
      cp_async4(dst + 4, n1 ? (const void*)(src + 4) : (const void*)p.scales, (uint32_t)n1);
    }
  }
  if (lane == 0) {
    // fmt 4 with sc_tma: the two boxes' scale runs (16 bytes x 32 rows each) by TMA too, in
    // place of 64 four-byte copies a stage
    constexpr uint32_t SC_BOX = FmtTraits<4>::SC_ROW * BOX_ROWS;
    const bool sc_tma = FMT == 4 && p.sc_tma;
    mbar_arrive_expect_tx(&full[s], W_STAGE_BYTES + (sc_tma ? 2 * SC_BOX : 0u));
    const int xb = FMT == 8 ? k0 : k0 / 2;
    uint8_t* wst = smem + L::W_OFF + s * W_STAGE_BYTES;
    tma_load_2d(wst, map, xb, it.wrow_a, &full[s]);
    tma_load_2d(wst + BOX_ROWS * BOX_BYTES, map, xb, it.wrow_b, &full[s]);
    if (sc_tma) {
      tma_load_2d(sst, smap, kb0 & ~15, it.sc_a, &full[s]);
      tma_load_2d(sst + SC_BOX, smap, kb0 & ~15, it.sc_b, &full[s]);
    }
  }
}

template <int FMT, int NT, int NSTAGE, int KS>
__device__ __forceinline__ void issue_acts(const GemmParams& p, const RouteSmem* rs,
                                           uint8_t* smem, uint64_t* full, const Item& it, int c,
                                           int s, int lane) {
  using L = GemmLayout<FMT, NT, NSTAGE, KS>;
  constexpr int KC = FmtTraits<FMT>::KC;
  constexpr int ASTR = FmtTraits<FMT>::ACT_STRIDE;
  constexpr int CPR = KC * 2 / 16;  // 16-byte chunks per activation row per stage
  const int k0 = it.k0 + c * KC;
  const int vbytes = min(KC, p.K - k0) * 2;
  uint8_t* ast = smem + L::ACT_OFF + s * L::ACT_BYTES;
  if (FMT == 4 && vbytes == KC * 2) {
    // expert rows (<= 8 of 512 bytes): one bulk copy per row, counted on the stage's barrier
    // before any lane's arrival below can complete the phase.  (The dense matrices' up to 48
    // rows of 256 bytes stream faster as 16-byte copies spread over the lanes.)
    if (lane == 0) mbar_expect_tx(&full[s], (uint32_t)(it.n * vbytes));
    __syncwarp();
    for (int i = lane; i < it.n; i += 32) {
      int arow = i;
      if (rs) arow = p.act_rowmap ? rs->rowmap[it.row0 + i] : it.row0 + i;
      bulk_load_g2s(ast + i * ASTR, p.act + (long long)arow * p.act_ld + k0, (uint32_t)vbytes,
                    &full[s]);
    }
  } else {  // 16-byte copies, zero-filled past the end of K
    for (int idx = lane; idx < it.n * CPR; idx += 32) {
      const int i = idx / CPR, ch = idx - i * CPR;
      int arow = i;
      if (rs) arow = p.act_rowmap ? rs->rowmap[it.row0 + i] : it.row0 + i;
      const bool ok = ch * 16 < vbytes;
      const __half* src = p.act + (long long)arow * p.act_ld + k0 + ch * 8;
      cp_async16(ast + i * ASTR + ch * 16, ok ? (const void*)src : (const void*)p.act,
                 ok ? 16u : 0u);
    }
  }
  cp_async_arrive_noinc(&full[s]);  // after this lane's scale copies (and any above) land
}

// The first item's first stages whose weights are issued before griddepcontrol.wait (dense
// matrices only); returns how many.
template <int FMT, int NT, int NSTAGE, int KS>
__device__ int prefetch_weights(const GemmParams& p, const CUtensorMap* map, uint8_t* smem,
                                uint64_t* full) {
  const int lane = threadIdx.x & 31;
  const int ks = split_of(p, nullptr);
  if (p.route || (int)blockIdx.x >= total_items(p, nullptr, ks)) return 0;
  Item it;
  decode_item<FMT>(p, nullptr, blockIdx.x, ks, it);
  const int pre = min(NSTAGE, it.nck);
  for (int c = 0; c < pre; ++c)
    issue_weights<FMT, NT, NSTAGE, KS>(p, map, map, smem, full, it, c, c, lane);
  return pre;
}

template <int FMT, int NT, int NSTAGE, int KS>
__device__ void gemm_producer(const GemmParams& p, const RouteSmem* rs, const CUtensorMap* map,
                              const CUtensorMap* smap, uint8_t* smem, uint64_t* full,
                              uint64_t* empty, volatile int* abort, int pre) {
  using L = GemmLayout<FMT, NT, NSTAGE, KS>;
  const int lane = threadIdx.x & 31;
  const int ks = split_of(p, rs);
  const int n_items = total_items(p, rs, ks);
  volatile int* slot_q = reinterpret_cast<volatile int*>(smem + L::SLOTQ_OFF);
  int iter = 0;
  // Large-step routed experts take their items from the launch's counter (a CTA that becomes
  // resident late, behind another stream's kernel, then finds little or no work left instead
  // of a fixed share), fetching the next index while the current item streams; the others
  // take every gridDim.x-th item.
  int q = blockIdx.x, qn = 0;
  if constexpr (DYNAMIC_ITEMS<FMT, KS>) {
    if (lane == 0) q = atomicAdd(p.item_next, 1);
    q = __shfl_sync(0xffffffffu, q, 0);
  }
  while (q < n_items) {
    if constexpr (DYNAMIC_ITEMS<FMT, KS>) {
      if (lane == 0) qn = atomicAdd(p.item_next, 1);
    }
    Item it;
    decode_item<FMT>(p, rs, q, ks, it);
    for (int c = 0; c < it.nck; ++c, ++iter) {
      const int s = iter % NSTAGE;
      const uint32_t ph = (iter / NSTAGE) & 1;
      if (!pipe_wait(&empty[s], ph ^ 1, p.status, abort)) goto drain;
      // published before lane 0's arrival on the stage's barrier (a release) in issue_weights
      if (DYNAMIC_ITEMS<FMT, KS> && c == 0 && lane == 0) slot_q[s] = q;
      if (iter >= pre) issue_weights<FMT, NT, NSTAGE, KS>(p, map, smap, smem, full, it, c, s, lane);
      issue_acts<FMT, NT, NSTAGE, KS>(p, rs, smem, full, it, c, s, lane);
    }
    if constexpr (DYNAMIC_ITEMS<FMT, KS>)
      q = __shfl_sync(0xffffffffu, qn, 0);
    else
      q += gridDim.x;
  }
  if constexpr (DYNAMIC_ITEMS<FMT, KS>) {
    // the end: one more stage that carries no data, only the end mark
    const int s = iter % NSTAGE;
    if (!pipe_wait(&empty[s], ((iter / NSTAGE) & 1) ^ 1, p.status, abort)) goto drain;
    if (lane == 0) {
      slot_q[s] = -1;
      mbar_arrive(&full[s]);
    }
    cp_async_arrive_noinc(&full[s]);  // the other 32 arrivals of the phase
  }
  return;
drain:
  // A wait failed: let the copies already issued land before the CTA exits.
  for (int k = 1; k <= NSTAGE && k <= iter; ++k) {
    const int j = iter - k;
    mbar_wait(&full[j % NSTAGE], (j / NSTAGE) & 1, p.status, 100000000ull);
  }
}

// ------------------------------------------------------------------------------ epilogue
__device__ __forceinline__ float swiglu_clamped(float g, float u, float c) {
  g = fminf(fmaxf(g, -c), c);
  u = fminf(fmaxf(u, -c), c);
  return g / (1.0f + expf(-g)) * u;
}

// Writes finished tile values to the output.  fin[m * EP_LD + i] holds the value of output
// row (row0 + i), column (col0 + m) -- for SwiGLU tiles (SW) the already combined gate/up
// value -- for m in [0, per), per = 32 (SW) or 64 a compile-time constant.  Four values per
// thread are in flight at a time, their residual reads issued before any store.
template <int EP_LD, int NTHR, bool SW>
__device__ void store_rows(const GemmParams& p, const Item& it, const float* fin, int tid) {
  constexpr int per = SW ? BOX_ROWS : TILE_M;
  const int total = per * it.n;
  const int ncols = SW ? p.swiglu_I : p.N;
  for (int base = tid; base < total; base += 4 * NTHR) {
    float v[4], r[4];
    size_t o[4];
    bool ok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * NTHR;
      const int i = idx / per, m = idx - (idx / per) * per;
      const int col = it.col0 + m;
      ok[u] = idx < total && col < ncols;
      o[u] = (size_t)(it.row0 + i) * p.out_ld + col;
      v[u] = ok[u] ? fin[m * EP_LD + i] : 0.0f;
      r[u] = ok[u] && p.epi == EPI_RESID_BF16
                 ? __bfloat162float(p.resid[(size_t)(it.row0 + i) * p.resid_ld + col])
                 : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!ok[u]) continue;
      switch (p.epi) {
        case EPI_BF16:
          reinterpret_cast<__nv_bfloat16*>(p.out)[o[u]] = __float2bfloat16_rn(v[u]);
          break;
        case EPI_F16:
        case EPI_SWIGLU_F16:
          reinterpret_cast<__half*>(p.out)[o[u]] = bf16_as_f16_sat(v[u], p.status);
          break;
        case EPI_RESID_BF16:
          reinterpret_cast<__nv_bfloat16*>(p.out)[o[u]] = __float2bfloat16_rn(r[u] + v[u]);
          break;
        default:
          reinterpret_cast<float*>(p.out)[o[u]] = v[u];
          break;
      }
    }
  }
}

// Epilogue of a tile whose full result sits in this CTA's shared memory.  SwiGLU tiles first
// combine each gate row m with its up row m + 32 in place.
template <int EP_LD, int NTHR>
__device__ void epilogue_local(const GemmParams& p, const Item& it, float* ep, int tid) {
  const bool sw = p.epi == EPI_SWIGLU_F16;
  if (sw) {
    for (int idx = tid; idx < BOX_ROWS * it.n; idx += NTHR) {
      const int i = idx / BOX_ROWS, m = idx - i * BOX_ROWS;
      ep[m * EP_LD + i] = swiglu_clamped(ep[m * EP_LD + i], ep[(m + BOX_ROWS) * EP_LD + i], p.clamp);
    }
    consumer_bar<NTHR>();
  }
  if (sw)
    store_rows<EP_LD, NTHR, true>(p, it, ep, tid);
  else
    store_rows<EP_LD, NTHR, false>(p, it, ep, tid);
}

// One finished value of output row orow, column col, as store_rows writes it.
__device__ __forceinline__ void store_value(const GemmParams& p, int orow, int col, float v) {
  const size_t o = (size_t)orow * p.out_ld + col;
  switch (p.epi) {
    case EPI_BF16:
      reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v);
      break;
    case EPI_F16:
    case EPI_SWIGLU_F16:
      reinterpret_cast<__half*>(p.out)[o] = bf16_as_f16_sat(v, p.status);
      break;
    case EPI_RESID_BF16:
      reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(
          __bfloat162float(p.resid[(size_t)orow * p.resid_ld + col]) + v);
      break;
    default:
      reinterpret_cast<float*>(p.out)[o] = v;
      break;
  }
}

// Epilogue straight from the accumulators (large-step routed experts: one K share, no
// cluster).  Thread (g, c) holds activation rows 8t + 2c and 8t + 2c + 1 of tile rows rowA
// (acc[t][0..1]) and rowB (acc[t][2..3]); with pair_gu those are a gate row and its up row,
// combined here into output column col0 + rowA.
template <int NT>
__device__ __forceinline__ void epilogue_regs(const GemmParams& p, const Item& it,
                                              const float (&acc)[NT][4], int rowA, int rowB,
                                              int c, bool pair_gu) {
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 8 * t + 2 * c + h;
      if (i >= it.n) continue;
      if (pair_gu) {
        const int col = it.col0 + rowA;
        if (col < p.swiglu_I)
          store_value(p, it.row0 + i, col, swiglu_clamped(acc[t][h], acc[t][2 + h], p.clamp));
      } else {
        const int ca = it.col0 + rowA, cb = it.col0 + rowB;
        if (ca < p.N) store_value(p, it.row0 + i, ca, acc[t][h]);
        if (cb < p.N) store_value(p, it.row0 + i, cb, acc[t][2 + h]);
      }
    }
  }
}

// owner_epilogue with the cluster size and the SwiGLU pairing as compile-time constants.
template <int EP_LD, int NTHR>
__device__ __forceinline__ void owner_epilogue_any(const GemmParams& p, const Item& it,
                                                   const float* recv, int tid, uint32_t rank);

// Accumulators of consumer warp (M-tile mt) into its K share's partial tile.
template <int NT, int EP_LD>
__device__ __forceinline__ void write_partial(const float (&acc)[NT][4], float* ep_mine, int mt,
                                              int g, int c, int ntl) {
  const int m0 = 16 * mt + g;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    if (NT == 1 || t < ntl) {
      const int col = t * 8 + 2 * c;
      ep_mine[m0 * EP_LD + col] = acc[t][0];
      ep_mine[m0 * EP_LD + col + 1] = acc[t][1];
      ep_mine[(m0 + 8) * EP_LD + col] = acc[t][2];
      ep_mine[(m0 + 8) * EP_LD + col + 1] = acc[t][3];
    }
  }
}

// The K shares' partial tiles added, in a fixed order, into the first.
template <int KS, int EP_LD, int NTHR>
__device__ __forceinline__ void sum_kshares(float* ep, int ntl, int tid) {
  (void)ntl;
  constexpr int cols = EP_LD - 1;  // every column of the tile (a compile-time divisor)
  for (int idx = tid; idx < TILE_M * cols; idx += NTHR) {
    const int m = idx / cols, col = idx - m * cols;
    float v = ep[m * EP_LD + col];
#pragma unroll
    for (int k = 1; k < KS; ++k) v += ep[k * TILE_M * EP_LD + m * EP_LD + col];
    ep[m * EP_LD + col] = v;
  }
}

// K-split tiles across a cluster of ks CTAs.  Rank o owns weight rows (output columns)
// [o * per, o * per + per) of the tile, per = 64 / ks -- for SwiGLU tiles per = 32 / ks gate
// rows together with their up rows 32 further.  Each CTA pushes the owner's rows of its
// partial tile into the owner's receive tile with bulk shared-to-shared copies that complete
// on the owner's mbarrier, so the reduction costs one asynchronous transfer instead of
// element-wise remote accesses; the owner adds the ks slots in rank order.  Receive tile:
// slot s (source rank) holds 64 / ks rows of EP_LD floats (SwiGLU: gate rows, then up rows).
template <int EP_LD>
__device__ __forceinline__ void push_slices(const GemmParams& p, const float* part, float* recv,
                                            uint64_t* red_full, uint32_t rank, int n) {
  const bool sw = p.epi == EPI_SWIGLU_F16;
  const int ks = p.ksplit;
  const int per = (sw ? BOX_ROWS : TILE_M) / ks;
  const uint32_t chunk = (uint32_t)(per * EP_LD * 4);  // bytes of one run of rows
  const uint32_t srows = (uint32_t)(TILE_M / ks);
  // this owner's slots arrive from every rank
  mbar_arrive_expect_tx(red_full, (uint32_t)ks * srows * EP_LD * 4);
  const uint32_t recv_u = smem_u32(recv), bar_u = smem_u32(red_full);
  for (int o = 0; o < ks; ++o) {
    const uint32_t dst = mapa_shared(recv_u + rank * srows * EP_LD * 4, (uint32_t)o);
    const uint32_t bar = mapa_shared(bar_u, (uint32_t)o);
    bulk_copy_s2s(dst, part + o * per * EP_LD, chunk, bar);
    if (sw) bulk_copy_s2s(dst + chunk, part + (BOX_ROWS + o * per) * EP_LD, chunk, bar);
  }
  bulk_commit();
  (void)n;
}

// The owner's share of a K-split tile: adds its receive slots in slot order and writes its
// columns out, two values per thread in flight at a time.
template <int EP_LD, int NTHR, int KSPLIT, bool SW>
__device__ void owner_epilogue(const GemmParams& p, const Item& it, const float* recv, int tid,
                               uint32_t rank) {
  constexpr bool sw = SW;
  constexpr int ks = KSPLIT;
  constexpr int per = (SW ? BOX_ROWS : TILE_M) / KSPLIT;
  constexpr int srows = TILE_M / KSPLIT;
  const int total = per * it.n;
  const int ncols = sw ? p.swiglu_I : p.N;
  constexpr int B = 2;
  for (int base = tid; base < total; base += B * NTHR) {
    float v[B], r[B];
    size_t o[B];
    bool ok[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int idx = base + u * NTHR;
      const int i = idx / per, lr = idx - (idx / per) * per;
      const int col = it.col0 + (int)rank * per + lr;
      ok[u] = idx < total && col < ncols;
      o[u] = (size_t)(it.row0 + i) * p.out_ld + col;
      r[u] = ok[u] && p.epi == EPI_RESID_BF16
                 ? __bfloat162float(p.resid[(size_t)(it.row0 + i) * p.resid_ld + col])
                 : 0.0f;
      float s = 0.0f, su = 0.0f;
      if (idx < total) {
#pragma unroll
        for (int sl = 0; sl < ks; ++sl) {
          const float* q = recv + (sl * srows + lr) * EP_LD + i;
          s += q[0];
          if (sw) su += q[per * EP_LD];
        }
      }
      v[u] = sw ? swiglu_clamped(s, su, p.clamp) : s;
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      if (!ok[u]) continue;
      switch (p.epi) {
        case EPI_BF16:
          reinterpret_cast<__nv_bfloat16*>(p.out)[o[u]] = __float2bfloat16_rn(v[u]);
          break;
        case EPI_F16:
        case EPI_SWIGLU_F16:
          reinterpret_cast<__half*>(p.out)[o[u]] = bf16_as_f16_sat(v[u], p.status);
          break;
        case EPI_RESID_BF16:
          reinterpret_cast<__nv_bfloat16*>(p.out)[o[u]] = __float2bfloat16_rn(r[u] + v[u]);
          break;
        default:
          reinterpret_cast<float*>(p.out)[o[u]] = v[u];
          break;
      }
    }
  }
}

template <int EP_LD, int NTHR>
__device__ __forceinline__ void owner_epilogue_any(const GemmParams& p, const Item& it,
                                                   const float* recv, int tid, uint32_t rank) {
  const bool sw = p.epi == EPI_SWIGLU_F16;
#define MONO_OWNER_CASE(K)                                                         \
  case K:                                                                          \
    if (sw) owner_epilogue<EP_LD, NTHR, K, true>(p, it, recv, tid, rank);          \
    else owner_epilogue<EP_LD, NTHR, K, false>(p, it, recv, tid, rank);            \
    break;
  switch (p.ksplit) {
    MONO_OWNER_CASE(2)
    MONO_OWNER_CASE(4)
    MONO_OWNER_CASE(8)
    default: break;  // ksplit in {2, 4, 8} for every clustered launch (host-checked)
  }
#undef MONO_OWNER_CASE
}

// E8M0 byte -> 2^(e-127) for e in 1..254 by placing the byte in the f32 exponent field
// (e = 0 gives 0 instead of 2^-127 and e = 255 infinity instead of NaN; scales of
// real weights lie far inside that range).
__device__ __forceinline__ float e8m0_fast(uint32_t word, int byte) {
  return __uint_as_float(__byte_perm(word, 0u, 0x4440u + byte) << 23);
}

// ------------------------------------------------------------------------------ consumer
template <int FMT, int NT, int NSTAGE, int KS>
__device__ void gemm_consumer(const GemmParams& p, const RouteSmem* rs, uint8_t* smem,
                              uint64_t* full, uint64_t* empty, uint64_t* red_full,
                              uint64_t* red_done, volatile int* abort) {
  using L = GemmLayout<FMT, NT, NSTAGE, KS>;
  constexpr int ASTR = FmtTraits<FMT>::ACT_STRIDE;
  constexpr int NB = FmtTraits<FMT>::KC / 32;  // 32-wide K blocks per stage
  constexpr int CONSUMER_WARPS = 4 * KS, NTHR = CONSUMER_WARPS * 32;
  constexpr int HB = NB / KS;                  // blocks per K share
  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const int mt = w & 3, kh = w >> 2;           // M-tile and K-half of this warp
  const int g = lane >> 2, c = lane & 3;
  // tile rows of this thread's two MMA row halves (MMA rows g and g + 8).  Warp mt takes tile
  // rows 16mt .. 16mt + 15, except in the large-step routed-expert kernel's SwiGLU tiles:
  // there it takes gate rows 8mt .. 8mt + 7 with their up rows (the same rows of the second
  // box), so that each thread holds a gate value and its up value and the epilogue needs no
  // exchange between warps.  Both choices keep row & 7 = g, the 128-byte swizzle's key.
  const bool pair_gu = KS == 1 && FMT == 4 && p.swiglu_I > 0;
  const int rowA = pair_gu ? 8 * mt + g : 16 * mt + g;
  const int rowB = pair_gu ? BOX_ROWS + 8 * mt + g : 16 * mt + g + 8;
  float* ep = reinterpret_cast<float*>(smem + L::EP_OFF);
  float* ep_mine = ep + kh * (TILE_M * L::EP_LD);
  // swizzled word offsets of this thread's K blocks (fmt 4: one chunk a block; fmt 8: two)
  int offs[FMT == 4 ? HB : 2 * HB];
#pragma unroll
  for (int j = 0; j < (FMT == 4 ? HB : 2 * HB); ++j)
    offs[j] = (((FMT == 4 ? kh * HB : 2 * kh * HB) + j) ^ g) * 16 + c * 4;
  const int ks = split_of(p, rs);
  const int n_items = total_items(p, rs, ks);
  const bool clustered = ks > 1;
  const uint32_t rank = clustered ? cluster_ctarank() : 0u;
  int iter = 0, tiles_done = 0;
  const volatile int* slot_q = reinterpret_cast<const volatile int*>(smem + L::SLOTQ_OFF);
  for (int q = blockIdx.x;; q += gridDim.x) {
    if constexpr (DYNAMIC_ITEMS<FMT, KS>) {
      // the next stage holds the next item's first K chunk and its index, or the end mark
      // (the stage loop below waits on it again, which then returns at once)
      const int s = iter % NSTAGE;
      if (!pipe_wait(&full[s], (iter / NSTAGE) & 1, p.status, abort)) return;
      q = slot_q[s];
      if (q < 0) break;
    } else if (q >= n_items) {
      break;
    }
    Item it;
    decode_item<FMT>(p, rs, q, ks, it);
    const int ntl = (it.n + 7) >> 3;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

    for (int ck = 0; ck < it.nck; ++ck, ++iter) {
      const int s = iter % NSTAGE;
      if (!pipe_wait(&full[s], (iter / NSTAGE) & 1, p.status, abort)) return;
      const uint8_t* wst = smem + L::W_OFF + s * W_STAGE_BYTES;  // the two boxes, rows 0..63
      const uint8_t* wr0 = wst + rowA * BOX_BYTES;
      const uint8_t* wr1 = wst + rowB * BOX_BYTES;
      const uint8_t* sc = smem + L::SC_OFF + s * L::SC_BYTES;
      const uint8_t* act = smem + L::ACT_OFF + s * L::ACT_BYTES + g * ASTR;
      if constexpr (FMT == 4) {
        // this stage's 8 scale bytes of a row sit at byte (k0 / 32) & 8 of its 16-byte run
        constexpr int SC_ROW = FmtTraits<4>::SC_ROW;
        const int soff = ((it.k0 + ck * FmtTraits<4>::KC) / 32) & 8;
        uint32_t sa[HB / 4], sb[HB / 4];
#pragma unroll
        for (int j = 0; j < HB / 4; ++j) {
          sa[j] = lds32(sc + rowA * SC_ROW + soff + 4 * (kh * HB / 4 + j));
          sb[j] = lds32(sc + rowB * SC_ROW + soff + 4 * (kh * HB / 4 + j));
        }
        uint32_t wa[HB], wb[HB];
#pragma unroll
        for (int j = 0; j < HB; ++j) {  // all of this warp's weight words first
          wa[j] = lds32(wr0 + offs[j]);
          wb[j] = lds32(wr1 + offs[j]);
        }
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          const int b = kh * HB + j;
          uint32_t ha[4], hb[4];
          e2m1x8_to_f16x8(wa[j], ha);
          e2m1x8_to_f16x8(wb[j], hb);
          const uint32_t A0[4] = {ha[0], hb[0], ha[1], hb[1]};
          const uint32_t A1[4] = {ha[2], hb[2], ha[3], hb[3]};
          const float fa = e8m0_fast(sa[j / 4], j % 4), fb = e8m0_fast(sb[j / 4], j % 4);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (NT == 1 || t < ntl) {
              const uint4 bv = lds128(act + t * 8 * ASTR + (32 * b + 8 * c) * 2);
              float d[4];
              mma_f16(d, A0, bv.x, bv.y);
              mma_f16_acc(d, A1, bv.z, bv.w);
              acc[t][0] = fmaf(fa, d[0], acc[t][0]);
              acc[t][1] = fmaf(fa, d[1], acc[t][1]);
              acc[t][2] = fmaf(fb, d[2], acc[t][2]);
              acc[t][3] = fmaf(fb, d[3], acc[t][3]);
            }
          }
        }
      } else {
        const uint32_t sc4 = lds32(sc + (mt >> 1) * 4);
        uint32_t wa0[HB], wb0[HB], wa1[HB], wb1[HB];
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          wa0[j] = lds32(wr0 + offs[2 * j]);
          wb0[j] = lds32(wr1 + offs[2 * j]);
          wa1[j] = lds32(wr0 + offs[2 * j + 1]);
          wb1[j] = lds32(wr1 + offs[2 * j + 1]);
        }
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          const int b = kh * HB + j;
          uint32_t ha0[2], hb0[2], ha1[2], hb1[2];
          e4m3x4_to_f16x4(wa0[j], ha0);
          e4m3x4_to_f16x4(wb0[j], hb0);
          e4m3x4_to_f16x4(wa1[j], ha1);
          e4m3x4_to_f16x4(wb1[j], hb1);
          const uint32_t A0[4] = {ha0[0], hb0[0], ha0[1], hb0[1]};
          const uint32_t A1[4] = {ha1[0], hb1[0], ha1[1], hb1[1]};
          const uint32_t e = __byte_perm(sc4, 0u, 0x4440u + b);  // the same for the whole warp
          if (NT >= 4 && e - 112u <= 22u) {
            // scale 2^-15 .. 2^7: the scaled weights are exact in f16, so the MMAs accumulate
            // every block straight into the tile accumulators
            const uint32_t hs = e >= 113u ? (e - 112u) << 10 : 0x0200u;  // f16 2^(e-127)
            const uint32_t s2 = hs | (hs << 16);
            uint32_t A0s[4], A1s[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) A0s[q] = hmul2(A0[q], s2), A1s[q] = hmul2(A1[q], s2);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < ntl) {
                const uint2 b0 = lds64(act + t * 8 * ASTR + (32 * b + 4 * c) * 2);
                const uint2 b1 = lds64(act + t * 8 * ASTR + (32 * b + 16 + 4 * c) * 2);
                mma_f16_acc(acc[t], A0s, b0.x, b0.y);
                mma_f16_acc(acc[t], A1s, b1.x, b1.y);
              }
            }
          } else {
            const float sf = __uint_as_float(e << 23);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (NT == 1 || t < ntl) {
                const uint2 b0 = lds64(act + t * 8 * ASTR + (32 * b + 4 * c) * 2);
                const uint2 b1 = lds64(act + t * 8 * ASTR + (32 * b + 16 + 4 * c) * 2);
                float d[4];
                mma_f16(d, A0, b0.x, b0.y);
                mma_f16_acc(d, A1, b1.x, b1.y);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[t][jj] = fmaf(sf, d[jj], acc[t][jj]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (clustered) {
      write_partial<NT, L::EP_LD>(acc, ep_mine, mt, g, c, ntl);
      if (*abort) return;
      if (KS > 1) {
        consumer_bar<NTHR>();
        sum_kshares<KS, L::EP_LD, NTHR>(ep, ntl, tid);
      }
      fence_proxy_async_shared();  // the partial is read by bulk copies next
      consumer_bar<NTHR>();
      float* recv = ep + KS * L::EP_TILE;
      if (tid == 0) {
        // every owner must have emptied its receive tile of the previous K-split tile
        if (tiles_done > 0 && !pipe_wait<true>(red_done, (tiles_done - 1) & 1, p.status, abort))
          return;
        push_slices<L::EP_LD>(p, ep, recv, red_full, rank, it.n);
      }
      if (!pipe_wait(red_full, tiles_done & 1, p.status, abort)) return;
      owner_epilogue_any<L::EP_LD, NTHR>(p, it, recv, tid, rank);
      if (tid == 0) bulk_wait_read();  // this CTA's pushes have read its partial tile
      consumer_bar<NTHR>();
      // tile free -- announced only when another tile follows: the CTAs of a cluster take the
      // same tiles, so after the last one nobody pushes again, and no CTA then touches a peer's
      // shared memory (each has received all of its slots before its epilogue)
      if (q + (int)gridDim.x < n_items && tid < p.ksplit)
        mbar_arrive_remote(mapa_shared(smem_u32(red_done), tid));
    } else if constexpr (KS == 1 && FMT == 4) {
      if (*abort) return;
      epilogue_regs<NT>(p, it, acc, rowA, rowB, c, pair_gu);
    } else {
      const int m0 = 16 * mt + g;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (NT == 1 || t < ntl) {
          const int col = t * 8 + 2 * c;
          ep_mine[m0 * L::EP_LD + col] = acc[t][0];
          ep_mine[m0 * L::EP_LD + col + 1] = acc[t][1];
          ep_mine[(m0 + 8) * L::EP_LD + col] = acc[t][2];
          ep_mine[(m0 + 8) * L::EP_LD + col + 1] = acc[t][3];
        }
      }
      if (*abort) return;
      if (KS > 1) {  // the K shares' tiles, added in a fixed order
        consumer_bar<NTHR>();
        const int cols = ntl * 8;
        for (int idx = tid; idx < TILE_M * cols; idx += NTHR) {
          const int m = idx / cols, col = idx - m * cols;
          float v = ep[m * L::EP_LD + col];
#pragma unroll
          for (int k = 1; k < KS; ++k) v += ep[k * TILE_M * L::EP_LD + m * L::EP_LD + col];
          ep[m * L::EP_LD + col] = v;
        }
      }
      consumer_bar<NTHR>();
      epilogue_local<L::EP_LD, NTHR>(p, it, ep, tid);
      consumer_bar<NTHR>();  // the tile is written out before the next partial overwrites it
    }
    ++tiles_done;
  }
}

template <int FMT, int NT, int NSTAGE, int KS>
__global__ void __launch_bounds__(gemm_threads(KS), FMT == 4 && KS == 1 ? 4 : 2)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map,
                   const __grid_constant__ CUtensorMap smap, const GemmParams p) {
  using L = GemmLayout<FMT, NT, NSTAGE, KS>;
  constexpr int CONSUMER_WARPS = 4 * KS, THREADS = gemm_threads(KS);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + NSTAGE;
  uint64_t* red_full = empty + NSTAGE;
  uint64_t* red_done = red_full + 1;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  const bool clustered = p.ksplit > 1;  // a cluster launch (routed experts may still not split)
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1 + 32);  // expect_tx arrival + one cp.async arrival per lane
      mbar_init(&empty[s], CONSUMER_WARPS);
    }
    mbar_init(red_full, 1);  // the owner's expect_tx arrival; the peers' slices complete_tx
    mbar_init(red_done, clustered ? p.ksplit : 1);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == CONSUMER_WARPS && (threadIdx.x & 31) == 0) {
    prefetch_tmap(&map);
    if (FMT == 4 && p.sc_tma) prefetch_tmap(&smap);
  }
  // every CTA of a cluster must have initialised its barriers before any remote arrival
  if (clustered)
    cluster_sync_all();
  else
    __syncthreads();
  // (the routed experts let their dependents in only after their own wait: the top-k is then
  // complete, and the final combine reads the routing before its wait)
  if (!L::EXPERT) pdl_trigger();
  // weights do not depend on the previous kernel: start streaming them before waiting on it
  int pre = 0;
  if (warp == CONSUMER_WARPS) pre = prefetch_weights<FMT, NT, NSTAGE, KS>(p, &map, smem, full);
  pdl_wait();
  if (L::EXPERT) pdl_trigger();
  RouteSmem* rs = nullptr;
  if constexpr (L::EXPERT) {
    if (p.route) {
      rs = reinterpret_cast<RouteSmem*>(smem + L::ROUTE_OFF);
      // every global read of the routing issued in one round (all MAX_EXPERTS entries, those
      // past the hit count ignored), so that the copy costs one memory latency
      constexpr int HPT = (MAX_EXPERTS + THREADS - 1) / THREADS;
      constexpr int RPT = (MAX_SLOTS + THREADS - 1) / THREADS;
      const int nh_raw = p.route->n_hit;
      int he[HPT], ho[HPT], hc[HPT], g0[HPT], g1[HPT], rm[RPT];
#pragma unroll
      for (int k = 0; k < HPT; ++k) {
        const int i = threadIdx.x + k * THREADS;
        const bool in = i < MAX_EXPERTS;
        he[k] = in ? p.route->hit_e[i] : 0;
        ho[k] = in ? p.route->hit_off[i] : 0;
        hc[k] = in ? p.route->hit_cnt[i] : 0;
        g0[k] = in ? p.route->rg_prefix[i] : 0;
        g1[k] = in ? p.route->rg_prefix[i + 1] : 0;
      }
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        const int i = threadIdx.x + k * THREADS;
        rm[k] = p.act_rowmap && i < min(p.n_slots, MAX_SLOTS) ? p.act_rowmap[i] : 0;
      }
      const int nh = min(nh_raw, MAX_EXPERTS);
#pragma unroll
      for (int k = 0; k < HPT; ++k) {
        const int i = threadIdx.x + k * THREADS;
        if (i < nh) {
          rs->hit_e[i] = he[k];
          rs->hit_off[i] = ho[k];
          rs->hit_cnt[i] = hc[k];
          for (int g = g0[k]; g < min(g1[k], MAX_SLOTS); ++g) rs->rg_expert[g] = (uint8_t)i;
        }
        if (i <= nh && i < MAX_EXPERTS) rs->rg_prefix[i] = g0[k];
        if (i == MAX_EXPERTS - 1 && nh == MAX_EXPERTS) rs->rg_prefix[MAX_EXPERTS] = g1[k];
      }
      if (p.act_rowmap) {
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
          const int i = threadIdx.x + k * THREADS;
          if (i < min(p.n_slots, MAX_SLOTS)) rs->rowmap[i] = rm[k];
        }
      }
      if (threadIdx.x == 0) {
        rs->n_hit = nh;
        rs->tile_shift = (p.n_tiles & (p.n_tiles - 1)) == 0 ? __ffs(p.n_tiles) - 1 : -1;
      }
      __syncthreads();
    }
  }
  if (warp == CONSUMER_WARPS)
    gemm_producer<FMT, NT, NSTAGE, KS>(p, rs, &map, &smap, smem, full, empty, abort, pre);
  else
    gemm_consumer<FMT, NT, NSTAGE, KS>(p, rs, smem, full, empty, red_full, red_done, abort);
}

}  // namespace mono
