// Routed-expert GEMMs of large steps on the 5th-generation tensor cores ("Mono decode layer
// for DeepSeek-V4.1-Flash on MI355X", launch table K2: "MXFP4 experts"; section Design: MXFP4
// routed experts with 1x32 E8M0 scales, read in place).
//
// tcgen05.mma kind::mxf4 (block-scaled, scale_vec::2X) multiplies the expert's e2m1 weights,
// TMA-loaded as stored (packed, 128-byte swizzle) with their E8M0 scales, by the routed rows'
// activations.  An activation row enters as the ACT_TERMS e2m1 terms of its split (see
// split_terms_x8 in common.cuh): row j of the item is MMA columns 8j .. 8j + 7, one per term,
// and the epilogue adds a row's eight accumulator columns in term order.  One M = 128, K = 64
// MMA covers 4 KB of packed weights whatever N (<= 64), so the weight stream, not the tensor
// core, sets the pace.
//
// Two CTAs per SM, six warps each: warp 0 loads (TMA for the weight tiles and their scale
// boxes, bulk copies for the term rows and term scales); warp 1 turns each stage's scales
// into the TMEM scale images (all lanes) and issues the copies and MMAs (one elected lane)
// into a double-buffered TMEM accumulator; warps 2-5 (one per TMEM lane quadrant) run the
// epilogue.  (A CTA's stage costs some 900 cycles of issue and bookkeeping across its two
// pipeline warps, so one pipeline per SM falls short of the SM's share of HBM bandwidth; two
// reach it.)  Items are (hit expert, group of up to 8 routed rows, weight tile), handed out
// by a per-launch counter, largest groups first (the order the top-k publishes).
// gate_up tiles are 64 gate rows with the 64 up rows they pair with; the epilogue forms
// SwiGLU and writes t (f16) and t's term split for the down GEMM.  Every wait is bounded.
#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"

namespace mono {
namespace {

using namespace tc;

constexpr int TC_M = 128;                    // weight rows per tile (the MMA's M)
constexpr int TC_KC = 256;                   // K elements per stage (128 packed bytes a row)
constexpr int TC_ROWS = 8;                   // routed rows per item
constexpr int TC_NMAX = TC_ROWS * ACT_TERMS; // MMA columns at most
constexpr int TC_THREADS = 192;
constexpr int TC_CTAS_PER_SM = 2;           // two pipelines per SM (shared memory, TMEM halves)
constexpr int TERM_ROW = 128;                // bytes of one term row per stage
constexpr int TERM_SC = ACT_TERMS * 8;       // term-scale bytes of one routed row per stage
constexpr int A_BYTES = TC_M * 128;
constexpr int B_BYTES = TC_NMAX * TERM_ROW;
constexpr int SA_BYTES = TC_M * 16;          // weight scale boxes: 16 bytes a row
constexpr int SB_BYTES = TC_ROWS * TERM_SC;
constexpr int IMG = 512;                     // one TMEM scale image: 32 lanes x 16 bytes
constexpr int A_OFF = 0, B_OFF = A_BYTES, SA_OFF = B_OFF + B_BYTES, SB_OFF = SA_OFF + SA_BYTES;
constexpr int IMG_OFF = SB_OFF + SB_BYTES;   // A word 0, A word 1, B word 0, B word 1
constexpr int STAGE = (IMG_OFF + 4 * IMG + 1023) / 1024 * 1024;
constexpr int NSTAGE = 3;
constexpr int XCH_OFF = NSTAGE * STAGE;      // gate_up: the up rows' values for the gate warps,
constexpr int XCH_BYTES = 2 * 64 * TC_ROWS * 4;  // one buffer per accumulator
constexpr int SMEM_BYTES = XCH_OFF + XCH_BYTES + 1024;  // + alignment slack
static_assert(STAGE % 1024 == 0, "stage buffers stay 1024-aligned for the 128-byte swizzle");
// TMEM: two accumulators of TC_NMAX columns, then 16 scale columns per ring stage
constexpr int SC_COL = 2 * TC_NMAX;
constexpr int TMEM_COLS = 256;
static_assert(SC_COL + 16 * NSTAGE <= TMEM_COLS, "TMEM columns");
static_assert(TMEM_COLS * TC_CTAS_PER_SM <= 512, "the co-resident CTAs' TMEM fits the SM's");
constexpr int MAX_GROUPS = MAX_SLOTS;        // row groups at most (<= routed slots)

// Items of a launch: hit expert d owns row groups [gpre[d], gpre[d + 1]) (ceil(rows / 16)
// each) and items [gpre[d] * n_tiles, gpre[d + 1] * n_tiles), tile fastest.
struct TcRoute {
  int n_hit;
  int e[MAX_EXPERTS], off[MAX_EXPERTS], cnt[MAX_EXPERTS];
  int gpre[MAX_EXPERTS + 1];
  uint8_t gexp[MAX_GROUPS];  // hit expert of each row group
  int rowmap[MAX_SLOTS];     // gate_up: sorted slot -> activation row
};
static_assert(MAX_EXPERTS <= 256, "gexp holds hit-expert indices in a byte");

struct TcItem {
  int e, tile, slot0, n;  // expert, weight tile, first sorted slot, routed rows (1 .. 16)
};
__device__ __forceinline__ TcItem tc_item(const TcRoute& rt, int n_tiles, int q) {
  const int g = q / n_tiles;
  const int d = rt.gexp[g];
  const int lg = g - rt.gpre[d];
  TcItem it;
  it.e = rt.e[d];
  it.tile = q - g * n_tiles;
  it.slot0 = rt.off[d] + lg * TC_ROWS;
  it.n = min(TC_ROWS, rt.cnt[d] - lg * TC_ROWS);
  return it;
}

// ---------------------------------------------------------------- shared-expert down items
// The down launch also runs the shared expert's down GEMM (MXFP8, e4m3 weights with 32 x 32
// E8M0 scales): items (128-row tile of H, a half of at most SH_ROWS activation rows), ahead
// of the routed items.  Their MMAs are kind::mxf8f6f4 (scale_vec::1X); the activations are
// t_s's e4m3 hi/lo split as the shared gate_up wrote it (common.cuh), a stage's B tile being
// the half's hi rows at rows [0, SH_ROWS) and its lo rows at [SH_ROWS, 2 SH_ROWS).
constexpr int SH_ROWS = 24;
static_assert(2 * SH_ROWS <= TC_NMAX && 2 * SH_ROWS * TERM_ROW <= B_BYTES, "a half's B tile");
static_assert(SPLIT_IMG_BYTES <= SB_BYTES && 4 * 16 <= SA_BYTES, "a half's scales");

struct ShItem {
  int tile, i0, nh;  // output tile, first activation row, rows (1 .. SH_ROWS)
};
__device__ __forceinline__ ShItem sh_item(const ExpertTcParams& p, int q) {
  ShItem it;
  it.tile = q / p.sh_halves;
  it.i0 = (q - it.tile * p.sh_halves) * SH_ROWS;
  it.nh = min(SH_ROWS, p.sh_rows - it.i0);
  return it;
}
// Producer: one stage of a shared item (elected lane).
__device__ __forceinline__ void sh_issue(const ExpertTcParams& p, const CUtensorMap* shmap,
                                         const ShItem& it, int c, uint8_t* st, uint64_t* full) {
  mbar_arrive_expect_tx(full, A_BYTES + 2 * it.nh * TERM_ROW + SPLIT_IMG_BYTES + 4 * 16);
  tma_load_2d(st + A_OFF, shmap, c * 128, it.tile * TC_M, full);
  // the tile's four 32-row scale blocks: the 16-byte runs holding this stage's 4 K blocks
#pragma unroll
  for (int g = 0; g < 4; ++g)
    bulk_load_g2s(st + SA_OFF + 16 * g,
                  p.sh_scales + (size_t)(it.tile * 4 + g) * p.sh_scale_ld + ((c * 4) & ~15), 16,
                  full);
  const uint8_t* src = p.sh_bsplit + (size_t)c * SPLIT_STAGE_BYTES;
  bulk_load_g2s(st + B_OFF, src + it.i0 * TERM_ROW, it.nh * TERM_ROW, full);
  bulk_load_g2s(st + B_OFF + SH_ROWS * TERM_ROW, src + (SPLIT_LO + it.i0) * TERM_ROW,
                it.nh * TERM_ROW, full);
  bulk_load_g2s(st + SB_OFF, p.sh_bimg + (size_t)c * SPLIT_IMG_BYTES, SPLIT_IMG_BYTES, full);
}
// MMA warp: one stage of a shared item -- the scale images (every lane), then the copies and
// MMAs (the elected lane).  A image: the tile's row block g's 4 scale bytes in column g of
// every lane; B image: MMA column n (hi row i0 + n, or lo row i0 + n - SH_ROWS) at lane n % 32,
// column n / 32, taken from the split's image (hi column j's word).
__device__ __forceinline__ void sh_mma(const ExpertTcParams& p, const ShItem& it, int c,
                                       uint8_t* st, uint32_t d0, uint32_t sc, int lane,
                                       bool first) {
  uint32_t wa[4], wb[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    wa[g] = *reinterpret_cast<const uint32_t*>(st + SA_OFF + 16 * g + ((c * 4) & 15));
    const int n = lane + 32 * g;
    const int j = it.i0 + (n < SH_ROWS ? n : n - SH_ROWS);
    wb[g] = n < 2 * SH_ROWS && j < p.sh_rows
                ? *reinterpret_cast<const uint32_t*>(st + SB_OFF + (j & 31) * 16 + (j >> 5) * 4)
                : 0x7F7F7F7Fu;
  }
  *reinterpret_cast<uint4*>(st + IMG_OFF + lane * 16) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
  *reinterpret_cast<uint4*>(st + IMG_OFF + 2 * IMG + lane * 16) =
      make_uint4(wb[0], wb[1], wb[2], wb[3]);
  fence_proxy_async_shared();
  __syncwarp();
  const uint32_t a0 = smem_u32(st + A_OFF), b0 = smem_u32(st + B_OFF);
  // kind::mxf8f6f4, A and B e4m3, E8M0 scales, M = 128, N = 2 SH_ROWS
  const uint32_t idesc = (1u << 23) | ((uint32_t)((2 * SH_ROWS) >> 3) << 17) |
                         ((uint32_t)(TC_M >> 4) << 24);
  if (elect_one()) {
    tc_fence_after();
    tc_cp_img(sc, st + IMG_OFF);
    tc_cp_img(sc + 8, st + IMG_OFF + 2 * IMG);
#pragma unroll
    for (int k = 0; k < 4; ++k)  // K = 32 each; scale byte k of the stage's words
      tc_mma_mxf8(d0, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k),
                  idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), sc, sc + 8,
                  (!first || k > 0) ? 1u : 0u);
  }
}
// Epilogue warp (TMEM lane quadrant quad) of a shared item: y_s rows i0 .. i0 + nh of its 32
// output columns, each the sum of the hi and lo accumulator columns.
__device__ __forceinline__ void sh_epilogue(const ExpertTcParams& p, const ShItem& it,
                                            uint32_t taddr, int quad, int lane) {
  uint32_t r0[32], r1[32];
  tc_ld32(taddr, r0);
  tc_ld32(taddr + 32, r1);
  tc_wait_ld();
  const int col = it.tile * TC_M + quad * 32 + lane;
#pragma unroll
  for (int j = 0; j < SH_ROWS; ++j) {
    const int n = SH_ROWS + j;
    const float v = __uint_as_float(r0[j]) + __uint_as_float(n < 32 ? r0[n & 31] : r1[n & 31]);
    if (j < it.nh) p.ys[(size_t)(it.i0 + j) * p.rows_per_mat + col] = v;
  }
}

// The setup of every CTA: the step's routing (written by the top-k kernel) into rt -- the hit
// experts in the order the items are handed out (decreasing row count) with the prefix of
// their row groups, and gate_up's row map -- checked, and the producer's first work item
// (thread 0's return value).  Every global read is issued in one round: the first work item,
// the hit count, all MAX_EXPERTS entries of the ordered hit arrays (those past the count are
// ignored) and the row map.  An entry that fails its check raises the status bit and leaves
// this CTA without routed items.
template <bool GU>
__device__ __forceinline__ int tc_setup(const ExpertTcParams& p, TcRoute& rt, int* s_bad) {
  const int tid = threadIdx.x;
  constexpr int HPT = (MAX_EXPERTS + TC_THREADS - 1) / TC_THREADS;  // hit entries per thread
  constexpr int RPT = (MAX_SLOTS + TC_THREADS - 1) / TC_THREADS;    // row-map entries per thread
  static_assert(TC_ROWS == EXPERT_ROWS, "the top-k's row groups are the items' row groups");
  if (tid == 0) *s_bad = 0;
  int q_first = 0;
  if (tid == 0) q_first = atomicAdd(p.item_next, 1);
  int n_hit = p.route->n_hit;
  int he[HPT], ho[HPT], hc[HPT], g0[HPT], g1[HPT], rm[RPT];
#pragma unroll
  for (int k = 0; k < HPT; ++k) {
    const int d = tid + k * TC_THREADS;
    const bool in = d < MAX_EXPERTS;
    he[k] = in ? p.route->lpt_e[d] : 0;
    ho[k] = in ? p.route->lpt_off[d] : 0;
    hc[k] = in ? p.route->lpt_cnt[d] : 0;
    g0[k] = in ? p.route->lpt_gpre[d] : 0;
    g1[k] = in ? p.route->lpt_gpre[d + 1] : 0;
  }
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int i = tid + k * TC_THREADS;
    rm[k] = GU && i < p.n_slots ? p.rowmap[i] : 0;
  }
  bool bad = n_hit < 0 || n_hit > MAX_EXPERTS;
  if (bad) n_hit = 0;
  __syncthreads();  // (s_bad cleared)
#pragma unroll
  for (int k = 0; k < HPT; ++k) {
    const int d = tid + k * TC_THREADS;
    if (d < n_hit) {
      const int e = he[k], off = ho[k], cnt = hc[k];
      bad |= e < 0 || e >= p.n_experts || cnt < 1 || off < 0 || off + cnt > p.n_slots ||
             g0[k] < 0 || g1[k] - g0[k] != (cnt + TC_ROWS - 1) / TC_ROWS || g1[k] > MAX_GROUPS;
      rt.e[d] = e, rt.off[d] = off, rt.cnt[d] = cnt, rt.gpre[d] = g0[k];
      if (d == n_hit - 1) rt.gpre[n_hit] = g1[k];
    }
  }
  if (GU) {
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int i = tid + k * TC_THREADS;
      if (i < p.n_slots) {
        bad |= rm[k] < 0 || rm[k] >= p.act_rows;
        rt.rowmap[i] = rm[k];
      }
    }
  }
  if (bad) *s_bad = 1;
  __syncthreads();
  if (*s_bad) {
    if (tid == 0) atomicOr(p.status, ST_BAD_ROUTE);
    n_hit = 0;
  }
  if (tid == 0) {
    rt.n_hit = n_hit;
    if (n_hit == 0) rt.gpre[0] = 0;
  }
  for (int d = tid; d < n_hit; d += TC_THREADS)
    for (int g = rt.gpre[d]; g < rt.gpre[d + 1]; ++g) rt.gexp[g] = (uint8_t)d;
  __syncthreads();
  return q_first;
}

template <bool GU>
__global__ void __launch_bounds__(TC_THREADS, TC_CTAS_PER_SM)
    expert_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                     const __grid_constant__ CUtensorMap smap,
                     const __grid_constant__ CUtensorMap shmap,
                     const __grid_constant__ ExpertTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[NSTAGE], empty[NSTAGE], tfull[2], tempty[2], drain;
  __shared__ __align__(8) uint64_t xfull[2], xempty[2];  // gate_up: the up-value exchange
  __shared__ TcRoute rt;
  __shared__ int s_bad;
  __shared__ int slot_q[NSTAGE], acc_q[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nck = p.K / TC_KC;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);   // the producer's expect_tx arrival; the copies complete_tx
      mbar_init(&empty[s], 1);  // the MMA thread's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 2);   // the item index published, then the MMAs' commit
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
      mbar_init(&xfull[b], 64);  // every lane of the two up-row warps
      mbar_init(&xempty[b], 64); // every lane of the two gate-row warps
    }
    mbar_init(&drain, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&wmap);
    prefetch_tmap(&smap);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "n"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  // Dependents are let in only now: everything the top-k wrote is complete, so the final
  // combine may read the routing (and anything older) before its own wait.
  pdl_trigger();
  const int q_first = tc_setup<GU>(p, rt, &s_bad);
  const int n_hit = rt.n_hit;
  // the shared expert's down items come first (each streams p.sh_nck stages, more than a
  // routed item's), then the routed items
  const int n_sh = GU ? 0 : p.sh_tiles * p.sh_halves;
  const int n_items = n_sh + min(rt.gpre[n_hit], MAX_GROUPS) * p.n_tiles;

  if (warp == 0) {
    // ---------------------------------------------------------------------------- producer
    int iter = 0;
    int q = __shfl_sync(0xffffffffu, q_first, 0);  // (thread 0's, fetched with the routing)
    while (q < n_items) {
      int qn = 0;  // the next item, fetched once this one's first stage is on its way
      if (!GU && q < n_sh) {
        const ShItem si = sh_item(p, q);
        for (int c = 0; c < p.sh_nck; ++c, ++iter) {
          const int s = iter % NSTAGE;
          if (!warp_wait(&empty[s], ((iter / NSTAGE) & 1) ^ 1, p.status, abort))
            goto producer_done;
          if (elect_one()) {
            if (c == 0) slot_q[s] = q;  // published by the arrival in sh_issue
            sh_issue(p, &shmap, si, c, smem + s * STAGE, &full[s]);
          }
          if (c == 0 && lane == 0) qn = atomicAdd(p.item_next, 1);
          __syncwarp();
        }
        q = __shfl_sync(0xffffffffu, qn, 0);
        continue;
      }
      const TcItem it = tc_item(rt, p.n_tiles, q - n_sh);
      int arow = 0;
      if (GU && lane < it.n) arow = rt.rowmap[it.slot0 + lane];
      const uint32_t tx = A_BYTES + SA_BYTES + it.n * (ACT_TERMS * TERM_ROW + TERM_SC);
      for (int c = 0; c < nck; ++c, ++iter) {
        const int s = iter % NSTAGE;
        if (!warp_wait(&empty[s], ((iter / NSTAGE) & 1) ^ 1, p.status, abort)) goto producer_done;
        uint8_t* st = smem + s * STAGE;
        if (elect_one()) {
          if (c == 0) slot_q[s] = q;  // published by the arrival below
          mbar_arrive_expect_tx(&full[s], tx);
          if constexpr (GU) {  // the tile's 64 gate rows, then the 64 up rows I further
            tma_load_4d(st + A_OFF, &wmap, c * 128, it.tile * 64, 0, it.e, &full[s]);
            tma_load_4d(st + SA_OFF, &smap, (c * 8) & ~15, it.tile * 64, 0, it.e, &full[s]);
          } else {
            const int row = it.e * p.rows_per_mat + it.tile * TC_M;
            tma_load_2d(st + A_OFF, &wmap, c * 128, row, &full[s]);
            tma_load_2d(st + SA_OFF, &smap, (c * 8) & ~15, row, &full[s]);
            // the item's slots are consecutive: their term rows and scales, one copy each
            const size_t rc = (size_t)c * p.n_slots + it.slot0;
            bulk_load_g2s(st + B_OFF, p.bterms + rc * (ACT_TERMS * TERM_ROW),
                          it.n * (ACT_TERMS * TERM_ROW), &full[s]);
            bulk_load_g2s(st + SB_OFF, p.bscales + rc * TERM_SC, it.n * TERM_SC, &full[s]);
          }
        }
        __syncwarp();
        if (GU && lane < it.n) {  // gathered rows of u: one pair of copies per row
          const size_t rc = (size_t)arow * nck + c;
          bulk_load_g2s(st + B_OFF + lane * (ACT_TERMS * TERM_ROW),
                        p.bterms + rc * (ACT_TERMS * TERM_ROW), ACT_TERMS * TERM_ROW, &full[s]);
          bulk_load_g2s(st + SB_OFF + lane * TERM_SC, p.bscales + rc * TERM_SC, TERM_SC, &full[s]);
        }
        if (c == 0 && lane == 0) qn = atomicAdd(p.item_next, 1);
      }
      q = __shfl_sync(0xffffffffu, qn, 0);
    }
    {  // the end: one more stage phase that carries no data, only the end mark
      const int s = iter % NSTAGE;
      if (!warp_wait(&empty[s], ((iter / NSTAGE) & 1) ^ 1, p.status, abort)) goto producer_done;
      if (lane == 0) {
        slot_q[s] = -1;
        mbar_arrive(&full[s]);
      }
    }
  producer_done:
    if (lane == 0 && *abort) {  // let the copies already issued land before the CTA exits
      for (int k = max(0, iter - NSTAGE); k < iter; ++k)
        mbar_wait(&full[k % NSTAGE], (k / NSTAGE) & 1, p.status, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale images + MMA issue
    int iter = 0;
    for (int li = 0;; ++li) {
      const int b = li & 1;
      int s = iter % NSTAGE;
      if (!warp_wait(&full[s], (iter / NSTAGE) & 1, p.status, abort)) break;
      const int q = slot_q[s];
      if (!warp_wait(&tempty[b], ((li >> 1) & 1) ^ 1, p.status, abort)) break;
      if (lane == 0) {
        acc_q[b] = q;
        mbar_arrive(&tfull[b]);  // publishes the item index (release)
      }
      if (q < 0) {
        if (elect_one()) tc_commit(&tfull[b]);  // (the issuing thread's commits)
        break;
      }
      const uint32_t d0 = tmem + b * TC_NMAX;
      if (!GU && q < n_sh) {
        const ShItem si = sh_item(p, q);
        bool sok = true;
        for (int c = 0; c < p.sh_nck; ++c, ++iter) {
          s = iter % NSTAGE;
          if (c > 0 && !warp_wait(&full[s], (iter / NSTAGE) & 1, p.status, abort)) {
            sok = false;
            break;
          }
          sh_mma(p, si, c, smem + s * STAGE, d0, tmem + SC_COL + s * 16, lane, c == 0);
          if (elect_one()) tc_commit(&empty[s]);
          __syncwarp();
        }
        if (!sok) break;
        if (elect_one()) tc_commit(&tfull[b]);
        continue;
      }
      const TcItem it = tc_item(rt, p.n_tiles, q - n_sh);
      const int ncol = (it.n * ACT_TERMS + 15) & ~15;
      const uint32_t idesc_base = (1u << 7) | (1u << 10) | ((uint32_t)(ncol >> 3) << 17) |
                                  (1u << 23) | ((uint32_t)(TC_M >> 4) << 24);
      bool ok = true;
      for (int c = 0; c < nck; ++c, ++iter) {
        s = iter % NSTAGE;
        if (c > 0 && !warp_wait(&full[s], (iter / NSTAGE) & 1, p.status, abort)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * STAGE;
        // scale images.  A word w: lane l, column g = weight row l + 32 g's K-block scales
        // 4w .. 4w + 3 of this stage, bytes (8c & 8) + 4w .. of the row's 16-byte box row.
        // B word w: lane l, column g = MMA column n = l + 32 g, routed row n / 8's term n % 8.
        {
          const bool hi = (c & 1) != 0;  // the stage's scales are the box row's second half
          uint32_t w0[4], w1[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 r = *reinterpret_cast<const uint4*>(st + SA_OFF + (lane + 32 * g) * 16);
            w0[g] = hi ? r.z : r.x;
            w1[g] = hi ? r.w : r.y;
          }
          *reinterpret_cast<uint4*>(st + IMG_OFF + lane * 16) =
              make_uint4(w0[0], w0[1], w0[2], w0[3]);
          *reinterpret_cast<uint4*>(st + IMG_OFF + IMG + lane * 16) =
              make_uint4(w1[0], w1[1], w1[2], w1[3]);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int n = lane + 32 * g;
            uint2 v = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);  // unused columns: scale 1
            if (n < it.n * ACT_TERMS)
              v = *reinterpret_cast<const uint2*>(st + SB_OFF + (n >> 3) * TERM_SC + (n & 7) * 8);
            w0[g] = v.x;
            w1[g] = v.y;
          }
          *reinterpret_cast<uint4*>(st + IMG_OFF + 2 * IMG + lane * 16) =
              make_uint4(w0[0], w0[1], w0[2], w0[3]);
          *reinterpret_cast<uint4*>(st + IMG_OFF + 3 * IMG + lane * 16) =
              make_uint4(w1[0], w1[1], w1[2], w1[3]);
        }
        fence_proxy_async_shared();  // the images, before the tensor core's copies read them
        __syncwarp();
        const uint32_t sc = tmem + SC_COL + s * 16;
        const uint32_t a0 = smem_u32(st + A_OFF), b0 = smem_u32(st + B_OFF);
        if (elect_one()) {
          tc_fence_after();
          tc_cp_img(sc, st + IMG_OFF);
          tc_cp_img(sc + 4, st + IMG_OFF + IMG);
          tc_cp_img(sc + 8, st + IMG_OFF + 2 * IMG);
          tc_cp_img(sc + 12, st + IMG_OFF + 3 * IMG);
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // K = 64 each; scale bytes 2j % 4 of word j / 2
            const uint32_t sf = 2u * (j & 1);
            tc_mma_mxf4(d0, desc_sw128(a0 + 32 * j), desc_sw128(b0 + 32 * j),
                        idesc_base | (sf << 4) | (sf << 29), sc + 4 * (j >> 1),
                        sc + 8 + 4 * (j >> 1), (c > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tfull[b]);
    }
    // every MMA issued has completed before the accumulators and TMEM are released
    if (elect_one()) {
      tc_commit(&drain);
      mbar_wait(&drain, 0, p.status, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // the TMEM lane quadrant this warp may read: tile rows 32 quad ..
    for (int li = 0;; ++li) {
      const int b = li & 1;
      const uint32_t ph = (li >> 1) & 1;
      float* xch = reinterpret_cast<float*>(smem + XCH_OFF) + b * 64 * TC_ROWS;  // [64][16]
      if (!warp_wait(&tfull[b], ph, p.status, abort)) break;
      tc_fence_after();
      const int q = acc_q[b];
      if (q < 0) break;
      if (!GU && q < n_sh) {
        sh_epilogue(p, sh_item(p, q), tmem + ((uint32_t)(quad * 32) << 16) + b * TC_NMAX, quad,
                    lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        continue;
      }
      const TcItem it = tc_item(rt, p.n_tiles, q - n_sh);
      // this lane's weight row's value for each routed row: the sum of its eight term columns
      float y[TC_ROWS];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + b * TC_NMAX;
#pragma unroll
      for (int c4 = 0; c4 < TC_NMAX / 32; ++c4) {
        if (c4 * 4 < it.n) {  // 32 columns = 4 routed rows
          uint32_t r[32];
          tc_ld32(taddr + c4 * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float v = 0.0f;
#pragma unroll
            for (int t = 0; t < ACT_TERMS; ++t) v += __uint_as_float(r[jj * 8 + t]);
            y[c4 * 4 + jj] = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
      if constexpr (GU) {
        // up rows (quadrants 2, 3) hand their values to the gate rows (quadrants 0, 1)
        if (quad >= 2) {
          if (!warp_wait(&xempty[b], ph ^ 1, p.status, abort)) break;
#pragma unroll
          for (int j = 0; j < TC_ROWS; ++j)
            if (j < it.n) xch[((quad - 2) * 32 + lane) * TC_ROWS + j] = y[j];
          mbar_arrive(&xfull[b]);
        } else {
          if (!warp_wait(&xfull[b], ph, p.status, abort)) break;
          const int col = it.tile * 64 + quad * 32 + lane;  // t's column (down's K index)
          const int kc = col / TC_KC, piece = (col % TC_KC) / 32;
#pragma unroll 1
          for (int j = 0; j < TC_ROWS; ++j) {
            if (j >= it.n) break;
            const size_t slot = (size_t)it.slot0 + j;
            const float t = round_bf16(
                swiglu_clamped(y[j], xch[(quad * 32 + lane) * TC_ROWS + j], p.clamp));
            p.t16[slot * p.I + col] = bf16_as_f16_sat(t, p.status);
            uint32_t words[ACT_TERMS], codes[ACT_TERMS];
            split_terms_lane(t, words, codes);
            const size_t base = ((size_t)kc * p.n_slots + slot) * ACT_TERMS;
#pragma unroll
            for (int tt = 0; tt < ACT_TERMS; ++tt) {
              if ((lane & 7) == 0)
                *reinterpret_cast<uint32_t*>(p.tterms + (base + tt) * TERM_ROW +
                                             ((piece ^ tt) << 4) + (lane >> 3) * 4) = words[tt];
              if (lane == 0) p.tscales[(base + tt) * 8 + piece] = (uint8_t)codes[tt];
            }
          }
          mbar_arrive(&xempty[b]);  // (the up values are read before the lanes arrive)
        }
      } else {
        const int col = it.tile * TC_M + quad * 32 + lane;
#pragma unroll
        for (int j = 0; j < TC_ROWS; ++j)
          if (j < it.n) p.y[((size_t)it.slot0 + j) * p.rows_per_mat + col] = y[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

cudaError_t expert_tc_prepare(int* ctas_per_sm) {
  // the largest shared-memory carveout, so that TC_CTAS_PER_SM rings fit on an SM
  cudaError_t e = cudaSuccess;
  for (const void* k : {reinterpret_cast<const void*>(expert_tc_kernel<true>),
                        reinterpret_cast<const void*>(expert_tc_kernel<false>)}) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  }
  // co-resident CTAs, from the kernel's registers and shared memory and the SM's totals (the
  // runtime's occupancy query answers 1 for this kernel; two CTAs do share an SM, which the
  // launch's time shows); never more than TC_CTAS_PER_SM, whose TMEM shares fill the SM's
  int n = 0;
  if (e == cudaSuccess) {
    int dev = 0;
    cudaDeviceProp pr;
    cudaFuncAttributes fa[2];
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaGetDeviceProperties(&pr, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa[0], expert_tc_kernel<true>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa[1], expert_tc_kernel<false>);
    if (e == cudaSuccess) {
      n = TC_CTAS_PER_SM;
      for (const cudaFuncAttributes& a : fa) {
        const size_t smem = SMEM_BYTES + a.sharedSizeBytes + pr.reservedSharedMemPerBlock;
        const int regs = ((a.numRegs * 32 + 255) / 256 * 256) * (TC_THREADS / 32);
        n = std::min(n, (int)std::min<size_t>(pr.sharedMemPerMultiprocessor / smem,
                                               (size_t)(pr.regsPerMultiprocessor / regs)));
      }
    }
  }
  *ctas_per_sm = n;
  return e;
}

cudaError_t launch_expert_tc(const Launch& L, bool gate_up, const CUtensorMap& wmap,
                             const CUtensorMap& smap, const CUtensorMap& shmap,
                             const ExpertTcParams& p, int grid) {
  if (p.K % TC_KC || (gate_up && (p.I % 64 || p.I % TC_KC)) || (!gate_up && p.rows_per_mat % TC_M) ||
      !p.item_next || !p.route || p.n_slots > MAX_SLOTS)
    return cudaErrorInvalidValue;
  if (!gate_up && p.sh_tiles > 0 &&
      (p.sh_rows < 1 || p.sh_halves != (p.sh_rows + SH_ROWS - 1) / SH_ROWS || p.sh_nck < 1 ||
       !p.sh_scales || !p.sh_bsplit || !p.sh_bimg || !p.ys || p.sh_scale_ld % 16 ||
       p.sh_nck * 4 > p.sh_scale_ld))
    return cudaErrorInvalidValue;
  if (gate_up)
    return launch_ex(L, dim3(grid), dim3(TC_THREADS), SMEM_BYTES, expert_tc_kernel<true>, wmap,
                     smap, shmap, p);
  return launch_ex(L, dim3(grid), dim3(TC_THREADS), SMEM_BYTES, expert_tc_kernel<false>, wmap,
                   smap, shmap, p);
}

}  // namespace mono
