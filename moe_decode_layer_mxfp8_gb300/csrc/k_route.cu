// Router and expert grouping ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", launch
// table K2: "router, top-6"; ATOM changes: "f32 router logits").
//
// router_kernel: z[r, e] = u[r] . W_r[e] in f32, split over K: CTA (8 experts x 2 warps,
// 1024-wide K slice, 16 rows) holds its experts' weight slices in registers (fetched before
// waiting on the previous kernel), stages the slice of its rows of u in shared memory and
// writes one partial per (slice, row, expert).  Rows go eight at a time: eight independent FMA chains
// per lane, then one transposing butterfly that leaves each of eight lanes with one row's
// sum.
//
// topk_kernel sums the partials in slice order (a fixed order, so results replay
// bit-exactly) into shared memory, picks the top-k per row (a group of 8 or 16 lanes per
// row: the largest (logit, lowest index) by a butterfly max per round) and sorts the
// (row, slot) pairs by expert, stably, for the grouped expert GEMMs: a row picks an expert
// at most once, so an entry's place among its expert's entries is the number of earlier
// rows in that expert's row mask.
#include "kernels.h"

namespace mono {

namespace {

constexpr int RT_EXPERTS = 8;    // experts per CTA
constexpr int RT_HALVES = 2;     // warps per expert, taking alternate groups of 8 rows
constexpr int RT_THREADS = RT_EXPERTS * RT_HALVES * 32;
constexpr int RT_J = ROUTER_KSLICE / 128;  // float4 weight chunks per lane
constexpr int RT_ROWS = 8 * RT_HALVES;     // rows per CTA (grid z = row groups)
constexpr int MAX_ROWS = 48, MAX_K = 8;

__global__ void __launch_bounds__(RT_THREADS) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t rt_smem[];
  __half* us = reinterpret_cast<__half*>(rt_smem);  // [rows][ROUTER_KSLICE]
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.y * ROUTER_KSLICE;
  const int klen = min(ROUTER_KSLICE, a.H - k0);
  // this lane's weights (k = k0 + 128 j + 4 lane + {0..3}): constant, so fetched first
  const int e = blockIdx.x * RT_EXPERTS + (warp % RT_EXPERTS);
  const int half = warp / RT_EXPERTS;
  float4 wv[RT_J];
#pragma unroll
  for (int j = 0; j < RT_J; ++j)
    wv[j] = e < a.E && 128 * j < klen
                ? *reinterpret_cast<const float4*>(a.wr + (size_t)e * a.H + k0 + 128 * j + 4 * lane)
                : make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_wait();
  // this CTA's rows [row0, row0 + nrows)
  const int row0 = blockIdx.z * RT_ROWS;
  const int nrows = min(RT_ROWS, a.rows - row0);
  const int chunks = klen / 8;  // 16-byte chunks per row
  for (int idx = tid; idx < nrows * chunks; idx += RT_THREADS) {
    const int r = idx / chunks, c = idx - r * chunks;
    cp_async16(us + r * ROUTER_KSLICE + c * 8, a.u + (size_t)(row0 + r) * a.H + k0 + c * 8, 16);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (e >= a.E) return;
  // lane l ends a group of eight rows with the sum of row 4 bit4(l) + 2 bit3(l) + bit2(l)
  const int my_row = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
  for (int r0 = 8 * half; r0 < nrows; r0 += 8 * RT_HALVES) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const int nr = min(8, nrows - r0);
#pragma unroll
    for (int j = 0; j < RT_J; ++j) {
      if (128 * j < klen) {
        // the eight rows' values of this chunk first, then eight independent FMA chains
        uint2 uv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          uv[i] = i < nr ? *reinterpret_cast<const uint2*>(us + (r0 + i) * ROUTER_KSLICE + 128 * j + 4 * lane)
                         : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&uv[i].x));
          const float2 u1 = __half22float2(*reinterpret_cast<const __half2*>(&uv[i].y));
          acc[i] = fmaf(u0.x, wv[j].x, acc[i]);
          acc[i] = fmaf(u0.y, wv[j].y, acc[i]);
          acc[i] = fmaf(u1.x, wv[j].z, acc[i]);
          acc[i] = fmaf(u1.y, wv[j].w, acc[i]);
        }
      }
    }
    // transposing butterfly: 8 values over 32 lanes -> 1 row sum per lane (9 shuffles)
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float s4[4], s3[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = b4 ? acc[i] : acc[i + 4];
      const float keep = b4 ? acc[i + 4] : acc[i];
      s4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = b3 ? s4[i] : s4[i + 2];
      const float keep = b3 ? s4[i + 2] : s4[i];
      s3[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float v = (b2 ? s3[1] : s3[0]) + __shfl_xor_sync(0xffffffffu, b2 ? s3[0] : s3[1], 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    if ((lane & 3) == 0 && r0 + my_row < nrows)
      a.partial[((size_t)blockIdx.y * a.rows + row0 + r0 + my_row) * a.E + e] = v;
  }
}

// f32 -> unsigned key with the same order (larger float, larger key)
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct Pick {
  int e;      // expert of slot li of the row (lanes li < k)
  float ex;   // its exp(z - z_max)
  float sum;  // the sum of exp(z - z_max) over the row's k picks
};

// Top-k of one row of logits by a group of lpr lanes, VPL logits per lane (lpr * VPL >= E:
// 8 x 16 for E <= 128 or 16 x 16 for E <= 256 when a warp takes several rows; a whole warp,
// 32 x 4 or 32 x 8, when the step has at most one row per warp), each packed with its expert
// index as (order key << 32 | 255 - e): the largest packed value is the largest logit, ties
// to the lowest expert index; k rounds of a local max and a butterfly over the group.  Not
// inlined, so that the kernel's call before griddepcontrol.wait (on no data, with live false)
// brings exactly this code into the instruction caches: the kernel runs once per step and its
// code is otherwise cold.
template <int VPL>
__device__ __noinline__ Pick select_topk(const float* z, int E, int k, int lpr, int li, bool live) {
  unsigned long long pv[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = li + lpr * j;
    pv[j] = live && e < E ? ((unsigned long long)order_key(z[e] + 0.0f) << 32) |
                                (unsigned long long)(255 - e)
                          : 0ull;  // (-0 -> +0 above); 0 sorts below every logit
  }
  Pick pk = {-1, 0.0f, 0.0f};
  float zsel0 = 0.0f;
#pragma unroll 1
  for (int kk = 0; kk < k; ++kk) {
    unsigned long long b = 0ull;
#pragma unroll
    for (int j = 0; j < VPL; ++j) b = max(b, pv[j]);
    for (int o = 1; o < lpr; o <<= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    const int be = 255 - (int)(b & 0xFFull);
    const float bv = key_value((uint32_t)(b >> 32));
    if (kk == 0) zsel0 = bv;
    const float ex = expf(bv - zsel0);
    pk.sum += ex;
    if (li == kk) pk.ex = ex, pk.e = be;  // lane kk of the group keeps slot kk
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (li + lpr * j == be) pv[j] = 0ull;
  }
  return pk;
}

constexpr int TOPK_THREADS = 512;
constexpr int TOPK_BATCH = 12;  // logits per thread in flight at once (48 rows x 128 experts)
template <int KSL>  // K slices of the router partials at most
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(TopkArgs a) {
  extern __shared__ float s_z[];  // [rows][E] logits
  __shared__ int s_idx[MAX_ROWS * MAX_K];
  __shared__ int s_pos[MAX_ROWS];
  __shared__ unsigned long long s_mask[MAX_EXPERTS];  // rows routed to each expert
  __shared__ int s_tot[3][MAX_EXPERTS / 32];          // per-warp totals of the expert scans
  // the hit experts by key = 63 - row count (a bit per expert), and per key the experts and the
  // row groups of all smaller keys
  __shared__ unsigned s_kmask[64][MAX_EXPERTS / 32];
  __shared__ int s_kstart[64], s_kgrp[64];
  static_assert(MAX_ROWS < 63, "a row count fits a key");
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = TOPK_THREADS / 32;
  for (int e = tid; e < MAX_EXPERTS; e += TOPK_THREADS) s_mask[e] = 0ull;
  for (int i = tid; i < 64 * (MAX_EXPERTS / 32); i += TOPK_THREADS) (&s_kmask[0][0])[i] = 0u;
  if (tid < a.rows) s_pos[tid] = a.positions[tid];  // a step input: read before the wait
  // at most one row per warp: a whole warp per row (shorter per-lane chains in each round)
  const bool wide = a.rows <= NW;
  if (warp == 0) {  // warm the selection code while the previous kernel finishes
    const Pick dry = !wide          ? select_topk<16>(s_z, a.E, a.k, a.E <= 128 ? 8 : 16, lane & 7, false)
                     : a.E <= 128 ? select_topk<4>(s_z, a.E, a.k, 32, lane, false)
                                  : select_topk<8>(s_z, a.E, a.k, 32, lane, false);
    if (dry.e == -2) s_pos[0] = 0;  // never true: keeps the call
  }
  pdl_wait();
  // the routed-expert GEMMs of this step take their work items from these counters; every
  // earlier kernel of the stream has completed once this CTA is past its wait
  if (tid == 0) a.route->item_next[0] = a.route->item_next[1] = 0;
  // phase 1a: logits = the K-slice partials summed in slice order
  const int nz = a.rows * a.E;
  for (int base = tid; base < nz; base += TOPK_BATCH * TOPK_THREADS) {
    float pz[TOPK_BATCH][KSL];
#pragma unroll
    for (int u = 0; u < TOPK_BATCH; ++u)
#pragma unroll
      for (int ks = 0; ks < KSL; ++ks) {
        const int i = base + u * TOPK_THREADS;
        pz[u][ks] = i < nz && ks < a.kslices ? a.partial[(size_t)ks * nz + i] : 0.0f;
      }
#pragma unroll
    for (int u = 0; u < TOPK_BATCH; ++u) {
      const int i = base + u * TOPK_THREADS;
      float z = 0.0f;
#pragma unroll
      for (int ks = 0; ks < KSL; ++ks)
        if (ks < a.kslices) z += pz[u][ks];
      if (i < nz) {
        s_z[i] = z;
        a.logits[i] = z;
      }
    }
  }
  __syncthreads();
  // phase 1b: selection, a group of 8 or 16 lanes per row, or a warp (select_topk)
  {
    const int lpr = wide ? 32 : a.E <= 128 ? 8 : 16;
    const int rpw = 32 / lpr;  // rows per warp
    const int li = lane & (lpr - 1), grp = lane / lpr;
    for (int r0 = warp * rpw; r0 < a.rows; r0 += NW * rpw) {
      const int r = r0 + grp;
      const bool live = r < a.rows;
      const float* zr = s_z + r * a.E;
      const Pick pk = !wide        ? select_topk<16>(zr, a.E, a.k, lpr, li, live)
                      : a.E <= 128 ? select_topk<4>(zr, a.E, a.k, lpr, li, live)
                                   : select_topk<8>(zr, a.E, a.k, lpr, li, live);
      const int my_e = pk.e;
      const float my_ex = pk.ex, ex_sum = pk.sum;
      if (live && li < a.k) {
        const bool pad = s_pos[r] < 0;
        const int e = pad ? -1 : my_e;
        const float wgt = pad ? 0.0f : my_ex / ex_sum * a.routed_scale;
        s_idx[r * a.k + li] = e;
        a.topk_idx[r * a.k + li] = e;
        a.topk_w[r * a.k + li] = wgt;
        if (a.user_idx) a.user_idx[r * a.k + li] = e;
        if (a.user_w) a.user_w[r * a.k + li] = wgt;
        if (e >= 0) atomicOr(&s_mask[e], 1ull << r);
      }
    }
  }
  __syncthreads();
  // phase 2: prefix sums over experts: warp w scans experts 32w..32w+31, then adds the
  // totals of the warps before it
  constexpr int SW = MAX_EXPERTS / 32;
  int c = 0, hit = 0, rg = 0, ic = 0, ih = 0, ir = 0;
  const int e = warp * 32 + lane;
  if (warp < SW) {
    c = e < a.E ? __popcll(s_mask[e]) : 0;
    hit = c > 0;
    rg = (c + EXPERT_ROWS - 1) / EXPERT_ROWS;
    ic = c, ih = hit, ir = rg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // inclusive warp scans
      const int tc = __shfl_up_sync(0xffffffffu, ic, o);
      const int th = __shfl_up_sync(0xffffffffu, ih, o);
      const int tr = __shfl_up_sync(0xffffffffu, ir, o);
      if (lane >= o) ic += tc, ih += th, ir += tr;
    }
    if (lane == 31) s_tot[0][warp] = ic, s_tot[1][warp] = ih, s_tot[2][warp] = ir;
    if (a.lpt && c > 0) atomicOr(&s_kmask[63 - c][e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  static_assert(SW < NW, "a spare warp for the key prefix");
  if (a.lpt && warp == SW) {  // per key: the experts and the row groups of all smaller keys
    int n[2], g[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int key = 2 * lane + i;
      n[i] = 0;
#pragma unroll
      for (int w = 0; w < MAX_EXPERTS / 32; ++w) n[i] += __popc(s_kmask[key][w]);
      g[i] = n[i] * ((63 - key + EXPERT_ROWS - 1) / EXPERT_ROWS);
    }
    int xn = n[0] + n[1], xg = g[0] + g[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yn = __shfl_up_sync(0xffffffffu, xn, o), yg = __shfl_up_sync(0xffffffffu, xg, o);
      if (lane >= o) xn += yn, xg += yg;
    }
    s_kstart[2 * lane] = xn - n[0] - n[1], s_kstart[2 * lane + 1] = xn - n[1];
    s_kgrp[2 * lane] = xg - g[0] - g[1], s_kgrp[2 * lane + 1] = xg - g[1];
  }
  __shared__ int s_off[MAX_EXPERTS];
  if (warp < SW) {
    int bo = 0, bh = 0, br = 0;
    for (int w = 0; w < warp; ++w) bo += s_tot[0][w], bh += s_tot[1][w], br += s_tot[2][w];
    const int off = bo + ic - c, d = bh + ih - hit, rgp = br + ir - rg;
    s_off[e] = off;
    if (c > 0) {
      a.route->hit_e[d] = e;
      a.route->hit_off[d] = off;
      a.route->hit_cnt[d] = c;
      a.route->rg_prefix[d] = rgp;
    }
    if (warp == SW - 1 && lane == 31) {
      a.route->n_hit = bh + ih;
      a.route->rg_prefix[bh + ih] = br + ir;
      if (a.lpt) a.route->lpt_gpre[bh + ih] = br + ir;
    }
  }
  __syncthreads();
  // phase 2b: the hit experts in decreasing row count, ties in expert order: an expert's
  // place is its key's start plus the experts of its key below it
  if (a.lpt && warp < SW && c > 0) {
    const int key = 63 - c, w0 = e >> 5;
    int rank = s_kstart[key] + __popc(s_kmask[key][w0] & ((1u << (e & 31)) - 1u));
    for (int w = 0; w < w0; ++w) rank += __popc(s_kmask[key][w]);
    a.route->lpt_e[rank] = e;
    a.route->lpt_off[rank] = s_off[e];
    a.route->lpt_cnt[rank] = c;
    a.route->lpt_gpre[rank] = s_kgrp[key] + (rank - s_kstart[key]) * rg;
  }
  // phase 3: stable placement -- an expert's entries in row order (a row picks an expert once)
  const int n = a.rows * a.k;
  for (int q = tid; q < n; q += TOPK_THREADS) {
    const int ex = s_idx[q];
    if (ex >= 0) {
      const int r = q / a.k;
      const int pos = s_off[ex] + __popcll(s_mask[ex] & ((1ull << r) - 1ull));
      a.slot_pos[q] = pos;
      a.perm[pos] = r;
    } else {
      a.slot_pos[q] = -1;
    }
  }
}

}  // namespace

int router_smem_bytes() { return RT_ROWS * ROUTER_KSLICE * 2; }
// The logits of the step in shared memory, [rows][E].
// The kernel is one latency-bound CTA: it asks for more shared memory than its logits need
// (200 KB) so that no GEMM CTA of the concurrently running shared expert lands on its SM and
// competes for its issue slots.
constexpr int TOPK_SMEM = 200 * 1024;
static_assert(TOPK_SMEM >= MAX_ROWS * MAX_EXPERTS * 4, "the logits must fit");
int topk_smem_bytes() { return TOPK_SMEM; }

// The limits are properties of the kernels, shared by every layer handle of the process: set
// them for the largest step any handle accepts.
cudaError_t router_prepare() {
  cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       router_smem_bytes());
  if (e != cudaSuccess) return e;
  for (auto k : {topk_kernel<1>, topk_kernel<2>, topk_kernel<4>, topk_kernel<8>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, topk_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_router(const Launch& L, const RouterArgs& a) {
  const dim3 grid((a.E + RT_EXPERTS - 1) / RT_EXPERTS, (a.H + ROUTER_KSLICE - 1) / ROUTER_KSLICE,
                  (a.rows + RT_ROWS - 1) / RT_ROWS);
  return launch_ex(L, grid, dim3(RT_THREADS), router_smem_bytes(), router_kernel, a);
}

cudaError_t launch_topk(const Launch& L, const TopkArgs& a) {
  const int smem = TOPK_SMEM;
  if (a.kslices <= 1) return launch_ex(L, dim3(1), dim3(TOPK_THREADS), smem, topk_kernel<1>, a);
  if (a.kslices <= 2) return launch_ex(L, dim3(1), dim3(TOPK_THREADS), smem, topk_kernel<2>, a);
  if (a.kslices <= 4) return launch_ex(L, dim3(1), dim3(TOPK_THREADS), smem, topk_kernel<4>, a);
  return launch_ex(L, dim3(1), dim3(TOPK_THREADS), smem, topk_kernel<8>, a);
}

}  // namespace mono
