// Router and expert grouping ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", launch
// table K2: "router, top-6"; ATOM changes: "f32 router logits").
//
// router_kernel: z[r, e] = u[r] . W_r[e] in f32, split over K: CTA (4 experts, 1024-wide K
// slice) stages the slice of every row of u in shared memory and writes one partial per
// (slice, row, expert).  topk_kernel sums the partials in slice order (a fixed order, so
// results replay bit-exactly), picks the top-k per row and sorts the (row, slot) pairs by
// expert, stably, for the grouped expert GEMMs.
#include "kernels.h"

namespace mono {

namespace {

constexpr int RT_EXPERTS = 4;    // experts per CTA, one warp each
constexpr int RT_THREADS = RT_EXPERTS * 32;
constexpr int MAX_ROWS = 48, MAX_K = 8;

__global__ void __launch_bounds__(RT_THREADS) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t rt_smem[];
  __half* us = reinterpret_cast<__half*>(rt_smem);  // [rows][ROUTER_KSLICE]
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.y * ROUTER_KSLICE;
  const int klen = min(ROUTER_KSLICE, a.H - k0);
  const int chunks = klen / 8;  // 16-byte chunks per row
  for (int idx = tid; idx < a.rows * chunks; idx += RT_THREADS) {
    const int r = idx / chunks, c = idx - r * chunks;
    cp_async16(us + r * ROUTER_KSLICE + c * 8, a.u + (size_t)r * a.H + k0 + c * 8, 16);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  // this lane's weights: k = k0 + 128 j + 4 lane + {0..3}
  const int e = blockIdx.x * RT_EXPERTS + warp;
  float4 wv[ROUTER_KSLICE / 128];
  if (e < a.E) {
    const float* wr = a.wr + (size_t)e * a.H + k0;
#pragma unroll
    for (int j = 0; j < ROUTER_KSLICE / 128; ++j)
      wv[j] = 128 * j < klen ? *reinterpret_cast<const float4*>(wr + 128 * j + 4 * lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  if (e >= a.E) return;
  for (int r = 0; r < a.rows; ++r) {
    const __half* ur = us + r * ROUTER_KSLICE + 4 * lane;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < ROUTER_KSLICE / 128; ++j) {
      if (128 * j < klen) {
        const uint2 uv = lds64(ur + 128 * j);
        const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&uv.x));
        const float2 u1 = __half22float2(*reinterpret_cast<const __half2*>(&uv.y));
        acc = fmaf(u0.x, wv[j].x, acc);
        acc = fmaf(u0.y, wv[j].y, acc);
        acc = fmaf(u1.x, wv[j].z, acc);
        acc = fmaf(u1.y, wv[j].w, acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) a.partial[((size_t)blockIdx.y * a.rows + r) * a.E + e] = acc;
  }
}

constexpr int TOPK_THREADS = 512;
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(TopkArgs a) {
  __shared__ int s_idx[MAX_ROWS * MAX_K];
  __shared__ int s_cnt[MAX_EXPERTS], s_off[MAX_EXPERTS], s_hit[MAX_EXPERTS], s_rg[MAX_EXPERTS];
  __shared__ int s_fill[MAX_EXPERTS];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = TOPK_THREADS / 32, ZJ = MAX_EXPERTS / 32;
  for (int e = tid; e < MAX_EXPERTS; e += TOPK_THREADS) s_cnt[e] = 0, s_fill[e] = 0;
  // phase 1: logits (sum of the K-slice partials in slice order) and selection, a warp a row
  for (int r = warp; r < a.rows; r += NW) {
    const bool pad = a.positions[r] < 0;
    float z[ZJ];
#pragma unroll
    for (int j = 0; j < ZJ; ++j) z[j] = 0.0f;
    for (int ks = 0; ks < a.kslices; ++ks) {
      float pz[ZJ];
#pragma unroll
      for (int j = 0; j < ZJ; ++j) {
        const int e = lane + 32 * j;
        pz[j] = e < a.E ? a.partial[((size_t)ks * a.rows + r) * a.E + e] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < ZJ; ++j) z[j] += pz[j];
    }
#pragma unroll
    for (int j = 0; j < ZJ; ++j) {
      const int e = lane + 32 * j;
      if (e < a.E) a.logits[(size_t)r * a.E + e] = z[j];
      else z[j] = -INFINITY;
    }
    float zsel0 = 0.0f, ex_sum = 0.0f, my_ex = 0.0f;
    int my_e = -1;
#pragma unroll
    for (int kk = 0; kk < MAX_K; ++kk) {
      if (kk < a.k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < ZJ; ++j) {
          const int e = lane + 32 * j;
          if (e < a.E && (z[j] > bv || (z[j] == bv && e < be))) bv = z[j], be = e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) bv = ov, be = oe;
        }
        if (kk == 0) zsel0 = bv;
        const float ex = expf(bv - zsel0);
        ex_sum += ex;
        if (lane == kk) my_ex = ex, my_e = be;  // lane kk keeps slot kk
#pragma unroll
        for (int j = 0; j < ZJ; ++j)
          if (lane + 32 * j == be) z[j] = -INFINITY;
      }
    }
    if (lane < a.k) {
      const int e = pad ? -1 : my_e;
      const float wgt = pad ? 0.0f : my_ex / ex_sum * a.routed_scale;
      s_idx[r * a.k + lane] = e;
      a.topk_idx[r * a.k + lane] = e;
      a.topk_w[r * a.k + lane] = wgt;
      if (a.user_idx) a.user_idx[r * a.k + lane] = e;
      if (a.user_w) a.user_w[r * a.k + lane] = wgt;
    }
  }
  __syncthreads();
  const int n = a.rows * a.k;
  for (int q = tid; q < n; q += TOPK_THREADS)
    if (s_idx[q] >= 0) atomicAdd(&s_cnt[s_idx[q]], 1);
  __syncthreads();
  // phase 2: prefix sums over experts (one warp; E <= 256)
  if (warp == 0) {
    int run_off = 0, run_hit = 0, run_rg = 0;
    for (int base = 0; base < MAX_EXPERTS; base += 32) {
      const int e = base + lane;
      const int c = e < a.E ? s_cnt[e] : 0;
      const int hit = c > 0, rg = (c + EXPERT_ROWS - 1) / EXPERT_ROWS;
      int ic = c, ih = hit, ir = rg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {  // inclusive warp scans
        const int tc = __shfl_up_sync(0xffffffffu, ic, o);
        const int th = __shfl_up_sync(0xffffffffu, ih, o);
        const int tr = __shfl_up_sync(0xffffffffu, ir, o);
        if (lane >= o) ic += tc, ih += th, ir += tr;
      }
      s_off[e] = run_off + ic - c;
      s_hit[e] = run_hit + ih - hit;
      s_rg[e] = run_rg + ir - rg;
      run_off += __shfl_sync(0xffffffffu, ic, 31);
      run_hit += __shfl_sync(0xffffffffu, ih, 31);
      run_rg += __shfl_sync(0xffffffffu, ir, 31);
    }
    if (lane == 0) {
      a.route->n_hit = run_hit;
      a.route->rg_prefix[run_hit] = run_rg;
    }
  }
  __syncthreads();
  for (int e = tid; e < a.E; e += TOPK_THREADS) {
    if (s_cnt[e] > 0) {
      const int d = s_hit[e];
      a.route->hit_e[d] = e;
      a.route->hit_off[d] = s_off[e];
      a.route->hit_cnt[d] = s_cnt[e];
      a.route->rg_prefix[d] = s_rg[e];
    }
  }
  // phase 3: stable placement in (row, slot) order within each expert, 32 entries at a time
  if (warp == 0) {
    for (int base = 0; base < n; base += 32) {
      const int q = base + lane;
      const int e = q < n ? s_idx[q] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int before = __popc(peers & ((1u << lane) - 1u));
      const int fill = e >= 0 ? s_fill[e] : 0;
      __syncwarp();
      if (q < n) {
        if (e >= 0) {
          const int pos = s_off[e] + fill + before;
          a.slot_pos[q] = pos;
          a.perm[pos] = q / a.k;
        } else {
          a.slot_pos[q] = -1;
        }
      }
      if (e >= 0 && before == 0) s_fill[e] = fill + __popc(peers);
      __syncwarp();
    }
  }
}

}  // namespace

int router_smem_bytes(int rows) { return rows * ROUTER_KSLICE * 2; }

// The limit is a property of the kernel, shared by every layer handle of the process: set it
// for the largest step any handle accepts.
cudaError_t router_prepare() {
  return cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              router_smem_bytes(MAX_ROWS));
}

cudaError_t launch_router(const Launch& L, const RouterArgs& a) {
  const dim3 grid((a.E + RT_EXPERTS - 1) / RT_EXPERTS, (a.H + ROUTER_KSLICE - 1) / ROUTER_KSLICE);
  return launch_ex(L, grid, dim3(RT_THREADS), router_smem_bytes(a.rows), router_kernel, a);
}

cudaError_t launch_topk(const Launch& L, const TopkArgs& a) {
  return launch_ex(L, dim3(1), dim3(TOPK_THREADS), 0, topk_kernel, a);
}

}  // namespace mono
