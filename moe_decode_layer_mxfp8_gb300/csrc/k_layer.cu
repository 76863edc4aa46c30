// The layer's non-GEMM kernels: RMSNorms, q/kv norm + fp8 KV insert, split sliding-window
// attention with a log-sum-exp combine, router logits, top-k with expert grouping, and the
// final residual combine ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", launch
// table rows K1 and K2).
#include <cuda_fp8.h>

#include "kernels.h"

namespace mono {

namespace {

constexpr int NORM_THREADS = 256;

// Block-wide sum / max over NORM_THREADS threads.
__device__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = l < (blockDim.x >> 5) ? red[l] : 0.0f;
  return warp_sum(t);
}
__device__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = l < (blockDim.x >> 5) ? red[l] : 0.0f;
  return warp_max(t);
}

// RMSNorm of one row (the attention-front norm and the FFN-seam norm): y = x / sqrt(mean(x^2)
// + eps) * gamma, rounded to bf16 and stored as its exact f16 copy for the tensor cores.
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(NormArgs a) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const __nv_bfloat16* x = a.in + (size_t)r * a.in_ld;
  float ss = 0.0f;
  for (int i = 2 * threadIdx.x; i < a.dim; i += 2 * NORM_THREADS) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + i));
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, ss));
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)a.dim + a.eps);
  __half* y = a.out + (size_t)r * a.out_ld;
  for (int i = 2 * threadIdx.x; i < a.dim; i += 2 * NORM_THREADS) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + i));
    const float2 gm = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a.gamma + i));
    y[i] = bf16_as_f16(v.x * inv * gm.x);
    y[i + 1] = bf16_as_f16(v.y * inv * gm.y);
  }
}

// Physical page of token t of request q, or -1 when the block table does not map it.
__device__ __forceinline__ int page_of(const int* table, int max_blocks, int n_req, long long nb,
                                       int q, int t, int bs) {
  const int lb = t / bs;
  if (q < 0 || q >= n_req || t < 0 || lb >= max_blocks) return -1;
  const int pb = table[(size_t)q * max_blocks + lb];
  return (pb < 0 || pb >= nb) ? -1 : pb;
}

// q-norm and kv-norm of one row, then the fp8 KV insert of the normed kv at the row's
// position: s = amax / 448 (1 when amax = 0), codes = e4m3(kv / s) rounded to nearest even
// and saturating, record = codes then s as f32.  Pad rows (position < 0) insert nothing.
__global__ void __launch_bounds__(NORM_THREADS) qkv_norm_insert_kernel(QkvNormInsertArgs a) {
  __shared__ float red[32];
  __shared__ float kvs[1024];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const __nv_bfloat16* row = a.qkv + (size_t)r * (a.q_rank + a.kv_dim);
  // q latent
  float ss = 0.0f;
  for (int i = threadIdx.x; i < a.q_rank; i += NORM_THREADS) {
    const float v = __bfloat162float(row[i]);
    ss = fmaf(v, v, ss);
  }
  ss = block_sum(ss, red);
  float inv = 1.0f / sqrtf(ss / (float)a.q_rank + a.eps);
  for (int i = threadIdx.x; i < a.q_rank; i += NORM_THREADS)
    a.qlatn[(size_t)r * a.q_rank + i] =
        bf16_as_f16(__bfloat162float(row[i]) * inv * __bfloat162float(a.gq[i]));
  // kv latent
  const __nv_bfloat16* kv = row + a.q_rank;
  ss = 0.0f;
  for (int i = threadIdx.x; i < a.kv_dim; i += NORM_THREADS) {
    const float v = __bfloat162float(kv[i]);
    ss = fmaf(v, v, ss);
  }
  ss = block_sum(ss, red);
  inv = 1.0f / sqrtf(ss / (float)a.kv_dim + a.eps);
  float amax = 0.0f;
  for (int i = threadIdx.x; i < a.kv_dim; i += NORM_THREADS) {
    const float v = round_bf16(__bfloat162float(kv[i]) * inv * __bfloat162float(a.gkv[i]));
    kvs[i] = v;
    a.kvn[(size_t)r * a.kv_dim + i] = __float2bfloat16_rn(v);
    amax = fmaxf(amax, fabsf(v));
  }
  amax = block_max(amax, red);  // (its barriers also publish kvs)
  const int p = a.positions[r];
  if (p < 0) return;
  const int pb = page_of(a.block_table, a.max_blocks, a.n_req, a.num_blocks, a.row_req[r], p,
                         a.block_size);
  if (pb < 0) {
    if (threadIdx.x == 0) atomicOr(a.status, ST_UNMAPPED_PAGE);
    return;
  }
  uint8_t* rec = a.cache + (size_t)pb * a.stride_block + (size_t)(p % a.block_size) * a.stride_tok;
  const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int i = 2 * threadIdx.x; i < a.kv_dim; i += 2 * NORM_THREADS) {
    const __nv_fp8x2_storage_t c2 =
        __nv_cvt_float2_to_fp8x2(make_float2(kvs[i] / s, kvs[i + 1] / s), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(rec + i) = c2;
  }
  if (threadIdx.x == 0) *reinterpret_cast<float*>(rec + a.kv_dim) = s;
}

// ------------------------------------------------------------------------------ attention
constexpr int ATTN_THREADS = 256;
constexpr int ATTN_KEYS = 128;  // keys per split at most
constexpr int ATTN_HEADS = 16;  // heads per kv group at most

// One (row, kv group, split): scores of the group's heads against the split's share of the
// row's window, a local softmax (max m, sum l, unnormalised o); the last split to finish
// combines all splits: o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.  The cached latent is
// both key and value; head h reads slice h / heads_per_group.  Scores scale 1/sqrt(head_dim).
template <int DH>
__global__ void __launch_bounds__(ATTN_THREADS) attn_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  __shared__ int s_flag;
  __shared__ float s_m[ATTN_HEADS], s_l[ATTN_HEADS];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, g = blockIdx.y, sp = blockIdx.z, S = a.splits;
  const int G = a.kv_dim / DH, hpg = a.n_q / G, h0 = g * hpg;
  const int tid = threadIdx.x;
  const int QW = a.n_q * DH;
  const int p = a.positions[r];
  if (p < 0) {  // pad row: attention output is zero
    if (sp == 0)
      for (int i = tid; i < hpg * DH; i += ATTN_THREADS)
        a.o[(size_t)r * QW + h0 * DH + i] = __float2half(0.0f);
    return;
  }
  const int req = a.row_req[r];
  int hi = p;
  if (!a.causal)
    for (int rr = 0; rr < a.rows; ++rr)
      if (a.row_req[rr] == req && a.positions[rr] > hi) hi = a.positions[rr];
  const int width = a.causal ? a.window : a.swa_width;
  const int lo = max(0, hi - width + 1);
  const int T = hi - lo + 1;
  const int per = (T + S - 1) / S;
  const int t0 = lo + sp * per;
  const int nt = max(0, min(per, hi + 1 - t0));

  float* qs = sm;                       // [hpg][DH]
  float* K = qs + ATTN_HEADS * DH;      // [ATTN_KEYS][DH + 1]
  float* P = K + ATTN_KEYS * (DH + 1);  // [hpg][ATTN_KEYS]
  for (int i = tid; i < hpg * DH; i += ATTN_THREADS)
    qs[i] = __bfloat162float(a.q[(size_t)r * QW + h0 * DH + i]);
  constexpr int CH = DH / 16;  // 16-byte chunks of the group's slice
  for (int idx = tid; idx < nt * CH; idx += ATTN_THREADS) {
    const int t = idx / CH, ch = idx - t * CH;
    const int pos = t0 + t;
    const int pb = page_of(a.block_table, a.max_blocks, a.n_req, a.num_blocks, req, pos,
                           a.block_size);
    float* kd = K + t * (DH + 1) + ch * 16;
    if (pb < 0) {
      if (ch == 0) atomicOr(a.status, ST_UNMAPPED_PAGE);
      for (int j = 0; j < 16; ++j) kd[j] = 0.0f;
      continue;
    }
    const uint8_t* rec =
        a.cache + (size_t)pb * a.stride_block + (size_t)(pos % a.block_size) * a.stride_tok;
    const float sc = *reinterpret_cast<const float*>(rec + a.kv_dim);
    const uint4 raw = *reinterpret_cast<const uint4*>(rec + g * DH + ch * 16);
    const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h2[2];
      e4m3x4_to_f16x4(wds[j], h2);
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h2[0]));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h2[1]));
      kd[4 * j + 0] = f0.x * sc;
      kd[4 * j + 1] = f0.y * sc;
      kd[4 * j + 2] = f1.x * sc;
      kd[4 * j + 3] = f1.y * sc;
    }
  }
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)DH);
  for (int idx = tid; idx < hpg * nt; idx += ATTN_THREADS) {
    const int h = idx / nt, t = idx - h * nt;
    const float* qh = qs + h * DH;
    const float* kt = K + t * (DH + 1);
    float d = 0.0f;
#pragma unroll 8
    for (int i = 0; i < DH; ++i) d = fmaf(qh[i], kt[i], d);
    P[h * ATTN_KEYS + t] = d * scale;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < hpg; h += ATTN_THREADS / 32) {
    float m = -INFINITY;
    for (int t = lane; t < nt; t += 32) m = fmaxf(m, P[h * ATTN_KEYS + t]);
    m = warp_max(m);
    float l = 0.0f;
    for (int t = lane; t < nt; t += 32) {
      const float e = expf(P[h * ATTN_KEYS + t] - m);
      P[h * ATTN_KEYS + t] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      s_m[h] = m;
      s_l[h] = l;
    }
  }
  __syncthreads();
  if (S == 1) {
    for (int idx = tid; idx < hpg * DH; idx += ATTN_THREADS) {
      const int h = idx / DH, d = idx - h * DH;
      float acc = 0.0f;
      for (int t = 0; t < nt; ++t) acc = fmaf(P[h * ATTN_KEYS + t], K[t * (DH + 1) + d], acc);
      a.o[(size_t)r * QW + (h0 + h) * DH + d] = bf16_as_f16(acc / s_l[h]);
    }
    return;
  }
  // partial of this split
  const int PW = DH + 2;
  for (int idx = tid; idx < hpg * DH; idx += ATTN_THREADS) {
    const int h = idx / DH, d = idx - h * DH;
    float acc = 0.0f;
    for (int t = 0; t < nt; ++t) acc = fmaf(P[h * ATTN_KEYS + t], K[t * (DH + 1) + d], acc);
    float* part = a.part + (((size_t)r * a.n_q + h0 + h) * S + sp) * PW;
    part[2 + d] = acc;
    if (d == 0) {
      part[0] = s_m[h];
      part[1] = s_l[h];
    }
  }
  __threadfence();
  __syncthreads();
  int* ctr = a.counters + r * G + g;
  if (tid == 0) s_flag = atomicAdd(ctr, 1) == S - 1;
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  for (int idx = tid; idx < hpg * DH; idx += ATTN_THREADS) {
    const int h = idx / DH, d = idx - h * DH;
    const float* base = a.part + ((size_t)r * a.n_q + h0 + h) * S * PW;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(base + s * PW));
    float num = 0.0f, den = 0.0f;
    for (int s = 0; s < S; ++s) {
      const float ms = __ldcg(base + s * PW);
      const float f = ms == -INFINITY ? 0.0f : expf(ms - M);
      num = fmaf(f, __ldcg(base + s * PW + 2 + d), num);
      den = fmaf(f, __ldcg(base + s * PW + 1), den);
    }
    a.o[(size_t)r * QW + (h0 + h) * DH + d] = bf16_as_f16(num / den);
  }
  if (tid == 0) *ctr = 0;
}

// -------------------------------------------------------------------------------- router
// f32 router logits z[r, e] = u[r] . W_r[e] ("f32 router logits"): one warp per expert, eight
// rows per CTA.
constexpr int ROUTER_ROWS = 8;
__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int r0 = blockIdx.y * ROUTER_ROWS;
  const int nr = min(ROUTER_ROWS, a.rows - r0);
  if (e >= a.E) return;
  float acc[ROUTER_ROWS];
#pragma unroll
  for (int j = 0; j < ROUTER_ROWS; ++j) acc[j] = 0.0f;
  const float* w = a.wr + (size_t)e * a.H;
  for (int k = lane * 4; k < a.H; k += 128) {
    const float4 wv = *reinterpret_cast<const float4*>(w + k);
#pragma unroll
    for (int j = 0; j < ROUTER_ROWS; ++j) {
      if (j < nr) {
        const uint2 uv = *reinterpret_cast<const uint2*>(a.u + (size_t)(r0 + j) * a.H + k);
        const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&uv.x));
        const float2 u1 = __half22float2(*reinterpret_cast<const __half2*>(&uv.y));
        acc[j] = fmaf(u0.x, wv.x, fmaf(u0.y, wv.y, fmaf(u1.x, wv.z, fmaf(u1.y, wv.w, acc[j]))));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < ROUTER_ROWS; ++j) {
    const float v = warp_sum(acc[j]);
    if (j < nr && lane == 0) a.logits[(size_t)(r0 + j) * a.E + e] = v;
  }
}

// Top-k per row (largest logits, ties to the lower expert index; weights = softmax over the
// chosen logits, which equals the full softmax renormalised over them, times routed_scale),
// then a stable counting sort of the (row, slot) pairs by expert for the grouped expert
// GEMMs.  One CTA.
constexpr int TOPK_THREADS = 512;
constexpr int MAX_ROWS = 48, MAX_K = 8;
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(TopkArgs a) {
  __shared__ int s_idx[MAX_ROWS * MAX_K];
  __shared__ int s_cnt[MAX_EXPERTS], s_off[MAX_EXPERTS], s_hit[MAX_EXPERTS], s_rg[MAX_EXPERTS];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nw = TOPK_THREADS / 32;
  for (int e = tid; e < MAX_EXPERTS; e += TOPK_THREADS) s_cnt[e] = 0;
  // phase 1: selection, one warp per row
  for (int r = warp; r < a.rows; r += nw) {
    const bool pad = a.positions[r] < 0;
    float z[MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MAX_EXPERTS / 32; ++j) {
      const int e = lane + 32 * j;
      z[j] = e < a.E ? a.logits[(size_t)r * a.E + e] : -INFINITY;
    }
    float zsel[MAX_K];
    int esel[MAX_K];
    for (int kk = 0; kk < a.k; ++kk) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < MAX_EXPERTS / 32; ++j) {
        const int e = lane + 32 * j;
        if (e < a.E && (z[j] > bv || (z[j] == bv && e < be))) {
          bv = z[j];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      zsel[kk] = bv;
      esel[kk] = be;
#pragma unroll
      for (int j = 0; j < MAX_EXPERTS / 32; ++j)
        if (lane + 32 * j == be) z[j] = -INFINITY;
    }
    if (lane == 0) {
      float sum = 0.0f, ex[MAX_K];
      for (int kk = 0; kk < a.k; ++kk) {
        ex[kk] = expf(zsel[kk] - zsel[0]);
        sum += ex[kk];
      }
      for (int kk = 0; kk < a.k; ++kk) {
        const int e = pad ? -1 : esel[kk];
        const float wgt = pad ? 0.0f : ex[kk] / sum * a.routed_scale;
        s_idx[r * a.k + kk] = e;
        a.topk_idx[r * a.k + kk] = e;
        a.topk_w[r * a.k + kk] = wgt;
        if (a.user_idx) a.user_idx[r * a.k + kk] = e;
        if (a.user_w) a.user_w[r * a.k + kk] = wgt;
      }
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
        if (lane >= o) {
          ic += tc;
          ih += th;
          ir += tr;
        }
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
  // phase 3: stable placement, (row, slot) order within each expert
  for (int q = tid; q < n; q += TOPK_THREADS) {
    const int e = s_idx[q];
    if (e < 0) {
      a.slot_pos[q] = -1;
      continue;
    }
    int rank = 0;
    for (int j = 0; j < q; ++j) rank += s_idx[j] == e;
    const int pos = s_off[e] + rank;
    a.slot_pos[q] = pos;
    a.perm[pos] = q / a.k;
  }
}

// out = bf16(h + y_shared + sum_j w_j y_j) in slot order; pad rows copy x.
__global__ void __launch_bounds__(256) final_kernel(FinalArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const bool pad = a.positions[r] < 0;
  for (int c = blockIdx.y * 512 + 2 * threadIdx.x; c < a.H; c += gridDim.y * 512) {
    const size_t o = (size_t)r * a.H + c;
    __nv_bfloat162 res;
    if (pad) {
      res = *reinterpret_cast<const __nv_bfloat162*>(a.x + o);
    } else {
      const float2 hv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a.h + o));
      const float2 sv = *reinterpret_cast<const float2*>(a.ys + o);
      float v0 = hv.x + sv.x, v1 = hv.y + sv.y;
      for (int j = 0; j < a.k; ++j) {
        const int pos = a.slot_pos[r * a.k + j];
        if (pos < 0) continue;
        const float wj = a.topk_w[r * a.k + j];
        const float2 yv = *reinterpret_cast<const float2*>(a.yr + (size_t)pos * a.H + c);
        v0 = fmaf(wj, yv.x, v0);
        v1 = fmaf(wj, yv.y, v1);
      }
      res = __floats2bfloat162_rn(v0, v1);
    }
    *reinterpret_cast<__nv_bfloat162*>(a.out + o) = res;
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const Launch& L, const NormArgs& a, int rows) {
  return launch_ex(L, dim3(rows), dim3(NORM_THREADS), 0, rmsnorm_kernel, a);
}

cudaError_t launch_qkv_norm_insert(const Launch& L, const QkvNormInsertArgs& a, int rows) {
  return launch_ex(L, dim3(rows), dim3(NORM_THREADS), 0, qkv_norm_insert_kernel, a);
}

int attention_smem_bytes(int head_dim) {
  return (ATTN_HEADS * head_dim + ATTN_KEYS * (head_dim + 1) + ATTN_HEADS * ATTN_KEYS) * 4;
}

cudaError_t attention_prepare(int head_dim) {
  const int smem = attention_smem_bytes(head_dim);
  if (head_dim == 128)
    return cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
  return cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int head_dim, int groups) {
  const dim3 grid(a.rows, groups, a.splits);
  const int smem = attention_smem_bytes(head_dim);
  if (head_dim == 128) return launch_ex(L, grid, dim3(ATTN_THREADS), smem, attn_kernel<128>, a);
  return launch_ex(L, grid, dim3(ATTN_THREADS), smem, attn_kernel<64>, a);
}

cudaError_t launch_router(const Launch& L, const RouterArgs& a) {
  const dim3 grid((a.E + 7) / 8, (a.rows + ROUTER_ROWS - 1) / ROUTER_ROWS);
  return launch_ex(L, grid, dim3(256), 0, router_kernel, a);
}

cudaError_t launch_topk(const Launch& L, const TopkArgs& a) {
  return launch_ex(L, dim3(1), dim3(TOPK_THREADS), 0, topk_kernel, a);
}

cudaError_t launch_final(const Launch& L, const FinalArgs& a) {
  const int ychunks = (a.H + 511) / 512;
  return launch_ex(L, dim3(a.rows, ychunks), dim3(256), 0, final_kernel, a);
}

}  // namespace mono
