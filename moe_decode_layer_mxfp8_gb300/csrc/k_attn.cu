// Sliding-window attention over the fp8 KV cache, split over the window with a
// log-sum-exp combine ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", launch table
// K2: "split attention, combine"; draft layers: non-causal rows 192 wide).
//
// CTA = (row, latent slice g, split s).  The cached kv_dim latent is both key and value; head
// h reads slice h / heads_per_slice, so one CTA serves the slice's (up to 16) heads against
// the split's share of the row's window.  Scores and the weighted sum of values run on the
// tensor cores (m16n8k16, f16 operands, f32 accumulation):
//   S[h, t] = (q_h . c_t) * s_t / sqrt(head_dim)      (c_t: e4m3 codes, exact in f16)
//   o_h     = sum_t p[h, t] * s_t * c_t,  p = exp(S - m)
// with p * s_t / s_max rounded to f16 for the second product (s_max, the split's largest
// scale, keeps that operand in f16's normal range) and s_max applied to the f32 result.
// The last split to finish a (row, slice) combines: o = sum_s e^(m_s - M) o_s / sum_s
// e^(m_s - M) l_s.
#include "kernels.h"

namespace mono {

namespace {

constexpr int ATTN_THREADS = 512;  // 16 warps: one 8-key score tile, head or 8-dim output tile each
constexpr int ATTN_KEYS = 128;     // keys per split at most
constexpr int ATTN_HEADS = 16;     // heads per latent slice at most (= the MMA's M)

template <int DH>
struct AttnSmem {
  static constexpr int QS = DH + 8;          // f16 row stride of q and codes (ldmatrix spread)
  static constexpr int PS = ATTN_KEYS + 8;   // f16 row stride of the probabilities
  static constexpr int SS = ATTN_KEYS + 4;   // f32 row stride of the scores
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + ATTN_HEADS * QS * 2;
  static constexpr int P_OFF = K_OFF + ATTN_KEYS * QS * 2;
  static constexpr int S_OFF = P_OFF + ATTN_HEADS * PS * 2;
  static constexpr int SC_OFF = S_OFF + ATTN_HEADS * SS * 4;
  static constexpr int BYTES = SC_OFF + ATTN_KEYS * 4;
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ int page_of(const int* table, int max_blocks, int n_req, long long nb,
                                       int q, int t, int bs) {
  const int lb = t / bs;
  if (q < 0 || q >= n_req || t < 0 || lb >= max_blocks) return -1;
  const int pb = table[(size_t)q * max_blocks + lb];
  return (pb < 0 || pb >= nb) ? -1 : pb;
}

// Writes this CTA's heads of output row r from a staged f32 copy (values already rounded to
// bf16): o in f16, and o's e4m3 split (every thread calls it).
template <int DH>
__device__ void store_o_staged(const AttnArgs& a, const float* stage, int r, int h0, int hpg) {
  const int QW = a.n_q * DH, items = hpg * (DH / 8);
  for (int base = 0; base < items; base += ATTN_THREADS) {
    const int idx = base + (int)threadIdx.x;
    const bool in = idx < items;
    const int h = in ? idx / (DH / 8) : 0, d = in ? 8 * (idx - h * (DH / 8)) : 0;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = in ? stage[h * DH + d + i] : 0.0f;
    if (in)
      *reinterpret_cast<uint4*>(a.o + (size_t)r * QW + (h0 + h) * DH + d) =
          make_uint4(pack_f16x2_sat(v[0], v[1], a.status), pack_f16x2_sat(v[2], v[3], a.status),
                     pack_f16x2_sat(v[4], v[5], a.status), pack_f16x2_sat(v[6], v[7], a.status));
    split_store8(v, in, r, (h0 + h) * DH + d, a.e4_data, a.e4_img);
  }
}

template <int DH>
__global__ void __launch_bounds__(ATTN_THREADS) attn_kernel(AttnArgs a) {
  using L = AttnSmem<DH>;
  extern __shared__ __align__(16) uint8_t sm[];
  __half* qs = reinterpret_cast<__half*>(sm + L::Q_OFF);   // [16][QS]
  __half* kc = reinterpret_cast<__half*>(sm + L::K_OFF);   // [128][QS] codes
  __half* pf = reinterpret_cast<__half*>(sm + L::P_OFF);   // [16][PS] p * s_t / s_max
  float* sc = reinterpret_cast<float*>(sm + L::S_OFF);     // [16][SS] scores
  float* ks = reinterpret_cast<float*>(sm + L::SC_OFF);    // [128] per-key scales
  __shared__ float s_m[ATTN_HEADS], s_l[ATTN_HEADS], red[32];
  __shared__ const uint8_t* s_rec[ATTN_KEYS];
  __shared__ int s_flag;
  pdl_trigger();
  // Everything up to griddepcontrol.wait reads only the step's inputs (positions, requests,
  // page table), none of which a kernel of the layer writes.
  const int r = blockIdx.x, g = blockIdx.y, sp = blockIdx.z, S = a.splits;
  const int G = a.kv_dim / DH, hpg = a.n_q / G, h0 = g * hpg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QW = a.n_q * DH;
  const int p = a.positions[r];
  if (p < 0) {  // pad row: attention output is zero
    pdl_wait();
    if (sp == 0) {
      if (a.e4_data) {
        for (int i = tid; i < hpg * DH; i += ATTN_THREADS) sc[i] = 0.0f;
        __syncthreads();
        store_o_staged<DH>(a, sc, r, h0, hpg);
      } else {
        for (int i = tid; i < hpg * DH; i += ATTN_THREADS)
          a.o[(size_t)r * QW + h0 * DH + i] = __float2half(0.0f);
      }
    }
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
  const int ntp = (nt + 15) & ~15;  // keys padded to whole MMA k-steps
  // the split's KV records (null: padding or an unmapped page)
  for (int t = tid; t < ntp; t += ATTN_THREADS) {
    const uint8_t* rec = nullptr;
    if (t < nt) {
      const int pos = t0 + t;
      const int pb = page_of(a.block_table, a.max_blocks, a.n_req, a.num_blocks, req, pos,
                             a.block_size);
      if (pb >= 0)
        rec = a.cache + (size_t)pb * a.stride_block + (size_t)(pos % a.block_size) * a.stride_tok;
      else
        atomicOr(a.status, ST_UNMAPPED_PAGE);
    }
    s_rec[t] = rec;
  }
  __syncthreads();
  pdl_wait();

  // q of the slice's heads (rows >= hpg zero), keys' codes and scales of the split
  constexpr int QC = DH / 8;  // 8-element chunks per head
  for (int idx = tid; idx < ATTN_HEADS * QC; idx += ATTN_THREADS) {
    const int h = idx / QC, c = idx - h * QC;
    uint4 o = {0u, 0u, 0u, 0u};
    if (h < hpg) {
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.q + (size_t)r * QW + (h0 + h) * DH + c * 8), f);
      o = make_uint4(pack_f16x2_sat(f[0], f[1], a.status), pack_f16x2_sat(f[2], f[3], a.status),
                     pack_f16x2_sat(f[4], f[5], a.status), pack_f16x2_sat(f[6], f[7], a.status));
    }
    *reinterpret_cast<uint4*>(qs + h * L::QS + c * 8) = o;
  }
  constexpr int KC = DH / 16;  // 16-byte code chunks per key
  constexpr int NL = ATTN_KEYS * KC / ATTN_THREADS;  // chunks per thread at most
  uint4 raw[NL];
  float scl[NL];
#pragma unroll
  for (int u = 0; u < NL; ++u) {  // every load in flight before the first use
    const int idx = tid + u * ATTN_THREADS;
    const int t = idx / KC, c = idx - t * KC;
    const uint8_t* rec = t < ntp ? s_rec[t] : nullptr;
    raw[u] = rec ? *reinterpret_cast<const uint4*>(rec + g * DH + c * 16) : make_uint4(0u, 0u, 0u, 0u);
    scl[u] = rec ? *reinterpret_cast<const float*>(rec + a.kv_dim) : 0.0f;
  }
  float smax = 0.0f;
#pragma unroll
  for (int u = 0; u < NL; ++u) {
    const int idx = tid + u * ATTN_THREADS;
    const int t = idx / KC, c = idx - t * KC;
    if (t < ntp) {
      uint4 lo16, hi16;
      uint32_t h2[2];
      e4m3x4_to_f16x4(raw[u].x, h2); lo16.x = h2[0]; lo16.y = h2[1];
      e4m3x4_to_f16x4(raw[u].y, h2); lo16.z = h2[0]; lo16.w = h2[1];
      e4m3x4_to_f16x4(raw[u].z, h2); hi16.x = h2[0]; hi16.y = h2[1];
      e4m3x4_to_f16x4(raw[u].w, h2); hi16.z = h2[0]; hi16.w = h2[1];
      *reinterpret_cast<uint4*>(kc + t * L::QS + c * 16) = lo16;
      *reinterpret_cast<uint4*>(kc + t * L::QS + c * 16 + 8) = hi16;
      if (c == 0) ks[t] = scl[u];
      smax = fmaxf(smax, scl[u]);
    }
  }
  smax = block_max(smax, red);  // (its barriers also publish q, codes and scales)
  const float inv_smax = smax > 0.0f ? 1.0f / smax : 0.0f;
  const float qk_scale = 1.0f / sqrtf((float)DH);
  const int gq = lane >> 2, cq = lane & 3;

  // scores: warps take 8-key tiles round robin
  for (int nt8 = warp; nt8 < ntp / 8; nt8 += ATTN_THREADS / 32) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      uint32_t af[4], bf[2];
      ldsm_x4(af, qs + (lane & 15) * L::QS + kk * 16 + (lane >> 4) * 8);
      ldsm_x2(bf, kc + (nt8 * 8 + (lane & 7)) * L::QS + kk * 16 + ((lane >> 3) & 1) * 8);
      mma_f16_acc(acc, af, bf[0], bf[1]);
    }
    const int t = nt8 * 8 + 2 * cq;
    const float s0 = ks[t] * qk_scale, s1 = ks[t + 1] * qk_scale;
    sc[gq * L::SS + t] = t < nt ? acc[0] * s0 : -INFINITY;
    sc[gq * L::SS + t + 1] = t + 1 < nt ? acc[1] * s1 : -INFINITY;
    sc[(gq + 8) * L::SS + t] = t < nt ? acc[2] * s0 : -INFINITY;
    sc[(gq + 8) * L::SS + t + 1] = t + 1 < nt ? acc[3] * s1 : -INFINITY;
  }
  __syncthreads();
  // per-head softmax statistics; probabilities (times s_t / s_max) to f16
  for (int h = warp; h < ATTN_HEADS; h += ATTN_THREADS / 32) {
    float m = -INFINITY;
    for (int t = lane; t < nt; t += 32) m = fmaxf(m, sc[h * L::SS + t]);
    m = warp_max(m);
    float l = 0.0f;
    for (int t = lane; t < ntp; t += 32) {
      const float e = t < nt ? expf(sc[h * L::SS + t] - m) : 0.0f;
      l += e;
      pf[h * L::PS + t] = __float2half_rn(e * ks[t] * inv_smax);
    }
    l = warp_sum(l);
    if (lane == 0) s_m[h] = m, s_l[h] = l;
  }
  __syncthreads();
  // o = P' . codes: warps take 8-dim tiles
  const int PW = DH + ATTN_PART_HEAD;
  for (int dt = warp; dt < DH / 8; dt += ATTN_THREADS / 32) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kk = 0; kk < ntp / 16; ++kk) {
      uint32_t af[4], bf[2];
      ldsm_x4(af, pf + (lane & 15) * L::PS + kk * 16 + (lane >> 4) * 8);
      ldsm_x2_trans(bf, kc + (kk * 16 + (lane & 15)) * L::QS + dt * 8);
      mma_f16_acc(acc, af, bf[0], bf[1]);
    }
    const int d = dt * 8 + 2 * cq;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int h = gq + 8 * half;
      if (h >= hpg) continue;
      const float v0 = acc[2 * half] * smax, v1 = acc[2 * half + 1] * smax;
      if (S == 1) {
        const float il = 1.0f / s_l[h];
        if (a.e4_data) {  // staged in the scores' memory (free since the softmax)
          sc[h * DH + d] = round_bf16(v0 * il);
          sc[h * DH + d + 1] = round_bf16(v1 * il);
        } else {
          *reinterpret_cast<uint32_t*>(a.o + (size_t)r * QW + (h0 + h) * DH + d) =
              pack_f16x2_sat(round_bf16(v0 * il), round_bf16(v1 * il), a.status);
        }
      } else {
        float* part = a.part + (((size_t)r * a.n_q + h0 + h) * S + sp) * PW;
        *reinterpret_cast<float2*>(part + ATTN_PART_HEAD + d) = make_float2(v0, v1);
        if (d == 0) part[0] = s_m[h], part[1] = s_l[h];
      }
    }
  }
  if (S == 1) {
    if (a.e4_data) {
      __syncthreads();
      store_o_staged<DH>(a, sc, r, h0, hpg);
    }
    return;
  }
  __threadfence();
  __syncthreads();
  int* ctr = a.counters + r * G + g;
  if (tid == 0) s_flag = atomicAdd(ctr, 1) == S - 1;
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  // a thread per (head, 4 dims); every split's values are in flight at once
  for (int idx = tid; idx < hpg * (DH / 4); idx += ATTN_THREADS) {
    const int h = idx / (DH / 4), d = 4 * (idx - h * (DH / 4));
    const float* base = a.part + ((size_t)r * a.n_q + h0 + h) * S * PW;
    float ms[ATTN_MAX_SPLITS], ls[ATTN_MAX_SPLITS];
    float4 os[ATTN_MAX_SPLITS];
#pragma unroll
    for (int s = 0; s < ATTN_MAX_SPLITS; ++s) {
      if (s < S) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + s * PW));
        ms[s] = ml.x;
        ls[s] = ml.y;
        os[s] = __ldcg(reinterpret_cast<const float4*>(base + s * PW + ATTN_PART_HEAD + d));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < ATTN_MAX_SPLITS; ++s)
      if (s < S) M = fmaxf(M, ms[s]);
    float n0 = 0.0f, n1 = 0.0f, n2 = 0.0f, n3 = 0.0f, den = 0.0f;
#pragma unroll
    for (int s = 0; s < ATTN_MAX_SPLITS; ++s) {
      if (s < S) {
        const float f = ms[s] == -INFINITY ? 0.0f : expf(ms[s] - M);
        n0 = fmaf(f, os[s].x, n0);
        n1 = fmaf(f, os[s].y, n1);
        n2 = fmaf(f, os[s].z, n2);
        n3 = fmaf(f, os[s].w, n3);
        den = fmaf(f, ls[s], den);
      }
    }
    if (a.e4_data) {
      sc[h * DH + d] = round_bf16(n0 / den);
      sc[h * DH + d + 1] = round_bf16(n1 / den);
      sc[h * DH + d + 2] = round_bf16(n2 / den);
      sc[h * DH + d + 3] = round_bf16(n3 / den);
    } else {
      *reinterpret_cast<uint2*>(a.o + (size_t)r * QW + (h0 + h) * DH + d) =
          make_uint2(pack_f16x2_sat(round_bf16(n0 / den), round_bf16(n1 / den), a.status),
                     pack_f16x2_sat(round_bf16(n2 / den), round_bf16(n3 / den), a.status));
    }
  }
  if (a.e4_data) {
    __syncthreads();
    store_o_staged<DH>(a, sc, r, h0, hpg);
  }
  if (tid == 0) *ctr = 0;
}

}  // namespace

cudaError_t attention_prepare(int head_dim) {
  if (head_dim == 128)
    return cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnSmem<128>::BYTES);
  return cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              AttnSmem<64>::BYTES);
}

cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int head_dim, int groups) {
  const dim3 grid(a.rows, groups, a.splits);
  if (head_dim == 128)
    return launch_ex(L, grid, dim3(ATTN_THREADS), AttnSmem<128>::BYTES, attn_kernel<128>, a);
  return launch_ex(L, grid, dim3(ATTN_THREADS), AttnSmem<64>::BYTES, attn_kernel<64>, a);
}

}  // namespace mono
