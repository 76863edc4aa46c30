// Row-wise kernels of the layer: the attention-front and FFN-seam RMSNorms, the q/kv norms
// with the fp8 KV-cache insert, and the final residual combine ("Mono decode layer for
// DeepSeek-V4.1-Flash on MI355X", launch table: K1 "q/kv norms, the KV insert", K2 "the FFN
// seam").  Every thread issues all of its global loads before it uses any of them, so a row
// costs about one memory latency.
#include <cuda_fp8.h>

#include "kernels.h"

namespace mono {

namespace {

constexpr int NORM_THREADS = 256;
constexpr int NORM_CHUNKS = 4;  // 8-element chunks per thread: rows up to 8192 wide

// RMSNorm: CTA (row r, 1024-column slice y) writes output elements 4q .. 4q + 3, q =
// RMS_THREADS y + t, from thread t, after computing the whole row's sum of squares itself (each
// of the row's CTAs reads the whole row; the row is in L2).  Spreading a row over several CTAs,
// and a 32-element block over 8 lanes, shortens the splits' serial per-block steps.
constexpr int RMS_THREADS = 256;
constexpr int RMS_COLS = RMS_THREADS * 4;  // output columns per CTA
constexpr int RMS_CHUNKS = 4;  // 8-element chunks per thread of the sum: rows up to 8192 wide

__device__ __forceinline__ void bf16x4_to_f32(uint2 v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x << 16), f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16), f[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

// Output elements i = 4q .. 4q + 3 of row r: v = bf16(x * inv * gamma) stored as its f16 copy,
// plus the optional e2m1 term split and e4m3 hi/lo split of v.  Every lane of the warp calls
// it (the splits' block maxima are shuffles).  Not inlined, so that the kernel's call before
// griddepcontrol.wait (live false: nothing is stored) brings exactly this code into the
// instruction caches: the kernel runs once per step and its code is otherwise cold.
__device__ __noinline__ void rms_out4(const NormArgs& a, int r, int q, uint2 xq, uint2 gq,
                                      float inv, bool live) {
  const int i = q * 4;
  const bool in = live && i < a.dim;
  float v[4];
  {
    float f[4], g[4];
    bf16x4_to_f32(xq, f);
    bf16x4_to_f32(gq, g);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = in ? round_bf16(f[j] * inv * g[j]) : 0.0f;
  }
  if (in)
    *reinterpret_cast<uint2*>(a.out + (size_t)r * a.out_ld + i) =
        make_uint2(pack_f16x2_sat(v[0], v[1], a.status), pack_f16x2_sat(v[2], v[3], a.status));
  if (a.terms) {  // (a whole warp's elements are in range or out of it: dim % 256 == 0)
    uint32_t words[ACT_TERMS], codes[ACT_TERMS];
    split_terms_x4(v, words, codes);
    if (in) {
      const int piece = (i & 255) >> 5;  // 16-byte piece (= 32-element block) in its row
      const size_t base = ((size_t)r * (a.dim / 256) + (i >> 8)) * ACT_TERMS;
#pragma unroll
      for (int t = 0; t < ACT_TERMS; ++t) {
        *reinterpret_cast<uint16_t*>(a.terms + (base + t) * 128 + ((piece ^ t) << 4) +
                                     ((i & 31) >> 1)) = (uint16_t)words[t];
        if ((i & 31) == 0) a.term_scales[(base + t) * 8 + piece] = (uint8_t)codes[t];
      }
    }
  }
  if (a.e4_data) split_store4(v, in, r, i, a.e4_data, a.e4_img);
}

__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_kernel(const __grid_constant__ NormArgs a) {
  __shared__ float red[32];
  pdl_trigger();
  const int r = blockIdx.x, tid = threadIdx.x;
  const int q = blockIdx.y * RMS_THREADS + tid;  // this thread's 4 output elements
  const bool mine_in = q * 4 < a.dim;
  const __nv_bfloat16* x = a.in + (size_t)r * a.in_ld;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint2 zero2 = make_uint2(0u, 0u);
  // gamma is constant: fetched before the wait (with the warm-up of the output code)
  const uint2 gq = mine_in ? *reinterpret_cast<const uint2*>(a.gamma + q * 4) : zero2;
  if (a.warm) rms_out4(a, r, q, zero2, zero2, 0.0f, false);
  pdl_wait();
  // the whole row in 8-element chunks for the sum, and this thread's own 4 elements
  uint4 xv[RMS_CHUNKS], rv[RMS_CHUNKS];
#pragma unroll
  for (int c = 0; c < RMS_CHUNKS; ++c) {
    const int i = (c * RMS_THREADS + tid) * 8;
    xv[c] = i < a.dim ? *reinterpret_cast<const uint4*>(x + i) : zero;
  }
  uint2 mine = mine_in ? *reinterpret_cast<const uint2*>(x + q * 4) : zero2;
  if (a.resid) {
    // residual first: h = bf16(x + resid).  The f32 sum of two bf16 values rounds to the
    // same bf16 as their exact sum (an f32 rounding error only arises when the exponents
    // differ by more than 16, far from any bf16 rounding midpoint).
    const __nv_bfloat16* rr = a.resid + (size_t)r * a.resid_ld;
#pragma unroll
    for (int c = 0; c < RMS_CHUNKS; ++c) {
      const int i = (c * RMS_THREADS + tid) * 8;
      rv[c] = i < a.dim ? *reinterpret_cast<const uint4*>(rr + i) : zero;
    }
    const uint2 rmine = mine_in ? *reinterpret_cast<const uint2*>(rr + q * 4) : zero2;
#pragma unroll
    for (int c = 0; c < RMS_CHUNKS; ++c) {
      float f[8], g[8];
      bf16x8_to_f32(xv[c], f);
      bf16x8_to_f32(rv[c], g);
      xv[c].x = pack_bf16x2(f[0] + g[0], f[1] + g[1]);
      xv[c].y = pack_bf16x2(f[2] + g[2], f[3] + g[3]);
      xv[c].z = pack_bf16x2(f[4] + g[4], f[5] + g[5]);
      xv[c].w = pack_bf16x2(f[6] + g[6], f[7] + g[7]);
    }
    float f[4], g[4];
    bf16x4_to_f32(mine, f);
    bf16x4_to_f32(rmine, g);
    mine = make_uint2(pack_bf16x2(f[0] + g[0], f[1] + g[1]), pack_bf16x2(f[2] + g[2], f[3] + g[3]));
    if (mine_in) *reinterpret_cast<uint2*>(a.sum_out + (size_t)r * a.sum_ld + q * 4) = mine;
  }
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < RMS_CHUNKS; ++c) {
    float f[8];
    bf16x8_to_f32(xv[c], f);  // (zero past the row's end)
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)a.dim + a.eps);
  rms_out4(a, r, q, mine, gq, inv, true);
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
// The two norms are independent: CTA (row, 0) normalises q (thread t owns q chunks t,
// t + 256, ...: 8 values each) and CTA (row, 1) kv (thread t owns kv chunk t) and inserts it.
constexpr int QKV_CHUNKS = 2;  // q latents up to 4096 wide
__global__ void __launch_bounds__(NORM_THREADS) qkv_norm_insert_kernel(QkvNormInsertArgs a) {
  __shared__ float red[32];
  pdl_trigger();
  const int r = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* row = a.qkv + (size_t)r * (a.q_rank + a.kv_dim);
  if (blockIdx.y == 0) {
    // ------------------------------------------------------------------------ q norm
    uint4 qv[QKV_CHUNKS], qg[QKV_CHUNKS];
#pragma unroll
    for (int c = 0; c < QKV_CHUNKS; ++c) {  // gamma before the wait
      const int i = (c * NORM_THREADS + tid) * 8;
      if (i < a.q_rank) qg[c] = *reinterpret_cast<const uint4*>(a.gq + i);
    }
    pdl_wait();
#pragma unroll
    for (int c = 0; c < QKV_CHUNKS; ++c) {
      const int i = (c * NORM_THREADS + tid) * 8;
      if (i < a.q_rank) qv[c] = *reinterpret_cast<const uint4*>(row + i);
    }
    float ssq = 0.0f;
#pragma unroll
    for (int c = 0; c < QKV_CHUNKS; ++c) {
      if ((c * NORM_THREADS + tid) * 8 < a.q_rank) {
        float f[8];
        bf16x8_to_f32(qv[c], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) ssq = fmaf(f[j], f[j], ssq);
      }
    }
    ssq = block_sum(ssq, red);
    const float invq = 1.0f / sqrtf(ssq / (float)a.q_rank + a.eps);
#pragma unroll
    for (int c = 0; c < QKV_CHUNKS; ++c) {
      const int i = (c * NORM_THREADS + tid) * 8;
      const bool in = i < a.q_rank;
      float v[8];
      if (in) {
        float f[8], g[8];
        bf16x8_to_f32(qv[c], f);
        bf16x8_to_f32(qg[c], g);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = round_bf16(f[j] * invq * g[j]);
        uint4 o;
        o.x = pack_f16x2_sat(v[0], v[1], a.status);
        o.y = pack_f16x2_sat(v[2], v[3], a.status);
        o.z = pack_f16x2_sat(v[4], v[5], a.status);
        o.w = pack_f16x2_sat(v[6], v[7], a.status);
        *reinterpret_cast<uint4*>(a.qlatn + (size_t)r * a.q_rank + i) = o;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.0f;
      }
      if (a.e4_data) split_store8(v, in, r, i, a.e4_data, a.e4_img);  // (every lane)
    }
    return;
  }
  // ------------------------------------------------------------------ kv norm, insert
  const bool has_kv = tid * 8 < a.kv_dim;  // kv_dim <= 2048: one chunk per thread at most
  uint4 kv = {}, kg = {};
  // the gamma and the step's inputs (position, page table) before the wait
  if (has_kv) kg = *reinterpret_cast<const uint4*>(a.gkv + tid * 8);
  const int p = a.positions[r];
  const int pb = p < 0 ? -1 : page_of(a.block_table, a.max_blocks, a.n_req, a.num_blocks,
                                     a.row_req[r], p, a.block_size);
  pdl_wait();
  if (has_kv) kv = *reinterpret_cast<const uint4*>(row + a.q_rank + tid * 8);
  float sskv = 0.0f;
  float kf[8];
  bf16x8_to_f32(kv, kf);
  if (has_kv)
#pragma unroll
    for (int j = 0; j < 8; ++j) sskv = fmaf(kf[j], kf[j], sskv);
  sskv = block_sum(sskv, red);
  const float invkv = 1.0f / sqrtf(sskv / (float)a.kv_dim + a.eps);
  float kn[8], g[8];
  bf16x8_to_f32(kg, g);
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    kn[j] = round_bf16(kf[j] * invkv * g[j]);
    amax = fmaxf(amax, fabsf(kn[j]));
  }
  if (has_kv) {
    uint4 o;
    o.x = pack_bf16x2(kn[0], kn[1]);
    o.y = pack_bf16x2(kn[2], kn[3]);
    o.z = pack_bf16x2(kn[4], kn[5]);
    o.w = pack_bf16x2(kn[6], kn[7]);
    *reinterpret_cast<uint4*>(a.kvn + (size_t)r * a.kv_dim + tid * 8) = o;
  } else {
    amax = 0.0f;
  }
  amax = block_max(amax, red);
  if (p < 0) return;
  if (pb < 0) {
    if (tid == 0) atomicOr(a.status, ST_UNMAPPED_PAGE);
    return;
  }
  uint8_t* rec = a.cache + (size_t)pb * a.stride_block + (size_t)(p % a.block_size) * a.stride_tok;
  const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  if (has_kv) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = __nv_cvt_float2_to_fp8x2(make_float2(kn[2 * j] / s, kn[2 * j + 1] / s),
                                      __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint2*>(rec + tid * 8) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
  }
  if (tid == 0) *reinterpret_cast<float*>(rec + a.kv_dim) = s;
}

// out = bf16(h + y_shared + sum_j w_j y_j) in slot order; pad rows copy x.  CTA = one row and
// FINAL_COLS columns; each thread owns 8 consecutive columns.
constexpr int FINAL_THREADS = 256;
constexpr int FINAL_COLS = FINAL_THREADS * 8;
constexpr int FINAL_MAX_K = 8;
__global__ void __launch_bounds__(FINAL_THREADS) final_kernel(FinalArgs a) {
  pdl_trigger();
  const int r = blockIdx.x;
  const int c = blockIdx.y * FINAL_COLS + threadIdx.x * 8;
  const bool pad = a.positions[r] < 0;  // a step input: read before the wait
  const bool in = c < a.H;
  const size_t o = (size_t)r * a.H + (in ? c : 0);
  // Read before the wait as well: the routing and h.  The routed-expert kernels let their
  // dependents in only after their own wait, when the top-k (and every earlier kernel, h's
  // writer included) has completed; the expert outputs y_s and y_r are read after it.
  int pos[FINAL_MAX_K];
  float wj[FINAL_MAX_K];
#pragma unroll
  for (int j = 0; j < FINAL_MAX_K; ++j) {
    pos[j] = j < a.k && !pad ? a.slot_pos[r * a.k + j] : -1;
    wj[j] = j < a.k && !pad ? a.topk_w[r * a.k + j] : 0.0f;
  }
  const uint4 hv = in ? *reinterpret_cast<const uint4*>((pad ? a.x : a.h) + o) : uint4{};
  pdl_wait();
  if (!in) return;
  if (pad) {
    *reinterpret_cast<uint4*>(a.out + o) = hv;  // (x: the layer input)
    return;
  }
  const float4 s0 = *reinterpret_cast<const float4*>(a.ys + o);
  const float4 s1 = *reinterpret_cast<const float4*>(a.ys + o + 4);
  float4 y0[FINAL_MAX_K], y1[FINAL_MAX_K];
#pragma unroll
  for (int j = 0; j < FINAL_MAX_K; ++j) {
    if (pos[j] >= 0) {
      const float* yr = a.yr + (size_t)pos[j] * a.H + c;
      y0[j] = *reinterpret_cast<const float4*>(yr);
      y1[j] = *reinterpret_cast<const float4*>(yr + 4);
    }
  }
  float v[8];
  bf16x8_to_f32(hv, v);
  v[0] += s0.x, v[1] += s0.y, v[2] += s0.z, v[3] += s0.w;
  v[4] += s1.x, v[5] += s1.y, v[6] += s1.z, v[7] += s1.w;
#pragma unroll
  for (int j = 0; j < FINAL_MAX_K; ++j) {
    if (pos[j] >= 0) {
      v[0] = fmaf(wj[j], y0[j].x, v[0]), v[1] = fmaf(wj[j], y0[j].y, v[1]);
      v[2] = fmaf(wj[j], y0[j].z, v[2]), v[3] = fmaf(wj[j], y0[j].w, v[3]);
      v[4] = fmaf(wj[j], y1[j].x, v[4]), v[5] = fmaf(wj[j], y1[j].y, v[5]);
      v[6] = fmaf(wj[j], y1[j].z, v[6]), v[7] = fmaf(wj[j], y1[j].w, v[7]);
    }
  }
  uint4 out;
  out.x = pack_bf16x2(v[0], v[1]);
  out.y = pack_bf16x2(v[2], v[3]);
  out.z = pack_bf16x2(v[4], v[5]);
  out.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(a.out + o) = out;
}

}  // namespace

cudaError_t launch_rmsnorm(const Launch& L, const NormArgs& a, int rows) {
  if (a.dim > RMS_CHUNKS * RMS_THREADS * 8 || a.dim % 8) return cudaErrorInvalidValue;
  const int slices = (a.dim + RMS_COLS - 1) / RMS_COLS;
  return launch_ex(L, dim3(rows, slices), dim3(RMS_THREADS), 0, rmsnorm_kernel, a);
}

cudaError_t launch_qkv_norm_insert(const Launch& L, const QkvNormInsertArgs& a, int rows) {
  if (a.q_rank > QKV_CHUNKS * NORM_THREADS * 8 || a.kv_dim > NORM_THREADS * 8)
    return cudaErrorInvalidValue;
  return launch_ex(L, dim3(rows, 2), dim3(NORM_THREADS), 0, qkv_norm_insert_kernel, a);
}

cudaError_t launch_final(const Launch& L, const FinalArgs& a) {
  const int ychunks = (a.H + FINAL_COLS - 1) / FINAL_COLS;
  return launch_ex(L, dim3(a.rows, ychunks), dim3(FINAL_THREADS), 0, final_kernel, a);
}

// One thread waits, through the pipelines' bounded mbarrier wait, on a barrier that nothing
// completes: the wait gives up after budget_ns, raises ST_WAIT_TIMEOUT and the kernel returns.
__global__ void wait_timeout_kernel(int* status, unsigned long long budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  (void)mbar_wait(&bar, 0, status, budget_ns);
}

cudaError_t launch_wait_timeout(cudaStream_t stream, int* status, unsigned long long budget_ns) {
  wait_timeout_kernel<<<1, 1, 0, stream>>>(status, budget_ns);
  return cudaGetLastError();
}

}  // namespace mono
