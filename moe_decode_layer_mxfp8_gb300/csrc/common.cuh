// Device helpers shared by the layer's kernels: PTX wrappers for mbarriers, TMA tile
// loads, cp.async, warp MMA and the MX element conversions; bounded waits that report
// through the device status word instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mono {

// Device status bits (mirrors MONO_STATUS_* in the public header).
constexpr int ST_UNMAPPED_PAGE = 1;
constexpr int ST_WAIT_TIMEOUT = 2;
constexpr int ST_BAD_ROUTE = 4;
constexpr int ST_F16_RANGE = 8;

// A pipeline wait that takes longer than this is treated as a fault (normal waits are
// microseconds).
constexpr uint64_t WAIT_BUDGET_NS = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- programmatic launch
// Wait until the previous kernel in the stream has completed and its writes are visible.
// A no-op when the kernel was launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of the given parity; gives up after WAIT_BUDGET_NS, sets the status
// bit and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint64_t budget_ns = WAIT_BUDGET_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > budget_ns) {
      atomicOr(status, ST_WAIT_TIMEOUT);
      return false;
    }
  }
  return true;
}

// --------------------------------------------------------------- clusters and DSMEM
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address, in the shared::cluster window, of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
// One arrival on an mbarrier that may live in another CTA of the cluster; releases this
// thread's (and, through the preceding barrier, its CTA's) earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}
// Raises an mbarrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Bulk copy global -> this CTA's shared memory, completing `bytes` on its mbarrier.
// Addresses and size multiples of 16.
__device__ __forceinline__ void bulk_load_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Bulk copy from this CTA's shared memory to (possibly) another CTA's of the cluster,
// completing `bytes` on the destination's mbarrier.  Addresses and size multiples of 16.
__device__ __forceinline__ void bulk_copy_s2s(uint32_t dst_cluster, const void* src,
                                              uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst_cluster), "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until this thread's committed bulk copies have read their sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
// Every thread of every CTA of the cluster arrives and waits (used once, at kernel start).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ------------------------------------------------------------------------- TMA / cp.async
// 2D tile load global -> shared through a tensor map; completion is counted in bytes on
// the mbarrier.  x is the innermost (byte) coordinate and must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// 16-byte copy; bytes beyond src_bytes (0..16) are zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// The mbarrier receives one arrival when all of this thread's earlier cp.async copies have
// landed (the arrival was counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// -------------------------------------------------------------------------- shared loads
__device__ __forceinline__ uint32_t lds32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// ---------------------------------------------------------------------------- MMA
// D = A * B (+ C) for one m16n8k16 tile, f16 operands, f32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ MX element decoding
// Four packed e2m1 pairs (one 32-bit word, element 2i in the low nibble of byte i) to
// eight f16 values: h[i] holds elements 2i (low half) and 2i+1 (high half).  Exact.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
// Four e4m3 bytes to four f16 values: h[0] = bytes 0,1 and h[1] = bytes 2,3.  Exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t (&h)[2]) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(w));
}
// f16x2 product, round to nearest, subnormals kept.
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// E8M0 scale byte to its f32 value 2^(e-127); 0 gives the subnormal 2^-127, 0xFF NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fc00000u : (e << 23));
  return __uint_as_float(bits);
}

// ----------------------------------------------------- e2m1 term split of activations
// The block-scaled FP4 tensor-core path takes an activation value v (a bf16 number) as a sum
// of ACT_TERMS e2m1 numbers, each 32-element block of a term under its own E8M0 scale:
// v = sum_t c_t * 2^(s_t - 127).  Term t's scale is the smallest power of two that brings
// the block's remaining residual within +-6 (the largest e2m1 magnitude), the codes round
// the residual to nearest (even), and the residual left after a term is exact in f32: every
// value is a bf16 number and each term removes a leading part of its bits.  Each term
// shrinks the block's largest residual at least threefold (the residual's magnitude a lies in
// (3s, 6s] and rounding leaves at most s), so eight leave less than 3^-8 of the block's
// largest magnitude; a bf16 value has 8 significant bits, and blocks of normal or
// heavy-tailed data come out exact (in a CPU simulation, 0 of 640,000 elements off; with
// log-normal magnitudes spread over e^+-4, 0.04 % off by at most 2.5e-8 of the block max).
constexpr int ACT_TERMS = 8;

// Two f32 values rounded to nearest-even e2m1 (saturating at +-6) in one byte, lo in the low
// nibble.
__device__ __forceinline__ uint32_t e2m1x2_of(float lo, float hi) {
  uint32_t out;
  asm("{\n .reg .b8 t;\n .reg .b16 w;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n"
      " mov.b16 w, {t, 0};\n cvt.u32.u16 %0, w;\n}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}
// E8M0 code of a term's scale: the smallest 2^(code - 127) with 6 * 2^(code - 127) >= a
// (127 for a = 0), within 1..253.
__device__ __forceinline__ uint32_t e2m1_term_code(float a) {
  if (!(a > 0.0f)) return 127u;
  const uint32_t b = __float_as_uint(a);
  const int code = (int)((b >> 23) & 0xFF) - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return (uint32_t)min(max(code, 1), 253);
}
__device__ __forceinline__ float e8m0_pow2(uint32_t code) { return __uint_as_float(code << 23); }
__device__ __forceinline__ float e8m0_inv_pow2(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}

// ----------------------------------------------------------------------- activations
// The layer's activations are bf16 at every rounding point.  Tensor-core operands are
// f16 copies of those bf16 values (exact for |v| in [2^-14, 65504]).
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ __half bf16_as_f16(float v) { return __float2half_rn(round_bf16(v)); }
// A bf16 value bound for an f16 tensor-core operand: magnitudes above f16's largest finite
// value are saturated to +-65504 and raise ST_F16_RANGE (below 2^-14 the copy is an f16
// subnormal, within 2^-25 of the value: no flag).  NaN passes through.
__device__ __forceinline__ float f16_range(float v, int* status) {
  if (fabsf(v) > 65504.0f) {
    if (status) atomicOr(status, ST_F16_RANGE);
    v = copysignf(65504.0f, v);
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// The largest of the warp's magnitudes (a >= 0, not NaN) in one reduction: non-negative
// floats order as their bit patterns.
__device__ __forceinline__ float warp_max_abs(float a) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
}

// Block-wide sum / max; `red` is a 32-float shared buffer; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  const float t = l < (int)(blockDim.x >> 5) ? red[l] : 0.0f;
  return warp_sum(t);
}
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  const float t = l < (int)(blockDim.x >> 5) ? red[l] : -INFINITY;
  return warp_max(t);
}

// 8 bf16 values in a 16-byte word <-> 8 floats
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  const __half2 h = __halves2half2(__float2half_rn(a), __float2half_rn(b));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// pack_f16x2 of two bf16 values through f16_range.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float a, float b, int* status) {
  return pack_f16x2(f16_range(a, status), f16_range(b, status));
}
__device__ __forceinline__ __half bf16_as_f16_sat(float v, int* status) {
  return __float2half_rn(f16_range(round_bf16(v), status));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace mono

namespace mono {

// The e2m1 term split of a 32-element block held 8 consecutive values per lane by an aligned
// group of 4 lanes (all 32 lanes of the warp call it): words[t] = this lane's 8 codes of term
// t (element 2i in the low nibble of byte i), codes[t] = the term's E8M0 scale code.
__device__ __forceinline__ void split_terms_x8(const float (&v)[8], uint32_t (&words)[ACT_TERMS],
                                               uint32_t (&codes)[ACT_TERMS]) {
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = v[i];
#pragma unroll
  for (int t = 0; t < ACT_TERMS; ++t) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(r[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const uint32_t code = e2m1_term_code(a);
    const float inv = e8m0_inv_pow2(code), sc = e8m0_pow2(code);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) w |= e2m1x2_of(r[2 * i] * inv, r[2 * i + 1] * inv) << (8 * i);
    uint32_t h[4];
    e2m1x8_to_f16x8(w, h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      r[2 * i] -= q.x * sc;
      r[2 * i + 1] -= q.y * sc;
    }
    words[t] = w;
    codes[t] = code;
  }
}

// The same split for a block held four consecutive values per lane by an aligned group of 8
// lanes: words[t] = this lane's 4 codes of term t in the low 16 bits (element 2i in the low
// nibble of byte i).
__device__ __forceinline__ void split_terms_x4(const float (&v)[4], uint32_t (&words)[ACT_TERMS],
                                               uint32_t (&codes)[ACT_TERMS]) {
  float r[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int t = 0; t < ACT_TERMS; ++t) {
    float a = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    const uint32_t code = e2m1_term_code(a);
    const float inv = e8m0_inv_pow2(code), sc = e8m0_pow2(code);
    const uint32_t w = e2m1x2_of(r[0] * inv, r[1] * inv) | (e2m1x2_of(r[2] * inv, r[3] * inv) << 8);
    uint32_t h0, h1;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    const float2 q0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
    const float2 q1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
    r[0] -= q0.x * sc, r[1] -= q0.y * sc, r[2] -= q1.x * sc, r[3] -= q1.y * sc;
    words[t] = w;
    codes[t] = code;
  }
}

// The same split for a 32-element block held one value per lane by a whole warp: words[t]
// = the codes of the 8-lane group this lane belongs to (lanes 8k .. 8k + 7 give bytes 0 .. 3
// of word k), codes[t] = the term's scale code.
__device__ __forceinline__ void split_terms_lane(float v, uint32_t (&words)[ACT_TERMS],
                                                 uint32_t (&codes)[ACT_TERMS]) {
  const int lane = threadIdx.x & 31;
  float r = v;
#pragma unroll
  for (int t = 0; t < ACT_TERMS; ++t) {
    const uint32_t code = e2m1_term_code(warp_max_abs(fabsf(r)));
    const uint32_t nib = e2m1x2_of(r * e8m0_inv_pow2(code), 0.0f) & 0xFu;
    uint32_t h[4];
    e2m1x8_to_f16x8(nib, h);
    r -= __low2float(*reinterpret_cast<const __half2*>(&h[0])) * e8m0_pow2(code);
    uint32_t w = nib << (4 * (lane & 7));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    w |= __shfl_xor_sync(0xffffffffu, w, 4);
    words[t] = w;
    codes[t] = code;
  }
}

}  // namespace mono

namespace mono {

// ------------------------------------------- e4m3 hi/lo split of a many-row activation
// The dense tensor-core GEMMs (k_dense_tc.cu) take an activation matrix (rows <= 48, K a
// multiple of 128) as an exact pair hi + lo of e4m3 numbers per element, under one E8M0
// scale per 32 consecutive K elements of a row (the scale puts the block's largest magnitude
// in [128, 256); hi = e4m3(v / s), lo = e4m3(v / s - hi), both rounded to nearest even).
// Every element at least 2^-10 of its block's maximum is reproduced exactly, the smaller ones
// to within 2^-17 of that maximum.  Its producers write it in the form the GEMM copies into
// shared memory as is: per 128-element K stage, 128 rows of 128 bytes (row j's hi codes in
// row j, its lo codes in row SPLIT_LO + j; 16-byte piece c of row n at piece c ^ (n % 8), the
// 128-byte swizzle), then per stage a 512-byte scale image (MMA column n's four K-block
// codes at byte (n % 32) * 16 + (n / 32) * 4 + kb).
constexpr int SPLIT_LO = 64;
constexpr int SPLIT_STAGE_BYTES = 128 * 128;
constexpr int SPLIT_IMG_BYTES = 512;
constexpr int SPLIT_MAX_ROWS = 48;

__device__ __forceinline__ uint32_t e4m3_block_code(float amax) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  return amax > 0.0f ? (uint32_t)max(eb - 7, 0) : 127u;
}
__device__ __forceinline__ float e8m0_inverse(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}
// v (already divided by the block scale) as hi and lo e4m3 codes.
__device__ __forceinline__ void e4m3_hilo(float v, uint32_t& hi, uint32_t& lo) {
  uint32_t h;
  asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}"
      : "=r"(h)
      : "f"(0.0f), "f"(v));
  uint32_t hf;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(hf) : "r"(h));
  const float hv = __low2float(*reinterpret_cast<const __half2*>(&hf));
  uint32_t l;
  asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}"
      : "=r"(l)
      : "f"(0.0f), "f"(v - hv));
  hi = h & 0xFFu;
  lo = l & 0xFFu;
}
// Byte offset of element k of row n (n = j for hi, SPLIT_LO + j for lo) in the split data.
__device__ __forceinline__ size_t split_off(int n, int k) {
  const int w = k & 127;
  return (size_t)(k >> 7) * SPLIT_STAGE_BYTES + n * 128 + ((((w >> 4) ^ (n & 7))) << 4) + (w & 15);
}
// Byte offset of the code of K block k / 32 for MMA column n in the scale images.
__device__ __forceinline__ size_t split_img_off(int n, int k) {
  return (size_t)(k >> 7) * SPLIT_IMG_BYTES + (n & 31) * 16 + (n >> 5) * 4 + ((k >> 5) & 3);
}

// One 32-element block held one element per lane by a whole warp (lane = k % 32): every lane
// calls it; lanes with !in give 0 and store nothing.
__device__ __forceinline__ void split_store1(float v, bool in, int row, int k, uint8_t* data,
                                             uint8_t* img) {
  const uint32_t code = e4m3_block_code(warp_max_abs(in ? fabsf(v) : 0.0f));
  uint32_t hi, lo;
  e4m3_hilo(in ? v * e8m0_inverse(code) : 0.0f, hi, lo);
  if (in) {
    data[split_off(row, k)] = (uint8_t)hi;
    data[split_off(SPLIT_LO + row, k)] = (uint8_t)lo;
    if ((threadIdx.x & 31) == 0) {
      img[split_img_off(row, k)] = (uint8_t)code;
      img[split_img_off(SPLIT_LO + row, k)] = (uint8_t)code;
    }
  }
}
// A block held eight consecutive elements per lane by an aligned group of four lanes (k8 =
// the first element, a multiple of 8): every lane of the warp calls it.
__device__ __forceinline__ void split_store8(const float (&v)[8], bool in, int row, int k8,
                                             uint8_t* data, uint8_t* img) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, in ? fabsf(v[i]) : 0.0f);
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  const uint32_t code = e4m3_block_code(a);
  const float inv = e8m0_inverse(code);
  uint32_t h[2] = {0, 0}, l[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t hb, lb;
    e4m3_hilo(in ? v[i] * inv : 0.0f, hb, lb);
    h[i >> 2] |= hb << (8 * (i & 3));
    l[i >> 2] |= lb << (8 * (i & 3));
  }
  if (in) {
    *reinterpret_cast<uint2*>(data + split_off(row, k8)) = make_uint2(h[0], h[1]);
    *reinterpret_cast<uint2*>(data + split_off(SPLIT_LO + row, k8)) = make_uint2(l[0], l[1]);
    if ((k8 & 31) == 0) {
      img[split_img_off(row, k8)] = (uint8_t)code;
      img[split_img_off(SPLIT_LO + row, k8)] = (uint8_t)code;
    }
  }
}

// The e4m3 split of a block held four consecutive elements per lane by an aligned group of 8
// lanes (k4 = the first element, a multiple of 4): every lane of the warp calls it.
__device__ __forceinline__ void split_store4(const float (&v)[4], bool in, int row, int k4,
                                             uint8_t* data, uint8_t* img) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) a = fmaxf(a, in ? fabsf(v[i]) : 0.0f);
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  const uint32_t code = e4m3_block_code(a);
  const float inv = e8m0_inverse(code);
  uint32_t h = 0, l = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t hb, lb;
    e4m3_hilo(in ? v[i] * inv : 0.0f, hb, lb);
    h |= hb << (8 * i);
    l |= lb << (8 * i);
  }
  if (in) {
    *reinterpret_cast<uint32_t*>(data + split_off(row, k4)) = h;
    *reinterpret_cast<uint32_t*>(data + split_off(SPLIT_LO + row, k4)) = l;
    if ((k4 & 31) == 0) {
      img[split_img_off(row, k4)] = (uint8_t)code;
      img[split_img_off(SPLIT_LO + row, k4)] = (uint8_t)code;
    }
  }
}

}  // namespace mono
