// Dense MXFP8 GEMMs of many-row steps on the 5th-generation tensor cores ("Mono decode layer
// for DeepSeek-V4.1-Flash on MI355X", launch table K1/K2: the MXFP8 attention linears and the
// shared expert; section Design: e4m3 weights with 32 x 32 E8M0 block scales).
//
// tcgen05.mma kind::mxf8f6f4 (block-scaled, scale_vec::1X) multiplies the e4m3 weights,
// TMA-loaded as stored, by the step's activations, which their producers have already split
// into exact e4m3 hi + lo pairs under E8M0 block scales (the split and its layout are in
// common.cuh): a stage's activation operand is two bulk copies (the hi rows, the lo rows) and
// its scale image a third.  hi rows are MMA columns [0, 64), lo rows [64, 128); the readout
// adds the two accumulator columns of a row.
//
// A CTA computes one 128-row weight tile over one K slice; the ks CTAs of a cluster split K
// and add their partial tiles through distributed shared memory: the tile's 32-row blocks
// have owners (block b: rank b % ks), each CTA pushes every owner its rows of that owner's
// blocks with bulk shared-to-shared copies, and an owner adds its slots in rank order and
// writes the block out -- a warp per activation row and block, so that the block's 32
// outputs of a row can also be split for the next GEMM.  Warp 0 streams the stages (the
// first ring's worth of weights before the previous kernel has finished: weights do not
// depend on it), warp 1 issues the tensor-core copies and MMAs from one elected lane, warps
// 0-3 read the accumulator out of TMEM.  Every wait is bounded.
#include "kernels.h"
#include "tc_common.cuh"

namespace mono {
namespace {

using namespace tc;

constexpr int DT_M = 128;                   // weight rows per tile (the MMA's M)
constexpr int DT_KC = 128;                  // K elements per stage (128 e4m3 bytes a row)
constexpr int DT_NST = 4;                   // ring stages
constexpr int DT_SMAX = 8;                  // stages of one CTA's K slice at most
constexpr int DT_RMAX = 48;                 // activation rows at most
constexpr int DT_THREADS = 192;
constexpr int A_ST = DT_M * DT_KC;          // 16 KB
constexpr int B_ST = 128 * DT_KC;           // hi rows [0, 64), lo rows [64, 128): 16 KB
constexpr int IMG = 512;                    // one scale image (see tc_cp_img)
constexpr int EP_LD = DT_RMAX + 1;          // floats per row of the partial and receive tiles
constexpr int A_OFF = 0;
constexpr int B_OFF = A_OFF + DT_NST * A_ST;
constexpr int AIMG_OFF = B_OFF + DT_NST * B_ST;  // the K slice's weight-scale images
constexpr int BIMG_OFF = AIMG_OFF + DT_SMAX * IMG;
constexpr int PART_OFF = BIMG_OFF + DT_NST * IMG;      // the CTA's partial tile [128][EP_LD]
constexpr int RECV_OFF = PART_OFF + DT_M * EP_LD * 4;  // an owner's receive slots
constexpr int RECV_BYTES = 2 * DT_M * EP_LD * 4;
constexpr int SMEM_BYTES = RECV_OFF + RECV_BYTES + 1024;  // + alignment slack
// larger receive sets (16-way K splits) go to the A and B rings once the owner's are idle
constexpr int RECV_MAX = DT_NST * (A_ST + B_ST);
static_assert(B_OFF % 1024 == 0 && A_ST % 1024 == 0 && B_ST % 1024 == 0, "swizzle atoms");
static_assert(SPLIT_LO == 64 && SPLIT_STAGE_BYTES == B_ST && SPLIT_IMG_BYTES == IMG &&
                  DT_RMAX <= SPLIT_MAX_ROWS,
              "the activation split is a B stage as stored");
constexpr int TMEM_COLS = 256;  // D: 128 columns; scale columns from SC_COL
constexpr int SC_COL = 128;     // stage slot s: weight image at SC_COL + 8 s, activations + 4
static_assert(SC_COL + 8 * DT_NST <= TMEM_COLS, "TMEM columns");

// Instruction descriptor of kind::mxf8f6f4: A and B e4m3, E8M0 scales, both K-major, M = 128;
// N and the scale-byte selectors are or-ed in per MMA.
constexpr uint32_t DT_IDESC = (0u << 7) | (0u << 10) | (1u << 23) | ((uint32_t)(DT_M >> 4) << 24);

// The owner's blocks: a warp per (owned block, four activation rows), lane = the block's row
// (output column); the K slots added in rank order.  recv holds, per owned block, KS slots of
// brows rows (gate rows, then up rows) of EP_LD floats; with KS = 1 it is the partial tile.
// The K split and the output form are compile-time, so that the loop is straight-line code.
// dry: one task whose loads read whatever recv holds and whose stores are all off -- run by
// an idle warp while the MMAs stream, it brings this code into the SM's instruction caches
// (the kernel runs once per step; the epilogue's first task otherwise took ~2,400 cycles
// against ~650 for the next).
template <int KS, int EPI>
__device__ __forceinline__ void owner_epilogue(const DenseTcParams& p, const float* recv,
                                               int tile, int rank, int nown, int warp, int lane,
                                               bool dry) {
  constexpr bool SW = EPI == EPI_SWIGLU_F16;
  constexpr int brows = SW ? 64 : 32, up = (KS > 1 ? 32 : 64) * EP_LD, U = 4;
  const int R = p.rows, RQ = (R + U - 1) / U;
  const int ncols = SW ? p.swiglu_I : p.N;
  const int ntask = dry ? 1 : nown * RQ;
  for (int task = dry ? 0 : warp; task < ntask; task += DT_THREADS / 32) {
    const int lb = task / RQ, i0 = U * (task - lb * RQ);
    const int b = lb * KS + rank;
    const int col = (SW ? tile * 64 : tile * DT_M) + 32 * b + lane;
    const bool ok = !dry && col < ncols;
    const float* q0 =
        KS > 1 ? recv + (lb * KS * brows + lane) * EP_LD : recv + (32 * b + lane) * EP_LD;
    float rv[U];  // the residual first: its loads are in flight while the slots are added
    if (EPI == EPI_RESID_BF16)
#pragma unroll
      for (int u = 0; u < U; ++u)
        rv[u] = ok ? __bfloat162float(p.resid[(size_t)min(i0 + u, R - 1) * p.resid_ld + col])
                   : 0.0f;
    float s[U], su[U];
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] = su[u] = 0.0f;
#pragma unroll
    for (int sl = 0; sl < KS; ++sl)  // slots in rank order
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float* q = q0 + sl * brows * EP_LD + min(i0 + u, R - 1);
        s[u] += q[0];
        if (SW) su[u] += q[up];
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u;
      if (i >= R) break;
      float v = SW ? swiglu_clamped(s[u], su[u], p.clamp) : s[u];
      const size_t o = (size_t)i * p.out_ld + col;
      if (EPI == EPI_BF16) {
        if (ok) reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v);
      } else if (EPI == EPI_F16 || EPI == EPI_SWIGLU_F16) {
        const __half hv = bf16_as_f16_sat(v, dry ? nullptr : p.status);
        if (ok) reinterpret_cast<__half*>(p.out)[o] = hv;
        v = __half2float(hv);
        if (p.osplit) split_store1(v, ok, i, col, p.osplit, p.oimg);  // (the whole warp)
      } else if (EPI == EPI_RESID_BF16) {
        if (ok) reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(rv[u] + v);
      } else {
        if (ok) reinterpret_cast<float*>(p.out)[o] = v;
      }
    }
  }
}

template <int KS>
__device__ __forceinline__ void owner_epilogue_epi(const DenseTcParams& p, const float* recv,
                                                   int tile, int rank, int nown, int warp,
                                                   int lane, bool dry) {
  switch (p.epi) {
    case EPI_BF16:
      owner_epilogue<KS, EPI_BF16>(p, recv, tile, rank, nown, warp, lane, dry);
      break;
    case EPI_F16: owner_epilogue<KS, EPI_F16>(p, recv, tile, rank, nown, warp, lane, dry); break;
    case EPI_SWIGLU_F16:
      owner_epilogue<KS, EPI_SWIGLU_F16>(p, recv, tile, rank, nown, warp, lane, dry);
      break;
    case EPI_RESID_BF16:
      owner_epilogue<KS, EPI_RESID_BF16>(p, recv, tile, rank, nown, warp, lane, dry);
      break;
    default: owner_epilogue<KS, EPI_F32>(p, recv, tile, rank, nown, warp, lane, dry); break;
  }
}

// The owners' epilogue for the launch's K split (dry: see owner_epilogue).
__device__ __forceinline__ void owner_epilogue_ks(const DenseTcParams& p, const float* recv,
                                                  int tile, int rank, int nown, int warp,
                                                  int lane, bool dry) {
  switch (p.ksplit) {
    case 1: owner_epilogue_epi<1>(p, recv, tile, rank, nown, warp, lane, dry); break;
    case 2: owner_epilogue_epi<2>(p, recv, tile, rank, nown, warp, lane, dry); break;
    case 4: owner_epilogue_epi<4>(p, recv, tile, rank, nown, warp, lane, dry); break;
    case 8: owner_epilogue_epi<8>(p, recv, tile, rank, nown, warp, lane, dry); break;
    default: owner_epilogue_epi<16>(p, recv, tile, rank, nown, warp, lane, dry); break;
  }
}

__global__ void __launch_bounds__(DT_THREADS, 1)
    dense_tc_kernel(const __grid_constant__ CUtensorMap wmap, const DenseTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t afull[DT_NST], bfull[DT_NST], empty[DT_NST], done, drain;
  __shared__ __align__(8) uint64_t aimg_ready;  // the weight-scale images are written
  __shared__ __align__(8) uint64_t red_ready, red_full;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = p.ksplit;
  const uint32_t rank = ks > 1 ? cluster_ctarank() : 0u;
  const int tile = (int)blockIdx.x / ks;
  const int S = p.K / (ks * DT_KC);  // stages of this CTA's K slice
  const int kc0 = (int)rank * S;     // its first K stage
  const int R = p.rows, RP = (R + 7) & ~7;
  const bool sw = p.swiglu_I > 0;

  if (tid == 0) {
    for (int s = 0; s < DT_NST; ++s) {
      mbar_init(&afull[s], 1);
      mbar_init(&bfull[s], 1);
      mbar_init(&empty[s], 1);  // the MMA thread's commit
    }
    mbar_init(&done, 1);
    mbar_init(&drain, 1);
    mbar_init(&aimg_ready, 4);  // one arrival per image-writing warp
    mbar_init(&red_ready, min(sw ? 2 : 4, ks));  // each owner's rings are free to receive
    mbar_init(&red_full, 1);  // the owner's expect_tx arrival; the pushed blocks complete_tx
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&wmap);
  }
  if (warp == 1) tmem_alloc<TMEM_COLS>(&s_tmem);
  tc_fence_before();
  // every CTA of the cluster has initialised its barriers before any remote arrival
  if (ks > 1)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_trigger();

  // weight stage c of the slice into ring slot c % DT_NST (tile rows: 128 rows, or 64 gate
  // rows and the 64 up rows I further)
  auto issue_weights = [&](int c) {
    const int s = c % DT_NST;
    mbar_arrive_expect_tx(&afull[s], A_ST);
    const int x = (kc0 + c) * DT_KC;
    if (sw)
      tma_load_3d(smem + A_OFF + s * A_ST, &wmap, x, tile * 64, 0, &afull[s]);
    else
      tma_load_2d(smem + A_OFF + s * A_ST, &wmap, x, tile * DT_M, &afull[s]);
  };
  // activation stage c: its hi rows, lo rows and scale image, as the producer stored them
  auto issue_acts = [&](int c) {
    const int s = c % DT_NST;
    const uint32_t rows = (uint32_t)RP * 128;
    mbar_arrive_expect_tx(&bfull[s], 2 * rows + IMG);
    const uint8_t* src = p.bsplit + (size_t)(kc0 + c) * SPLIT_STAGE_BYTES;
    uint8_t* dst = smem + B_OFF + s * B_ST;
    bulk_load_g2s(dst, src, rows, &bfull[s]);
    bulk_load_g2s(dst + SPLIT_LO * 128, src + SPLIT_LO * 128, rows, &bfull[s]);
    bulk_load_g2s(smem + BIMG_OFF + s * IMG, p.bimg + (size_t)(kc0 + c) * SPLIT_IMG_BYTES, IMG,
                  &bfull[s]);
  };
  if (warp == 0 && elect_one())
    for (int c = 0; c < min(S, DT_NST); ++c) issue_weights(c);
  // the weight-scale images of the slice (lane l, column g = tile row l + 32 g: one 32 x 32
  // block's four K-block scales, the same for every lane)
  if (warp >= 2) {
    for (int c = warp - 2; c < S; c += 4) {
      uint32_t w[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        int row = sw ? (g < 2 ? tile * 64 + 32 * g : p.swiglu_I + tile * 64 + 32 * (g - 2))
                     : tile * DT_M + 32 * g;
        row = min(row, p.N - 1) / 32;
        w[g] = *reinterpret_cast<const uint32_t*>(p.scales + (size_t)row * p.scale_ld +
                                                  (kc0 + c) * 4);
      }
      *reinterpret_cast<uint4*>(smem + AIMG_OFF + c * IMG + lane * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_shared();  // read by the tensor core's copies
    __syncwarp();
    if (lane == 0) mbar_arrive(&aimg_ready);
  }
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------- stage loads (TMA, bulk)
    for (int c = 0; c < S; ++c) {
      const int s = c % DT_NST;
      if (c >= DT_NST && !warp_wait(&empty[s], ((c / DT_NST) - 1) & 1, p.status, abort)) break;
      if (elect_one()) {
        if (c >= DT_NST) issue_weights(c);
        issue_acts(c);
      }
      __syncwarp();
    }
  } else if (warp == 4) {
    // warm the epilogue's code while the stages stream (reads only; every store is off)
    owner_epilogue_ks(p, reinterpret_cast<const float*>(smem + A_OFF), tile, (int)rank, 1, 0,
                      lane, true);
  } else if (warp == 1) {
    // ------------------------------------------------------- scale copies and MMA issue
    const uint32_t idesc = DT_IDESC | ((uint32_t)(128 >> 3) << 17);
    bool ok = warp_wait(&aimg_ready, 0, p.status, abort);
    for (int c = 0; c < S && ok; ++c) {
      const int s = c % DT_NST;
      const uint32_t ph = (c / DT_NST) & 1;
      ok = warp_wait(&afull[s], ph, p.status, abort) && warp_wait(&bfull[s], ph, p.status, abort);
      if (!ok) break;
      const uint32_t sc = tmem + SC_COL + 8 * s;
      const uint32_t a0 = smem_u32(smem + A_OFF + s * A_ST), b0 = smem_u32(smem + B_OFF + s * B_ST);
      if (elect_one()) {
        tc_fence_after();
        tc_cp_img(sc, smem + AIMG_OFF + c * IMG);
        tc_cp_img(sc + 4, smem + BIMG_OFF + s * IMG);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 32 each; scale byte k of the stage's words
          tc_mma_mxf8(tmem, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k),
                      idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), sc, sc + 4,
                      (c > 0 || k > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (elect_one()) {
      tc_commit(ok ? &done : &drain);  // every MMA issued has completed at this arrival
      if (!ok) mbar_wait(&drain, 0, p.status, 100000000ull);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------- accumulator readout
  float* part = reinterpret_cast<float*>(smem + PART_OFF);  // [128][EP_LD]
  if (warp < 4) {
    if (warp_wait(&done, 0, p.status, abort)) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
      float* prow = part + (32 * warp + lane) * EP_LD;
      for (int x = 0; x * 32 < R; ++x) {
        uint32_t h[32], l[32];
        tc_ld32(taddr + 32 * x, h);
        tc_ld32(taddr + SPLIT_LO + 32 * x, l);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (32 * x + i < R) prow[32 * x + i] = __uint_as_float(h[i]) + __uint_as_float(l[i]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------- reduction and epilogue
  // 32-row blocks of the tile: NB = 4 (SwiGLU: 2 blocks of gate rows, each with the up rows
  // 64 on); block b belongs to rank b % ks, as that owner's block b / ks
  const int NB = sw ? 2 : 4;
  const int brows = sw ? 64 : 32;  // rows of a block's slot (gate rows, then up rows)
  const int nown = (int)rank < NB ? (NB - (int)rank + ks - 1) / ks : 0;
  const float* recv = part;
  // receive slots: the dedicated region, or the idle rings when they do not fit it (the same
  // choice on every CTA: rank 0 owns the most blocks)
  const int recv_max = (NB + ks - 1) / ks * ks * brows * EP_LD * 4;
  const bool in_rings = recv_max > RECV_BYTES;
  float* rbuf = reinterpret_cast<float*>(smem + (in_rings ? A_OFF : RECV_OFF));
  if (ks > 1) {
    fence_proxy_async_shared();  // the partial tile is read by bulk copies next
    __syncthreads();
    if (in_rings) {
      // owners: the rings are idle (this CTA's MMAs have completed); every peer may push
      if (nown > 0 && tid < ks)
        mbar_arrive_remote(mapa_shared(smem_u32(&red_ready), (uint32_t)tid));
      if (tid == 0 && !mbar_wait(&red_ready, 0, p.status)) *abort = 1;
      __syncthreads();
    }
    if (tid == 0 && !*abort) {
      mbar_arrive_expect_tx(&red_full, (uint32_t)(nown * ks * brows * EP_LD * 4));
      const uint32_t chunk = 32 * EP_LD * 4;
      for (int b = 0; b < NB; ++b) {
        const uint32_t o = (uint32_t)(b % ks), lb = (uint32_t)(b / ks);
        const uint32_t dst = mapa_shared(
            smem_u32(rbuf) + ((lb * ks + rank) * brows) * EP_LD * 4, o);
        const uint32_t bar = mapa_shared(smem_u32(&red_full), o);
        bulk_copy_s2s(dst, part + 32 * b * EP_LD, chunk, bar);
        if (sw) bulk_copy_s2s(dst + chunk, part + (64 + 32 * b) * EP_LD, chunk, bar);
      }
      bulk_commit();
    }
    if (!warp_wait(&red_full, 0, p.status, abort)) goto finish;
    recv = rbuf;
  }
  owner_epilogue_ks(p, recv, tile, (int)rank, nown, warp, lane, false);
finish:
  // A CTA leaves once its pushes have read its partial tile: every push into an owner has
  // landed when its receive barrier completes, before its epilogue, and a CTA that owns no
  // block receives none (so no cluster-wide handshake at the end).
  if (ks > 1 && tid == 0) bulk_wait_read();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<TMEM_COLS>(tmem);
  }
}

}  // namespace

cudaError_t dense_tc_prepare() {
  cudaError_t e =
      cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

int dense_tc_max_clusters(int ks) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks);
  cfg.blockDim = dim3(DT_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, dense_tc_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_dense_tc(const Launch& L, const CUtensorMap& wmap, const DenseTcParams& p) {
  const int ks = p.ksplit;
  if (p.rows < 1 || p.rows > DT_RMAX || ks < 1 || ks > 16 || (ks & (ks - 1)) ||
      p.K % (ks * DT_KC) || p.K / (ks * DT_KC) > DT_SMAX || p.K / (ks * DT_KC) < 1 ||
      p.n_tiles < 1 || !p.bsplit || !p.bimg || (p.osplit && !p.oimg))
    return cudaErrorInvalidValue;
  // an owner's receive slots fit its idle rings
  const int nb = p.swiglu_I > 0 ? 2 : 4, brows = p.swiglu_I > 0 ? 64 : 32;
  if (ks > 1 && (nb + ks - 1) / ks * ks * brows * EP_LD * 4 > RECV_MAX) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_tiles * ks);
  cfg.blockDim = dim3(DT_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = ks;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (L.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, dense_tc_kernel, wmap, p);
}

}  // namespace mono
