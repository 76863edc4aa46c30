// Instantiations and launcher of the MX block-scaled GEMM (mx_gemm.cuh).
#include "kernels.h"

namespace mono {

namespace {

// Ring depth per variant.  Dense matrices (few CTAs per SM) give each stage to two warps
// per M-tile; the routed experts fill the SMs with CTAs instead, except in small steps,
// whose few expert items also split K across a cluster.
template <int FMT, int NT, int KS>
struct Var;
template <> struct Var<8, 1, 2> { static constexpr int NSTAGE = 6; };
template <> struct Var<8, 2, 2> { static constexpr int NSTAGE = 6; };
template <> struct Var<8, 4, 2> { static constexpr int NSTAGE = 4; };
template <> struct Var<8, 6, 2> { static constexpr int NSTAGE = 3; };
template <> struct Var<4, 1, 1> { static constexpr int NSTAGE = 3; };  // 4 CTAs per SM
template <> struct Var<4, 1, 2> { static constexpr int NSTAGE = 4; };

template <int FMT, int NT, int KS>
constexpr int smem_of() {
  return GemmLayout<FMT, NT, Var<FMT, NT, KS>::NSTAGE, KS>::BYTES;
}

template <int FMT, int NT, int KS>
void* kernel_of(int* smem, int* threads) {
  *smem = smem_of<FMT, NT, KS>();
  *threads = gemm_threads(KS);
  return reinterpret_cast<void*>(&mx_gemm_kernel<FMT, NT, Var<FMT, NT, KS>::NSTAGE, KS>);
}

int ks_of(GemmVariant v) { return v.ks ? v.ks : (v.fmt == 8 ? 2 : 1); }

void* variant_kernel(GemmVariant v, int* smem, int* threads) {
  const int ks = ks_of(v);
  if (v.fmt == 8 && ks == 2) {
    switch (v.nt) {
      case 1: return kernel_of<8, 1, 2>(smem, threads);
      case 2: return kernel_of<8, 2, 2>(smem, threads);
      case 4: return kernel_of<8, 4, 2>(smem, threads);
      case 6: return kernel_of<8, 6, 2>(smem, threads);
      default: return nullptr;
    }
  }
  if (v.fmt == 4 && v.nt == 1) {
    if (ks == 1) return kernel_of<4, 1, 1>(smem, threads);
    if (ks == 2) return kernel_of<4, 1, 2>(smem, threads);
  }
  return nullptr;
}

cudaLaunchConfig_t config(const Launch& L, int grid, int threads, int smem, int cluster,
                          cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  int n = 0;
  if (L.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

}  // namespace

int gemm_smem_bytes(GemmVariant v) {
  int s = 0, t = 0;
  return variant_kernel(v, &s, &t) ? s : -1;
}

cudaError_t gemm_prepare(GemmVariant v) {
  int smem = 0, t = 0;
  void* k = variant_kernel(v, &smem, &t);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
}

int gemm_ctas_per_sm(GemmVariant v) {
  int smem = 0, t = 0, n = 0;
  void* k = variant_kernel(v, &smem, &t);
  if (!k) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, t, smem) != cudaSuccess) return 0;
  return n;
}

int gemm_max_clusters(GemmVariant v, int cluster) {
  int smem = 0, t = 0, n = 0;
  void* k = variant_kernel(v, &smem, &t);
  if (!k) return 0;
  cudaLaunchAttribute attr[2];
  const Launch L{nullptr, false};
  cudaLaunchConfig_t cfg = config(L, cluster * 1024, t, smem, cluster, attr);
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int FMT, int NT, int KS>
cudaError_t launch_variant(const cudaLaunchConfig_t& cfg, const CUtensorMap& map,
                           const CUtensorMap& smap, const GemmParams& p) {
  return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<FMT, NT, Var<FMT, NT, KS>::NSTAGE, KS>, map, smap,
                            p);
}

cudaError_t launch_gemm(const Launch& L, GemmVariant v, const CUtensorMap& map,
                        const CUtensorMap* smap, const GemmParams& p, int grid, int cluster) {
  int smem = 0, t = 0;
  if (!variant_kernel(v, &smem, &t)) return cudaErrorInvalidValue;
  if (p.sc_tma && (v.fmt != 4 || !smap)) return cudaErrorInvalidValue;
  // the large-step routed-expert variant: no cluster, and a work counter
  if (v.fmt == 4 && ks_of(v) == 1 && (cluster != 1 || p.ksplit != 1 || !p.item_next))
    return cudaErrorInvalidValue;
  const CUtensorMap& sm = smap ? *smap : map;  // unread unless p.sc_tma
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = config(L, grid, t, smem, cluster, attr);
  if (v.fmt == 8) {
    switch (v.nt) {
      case 1: return launch_variant<8, 1, 2>(cfg, map, sm, p);
      case 2: return launch_variant<8, 2, 2>(cfg, map, sm, p);
      case 4: return launch_variant<8, 4, 2>(cfg, map, sm, p);
      default: return launch_variant<8, 6, 2>(cfg, map, sm, p);
    }
  }
  return ks_of(v) == 2 ? launch_variant<4, 1, 2>(cfg, map, sm, p)
                        : launch_variant<4, 1, 1>(cfg, map, sm, p);
}

}  // namespace mono
