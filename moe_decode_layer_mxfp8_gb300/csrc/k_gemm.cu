// Instantiations and launcher of the MX block-scaled GEMM (mx_gemm.cuh).
#include "kernels.h"

namespace mono {

namespace {

// Ring depth and K-shares per variant: dense matrices (few CTAs per SM) give each stage to
// two warps per M-tile; the routed experts fill the SMs with CTAs instead.
template <int FMT, int NT>
struct Var;
template <> struct Var<8, 1> { static constexpr int NSTAGE = 6, KS = 2; };
template <> struct Var<8, 2> { static constexpr int NSTAGE = 6, KS = 2; };
template <> struct Var<8, 4> { static constexpr int NSTAGE = 4, KS = 2; };
template <> struct Var<8, 6> { static constexpr int NSTAGE = 3, KS = 2; };
template <> struct Var<4, 1> { static constexpr int NSTAGE = 4, KS = 1; };

template <int FMT, int NT>
constexpr int smem_of() {
  return GemmLayout<FMT, NT, Var<FMT, NT>::NSTAGE, Var<FMT, NT>::KS>::BYTES;
}

template <int FMT, int NT>
void* kernel_of() {
  return reinterpret_cast<void*>(&mx_gemm_kernel<FMT, NT, Var<FMT, NT>::NSTAGE, Var<FMT, NT>::KS>);
}

void* variant_kernel(GemmVariant v, int* smem, int* threads) {
  if (v.fmt == 8) {
    switch (v.nt) {
      case 1: *smem = smem_of<8, 1>(); *threads = gemm_threads(Var<8, 1>::KS); return kernel_of<8, 1>();
      case 2: *smem = smem_of<8, 2>(); *threads = gemm_threads(Var<8, 2>::KS); return kernel_of<8, 2>();
      case 4: *smem = smem_of<8, 4>(); *threads = gemm_threads(Var<8, 4>::KS); return kernel_of<8, 4>();
      case 6: *smem = smem_of<8, 6>(); *threads = gemm_threads(Var<8, 6>::KS); return kernel_of<8, 6>();
      default: return nullptr;
    }
  }
  if (v.fmt == 4 && v.nt == 1) {
    *smem = smem_of<4, 1>();
    *threads = gemm_threads(Var<4, 1>::KS);
    return kernel_of<4, 1>();
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

template <int FMT, int NT>
cudaError_t launch_variant(const cudaLaunchConfig_t& cfg, const CUtensorMap& map,
                           const GemmParams& p) {
  return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<FMT, NT, Var<FMT, NT>::NSTAGE, Var<FMT, NT>::KS>,
                            map, p);
}

cudaError_t launch_gemm(const Launch& L, GemmVariant v, const CUtensorMap& map,
                        const GemmParams& p, int grid, int cluster) {
  int smem = 0, t = 0;
  if (!variant_kernel(v, &smem, &t)) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = config(L, grid, t, smem, cluster, attr);
  if (v.fmt == 8) {
    switch (v.nt) {
      case 1: return launch_variant<8, 1>(cfg, map, p);
      case 2: return launch_variant<8, 2>(cfg, map, p);
      case 4: return launch_variant<8, 4>(cfg, map, p);
      default: return launch_variant<8, 6>(cfg, map, p);
    }
  }
  return launch_variant<4, 1>(cfg, map, p);
}

}  // namespace mono
