// Instantiations and launcher of the MX block-scaled GEMM (mx_gemm.cuh).
#include "kernels.h"

namespace mono {

namespace {

// Ring depth per variant, chosen so that two or three CTAs fit on one SM.
template <int FMT, int NT>
struct Stages;
template <> struct Stages<8, 1> { static constexpr int value = 6; };
template <> struct Stages<8, 2> { static constexpr int value = 6; };
template <> struct Stages<8, 4> { static constexpr int value = 4; };
template <> struct Stages<8, 6> { static constexpr int value = 4; };
template <> struct Stages<4, 1> { static constexpr int value = 4; };

template <int FMT, int NT>
constexpr int smem_of() {
  return GemmLayout<FMT, NT, Stages<FMT, NT>::value>::BYTES;
}

template <int FMT, int NT>
void* kernel_of() {
  return reinterpret_cast<void*>(&mx_gemm_kernel<FMT, NT, Stages<FMT, NT>::value>);
}

void* variant_kernel(GemmVariant v, int* smem) {
  if (v.fmt == 8) {
    switch (v.nt) {
      case 1: *smem = smem_of<8, 1>(); return kernel_of<8, 1>();
      case 2: *smem = smem_of<8, 2>(); return kernel_of<8, 2>();
      case 4: *smem = smem_of<8, 4>(); return kernel_of<8, 4>();
      case 6: *smem = smem_of<8, 6>(); return kernel_of<8, 6>();
      default: return nullptr;
    }
  }
  if (v.fmt == 4 && v.nt == 1) {
    *smem = smem_of<4, 1>();
    return kernel_of<4, 1>();
  }
  return nullptr;
}

cudaLaunchConfig_t config(const Launch& L, int grid, int smem, int cluster,
                          cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(GEMM_THREADS);
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
  int s = 0;
  return variant_kernel(v, &s) ? s : -1;
}

cudaError_t gemm_prepare(GemmVariant v) {
  int smem = 0;
  void* k = variant_kernel(v, &smem);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
}

int gemm_ctas_per_sm(GemmVariant v) {
  int smem = 0, n = 0;
  void* k = variant_kernel(v, &smem);
  if (!k) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, GEMM_THREADS, smem) != cudaSuccess)
    return 0;
  return n;
}

int gemm_max_clusters(GemmVariant v, int cluster) {
  int smem = 0, n = 0;
  void* k = variant_kernel(v, &smem);
  if (!k) return 0;
  cudaLaunchAttribute attr[2];
  const Launch L{nullptr, false};
  cudaLaunchConfig_t cfg = config(L, cluster * 1024, smem, cluster, attr);
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemm(const Launch& L, GemmVariant v, const CUtensorMap& map,
                        const GemmParams& p, int grid, int cluster) {
  int smem = 0;
  if (!variant_kernel(v, &smem)) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = config(L, grid, smem, cluster, attr);
  if (v.fmt == 8) {
    switch (v.nt) {
      case 1: return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<8, 1, Stages<8, 1>::value>, map, p);
      case 2: return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<8, 2, Stages<8, 2>::value>, map, p);
      case 4: return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<8, 4, Stages<8, 4>::value>, map, p);
      default: return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<8, 6, Stages<8, 6>::value>, map, p);
    }
  }
  return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<4, 1, Stages<4, 1>::value>, map, p);
}

}  // namespace mono
