// Instantiations of the tensor-core tile region kernels for fp16 (one
// translation unit per activation type so the library builds in parallel).
#include <mutex>

#include "dense_launch.cuh"

namespace ds {

cudaError_t launch_dense_f16(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                             cudaStream_t st, bool pdl) {
  return launch_dense_t<__half>(r, a, xh, xl, st, pdl);
}

cudaError_t prepare_dense_f16(int max_smem) { return prepare_dense_t<__half>(max_smem); }

// Clusters of `size` tile CTAs (max_smem bytes of shared memory each: one CTA
// per SM, as every tile CTA) that the current device holds at once -- a
// cluster lives within one GPC, so e.g. clusters of 7 leave SMs of every GPC
// idle.  0 if the query fails.  Cached per device.
int dense_cluster_capacity(int size, int max_smem) {
  static std::mutex mu;
  static int cache[64][9];
  static bool init = false;
  int dev = 0;
  if (size < 1 || size > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  if (cache[dev][size] >= 0) return cache[dev][size];
  auto k = &dense_region_kernel<Region::FfnDown, __half, false, 1>;
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(size * 64));
    cfg.blockDim = dim3(dense_threads(false, 1));
    cfg.dynamicSmemBytes = (size_t)max_smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)size;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
      n = 0;
      (void)cudaGetLastError();
    }
  }
  cache[dev][size] = n;
  return n;
}

}  // namespace ds
