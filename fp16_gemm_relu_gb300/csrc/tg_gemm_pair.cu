// Instantiation and launch of the CTA-pair (cta_group::2) kernel, 256 x 256 output tiles.
#include "tg_internal.h"

namespace tg {

namespace {
template <bool OUT_F32, bool GENERAL>
cudaError_t launch_one(const GemmLaunch& l) {
  auto kern = tg_gemm_pair_kernel<OUT_F32, GENERAL>;
  constexpr int smem = PairCfgT<GENERAL ? 1 : 2>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<l.grid, kThreads, smem, l.stream>>>(l.a, l.b, l.out, l.p);  // grid is a multiple of 2
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_pair(const GemmLaunch& l, bool out_f32) {
  if (l.grid <= 0 || (l.grid & 1)) return cudaErrorInvalidConfiguration;
  const bool general = l.p.a_mn || l.p.b_k;
  if (out_f32) return general ? launch_one<true, true>(l) : launch_one<true, false>(l);
  return general ? launch_one<false, true>(l) : launch_one<false, false>(l);
}

cudaError_t gemm_pair_max_clusters(int* out) {
  auto kern = tg_gemm_pair_kernel<false, false>;
  constexpr int smem = PairCfgFwd::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, reinterpret_cast<const void*>(kern), &cfg);
}

}  // namespace tg
