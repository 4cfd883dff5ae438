// Instantiation and launch of the CTA-pair (cta_group::2) kernel, 256 x 256 output tiles.
#include "tg_internal.h"

namespace tg {

namespace {
template <bool OUT_F32, bool A_MN, bool B_K>
cudaError_t launch_one(const GemmLaunch& l) {
  auto kern = tg_gemm_pair_kernel<OUT_F32, A_MN, B_K>;
  constexpr int smem = PairCfgFwd::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<l.grid, kThreads, smem, l.stream>>>(l.a, l.b, l.out, l.p);  // grid is a multiple of 2
  return cudaGetLastError();
}

template <bool OUT_F32>
cudaError_t launch_layout(const GemmLaunch& l) {
  if (l.p.a_mn) return l.p.b_k ? launch_one<OUT_F32, true, true>(l) : launch_one<OUT_F32, true, false>(l);
  return l.p.b_k ? launch_one<OUT_F32, false, true>(l) : launch_one<OUT_F32, false, false>(l);
}
}  // namespace

cudaError_t launch_gemm_pair(const GemmLaunch& l, bool out_f32) {
  if (l.grid <= 0 || (l.grid & 1)) return cudaErrorInvalidConfiguration;
  return out_f32 ? launch_layout<true>(l) : launch_layout<false>(l);
}

cudaError_t launch_gemm_pair_cls(const AClassMaps& cls, const GemmLaunch& l) {
  if (l.grid <= 0 || (l.grid & 1)) return cudaErrorInvalidConfiguration;
  auto kern = tg_gemm_pair_cls_kernel<kARowClasses>;
  constexpr int smem = PairCfgFwd::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<l.grid, kThreads, smem, l.stream>>>(cls, l.b, l.out, l.p);
  return cudaGetLastError();
}

cudaError_t gemm_pair_max_clusters(int* out) {
  auto kern = tg_gemm_pair_kernel<false, false, false>;
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
