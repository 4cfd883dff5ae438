// Instantiation of the tcgen05 kernel for 192-wide output tiles (its own translation unit
// so that the tile widths compile in parallel).
#include "tg_internal.h"

namespace tg {

namespace {
template <bool OUT_F32, bool GENERAL>
cudaError_t launch_one(const GemmLaunch& l) {
  auto kern = tg_gemm_tc_kernel<192, OUT_F32, GENERAL>;
  constexpr int smem = TileCfg<192>::kSmemBytes;
  // per device and per function; cheap enough to repeat on every launch
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<l.grid, kThreads, smem, l.stream>>>(l.a, l.b, l.out, l.p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_bn192(const GemmLaunch& l, bool out_f32) {
  const bool general = l.p.a_mn || l.p.b_k;
  if (out_f32) return general ? launch_one<true, true>(l) : launch_one<true, false>(l);
  return general ? launch_one<false, true>(l) : launch_one<false, false>(l);
}

}  // namespace tg
