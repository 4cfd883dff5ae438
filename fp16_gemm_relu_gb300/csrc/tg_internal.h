// tg_internal.h — launchers shared between the C-ABI translation unit and the kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tg_gemm_kernel.cuh"

namespace tg {

struct GemmLaunch {
  CUtensorMap a, b, out;  // see tg_gemm_tc_kernel for the layouts each map describes
  GemmParams p;
  int grid;
  cudaStream_t stream;
};

// Shared-memory bytes and stage count of the kernel for a tile width.
int gemm_smem_bytes(int block_n);
int gemm_stages(int block_n);

// Launch tg_gemm_tc_kernel<block_n, out_f32>; returns the launch error (cudaSuccess if queued).
cudaError_t launch_gemm_bn256(const GemmLaunch& l, bool out_f32);
cudaError_t launch_gemm_bn192(const GemmLaunch& l, bool out_f32);
cudaError_t launch_gemm_bn128(const GemmLaunch& l, bool out_f32);

}  // namespace tg
