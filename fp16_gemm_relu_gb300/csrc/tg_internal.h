// tg_internal.h — launchers shared between the C-ABI translation unit and the kernel units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tg_gemm_kernel.cuh"
#include "tg_gemm_relu.h"

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

// CTA-pair kernel (256 x 256 tiles; l.grid must be even, l.p counts pair tiles).
cudaError_t launch_gemm_pair(const GemmLaunch& l, bool out_f32);
// The CTA-pair kernel with A read in place through row classes (float32 output only; l.a is
// unused, l.p.cls_* describe the classes).
cudaError_t launch_gemm_pair_cls(const AClassMaps& cls, const GemmLaunch& l);
// Clusters of two that can be resident at once on the current device.
cudaError_t gemm_pair_max_clusters(int* out);

// Makes the runtime's context for `dev` current in the calling thread (once per thread), so that
// driver-API calls (tensor-map encoding) work from any host thread.
cudaError_t bind_thread_context(int dev);

// Records `e` as the calling thread's last CUDA error (what tg_last_cuda_error reports) and
// returns TG_ERR_CUDA, for entry points defined outside tg_api.cu.
tg_status record_cuda_error(cudaError_t e);

// Current device's SM count and error word (checks the device; sets up library state).
tg_status device_info(int* sm_count, unsigned int** err);

// Address of the device error word that kernels set when a pipeline wait runs out.
cudaError_t error_word_address(unsigned int** out);

// Stream-ordered scratch of `bytes` from the library's pool on the current device; give it back
// with cudaFreeAsync on the same stream.  TG_ERR_NO_WORKSPACE if the pool cannot supply it.
tg_status scratch_alloc(size_t bytes, cudaStream_t stream, void** out);

// cuTensorMapEncodeTiled from the driver (false if the driver does not provide it).
bool tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn);

// Deterministic split-K reduction: C = fp16(epi(sum_s W[s])) (see tg_splitk_reduce_kernel).
// p supplies the epilogue (act, bias, residual, ldr) and the shape (M, N).
cudaError_t launch_splitk_reduce(const float* ws, int64_t ldw, int64_t split_stride, int splits,
                                 void* C, int64_t ldc, const GemmParams& p, int num_sms,
                                 cudaStream_t stream);

}  // namespace tg
