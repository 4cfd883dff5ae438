// tg_no_alloc.cu — tg_gemm_relu_f16_splitk_noalloc: the split-K path with its float32
// workspace in a fixed array of device memory that belongs to the library, for callers that
// cannot allocate while they run a GEMM.  It launches the same split-K GEMM kernel and the
// same ordered reduction as tg_gemm_relu_f16; only where the workspace comes from differs.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "tg_gemm_relu.h"
#include "tg_internal.h"

// The workspace.  In host code this name only stands for the symbol; it is not a device
// address.  The address that kernels use comes from cudaGetSymbolAddress at set-up.
static __device__ __align__(256) unsigned char g_tg_static_workspace[TG_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBlockN = 256;
constexpr int kPanel = 16;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

struct StaticSetup {
  bool done = false;
  tg_status status = TG_OK;
  float* workspace = nullptr;     // device address of g_tg_static_workspace on this device
  unsigned int* err = nullptr;    // device error word
  int sm_count = 0;
};

StaticSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One-time set-up for the current device: checks the device and looks up device addresses.
// Allocates nothing.  Every CUDA failure is recorded for tg_last_cuda_error.
tg_status setup_current_device(StaticSetup** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tg::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
  if ((e = tg::bind_thread_context(dev)) != cudaSuccess) return tg::record_cuda_error(e);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  StaticSetup& s = g_setup[dev];
  if (!s.done) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return tg::record_cuda_error(e);
    if (major != 10 || minor != 3) {
      s.status = TG_ERR_UNSUPPORTED_DEVICE;
    } else {
      void* ws = nullptr;
      if ((e = cudaGetSymbolAddress(&ws, g_tg_static_workspace)) != cudaSuccess)
        return tg::record_cuda_error(e);
      unsigned int* err = nullptr;
      if ((e = tg::error_word_address(&err)) != cudaSuccess) return tg::record_cuda_error(e);
      s.workspace = static_cast<float*>(ws);
      s.err = err;
      s.sm_count = sms;
      s.status = TG_OK;
    }
    s.done = true;
  }
  *out = &s;
  return s.status;
}

// True when splits x M x ldw float32 values fit in the fixed workspace.  Each product is
// checked by division first, so no intermediate can overflow (M and ldw may each approach
// 2^31).
bool fits_workspace(int64_t splits, int64_t M, int64_t ldw) {
  const uint64_t limit = TG_STATIC_WORKSPACE_BYTES;
  const uint64_t row = static_cast<uint64_t>(ldw) * 4u;  // ldw < 2^31: no overflow
  if (row == 0 || row > limit) return false;
  if (static_cast<uint64_t>(M) > limit / row) return false;
  const uint64_t per_split = static_cast<uint64_t>(M) * row;  // <= limit
  if (per_split == 0) return true;
  return static_cast<uint64_t>(splits) <= limit / per_split;
}

CUresult encode(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, CUtensorMapDataType dt,
                const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box) {
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

extern "C" tg_status tg_gemm_relu_f16_splitk_noalloc(const void* A, const void* B, void* C,
                                                     int64_t M, int64_t N, int64_t K,
                                                     int64_t lda, int64_t ldb, int64_t ldc,
                                                     int epilogue_flag, int split_k,
                                                     tg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int64_t max_dim = (int64_t{1} << 31) - 1024;
  if (M < 0 || N < 0 || K < 0 || split_k < 0) return TG_ERR_INVALID_ARG;
  if (M > max_dim || N > max_dim || K > max_dim) return TG_ERR_INVALID_ARG;
  if (epilogue_flag != TG_EPILOGUE_NONE && epilogue_flag != TG_EPILOGUE_RELU)
    return TG_ERR_INVALID_ARG;
  if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) ||
      ldc < std::max<int64_t>(1, N))
    return TG_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))))
    return TG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(C) & 1u) return TG_ERR_MISALIGNED;
  if (M == 0 || N == 0) return TG_OK;
  const bool operands_aligned =
      ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) == 0 &&
      lda % 8 == 0 && ldb % 8 == 0;
  if (K > 0 && !operands_aligned) return TG_ERR_MISALIGNED;

  const int64_t kblocks = cdiv(K, tg::kBK);
  const int64_t want = std::max<int64_t>(split_k == 0 ? 2 : split_k, 1);
  const int64_t kbps = kblocks > 0 ? cdiv(kblocks, std::min(want, kblocks)) : 1;
  const int64_t splits = kblocks > 0 ? cdiv(kblocks, kbps) : 1;  // every split is non-empty
  const int64_t ldw = cdiv(N, 4) * 4;
  if (K > 0 && !fits_workspace(splits, M, ldw)) return TG_ERR_NO_WORKSPACE;

  StaticSetup* su = nullptr;
  tg_status st = setup_current_device(&su);
  if (st != TG_OK) return st;
  if (K == 0) {  // the empty sum: C = +0
    const cudaError_t e =
        cudaMemset2DAsync(C, size_t(ldc) * 2, 0, size_t(N) * 2, size_t(M), stream);
    return e == cudaSuccess ? TG_OK : tg::record_cuda_error(e);
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!tg::tensor_map_encoder(&enc)) return tg::record_cuda_error(cudaErrorNotSupported);

  tg::GemmLaunch L;
  std::memset(&L, 0, sizeof(L));
  const cuuint64_t a_dims[2] = {cuuint64_t(K), cuuint64_t(M)};
  const cuuint64_t a_str[1] = {cuuint64_t(lda) * 2};
  const cuuint32_t a_box[2] = {tg::kBK, tg::kBM};
  const cuuint64_t b_dims[2] = {cuuint64_t(N), cuuint64_t(K)};
  const cuuint64_t b_str[1] = {cuuint64_t(ldb) * 2};
  const cuuint32_t b_box[2] = {64, tg::kBK};
  const cuuint64_t w_dims[3] = {cuuint64_t(N), cuuint64_t(M), cuuint64_t(splits)};
  const cuuint64_t w_str[2] = {cuuint64_t(ldw) * 4, cuuint64_t(ldw) * 4 * cuuint64_t(M)};
  const cuuint32_t w_box[3] = {32, 32, 1};
  if (encode(enc, &L.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, 2, a_dims, a_str, a_box) !=
          CUDA_SUCCESS ||
      encode(enc, &L.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, 2, b_dims, b_str, b_box) !=
          CUDA_SUCCESS ||
      encode(enc, &L.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, su->workspace, 3, w_dims, w_str,
             w_box) != CUDA_SUCCESS)
    return tg::record_cuda_error(cudaErrorInvalidValue);

  const int64_t tiles_m = cdiv(M, tg::kBM);
  const int64_t tiles_n = cdiv(N, kBlockN);
  const int64_t units = tiles_m * tiles_n * splits;
  if (units >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
  tg::GemmParams& p = L.p;
  p.tiles_m = static_cast<int>(tiles_m);
  p.tiles_n = static_cast<int>(tiles_n);
  p.num_kb = static_cast<int>(kblocks);
  p.kb_per_split = static_cast<int>(kbps);
  p.splits = static_cast<int>(splits);
  p.units = static_cast<int>(units);
  p.panel_m = static_cast<int>(std::min<int64_t>(kPanel, tiles_m));
  p.act = epilogue_flag == TG_EPILOGUE_RELU ? tg::kActRelu : tg::kActNone;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.debug_flags = 0;
  p.timeout_ns = kTimeoutNs;
  p.err = su->err;
  L.grid = static_cast<int>(std::min<int64_t>(units, su->sm_count));
  L.stream = stream;
  cudaError_t e = tg::launch_gemm_bn256(L, /*out_f32=*/true);
  if (e != cudaSuccess) return tg::record_cuda_error(e);
  e = tg::launch_splitk_reduce(su->workspace, ldw, M * ldw, static_cast<int>(splits), C, ldc, p,
                               su->sm_count, stream);
  if (e != cudaSuccess) return tg::record_cuda_error(e);
  return TG_OK;
}
