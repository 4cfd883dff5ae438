// tg_gemm_w4a16_f16: the int4-weight dequantising GEMM (see tg_gemm_w4.cuh for the kernel).
#include <algorithm>
#include <atomic>
#include <cstring>

#include "tg_gemm_w4.cuh"
#include "tg_internal.h"

namespace {

// Smallest M for which the decode-first plan is chosen by default, per weight format.  On
// GB300 (L2 flushed, fused against decode-first, with the decode pass at 28.6 us for
// 8192 x 8192): int4 at M = 256 65.6 / 78.8 us (N = K = 8192) and 180 / 214 us
// (N = 28672); at M = 512 92.2 / 91.5, 38.2 / 38.5 (N = K = 4096), 254 / 249 (N = 28672) and
// 287 / 258 (K = 28672); at M = 640 166 / 114.  NF4, whose fused decode costs more: at
// M = 384 97.4 / 91.8; at M = 256 79.9 / 79.6, 45.1 / 37.0 (N = K = 4096) and 193 / 218
// (N = 28672).
constexpr int64_t kDecodeFirstMinMInt4 = 512;
constexpr int64_t kDecodeFirstMinMNf4 = 384;


int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int BMT, int FMT, bool TDEC = false>
cudaError_t launch_w4t(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& s,
                       const tg::GemmParams& p, int grid, cudaStream_t stream) {
  auto kern = tg::tg_gemm_w4t_kernel<BMT, FMT, TDEC>;
  constexpr int smem = tg::W4TCfg<BMT, TDEC>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, tg::kW4TThreads, smem, stream>>>(a, q, s, p);
  return cudaGetLastError();
}

template <int BN, int FMT>
cudaError_t launch_w4(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& s,
                      const CUtensorMap& out, const tg::GemmParams& p, int grid,
                      cudaStream_t stream) {
  auto kern = tg::tg_gemm_w4_kernel<BN, FMT>;
  constexpr int smem = tg::W4Cfg<BN>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, tg::kW4Threads, smem, stream>>>(a, q, s, out, p);
  return cudaGetLastError();
}

int w4_pair_query_clusters();

template <int FMT>
cudaError_t launch_w4_pair(const CUtensorMap& a, const CUtensorMap& q, const CUtensorMap& s,
                           const CUtensorMap& out, const tg::GemmParams& p, int grid,
                           cudaStream_t stream) {
  constexpr int smem = tg::W4PairCfg::kSmemBytes;
  auto kern = tg::tg_gemm_w4_pair_kernel<FMT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, tg::W4PairCfg::kThreads, smem, stream>>>(a, q, s, out, p);
  return cudaGetLastError();
}

// Clusters of two that can be resident at once (0 if the query fails), queried once per device.
int w4_pair_max_clusters() {
  static std::atomic<int> cached[64];  // value + 1; 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c - 1;
  }
  const int n = w4_pair_query_clusters();
  if (dev >= 0 && dev < 64) cached[dev].store(n + 1, std::memory_order_relaxed);
  return n;
}

int w4_pair_query_clusters() {
  constexpr int smem = tg::W4PairCfg::kSmemBytes;
  // both formats' instances use the same threads and shared memory
  auto kern = tg::tg_gemm_w4_pair_kernel<tg::kFmtInt4>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(tg::W4PairCfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

CUresult encode(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, CUtensorMapDataType dt,
                const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Both dequantising GEMMs (int4 and NF4 weights): same packing, arguments and plans; only
// the per-nibble decode in the kernels differs.
template <int FMT>
tg_status run_dequant(const void* A, const void* Wq, const void* scales, void* C, int64_t M,
                      int64_t N, int64_t K, int64_t lda, int64_t ldq, int64_t lds, int64_t ldc,
                      int group_size, const tg_epilogue* epi, const tg_options* opt,
                      tg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int64_t max_dim = (int64_t{1} << 31) - 1024;
  if (M < 0 || N < 0 || K < 0 || M > max_dim || N > max_dim || K > max_dim)
    return TG_ERR_INVALID_ARG;
  if (group_size < 64 || group_size % 64 != 0) return TG_ERR_INVALID_ARG;
  if (lda < std::max<int64_t>(1, K) || ldq < cdiv(N, 8) || lds < std::max<int64_t>(1, N) ||
      ldc < std::max<int64_t>(1, N))
    return TG_ERR_INVALID_ARG;
  tg_epilogue e;
  std::memset(&e, 0, sizeof(e));
  if (epi) e = *epi;
  if (e.activation < TG_ACT_NONE || e.activation > TG_ACT_GELU_TANH) return TG_ERR_INVALID_ARG;
  if (e.residual && (e.ldr < std::max<int64_t>(1, N) || (e.residual == C && e.ldr != ldc)))
    return TG_ERR_INVALID_ARG;
  tg_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.block_n != 0 && o.block_n != 128 && o.block_n != 256) return TG_ERR_INVALID_ARG;
  if (o.max_ctas < 0 || o.panel_m < 0 || o.timeout_ms < 0 || o.swap_ab < -1 || o.swap_ab > 1 ||
      o.pair < -1 || o.pair > 1 || o.tail < -1 || o.tail > 1 || o.tmem_decode < 0 ||
      o.tmem_decode > 1 || o.dequant_first < -1 || o.dequant_first > 1)
    return TG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TG_OK;
  if (C == nullptr) return TG_ERR_INVALID_ARG;
  if (K == 0)  // no weights are read: the empty sum through the ordinary entry point
    return tg_gemm_f16_epilogue(nullptr, nullptr, C, M, N, 0, 1, N, ldc, &e, nullptr, stream_);
  if (!A || !Wq || !scales) return TG_ERR_INVALID_ARG;
  const uintptr_t bits = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Wq) |
                         reinterpret_cast<uintptr_t>(scales) | reinterpret_cast<uintptr_t>(C);
  if ((bits & 15u) || lda % 8 || ldq % 4 || lds % 8 || ldc % 8) return TG_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(e.bias) | reinterpret_cast<uintptr_t>(e.residual)) & 1u)
    return TG_ERR_MISALIGNED;

  int sms = 0;
  unsigned int* err = nullptr;
  tg_status st = tg::device_info(&sms, &err);
  if (st != TG_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!tg::tensor_map_encoder(&enc)) return tg::record_cuda_error(cudaErrorNotSupported);

  // Decode first: for large M the GEMM is compute-bound, and one pass that writes the weights
  // as fp16 (K x N x 2 bytes) costs less than decoding every weight tile inside the GEMM.
  const bool fused_override = o.swap_ab != 0 || o.pair != 0 || o.block_n != 0 ||
                              o.tmem_decode != 0;
  const int64_t min_m = FMT == tg::kFmtInt4 ? kDecodeFirstMinMInt4 : kDecodeFirstMinMNf4;
  if (o.dequant_first > 0 || (o.dequant_first == 0 && !fused_override && M >= min_m)) {
    const int64_t ldw = (N + 7) / 8 * 8;
    void* w16 = nullptr;
    st = tg::scratch_alloc(size_t(K) * size_t(ldw) * 2, stream, &w16);
    if (st != TG_OK && o.dequant_first > 0) return st;
    if (st == TG_OK) {
      const int64_t words = cdiv(N, 8);
      const dim3 grid(static_cast<unsigned>(cdiv(words, 256)),
                      static_cast<unsigned>(std::min<int64_t>(cdiv(K, tg::kDequantRows), 65535)));
      tg::tg_dequant_kernel<FMT><<<grid, 256, 0, stream>>>(
          static_cast<const uint32_t*>(Wq), ldq, static_cast<const uint16_t*>(scales), lds,
          group_size, K, N, static_cast<uint16_t*>(w16), ldw);
      const cudaError_t ce = cudaGetLastError();
      if (ce == cudaSuccess) {
        tg_options go;  // the options the fp16 GEMM knows; the int4-kernel ones do not apply
        std::memset(&go, 0, sizeof(go));
        go.max_ctas = o.max_ctas;
        go.panel_m = o.panel_m;
        go.tail = o.tail;
        go.timeout_ms = o.timeout_ms;
        go.debug_flags = o.debug_flags;
        st = tg_gemm_f16_epilogue(A, w16, C, M, N, K, lda, ldw, ldc, &e, &go, stream_);
      } else {
        st = tg::record_cuda_error(ce);
      }
      const cudaError_t fe = cudaFreeAsync(w16, stream);
      if (st == TG_OK && fe != cudaSuccess) st = tg::record_cuda_error(fe);
      return st;
    }
    st = TG_OK;  // no scratch: the fused kernels need none for most plans
  }

  const int grid_cap0 = o.max_ctas > 0 ? std::min(o.max_ctas, sms) : sms;
  const bool swap = o.swap_ab > 0 || (o.swap_ab == 0 && M <= 128);
  if (swap) {
    // C^T = W^T A^T: 128 output columns per tile on the MMA's M side, BMT rows of A on its N side
    const int bmt = M <= 64 ? 64 : 128;
    const int64_t tm = cdiv(M, bmt), tn = cdiv(N, 128);
    if (tm * tn >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
    CUtensorMap ta, tq, ts;
    if (encode(enc, &ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, uint64_t(K), uint64_t(M),
               uint64_t(lda) * 2, tg::kBK, uint32_t(bmt), CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode(enc, &tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, Wq, uint64_t(cdiv(N, 8)), uint64_t(K),
               uint64_t(ldq) * 4, 16, tg::kBK, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
        encode(enc, &ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, uint64_t(N),
               uint64_t(cdiv(K, group_size)), uint64_t(lds) * 2, 128, 1,
               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return tg::record_cuda_error(cudaErrorInvalidValue);
    tg::GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.tiles_m = static_cast<int>(tm);
    p.tiles_n = static_cast<int>(tn);
    p.num_kb = static_cast<int>(cdiv(K, tg::kBK));
    p.kb_per_split = p.num_kb;
    p.splits = 1;
    p.units = static_cast<int>(tm * tn);
    p.panel_m = static_cast<int>(std::min<int64_t>(o.panel_m ? o.panel_m : 16, tm));
    p.act = e.activation;
    p.group_kb = group_size / tg::kBK;
    p.timeout_ns = 1000000ull * static_cast<unsigned long long>(o.timeout_ms > 0 ? o.timeout_ms : 2000);
    p.debug_flags = o.debug_flags;
    p.err = err;
    p.c = static_cast<__half*>(C);
    p.ldc = ldc;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.bias = static_cast<const __half*>(e.bias);
    p.residual = static_cast<const __half*>(e.residual);
    p.ldr = e.residual ? e.ldr : 0;
    // The tiles of a last partial wave that holds at most half a grid run as two K halves,
    // which halves that wave's time (e.g. 224 tiles on 152 SMs: 1.5 tile-times instead of 2).
    const int64_t tiles = p.units;
    const int64_t r = tiles % grid_cap0;
    const bool split_tail = p.num_kb >= 2 && r > 0 && tiles + r < (int64_t{1} << 31) &&
                            (o.tail > 0 || (o.tail == 0 && 2 * r <= grid_cap0));
    uint8_t* scratch = nullptr;
    size_t cnt_off = 0;
    if (split_tail) {
      const size_t ws_bytes = size_t(r) * 2 * 4 * 32 * bmt * sizeof(float);
      cnt_off = ws_bytes;
      const tg_status sst = tg::scratch_alloc(ws_bytes + size_t(r) * 4 * sizeof(int), stream,
                                              reinterpret_cast<void**>(&scratch));
      if (sst != TG_OK) return sst;
      p.tail = 1;
      p.n_full = static_cast<int>(tiles - r);
      p.units = static_cast<int>(tiles + r);
      p.tail_ws = reinterpret_cast<float*>(scratch);
      p.tail_cnt = reinterpret_cast<int*>(scratch + cnt_off);
      const cudaError_t me = cudaMemsetAsync(p.tail_cnt, 0, size_t(r) * 4 * sizeof(int), stream);
      if (me != cudaSuccess) {
        cudaFreeAsync(scratch, stream);
        return tg::record_cuda_error(me);
      }
    }
    const int grid = static_cast<int>(std::min<int64_t>(p.units, grid_cap0));
    // on request, with 64 rows of A (the accumulators then leave half of tensor memory for
    // decoded stages), the weights are decoded into tensor memory
    const bool tdec = bmt == 64 && o.tmem_decode > 0;
    const cudaError_t ce = bmt == 128 ? launch_w4t<128, FMT>(ta, tq, ts, p, grid, stream)
                           : tdec     ? launch_w4t<64, FMT, true>(ta, tq, ts, p, grid, stream)
                                      : launch_w4t<64, FMT>(ta, tq, ts, p, grid, stream);
    const cudaError_t fe = scratch ? cudaFreeAsync(scratch, stream) : cudaSuccess;
    if (ce != cudaSuccess) return tg::record_cuda_error(ce);
    return fe == cudaSuccess ? TG_OK : tg::record_cuda_error(fe);
  }

  // many rows: 256 x 256 tiles on CTA pairs, each CTA decoding half of the weight tile
  // (an explicit block_n asks for the single-CTA kernel's tile width).  By default the pair
  // kernel runs when its tiles occupy at least half of the clusters that fit at once: with
  // fewer, the single-CTA kernel's smaller tiles spread the work over more SMs.
  const bool want_pair = o.pair > 0 || (o.pair == 0 && o.block_n == 0 && M >= 256);
  const int pair_clusters = want_pair ? w4_pair_max_clusters() : 0;
  const int64_t pair_tiles = cdiv(M, 2 * tg::kBM) * cdiv(N, tg::W4PairCfg::kBN);
  if (pair_clusters > 0 && (o.pair > 0 || 2 * pair_tiles >= pair_clusters)) {
    const int64_t tm = cdiv(M, 2 * tg::kBM), tn = cdiv(N, tg::W4PairCfg::kBN);
    if (tm * tn >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
    CUtensorMap ta, tq, ts, tc;
    if (encode(enc, &ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, uint64_t(K), uint64_t(M),
               uint64_t(lda) * 2, tg::kBK, tg::kBM, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode(enc, &tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, Wq, uint64_t(cdiv(N, 8)), uint64_t(K),
               uint64_t(ldq) * 4, tg::W4PairCfg::kHalfN / 8, tg::kBK, CU_TENSOR_MAP_SWIZZLE_NONE) !=
            CUDA_SUCCESS ||
        encode(enc, &ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, uint64_t(N),
               uint64_t(cdiv(K, group_size)), uint64_t(lds) * 2, tg::W4PairCfg::kHalfN, 1,
               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
        encode(enc, &tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C,
               uint64_t(std::max<int64_t>(N & ~int64_t{7}, 8)), uint64_t(M), uint64_t(ldc) * 2, 64,
               32, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return tg::record_cuda_error(cudaErrorInvalidValue);
    tg::GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.tiles_m = static_cast<int>(tm);
    p.tiles_n = static_cast<int>(tn);
    p.num_kb = static_cast<int>(cdiv(K, tg::kBK));
    p.kb_per_split = p.num_kb;
    p.splits = 1;
    p.units = static_cast<int>(tm * tn);
    p.panel_m = static_cast<int>(std::min<int64_t>(o.panel_m ? o.panel_m : 8, tm));
    p.act = e.activation;
    p.group_kb = group_size / tg::kBK;
    p.timeout_ns = 1000000ull * static_cast<unsigned long long>(o.timeout_ms > 0 ? o.timeout_ms : 2000);
    p.debug_flags = o.debug_flags;
    p.err = err;
    p.c = static_cast<__half*>(C);
    p.ldc = ldc;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.n_tma = static_cast<int>(N & ~int64_t{7});
    p.bias = static_cast<const __half*>(e.bias);
    p.residual = static_cast<const __half*>(e.residual);
    p.ldr = e.residual ? e.ldr : 0;
    int clusters = std::min<int64_t>(p.units, pair_clusters);
    if (o.max_ctas > 0) clusters = std::min(clusters, std::max(1, o.max_ctas / 2));
    const cudaError_t ce = launch_w4_pair<FMT>(ta, tq, ts, tc, p, 2 * clusters, stream);
    return ce == cudaSuccess ? TG_OK : tg::record_cuda_error(ce);
  }

  const int64_t tiles_m = cdiv(M, tg::kBM);
  int bn = o.block_n;
  if (bn == 0) bn = (tiles_m * cdiv(N, 256) >= (9 * sms) / 10) ? 256 : 128;
  const int64_t tiles_n = cdiv(N, bn);
  const int64_t units = tiles_m * tiles_n;
  if (units >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
  const int grid_cap = o.max_ctas > 0 ? std::min(o.max_ctas, sms) : sms;

  CUtensorMap ta, tq, ts, tc;
  if (encode(enc, &ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, uint64_t(K), uint64_t(M),
             uint64_t(lda) * 2, tg::kBK, tg::kBM, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode(enc, &tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, Wq, uint64_t(cdiv(N, 8)), uint64_t(K),
             uint64_t(ldq) * 4, uint32_t(bn / 8), tg::kBK, CU_TENSOR_MAP_SWIZZLE_NONE) !=
          CUDA_SUCCESS ||
      encode(enc, &ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, uint64_t(N),
             uint64_t(cdiv(K, group_size)), uint64_t(lds) * 2, uint32_t(bn), 1,
             CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      encode(enc, &tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C,
             uint64_t(std::max<int64_t>(N & ~int64_t{7}, 8)), uint64_t(M), uint64_t(ldc) * 2, 64,
             32, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return tg::record_cuda_error(cudaErrorInvalidValue);

  tg::GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.tiles_m = static_cast<int>(tiles_m);
  p.tiles_n = static_cast<int>(tiles_n);
  p.num_kb = static_cast<int>(cdiv(K, tg::kBK));
  p.kb_per_split = p.num_kb;
  p.splits = 1;
  p.units = static_cast<int>(units);
  p.panel_m = static_cast<int>(std::min<int64_t>(o.panel_m ? o.panel_m : 16, tiles_m));
  p.act = e.activation;
  p.group_kb = group_size / tg::kBK;
  p.timeout_ns = 1000000ull * static_cast<unsigned long long>(o.timeout_ms > 0 ? o.timeout_ms : 2000);
  p.debug_flags = o.debug_flags;
  p.err = err;
  p.c = static_cast<__half*>(C);
  p.ldc = ldc;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.n_tma = static_cast<int>(N & ~int64_t{7});
  p.bias = static_cast<const __half*>(e.bias);
  p.residual = static_cast<const __half*>(e.residual);
  p.ldr = e.residual ? e.ldr : 0;
  const int grid = static_cast<int>(std::min<int64_t>(units, grid_cap));
  const cudaError_t ce = bn == 256 ? launch_w4<256, FMT>(ta, tq, ts, tc, p, grid, stream)
                                   : launch_w4<128, FMT>(ta, tq, ts, tc, p, grid, stream);
  return ce == cudaSuccess ? TG_OK : tg::record_cuda_error(ce);
}

}  // namespace

extern "C" tg_status tg_gemm_w4a16_f16(const void* A, const void* Wq, const void* scales,
                                       void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                       int64_t ldq, int64_t lds, int64_t ldc, int group_size,
                                       const tg_epilogue* epi, const tg_options* opt,
                                       tg_stream_t stream) {
  return run_dequant<tg::kFmtInt4>(A, Wq, scales, C, M, N, K, lda, ldq, lds, ldc, group_size,
                                   epi, opt, stream);
}

extern "C" tg_status tg_gemm_nf4a16_f16(const void* A, const void* Wq, const void* scales,
                                        void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                        int64_t ldq, int64_t lds, int64_t ldc, int group_size,
                                        const tg_epilogue* epi, const tg_options* opt,
                                        tg_stream_t stream) {
  return run_dequant<tg::kFmtNf4>(A, Wq, scales, C, M, N, K, lda, ldq, lds, ldc, group_size,
                                  epi, opt, stream);
}
