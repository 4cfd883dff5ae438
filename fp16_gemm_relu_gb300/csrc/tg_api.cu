// tg_api.cu — the C ABI declared in include/tg_gemm_relu.h.
//
// Host side of every call: validate -> plan (tile width, K splits, repack/workspace needs)
// -> scratch from a stream-ordered pool -> optional operand repack -> TMA tensor maps ->
// the persistent tcgen05 kernel -> optional deterministic split-K reduction.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "tg_gemm_relu.h"
#include "tg_internal.h"

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1024;  // TMA coordinates are 32-bit
// L2 panel height in M-tiles (units walk the M-tiles of a panel fastest).  Measured against 16,
// best of two runs with L2 flushed: 2048^3 20.4 against 21.4 us, 5000x4000x1000 49.3 against
// 51.2 us, ragged 4095x3073x65537 1.320 against 1.331 ms, 8192^3 and 64x28672x8192 unchanged;
// 8192^3 reads 1.05 GB of DRAM per launch against 1.26 GB (4 and 32 are slower and read more).
constexpr int kDefaultPanel = 8;
constexpr int kDefaultTimeoutMs = 2000;
constexpr int kBlockNs[3] = {256, 192, 128};
constexpr int kMaxOverlapSplits = 32;  // the plan's largest split count

thread_local int t_last_cuda_error = 0;

tg_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return TG_ERR_CUDA;
}

// Set by kernels whose pipeline wait ran out (see tg_device_error_check).
__device__ unsigned int g_tg_error_word;

struct DeviceState {
  bool ready = false;
  tg_status status = TG_OK;
  int sm_count = 0;
  cudaMemPool_t pool = nullptr;
  unsigned int* err = nullptr;
  int pair_clusters = 0;  // co-resident clusters of the CTA-pair kernel (0: do not use it)
};

// Library streams and events of the overlapped operand copies (one set per device, created on
// first use): `copy` makes the split-by-split copies, gemm[0] / gemm[1] take the splits' GEMMs
// in turn so that one split's last partial wave can share the SMs with the next split's
// first.  Calls enqueue under `mu`; each joins every stream back to the caller's before it
// returns, so work of different calls only meets in stream order.
struct OverlapStreams {
  bool ready = false;
  cudaStream_t copy = nullptr, gemm[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, copied[kMaxOverlapSplits] = {}, done[3] = {};
  std::mutex mu;
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
OverlapStreams g_overlap[kMaxDevices];
std::mutex g_mutex;

tg_status overlap_streams(OverlapStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  OverlapStreams& o = g_overlap[dev];
  if (!o.ready) {
    const unsigned ev = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&o.copy, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&o.gemm[0], cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&o.gemm[1], cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&o.start, ev)) != cudaSuccess)
      return cuda_fail(e);
    for (int i = 0; i < kMaxOverlapSplits; ++i)
      if ((e = cudaEventCreateWithFlags(&o.copied[i], ev)) != cudaSuccess) return cuda_fail(e);
    for (int i = 0; i < 3; ++i)
      if ((e = cudaEventCreateWithFlags(&o.done[i], ev)) != cudaSuccess) return cuda_fail(e);
    o.ready = true;
  }
  *out = &o;
  return TG_OK;
}

tg_status current_device(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
  if ((e = tg::bind_thread_context(dev)) != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      s.status = TG_ERR_UNSUPPORTED_DEVICE;
    } else {
      cudaMemPoolProps props;
      std::memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if ((e = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess) return cuda_fail(e);
      uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse instead of returning them
      if ((e = cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
        return cuda_fail(e);
      if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_tg_error_word)) != cudaSuccess)
        return cuda_fail(e);
      s.sm_count = sms;
      int clusters = 0;
      if (tg::gemm_pair_max_clusters(&clusters) != cudaSuccess) {
        clusters = 0;
        cudaGetLastError();  // a failed occupancy query only disables the pair kernel
      }
      s.pair_clusters = clusters;
      s.status = TG_OK;
    }
    s.ready = true;
  }
  *out = &s;
  return s.status;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

tg_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!g_encode) return cuda_fail(cudaErrorNotSupported);
  *fn = g_encode;
  return TG_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// ta / tb: A stored K x M (row length M) / B stored N x K (row length K) instead of M x K / K x N.
tg_status validate(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, int flag, int ta = 0, int tb = 0) {
  if (M < 0 || N < 0 || K < 0) return TG_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TG_ERR_INVALID_ARG;
  if (flag != TG_EPILOGUE_NONE && flag != TG_EPILOGUE_RELU) return TG_ERR_INVALID_ARG;
  if ((ta != 0 && ta != 1) || (tb != 0 && tb != 1)) return TG_ERR_INVALID_ARG;
  if (lda < std::max<int64_t>(1, ta ? M : K) || ldb < std::max<int64_t>(1, tb ? K : N) ||
      ldc < std::max<int64_t>(1, N))
    return TG_ERR_INVALID_ARG;
  if (lda > (int64_t{1} << 36) || ldb > (int64_t{1} << 36) || ldc > (int64_t{1} << 36))
    return TG_ERR_INVALID_ARG;
  if (M > 0 && N > 0) {
    if (C == nullptr) return TG_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return TG_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 1u)
    return TG_ERR_MISALIGNED;
  return TG_OK;
}

struct Plan {
  tg_plan pub;
  int64_t lda_p, ldb_p, ldw;     // leading dimensions of the scratch copies / workspace
  int64_t off_a, off_b, off_w;   // byte offsets inside the scratch block
  int64_t off_tail_ws, off_tail_cnt, tail_cnt_bytes;  // tail-split partials and counters
  // A read by row classes: rows per class (a multiple of the 256-row pair tile), each class's
  // element shift past a 32-byte boundary, and the first-window copy's offset in scratch
  int64_t cls_rows, off_first;
  int cls_shift[tg::kARowClasses];
};

// Per-k-block cost in SM cycles of an output tile 128 x bn: the tensor-core time (a
// 128 x bn x 16 MMA takes bn/8 cycles, four per k-block) or the time to bring the stage's
// bytes in from L2, whichever is longer.  The L2 feed rate, ~87 B/cycle per SM, is what the
// 128 x 256 tile sustains on 8192^3 (~1630 TFLOP/s, ~10% below the CTA-pair tile, whose
// 32 KB per SM and k-block stay within it: the pair's 512 cycles below).
double kblock_cycles(int bn) {
  const double mma = 2.0 * bn;
  const double load = (16384.0 + 128.0 * bn) / 87.0;
  return std::max(mma, load);
}

// Plan selection (host only): tries every tile width and split count and keeps the fastest
// by a simple model.  Compute time = waves x k-blocks per unit x kblock_cycles / 1.9 GHz
// (a tail-split last wave counts half); memory time = the algorithmic bytes at 6.8 TB/s,
// inflated when a wave keeps fewer than 60% of the SMs busy; plus the float32 workspace
// traffic of split-K and its extra launch, and the operand copies of unaligned operands.
tg_status make_plan(uintptr_t a, uintptr_t b, uintptr_t c, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int num_sms, int pair_clusters,
                    const tg_options* opt, Plan* out, int ta = 0, int tb = 0) {
  tg_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (num_sms <= 0) return TG_ERR_INVALID_ARG;
  if (o.block_n != 0 && o.block_n != 128 && o.block_n != 192 && o.block_n != 256)
    return TG_ERR_INVALID_ARG;
  if (o.split_k < 0 || o.panel_m < 0 || o.max_ctas < 0 || o.timeout_ms < 0 || o.pair < -1 ||
      o.pair > 1 || o.tail < -1 || o.tail > 1 || o.a_in_place < 0 || o.a_in_place > 1 ||
      o.repack_overlap < -1 || o.repack_overlap > 0)
    return TG_ERR_INVALID_ARG;
  if (o.pair == 1 && o.block_n != 0 && o.block_n != 256) return TG_ERR_INVALID_ARG;

  Plan pl;
  std::memset(&pl, 0, sizeof(pl));
  tg_plan& P = pl.pub;
  P.block_m = tg::kBM;
  P.block_k = tg::kBK;
  P.repack_a = (a % 16 != 0 || lda % 8 != 0 || o.force_repack) ? 1 : 0;
  P.repack_b = (b % 16 != 0 || ldb % 8 != 0 || o.force_repack) ? 1 : 0;
  const bool c_direct = (c % 16 == 0) && (ldc % 8 == 0) && !o.force_workspace;
  P.kblocks = cdiv(K, tg::kBK);
  P.tiles_m = cdiv(M, tg::kBM);
  if (M == 0 || N == 0) {
    *out = pl;
    return TG_OK;
  }
  if (K == 0) {  // C = +0: one memset
    P.kernels = 1;
    *out = pl;
    return TG_OK;
  }
  const int grid_cap = o.max_ctas > 0 ? std::min(o.max_ctas, num_sms) : num_sms;
  const double clk = 1.9e9, hbm = 6.8e12;
  const double alg_bytes = 2.0 * (double(M) * K + double(K) * N + double(M) * N);
  // Operand copies (each element read once, written once).  Made first, they add their full
  // time.  Overlapped split by split (split-K only), the first split's copy runs alone and the
  // others still cost ~3/4 of their time, since they share DRAM and L2 with the GEMMs; every
  // further split also adds a launch and two copies (~5 us).  Calibrated on unaligned shapes
  // from 1 x 4096 x 8192 to 4095 x 3073 x 65537, timed with each plan forced.
  const double copy_time = 4.0 * ((P.repack_a ? double(M) * K : 0.0) +
                                  (P.repack_b ? double(K) * N : 0.0)) / hbm;
  const bool may_overlap = copy_time > 0.0 && o.repack_overlap >= 0 && o.a_in_place == 0;

  struct Cand {
    double t;
    int bn, s, active, pair;
  };
  Cand cands[4 * 32];
  int nc = 0;
  // tile kinds: the 256x256 CTA-pair tile, then single-CTA 128 x {256, 192, 128}
  const int pair_cap = std::min(o.max_ctas > 0 ? o.max_ctas / 2 : num_sms / 2,
                                pair_clusters > 0 ? pair_clusters : num_sms / 2);
  for (int kind = 0; kind < 4; ++kind) {
    const int pair = kind == 0 ? 1 : 0;
    const int bn = pair ? 256 : kBlockNs[kind - 1];
    if (pair && (o.pair < 0 || pair_cap < 1)) continue;
    if (!pair && o.pair > 0) continue;
    if (o.block_n && bn != o.block_n) continue;
    const int bm = pair ? 2 * tg::kBM : tg::kBM;
    const int64_t tiles = cdiv(M, bm) * cdiv(N, bn);
    const int64_t s_max = o.split_k ? std::min<int64_t>(o.split_k, P.kblocks)
                                    : std::min<int64_t>(P.kblocks, 32);
    const int64_t s_min = o.split_k ? s_max : 1;
    for (int64_t s = s_min; s <= s_max; ++s) {
      const int64_t kbps = cdiv(P.kblocks, s);
      const int64_t s_eff = cdiv(P.kblocks, kbps);
      if (!o.split_k && s_eff != s) continue;  // same plan as a smaller s
      const int64_t units = tiles * s_eff;
      // a pair unit occupies two SMs; the per-SM k-block cost of the pair tile is the MMA
      // time alone (each SM loads 32 KB per k-block, well under the L2 budget)
      const int64_t slots_cap = pair ? pair_cap : grid_cap;
      const int64_t grid = std::min<int64_t>(units, slots_cap);
      const bool ws = s_eff > 1 || !c_direct;
      // the pair kernel's tail split (below) runs a last wave of at most half the clusters as
      // K halves on twice as many clusters, in half a wave's time
      const bool tail = pair && s_eff == 1 && !ws && o.tail >= 0 && P.kblocks >= 2 &&
                        units > grid && units % grid != 0 && 2 * (units % grid) <= grid;
      const double waves = tail ? double(units / grid) + 0.5 : double(cdiv(units, grid));
      const double kb_cycles = pair ? 512.0 : kblock_cycles(bn);
      // the pair kernel's cluster launch and its first 64 KB stage per CTA cost ~2 us more
      // before the first MMA than the single-CTA kernel's start (measured on 2048^3, one wave
      // either way: 22.6 us against 20.5 us)
      const double t_start = pair ? 2.1e-6 : 0.0;
      // the tail's K halves meet through a float32 workspace: ~5 us, which short K does not win
      // back
      const double t_mma = waves * double(kbps) * kb_cycles / clk + t_start + (tail ? 5e-6 : 0.0);
      const bool overlap = may_overlap && s_eff >= 2 && s_eff <= kMaxOverlapSplits;
      const double t_copy =
          overlap ? copy_time * (1.0 / s_eff + 0.75 * (1.0 - 1.0 / s_eff)) + (s_eff - 1) * 5e-6
                  : copy_time;
      double slots = 0.0;  // wave-by-wave occupancy penalty on the memory time
      for (int64_t wv = 0; wv < cdiv(units, grid); ++wv) {
        const int64_t active = (pair ? 2 : 1) * std::min<int64_t>(grid, units - wv * grid);
        slots += std::max<double>(double(active), 0.6 * num_sms);
      }
      const double t_hbm = alg_bytes / hbm * (slots / double((pair ? 2 : 1) * units));
      // workspace traffic plus the extra launch of the reduction kernel (~3 us)
      const double t_ws = ws ? (2.0 * 4.0 * double(s_eff) * M * N + 2.0 * M * N) / hbm + 3e-6 : 0.0;
      cands[nc++] = Cand{std::max(t_mma, t_hbm) + t_ws + t_copy, bn, static_cast<int>(s_eff),
                         static_cast<int>((pair ? 2 : 1) * grid), pair};
    }
  }
  if (nc == 0) return TG_ERR_INVALID_ARG;
  double best_t = cands[0].t;
  for (int i = 1; i < nc; ++i) best_t = std::min(best_t, cands[i].t);
  // among plans within 2% of the fastest: most SMs busy, then the wider tile, then fewer splits
  int pick = -1;
  for (int i = 0; i < nc; ++i) {
    if (cands[i].t > best_t * 1.02) continue;
    if (pick < 0 || cands[i].active > cands[pick].active) pick = i;
  }
  const int best_bn = cands[pick].bn;
  const int best_s = cands[pick].s;
  const int best_pair = cands[pick].pair;
  P.cta_pair = best_pair;
  P.block_m = best_pair ? 2 * tg::kBM : tg::kBM;
  P.block_n = best_bn;
  P.stages = best_pair ? tg::PairCfgFwd::kStages : tg::gemm_stages(best_bn);
  P.kblocks_per_split = cdiv(P.kblocks, best_s);
  P.split_k = static_cast<int>(cdiv(P.kblocks, P.kblocks_per_split));
  P.tiles_m = cdiv(M, P.block_m);
  P.tiles_n = cdiv(N, best_bn);
  P.units = P.tiles_m * P.tiles_n * P.split_k;
  if (P.units >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
  P.grid = best_pair ? 2 * static_cast<int>(std::min<int64_t>(P.units, pair_cap))
                     : static_cast<int>(std::min<int64_t>(P.units, grid_cap));
  P.panel_m = static_cast<int>(std::min<int64_t>(o.panel_m ? o.panel_m : kDefaultPanel, P.tiles_m));
  P.workspace_epilogue = (P.split_k > 1 || !c_direct) ? 1 : 0;
  // On request (tg_options.a_in_place), an A whose rows TMA cannot describe (lda not a
  // multiple of 8) is read in place through 16 row classes (AClassMaps) instead of being
  // copied, when A itself is 32-byte aligned, the plan uses CTA pairs on the forward layout and
  // the class-major row order adds at most 3% of M tiles.  The partial sums then go through the
  // float32 workspace in class-major row order and the reduction writes them back to C's rows.
  // Each class's K windows start up to 15 elements early, which can add one k-block.  It saves
  // the copy's scratch, but is not the default: a class's rows lie 32 lda bytes apart, so
  // three in four start inside a 128-byte line and every box row spans two lines, which on
  // 4095 x 3073 x 65537 made the GEMM 29% slower (1226 against 952 us) than on the aligned copy.
  if (o.a_in_place > 0 && P.repack_a && !o.force_repack && !ta && !tb && P.cta_pair &&
      lda % 8 != 0 && a % 32 == 0 && K >= tg::kBK && M >= 2 * tg::kBM) {
    const int64_t rows = round_up(cdiv(M, tg::kARowClasses), 2 * tg::kBM);
    const int64_t tiles_cls = tg::kARowClasses * rows / (2 * tg::kBM);
    if (tiles_cls * 100 <= P.tiles_m * 103) {
      int emax = 0;
      for (int r = 0; r < tg::kARowClasses; ++r) {
        pl.cls_shift[r] = static_cast<int>((int64_t(r) * lda) % tg::kARowClasses);
        emax = std::max(emax, pl.cls_shift[r]);
      }
      pl.cls_rows = rows;
      P.a_row_classes = tg::kARowClasses;
      P.repack_a = 0;
      P.workspace_epilogue = 1;
      P.kblocks = cdiv(K + emax, tg::kBK);
      P.kblocks_per_split = cdiv(P.kblocks, P.split_k);
      P.split_k = static_cast<int>(cdiv(P.kblocks, P.kblocks_per_split));
      P.tiles_m = tiles_cls;
      P.units = P.tiles_m * P.tiles_n * P.split_k;
      if (P.units >= (int64_t{1} << 31)) return TG_ERR_INVALID_ARG;
      P.grid = 2 * static_cast<int>(std::min<int64_t>(P.units, pair_cap));
      P.panel_m = static_cast<int>(std::min<int64_t>(o.panel_m ? o.panel_m : kDefaultPanel, P.tiles_m));
    }
  }
  // Tail split (tg_options.tail: 0 chooses, 1 forces, -1 never): when the last wave of pair
  // tiles would leave more than half the clusters idle, its r tiles run as 2r K halves
  // instead.  On 8192^3 (36 tiles left for 76 clusters) launches interleaved with whole-tile
  // launches measured ~8 us (1.3%) faster; under the power cap the idle SMs of a partial wave
  // let the busy ones clock higher, which is why the gain is below the 3.8% the cycle count
  // predicts.
  if (P.cta_pair && P.split_k == 1 && !P.workspace_epilogue && o.tail >= 0 && P.kblocks >= 2) {
    const int64_t clusters = P.grid / 2;
    const int64_t r = P.units % clusters;
    if (r > 0 && 2 * r <= clusters && P.units > clusters) {
      P.tail_tiles = r;
      P.units += r;
    }
  }

  int64_t off = 0;
  if (P.repack_a) {  // A is stored (ta ? K x M : M x K)
    // rows of the copies start on 128-byte lines: a 128-byte TMA box row then reads four
    // 32-byte sectors of L2, where a row only 16-byte aligned spans five
    pl.lda_p = round_up(ta ? M : K, 64);
    pl.off_a = off;
    off += round_up((ta ? K : M) * pl.lda_p * 2, 256);
  }
  if (P.repack_b) {  // B is stored (tb ? N x K : K x N)
    pl.ldb_p = round_up(tb ? K : N, 64);
    pl.off_b = off;
    off += round_up((tb ? N : K) * pl.ldb_p * 2, 256);
  }
  if (P.a_row_classes) {  // the first 64-k window of every class-major row, pre-shifted
    pl.off_first = off;
    off += round_up(P.a_row_classes * pl.cls_rows * tg::kBK * 2, 256);
  }
  if (P.workspace_epilogue) {
    pl.ldw = round_up(N, 32);  // 128-byte rows for the same reason
    pl.off_w = off;
    const int64_t ws_rows = P.a_row_classes ? P.a_row_classes * pl.cls_rows : M;
    off += round_up(int64_t(P.split_k) * ws_rows * pl.ldw * 4, 256);
  }
  if (P.tail_tiles) {
    pl.off_tail_ws = off;
    off += round_up(P.tail_tiles * 2 * 256 * 256 * 4, 256);
    pl.off_tail_cnt = off;
    pl.tail_cnt_bytes = round_up(P.tail_tiles * 8 * 4, 256);
    off += pl.tail_cnt_bytes;
  }
  P.workspace_bytes = off;
  // Operand copies overlap the GEMM split by split: split s's slice of A and B is copied on a
  // library stream while the GEMMs of earlier splits run (the copies use DRAM bandwidth that
  // the L2-bound GEMM leaves idle), and each split's GEMM starts once its slice is in place.
  P.repack_overlap = (P.repack_a || P.repack_b) && P.split_k >= 2 && P.workspace_epilogue &&
                     !P.tail_tiles && !P.a_row_classes && o.repack_overlap >= 0 &&
                     P.split_k <= kMaxOverlapSplits;
  if (P.repack_overlap)
    P.kernels = P.split_k * (1 + P.repack_a + P.repack_b) + 1;
  else
    P.kernels = 1 + P.repack_a + P.repack_b + P.workspace_epilogue + (P.a_row_classes ? 1 : 0);
  *out = pl;
  return TG_OK;
}

// ------------------------------ auxiliary kernels ------------------------------

// dst (rows x ld_dst, 16-byte aligned rows) <- src (rows x ld_src, any 2-byte alignment).
// Output chunk c of a row is elements [8c, 8c + 8); columns in [cols, round_up(cols, 8)) are
// written as zero.  A warp copies 32 consecutive chunks of one row.  Element 0 of a row sits
// b bytes into an aligned 16-byte block (b even, the same for every chunk of the row), so
// chunk c lies in blocks c and c + 1 from there: a lane loads block c, loads block c + 1 only
// when it holds one of the chunk's elements (so no load leaves a block that holds valid data),
// and shifts the pair by b bytes in registers.
__global__ void tg_pack_rows_kernel(const uint16_t* __restrict__ src, int64_t ld_src,
                                    uint16_t* __restrict__ dst, int64_t ld_dst, int64_t rows,
                                    int64_t cols) {
  const int64_t cpr = (cols + 7) >> 3;
  const int64_t gpr = (cpr + 31) >> 5;  // 32-chunk groups per row
  const int64_t items = rows * gpr;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t it = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const int64_t r = it / gpr;
    const int64_t c = ((it - r * gpr) << 5) + lane;
    if (c >= cpr) continue;
    const uintptr_t row = reinterpret_cast<uintptr_t>(src + r * ld_src);
    const uint32_t b = static_cast<uint32_t>(row & 15u);
    const uint4* blk = reinterpret_cast<const uint4*>(row - b) + c;
    const int nvalid = static_cast<int>(cols - (c << 3) < 8 ? cols - (c << 3) : 8);
    const uint4 lo = __ldg(blk);
    const uint4 hi = (b + 2u * static_cast<uint32_t>(nvalid - 1) >= 16u) ? __ldg(blk + 1)
                                                                          : make_uint4(0, 0, 0, 0);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t q = b >> 2;  // whole words to skip
    uint32_t t[7], u[5];
#pragma unroll
    for (int i = 0; i < 7; ++i) t[i] = (q & 1u) ? w[i + 1] : w[i];
#pragma unroll
    for (int i = 0; i < 5; ++i) u[i] = (q & 2u) ? t[i + 2] : t[i];
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[j] = (b & 2u) ? __funnelshift_r(u[j], u[j + 1], 16) : u[j];
      if (2 * j >= nvalid) o[j] = 0u;
      else if (2 * j + 1 >= nvalid) o[j] &= 0xFFFFu;
    }
    *reinterpret_cast<uint4*>(dst + r * ld_dst + (c << 3)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The same copy with each lane taking kPackItems chunks (of warp items nwarps apart) per pass,
// all of their loads issued before its first store: for large copies, where every warp has
// at least that many items (launch_pack).
constexpr int kPackItems = 4;

__global__ void tg_pack_rows4_kernel(const uint16_t* __restrict__ src, int64_t ld_src,
                                     uint16_t* __restrict__ dst, int64_t ld_dst, int64_t rows,
                                     int64_t cols) {
  const int64_t cpr = (cols + 7) >> 3;
  const int64_t gpr = (cpr + 31) >> 5;  // 32-chunk groups per row
  const int64_t items = rows * gpr;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t it0 = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; it0 < items;
       it0 += kPackItems * nwarps) {
    uint4 lo[kPackItems], hi[kPackItems];
    uint32_t bs[kPackItems];
    int nv[kPackItems];
    int64_t out[kPackItems];  // element offset of the chunk in dst, or -1 when there is none
#pragma unroll
    for (int i = 0; i < kPackItems; ++i) {
      const int64_t it = it0 + i * nwarps;
      out[i] = -1;
      if (it >= items) continue;
      const int64_t r = it / gpr;
      const int64_t c = ((it - r * gpr) << 5) + lane;
      if (c >= cpr) continue;
      const uintptr_t row = reinterpret_cast<uintptr_t>(src + r * ld_src);
      const uint32_t b = static_cast<uint32_t>(row & 15u);
      const uint4* blk = reinterpret_cast<const uint4*>(row - b) + c;
      const int nvalid = static_cast<int>(cols - (c << 3) < 8 ? cols - (c << 3) : 8);
      lo[i] = __ldg(blk);
      hi[i] = (b + 2u * static_cast<uint32_t>(nvalid - 1) >= 16u) ? __ldg(blk + 1)
                                                                 : make_uint4(0, 0, 0, 0);
      bs[i] = b;
      nv[i] = nvalid;
      out[i] = r * ld_dst + (c << 3);
    }
#pragma unroll
    for (int i = 0; i < kPackItems; ++i) {
      if (out[i] < 0) continue;
      const uint32_t b = bs[i];
      const uint32_t w[8] = {lo[i].x, lo[i].y, lo[i].z, lo[i].w,
                             hi[i].x, hi[i].y, hi[i].z, hi[i].w};
      const uint32_t q = b >> 2;  // whole words to skip
      uint32_t t[7], u[5];
#pragma unroll
      for (int k = 0; k < 7; ++k) t[k] = (q & 1u) ? w[k + 1] : w[k];
#pragma unroll
      for (int k = 0; k < 5; ++k) u[k] = (q & 2u) ? t[k + 2] : t[k];
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[j] = (b & 2u) ? __funnelshift_r(u[j], u[j + 1], 16) : u[j];
        if (2 * j >= nv[i]) o[j] = 0u;
        else if (2 * j + 1 >= nv[i]) o[j] &= 0xFFFFu;
      }
      *reinterpret_cast<uint4*>(dst + out[i]) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Element shifts of the 16 row classes of A (AClassMaps), passed by value.
struct ClassShifts {
  int e[tg::kARowClasses];
};

// The first 64-k window of every row of A in class-major order, shifted like the class's
// windows: F[(r * cls_rows + j) * 64 + t] = A[16 j + r][t - e_r] where 0 <= t - e_r < K and
// 16 j + r < M, else +0 (so the window's elements before k = 0 are zero).
__global__ void tg_first_window_kernel(const uint16_t* __restrict__ A, int64_t lda, int64_t M,
                                       int64_t K, int64_t cls_rows, ClassShifts sh,
                                       uint16_t* __restrict__ F) {
  const int64_t total = tg::kARowClasses * cls_rows * tg::kBK;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = idx / tg::kBK;
    const int t = static_cast<int>(idx - row * tg::kBK);
    const int r = static_cast<int>(row / cls_rows);
    const int64_t i = (row - r * cls_rows) * tg::kARowClasses + r;
    const int64_t k = t - sh.e[r];
    F[idx] = (i < M && k >= 0 && k < K) ? A[i * lda + k] : uint16_t(0);
  }
}

// C[i, j] = fp16(epilogue(sum_{s=0}^{splits-1} W[s][i][j])), the splits added in increasing s
// (deterministic), then the same fused epilogue as the GEMM kernel (bias, activation,
// residual).  W rows are ldw floats (multiple of 4, 16-byte aligned); C may have any 2-byte
// alignment and leading dimension.  p supplies act, bias, residual, ldr, M and N.
// With cls_rows > 0 the workspace rows are in class-major order (A read by row classes): row i
// of C is workspace row (i mod 16) * cls_rows + i / 16.  Thread g of the x range takes columns
// 4g .. 4g + 3 of kReduceRows rows at a time, loading one split of all of them before adding
// (a flat index split by a 64-bit division per item, one row at a time, ran at 0.67 of HBM).
constexpr int kReduceRows = 4;
constexpr int kReduceThreads = 128;
__global__ void __launch_bounds__(kReduceThreads)
    tg_splitk_reduce_kernel(const float* __restrict__ ws, int64_t ldw, int64_t split_stride,
                            int splits, __half* C, int64_t ldc, const tg::GemmParams p,
                            int64_t cls_rows) {
  const int64_t M = p.M, N = p.N;
  const int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;  // group of 4 columns
  if (g >= (N + 3) >> 2) return;
  const int64_t c0 = g << 2;
  for (int64_t r0 = int64_t(blockIdx.y) * kReduceRows; r0 < M;
       r0 += int64_t(gridDim.y) * kReduceRows) {
    // rows past M read row M - 1 (in bounds) and are never stored
    const float* w[kReduceRows];
    float4 acc[kReduceRows];
#pragma unroll
    for (int i = 0; i < kReduceRows; ++i) {
      const int64_t r = r0 + i < M ? r0 + i : M - 1;
      const int64_t wr =
          cls_rows > 0 ? (r % tg::kARowClasses) * cls_rows + r / tg::kARowClasses : r;
      w[i] = ws + wr * ldw + c0;
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);  // splits == 0: the empty sum (K == 0)
    }
    for (int s = 0; s < splits; ++s) {
      float4 v[kReduceRows];
#pragma unroll
      for (int i = 0; i < kReduceRows; ++i)
        v[i] = __ldg(reinterpret_cast<const float4*>(w[i] + s * split_stride));
#pragma unroll
      for (int i = 0; i < kReduceRows; ++i) {
        if (s == 0) {
          acc[i] = v[i];
        } else {
          acc[i].x += v[i].x;
          acc[i].y += v[i].y;
          acc[i].z += v[i].z;
          acc[i].w += v[i].w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kReduceRows; ++i) {
      const int64_t r = r0 + i;
      if (r >= M) break;
      const float a[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
      __half h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        h[e] = __float2half_rn(c0 + e < N ? tg::epilogue_value(a[e], int(r), int(c0 + e), p)
                                          : 0.0f);
      __half* d = C + r * ldc + c0;
      if (c0 + 4 <= N && (reinterpret_cast<uintptr_t>(d) & 7u) == 0) {
        uint2 v;
        v.x = uint32_t(__half_as_ushort(h[0])) | (uint32_t(__half_as_ushort(h[1])) << 16);
        v.y = uint32_t(__half_as_ushort(h[2])) | (uint32_t(__half_as_ushort(h[3])) << 16);
        *reinterpret_cast<uint2*>(d) = v;
      } else {
        for (int e = 0; e < 4 && c0 + e < N; ++e) d[e] = h[e];
      }
    }
  }
}

// Grid of the reduction: x over the groups of 4 columns, y over chunks of kReduceRows rows.
dim3 reduce_grid(int64_t M, int64_t N) {
  return dim3(static_cast<unsigned>(cdiv(cdiv(std::max<int64_t>(N, 1), 4), kReduceThreads)),
              static_cast<unsigned>(std::min<int64_t>(cdiv(std::max<int64_t>(M, 1), kReduceRows),
                                                      65535)));
}

// dZ[i, j] = C[i, j] > 0 ? dC[i, j] : +0 (the relu derivative taken on the forward output C;
// NaN or -0 in C gives +0).  Any 2-byte alignment: row r of the grid's y range at a time, the
// columns spread over the x range (2-D, so no index division per element).
__global__ void tg_relu_backward_kernel(const uint16_t* __restrict__ dC, int64_t lddc,
                                        const uint16_t* __restrict__ C, int64_t ldc,
                                        uint16_t* __restrict__ dZ, int64_t lddz, int64_t M,
                                        int64_t N) {
  for (int64_t r = blockIdx.y; r < M; r += gridDim.y) {
    for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < N;
         c += int64_t(gridDim.x) * blockDim.x) {
      const uint16_t cv = __ldg(C + r * ldc + c);
      const bool pos = (cv & 0x8000u) == 0 && cv != 0 && (cv & 0x7FFFu) <= 0x7C00u;
      dZ[r * lddz + c] = pos ? __ldg(dC + r * lddc + c) : uint16_t(0);
    }
  }
}

// Both fp16 lanes of a 32-bit word: d's lane where c's lane is positive (sign clear, nonzero,
// not NaN), else +0.
__device__ __forceinline__ uint32_t relu_grad2(uint32_t c, uint32_t d) {
  const uint32_t lo = c & 0xFFFFu, hi = c >> 16;
  uint32_t out = 0;
  if ((lo & 0x8000u) == 0 && lo != 0 && (lo & 0x7FFFu) <= 0x7C00u) out |= d & 0x0000FFFFu;
  if ((hi & 0x8000u) == 0 && hi != 0 && (hi & 0x7FFFu) <= 0x7C00u) out |= d & 0xFFFF0000u;
  return out;
}

// The same for rows that all start 16-byte aligned (the three pointers 16-byte aligned, the
// leading dimensions multiples of 8): thread j of the x range takes 16-byte chunk j of
// kMaskRows rows at a time, with all of their loads issued before the first store (one chunk
// of one row per thread left the pass latency-bound); thread j == N / 8 takes the rows' last
// N mod 8 columns one by one.
constexpr int kMaskRows = 8;

__global__ void __launch_bounds__(256)
    tg_relu_backward_vec_kernel(const uint16_t* __restrict__ dC, int64_t lddc,
                                const uint16_t* __restrict__ C, int64_t ldc,
                                uint16_t* __restrict__ dZ, int64_t lddz, int64_t M, int64_t N) {
  const int64_t chunks = N >> 3;
  const int64_t j = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (j > chunks) return;
  for (int64_t r0 = int64_t(blockIdx.y) * kMaskRows; r0 < M;
       r0 += int64_t(gridDim.y) * kMaskRows) {
    if (j < chunks) {
      uint4 cv[kMaskRows], dv[kMaskRows];
#pragma unroll
      for (int i = 0; i < kMaskRows; ++i) {
        if (r0 + i < M) {
          cv[i] = __ldg(reinterpret_cast<const uint4*>(C + (r0 + i) * ldc) + j);
          dv[i] = __ldg(reinterpret_cast<const uint4*>(dC + (r0 + i) * lddc) + j);
        }
      }
#pragma unroll
      for (int i = 0; i < kMaskRows; ++i) {
        if (r0 + i < M) {
          const uint4 o = make_uint4(relu_grad2(cv[i].x, dv[i].x), relu_grad2(cv[i].y, dv[i].y),
                                     relu_grad2(cv[i].z, dv[i].z), relu_grad2(cv[i].w, dv[i].w));
          *(reinterpret_cast<uint4*>(dZ + (r0 + i) * lddz) + j) = o;
        }
      }
    } else {
      for (int i = 0; i < kMaskRows && r0 + i < M; ++i) {
        for (int64_t c = chunks * 8; c < N; ++c) {
          const uint16_t cv = __ldg(C + (r0 + i) * ldc + c);
          const bool pos = (cv & 0x8000u) == 0 && cv != 0 && (cv & 0x7FFFu) <= 0x7C00u;
          dZ[(r0 + i) * lddz + c] = pos ? __ldg(dC + (r0 + i) * lddc + c) : uint16_t(0);
        }
      }
    }
  }
}

int aux_grid(int64_t work_items, int num_sms, int per_sm = 8) {
  const int64_t blocks = cdiv(std::max<int64_t>(work_items, 1), 256);
  return static_cast<int>(std::min<int64_t>(blocks, int64_t(num_sms) * per_sm));
}

// One operand copy on `per_sm` blocks of 256 threads per SM at most.  For the copies made
// before a single GEMM (`copies_first`), tg_pack_rows4_kernel takes kPackItems 32-chunk
// items per pass, their loads together, when every warp has at least that many: 4096^3 with
// odd strides ran 154 against 165 us per call (one process, one box).  Copies split by split
// beside the GEMMs keep one item per pass: unrolled, 4095 x 3073 x 65537 measured 0-3% faster
// depending on the box, and 300 x 1030 x 65537 2-4% slower.
void launch_pack(const uint16_t* src, int64_t ld_src, uint16_t* dst, int64_t ld_dst,
                 int64_t rows, int64_t cols, int num_sms, int per_sm, bool copies_first,
                 cudaStream_t st) {
  const int64_t cpr = cdiv(cols, 8);
  const int grid = aux_grid(rows * cpr, num_sms, per_sm);
  const int64_t items = rows * cdiv(cpr, 32);
  if (copies_first && items >= kPackItems * int64_t(grid) * 8)
    tg_pack_rows4_kernel<<<grid, 256, 0, st>>>(src, ld_src, dst, ld_dst, rows, cols);
  else
    tg_pack_rows_kernel<<<grid, 256, 0, st>>>(src, ld_src, dst, ld_dst, rows, cols);
}

// Blocks per SM of the operand copies that run beside the GEMM (overlapped copies).  On
// 4095 x 3073 x 65537 (two runs each): 1 block 1.62 ms per step, 2: 1.43, 4: 1.32, 8: 1.33;
// copies first, no overlap: 1.33-1.38.  With fewer blocks the copies themselves become the
// critical path.
constexpr int kOverlapCopyBlocksPerSm = 4;

CUresult encode_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m,
                   CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_ws_3d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base,
                      uint64_t n, uint64_t rows, uint64_t splits, uint64_t ldw) {
  cuuint64_t dims[3] = {n, rows, splits};
  cuuint64_t strides[2] = {ldw * 4, ldw * 4 * rows};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

tg_epilogue epilogue_from_flag(int flag) {
  tg_epilogue e;
  std::memset(&e, 0, sizeof(e));
  e.activation = flag;
  return e;
}

tg_status validate_epilogue(const tg_epilogue& e, const void* C, int64_t N, int64_t ldc) {
  if (e.activation < TG_ACT_NONE || e.activation > TG_ACT_GELU_TANH) return TG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(e.bias) | reinterpret_cast<uintptr_t>(e.residual)) & 1u)
    return TG_ERR_MISALIGNED;
  if (e.residual) {
    if (e.ldr < std::max<int64_t>(1, N) || e.ldr > (int64_t{1} << 36)) return TG_ERR_INVALID_ARG;
    if (e.residual == C && e.ldr != ldc) return TG_ERR_INVALID_ARG;
  }
  return TG_OK;
}

tg_status run_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, const tg_epilogue& epi,
                   const tg_options* opt, cudaStream_t stream, int ta = 0, int tb = 0) {
  tg_status st = validate(A, B, C, M, N, K, lda, ldb, ldc, TG_EPILOGUE_NONE, ta, tb);
  if (st != TG_OK) return st;
  if ((st = validate_epilogue(epi, C, N, ldc)) != TG_OK) return st;
  if (M == 0 || N == 0) return TG_OK;
  DeviceState* ds = nullptr;
  if ((st = current_device(&ds)) != TG_OK) return st;
  cudaError_t e;
  if (K == 0 && epi.bias == nullptr && epi.residual == nullptr) {
    // act(+0) is +0 for every activation: the empty sum writes +0
    e = cudaMemset2DAsync(C, size_t(ldc) * 2, 0, size_t(N) * 2, size_t(M), stream);
    return e == cudaSuccess ? TG_OK : cuda_fail(e);
  }
  if (K == 0) {  // C = act(0 + bias) + residual: the reduction pass over zero splits
    tg::GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.act = epi.activation;
    gp.bias = static_cast<const __half*>(epi.bias);
    gp.residual = static_cast<const __half*>(epi.residual);
    gp.ldr = epi.residual ? epi.ldr : 0;
    gp.M = static_cast<int>(M);
    gp.N = static_cast<int>(N);
    tg_splitk_reduce_kernel<<<reduce_grid(M, N), kReduceThreads, 0, stream>>>(
        nullptr, 0, 0, 0, static_cast<__half*>(C), ldc, gp, 0);
    e = cudaGetLastError();
    return e == cudaSuccess ? TG_OK : cuda_fail(e);
  }
  Plan pl;
  st = make_plan(reinterpret_cast<uintptr_t>(A), reinterpret_cast<uintptr_t>(B),
                 reinterpret_cast<uintptr_t>(C), M, N, K, lda, ldb, ldc, ds->sm_count,
                 ds->pair_clusters, opt, &pl, ta, tb);
  if (st != TG_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((st = encode_fn(&enc)) != TG_OK) return st;
  const tg_plan& P = pl.pub;

  uint8_t* scratch = nullptr;
  if (P.workspace_bytes > 0) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), size_t(P.workspace_bytes),
                                ds->pool, stream);
    if (e != cudaSuccess) {
      t_last_cuda_error = static_cast<int>(e);
      return TG_ERR_NO_WORKSPACE;
    }
  }
  auto fail = [&](tg_status s) {
    if (scratch) cudaFreeAsync(scratch, stream);
    return s;
  };

  const void* Ae = A;
  const void* Be = B;
  int64_t lda_e = lda, ldb_e = ldb;
  uint16_t* Ap = P.repack_a ? reinterpret_cast<uint16_t*>(scratch + pl.off_a) : nullptr;
  uint16_t* Bp = P.repack_b ? reinterpret_cast<uint16_t*>(scratch + pl.off_b) : nullptr;
  // Copies of the K range [k0, k1) of A and B into their aligned scratch (A stored M x K:
  // columns k0..k1 of every row; stored K x M: rows k0..k1; B likewise).
  auto copy_k_range = [&](int64_t k0, int64_t k1, cudaStream_t st, int per_sm,
                          bool copies_first) -> cudaError_t {
    const uint16_t* a16 = static_cast<const uint16_t*>(A);
    const uint16_t* b16 = static_cast<const uint16_t*>(B);
    if (P.repack_a) {
      if (ta)
        launch_pack(a16 + k0 * lda, lda, Ap + k0 * pl.lda_p, pl.lda_p, k1 - k0, M, ds->sm_count,
                    per_sm, copies_first, st);
      else
        launch_pack(a16 + k0, lda, Ap + k0, pl.lda_p, M, k1 - k0, ds->sm_count, per_sm,
                    copies_first, st);
      const cudaError_t ce = cudaGetLastError();
      if (ce != cudaSuccess) return ce;
    }
    if (P.repack_b) {
      if (tb)
        launch_pack(b16 + k0, ldb, Bp + k0, pl.ldb_p, N, k1 - k0, ds->sm_count, per_sm,
                    copies_first, st);
      else
        launch_pack(b16 + k0 * ldb, ldb, Bp + k0 * pl.ldb_p, pl.ldb_p, k1 - k0, N, ds->sm_count,
                    per_sm, copies_first, st);
      return cudaGetLastError();
    }
    return cudaSuccess;
  };
  if (P.repack_a) {
    Ae = Ap;
    lda_e = pl.lda_p;
  }
  if (P.repack_b) {
    Be = Bp;
    ldb_e = pl.ldb_p;
  }
  // Under stream capture the library's side streams would join the caller's graph (and could
  // meet another thread's eager calls there): a captured call takes the sequential path.
  bool overlap = P.repack_overlap != 0;
  if (overlap) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(stream, &cap)) != cudaSuccess) return fail(cuda_fail(e));
    overlap = cap == cudaStreamCaptureStatusNone;
  }
  if (!overlap && (P.repack_a || P.repack_b)) {
    if ((e = copy_k_range(0, K, stream, 8, true)) != cudaSuccess) return fail(cuda_fail(e));
  }

  tg::GemmLaunch L;
  std::memset(&L, 0, sizeof(L));
  // A read in place by row classes: the pre-shifted first windows, then one map per class
  // (class r: base 2 (r lda - e_r) bytes past A, 32-byte aligned because A is and e_r =
  // r lda mod 16; rows 32 lda bytes apart; x = k + e_r)
  tg::AClassMaps cls;
  std::memset(&cls, 0, sizeof(cls));
  const int64_t ws_rows = P.a_row_classes ? P.a_row_classes * pl.cls_rows : M;
  if (P.a_row_classes) {
    uint16_t* first = reinterpret_cast<uint16_t*>(scratch + pl.off_first);
    ClassShifts sh;
    for (int r = 0; r < tg::kARowClasses; ++r) sh.e[r] = pl.cls_shift[r];
    tg_first_window_kernel<<<aux_grid(ws_rows * tg::kBK, ds->sm_count), 256, 0, stream>>>(
        static_cast<const uint16_t*>(A), lda, M, K, pl.cls_rows, sh, first);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(cuda_fail(e));
    CUresult cr = encode_2d(enc, &cls.first, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, first,
                            uint64_t(tg::kBK), uint64_t(ws_rows), uint64_t(tg::kBK) * 2, tg::kBK,
                            tg::kBM);
    for (int r = 0; r < tg::kARowClasses && cr == CUDA_SUCCESS; ++r) {
      const int64_t rows_r = (M - r + tg::kARowClasses - 1) / tg::kARowClasses;  // M >= 256 > r
      const uint16_t* base = static_cast<const uint16_t*>(A) + (int64_t(r) * lda - pl.cls_shift[r]);
      cr = encode_2d(enc, &cls.cls[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base,
                     uint64_t(K + pl.cls_shift[r]), uint64_t(rows_r),
                     uint64_t(lda) * 2 * tg::kARowClasses, tg::kBK, tg::kBM);
    }
    if (cr != CUDA_SUCCESS) return fail(cuda_fail(cudaErrorInvalidValue));
  }
  // A: K-major box {64 K, 128 rows} or, stored K x M, two MN-major boxes {64 M, 64 K};
  // B: MN-major boxes {64 N, 64 K} or, stored N x K, one K-major box {64 K, BN (or 128) rows}
  // the CTA-pair kernel stages 128 k: its MN-major boxes are {64, 128 K}
  const uint32_t mn_box_k = P.cta_pair ? uint32_t(tg::PairCfgFwd::kKB * tg::kBK) : tg::kBK;
  CUresult cr = P.a_row_classes ? CUDA_SUCCESS  // A comes through cls
                : ta ? encode_2d(enc, &L.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Ae, uint64_t(M),
                                 uint64_t(K), uint64_t(lda_e) * 2, 64, mn_box_k)
                     : encode_2d(enc, &L.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Ae, uint64_t(K),
                                 uint64_t(M), uint64_t(lda_e) * 2, tg::kBK, tg::kBM);
  if (cr == CUDA_SUCCESS)
    cr = tb ? encode_2d(enc, &L.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Be, uint64_t(K), uint64_t(N),
                        uint64_t(ldb_e) * 2, tg::kBK, P.cta_pair ? 128u : uint32_t(P.block_n))
            : encode_2d(enc, &L.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Be, uint64_t(N), uint64_t(K),
                        uint64_t(ldb_e) * 2, 64, mn_box_k);
  float* ws = P.workspace_epilogue ? reinterpret_cast<float*>(scratch + pl.off_w) : nullptr;
  if (cr == CUDA_SUCCESS) {
    if (ws)
      cr = encode_ws_3d(enc, &L.out, ws, uint64_t(N), uint64_t(ws_rows), uint64_t(P.split_k),
                        uint64_t(pl.ldw));
    else  // a tile store writes whole 16-byte chunks: the map stops at N rounded down to 8
      cr = encode_2d(enc, &L.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C,
                     uint64_t(std::max<int64_t>(N & ~int64_t{7}, 8)), uint64_t(M),
                     uint64_t(ldc) * 2, 64, 32);
  }
  if (cr != CUDA_SUCCESS) return fail(cuda_fail(cudaErrorInvalidValue));

  tg_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  tg::GemmParams& gp = L.p;
  gp.tiles_m = static_cast<int>(P.tiles_m);
  gp.tiles_n = static_cast<int>(P.tiles_n);
  gp.num_kb = static_cast<int>(P.kblocks);
  gp.kb_per_split = static_cast<int>(P.kblocks_per_split);
  gp.splits = P.split_k;
  gp.units = static_cast<int>(P.units);
  gp.panel_m = P.panel_m;
  gp.act = epi.activation;
  gp.bias = static_cast<const __half*>(epi.bias);
  gp.residual = static_cast<const __half*>(epi.residual);
  gp.ldr = epi.residual ? epi.ldr : 0;
  gp.a_mn = ta;
  gp.b_k = tb;
  if (P.tail_tiles) {
    gp.tail = 1;
    gp.n_full = static_cast<int>(P.units - 2 * P.tail_tiles);
    gp.tail_ws = reinterpret_cast<float*>(scratch + pl.off_tail_ws);
    gp.tail_cnt = reinterpret_cast<int*>(scratch + pl.off_tail_cnt);
    e = cudaMemsetAsync(gp.tail_cnt, 0, size_t(pl.tail_cnt_bytes), stream);
    if (e != cudaSuccess) return fail(cuda_fail(e));
  }
  gp.debug_flags = o.debug_flags;
  gp.timeout_ns = 1000000ull * static_cast<unsigned long long>(o.timeout_ms > 0 ? o.timeout_ms : kDefaultTimeoutMs);
  gp.err = ds->err;
  gp.c = static_cast<__half*>(C);
  gp.ldc = ldc;
  gp.M = static_cast<int>(M);
  gp.N = static_cast<int>(N);
  gp.n_tma = static_cast<int>(N & ~int64_t{7});
  const tg::GemmParams reduce_params = gp;  // the reduction writes C's M rows
  if (P.a_row_classes) {
    gp.M = static_cast<int>(ws_rows);  // the GEMM writes class-major workspace rows
    gp.cls_tiles = static_cast<int>(pl.cls_rows / (2 * tg::kBM));
    for (int r = 0; r < tg::kARowClasses; ++r)
      gp.cls_shift[r] = static_cast<unsigned char>(pl.cls_shift[r]);
  }
  L.grid = P.grid;
  L.stream = stream;
  auto launch = [&](const tg::GemmLaunch& l) -> cudaError_t {
    if (P.a_row_classes) return tg::launch_gemm_pair_cls(cls, l);
    if (P.cta_pair) return tg::launch_gemm_pair(l, ws != nullptr);
    switch (P.block_n) {
      case 256: return tg::launch_gemm_bn256(l, ws != nullptr);
      case 192: return tg::launch_gemm_bn192(l, ws != nullptr);
      default: return tg::launch_gemm_bn128(l, ws != nullptr);
    }
  };
  if (!overlap) {
    if ((e = launch(L)) != cudaSuccess) return fail(cuda_fail(e));
  } else {
    // split s: copy its K slice on ov->copy, then its GEMM (the tiles of split s only) on
    // ov->gemm[s & 1] once the slice is in place; every stream joins back to `stream` before
    // the reduction, on success and on error alike (the scratch is freed on `stream`).
    OverlapStreams* ov = nullptr;
    if ((st = overlap_streams(&ov)) != TG_OK) return fail(st);
    std::lock_guard<std::mutex> lock(ov->mu);
    cudaError_t ce = cudaEventRecord(ov->start, stream);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(ov->copy, ov->start, 0);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(ov->gemm[0], ov->start, 0);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(ov->gemm[1], ov->start, 0);
    const int64_t tiles = P.tiles_m * P.tiles_n;
    const int64_t kspan = P.kblocks_per_split * tg::kBK;
    for (int sp = 0; sp < P.split_k && ce == cudaSuccess; ++sp) {
      const int64_t k0 = sp * kspan, k1 = std::min<int64_t>(K, k0 + kspan);
      cudaStream_t g = ov->gemm[sp & 1];
      // the first split's copy has the GPU to itself
      ce = copy_k_range(k0, k1, ov->copy, sp == 0 ? 8 : kOverlapCopyBlocksPerSm, false);
      if (ce == cudaSuccess) ce = cudaEventRecord(ov->copied[sp], ov->copy);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(g, ov->copied[sp], 0);
      if (ce != cudaSuccess) break;
      tg::GemmLaunch ls = L;
      ls.p.unit_base = static_cast<int>(sp * tiles);
      ls.p.units = static_cast<int>(tiles);
      ls.grid = P.cta_pair ? 2 * static_cast<int>(std::min<int64_t>(tiles, P.grid / 2))
                           : static_cast<int>(std::min<int64_t>(tiles, P.grid));
      ls.stream = g;
      ce = launch(ls);
    }
    cudaError_t je = cudaEventRecord(ov->done[0], ov->copy);
    if (je == cudaSuccess) je = cudaEventRecord(ov->done[1], ov->gemm[0]);
    if (je == cudaSuccess) je = cudaEventRecord(ov->done[2], ov->gemm[1]);
    for (int i = 0; i < 3 && je == cudaSuccess; ++i) je = cudaStreamWaitEvent(stream, ov->done[i], 0);
    if (je != cudaSuccess) {  // cannot order the side streams: wait for them here
      cudaStreamSynchronize(ov->copy);
      cudaStreamSynchronize(ov->gemm[0]);
      cudaStreamSynchronize(ov->gemm[1]);
    }
    if (ce == cudaSuccess) ce = je;
    if (ce != cudaSuccess) return fail(cuda_fail(ce));
  }

  if (ws) {
    tg_splitk_reduce_kernel<<<reduce_grid(M, N), kReduceThreads, 0, stream>>>(
        ws, pl.ldw, ws_rows * pl.ldw, P.split_k, static_cast<__half*>(C), ldc, reduce_params,
        P.a_row_classes ? pl.cls_rows : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(cuda_fail(e));
  }
  if (scratch && (e = cudaFreeAsync(scratch, stream)) != cudaSuccess) return cuda_fail(e);
  return TG_OK;
}

// Library-owned streams and events of the host-buffer entry point, one set per device.
constexpr int kMaxPanels = 8;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done_h2d = nullptr, done_d2h = nullptr;
  cudaEvent_t a_ready[kMaxPanels] = {}, c_ready[kMaxPanels] = {};
  std::mutex mu;
};
HostPipe g_pipes[kMaxDevices];

tg_status host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  HostPipe& hp = g_pipes[dev];
  if (!hp.ready) {
    const unsigned ev = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.start, ev)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.done_h2d, ev)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.done_d2h, ev)) != cudaSuccess)
      return cuda_fail(e);
    for (int i = 0; i < kMaxPanels; ++i)
      if ((e = cudaEventCreateWithFlags(&hp.a_ready[i], ev)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&hp.c_ready[i], ev)) != cudaSuccess)
        return cuda_fail(e);
    hp.ready = true;
  }
  *out = &hp;
  return TG_OK;
}

// rows x width_bytes between pitched buffers: one linear copy when both are dense.
cudaError_t copy_rows(void* dst, int64_t dpitch, const void* src, int64_t spitch,
                      int64_t width_bytes, int64_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (rows <= 0 || width_bytes <= 0) return cudaSuccess;
  if (dpitch == width_bytes && spitch == width_bytes)
    return cudaMemcpyAsync(dst, src, size_t(width_bytes * rows), kind, s);
  return cudaMemcpy2DAsync(dst, size_t(dpitch), src, size_t(spitch), size_t(width_bytes),
                           size_t(rows), kind, s);
}

}  // namespace

namespace tg {
// Hooks for other translation units of this library (not part of the C ABI).
// The tensor maps are encoded with the driver API, which works on the calling thread's
// current context.  cudaGetDevice does not make one current, so a host thread whose first CUDA
// call enters this library would have none: bind the runtime's context for the device once per
// thread (cudaFree(nullptr) initialises it without changing the selected device).
cudaError_t bind_thread_context(int dev) {
  thread_local int bound = -1;
  if (bound == dev) return cudaSuccess;
  const cudaError_t e = cudaFree(nullptr);
  if (e == cudaSuccess) bound = dev;
  return e;
}

tg_status record_cuda_error(cudaError_t e) { return cuda_fail(e); }

tg_status device_info(int* sm_count, unsigned int** err) {
  DeviceState* ds = nullptr;
  tg_status st = current_device(&ds);
  if (st != TG_OK) return st;
  *sm_count = ds->sm_count;
  *err = ds->err;
  return TG_OK;
}

tg_status scratch_alloc(size_t bytes, cudaStream_t stream, void** out) {
  DeviceState* ds = nullptr;
  tg_status st = current_device(&ds);
  if (st != TG_OK) return st;
  const cudaError_t e = cudaMallocFromPoolAsync(out, bytes, ds->pool, stream);
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    return TG_ERR_NO_WORKSPACE;
  }
  return TG_OK;
}

cudaError_t error_word_address(unsigned int** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_tg_error_word);
}

bool tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) { return encode_fn(fn) == TG_OK; }

cudaError_t launch_splitk_reduce(const float* ws, int64_t ldw, int64_t split_stride, int splits,
                                 void* C, int64_t ldc, const GemmParams& p, int num_sms,
                                 cudaStream_t stream) {
  tg_splitk_reduce_kernel<<<reduce_grid(p.M, p.N), kReduceThreads, 0, stream>>>(
      ws, ldw, split_stride, splits, static_cast<__half*>(C), ldc, p, 0);
  return cudaGetLastError();
}

int gemm_stages(int block_n) {
  switch (block_n) {
    case 256: return TileCfg<256>::kStages;
    case 192: return TileCfg<192>::kStages;
    default: return TileCfg<128>::kStages;
  }
}
int gemm_smem_bytes(int block_n) {
  switch (block_n) {
    case 256: return TileCfg<256>::kSmemBytes;
    case 192: return TileCfg<192>::kSmemBytes;
    default: return TileCfg<128>::kSmemBytes;
  }
}
}  // namespace tg

// ------------------------------ exported C ABI ------------------------------
extern "C" {

tg_status tg_gemm_relu_f16(const void* A, const void* B, void* C, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int epilogue_flag,
                           tg_stream_t stream) {
  if (epilogue_flag != TG_EPILOGUE_NONE && epilogue_flag != TG_EPILOGUE_RELU)
    return TG_ERR_INVALID_ARG;
  return run_gemm(A, B, C, M, N, K, lda, ldb, ldc, epilogue_from_flag(epilogue_flag), nullptr,
                  reinterpret_cast<cudaStream_t>(stream));
}

tg_status tg_gemm_relu_f16_ex(const void* A, const void* B, void* C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              int epilogue_flag, const tg_options* opt, tg_stream_t stream) {
  if (epilogue_flag != TG_EPILOGUE_NONE && epilogue_flag != TG_EPILOGUE_RELU)
    return TG_ERR_INVALID_ARG;
  return run_gemm(A, B, C, M, N, K, lda, ldb, ldc, epilogue_from_flag(epilogue_flag), opt,
                  reinterpret_cast<cudaStream_t>(stream));
}

tg_status tg_gemm_f16_epilogue(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                               const tg_epilogue* epi, const tg_options* opt,
                               tg_stream_t stream) {
  return run_gemm(A, B, C, M, N, K, lda, ldb, ldc,
                  epi ? *epi : epilogue_from_flag(TG_EPILOGUE_NONE), opt,
                  reinterpret_cast<cudaStream_t>(stream));
}

tg_status tg_gemm_f16_t(int trans_a, int trans_b, const void* A, const void* B, void* C,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        const tg_epilogue* epi, const tg_options* opt, tg_stream_t stream) {
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return TG_ERR_INVALID_ARG;
  return run_gemm(A, B, C, M, N, K, lda, ldb, ldc,
                  epi ? *epi : epilogue_from_flag(TG_EPILOGUE_NONE), opt,
                  reinterpret_cast<cudaStream_t>(stream), trans_a, trans_b);
}

tg_status tg_relu_backward_f16(const void* dC, const void* C, void* dZ, int64_t M, int64_t N,
                               int64_t lddc, int64_t ldc, int64_t lddz, tg_stream_t stream) {
  if (M < 0 || N < 0) return TG_ERR_INVALID_ARG;
  if (lddc < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N) ||
      lddz < std::max<int64_t>(1, N))
    return TG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TG_OK;
  if (!dC || !C || !dZ) return TG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dC) | reinterpret_cast<uintptr_t>(C) |
       reinterpret_cast<uintptr_t>(dZ)) & 1u)
    return TG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  tg_status st = current_device(&ds);
  if (st != TG_OK) return st;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = ((reinterpret_cast<uintptr_t>(dC) | reinterpret_cast<uintptr_t>(C) |
                     reinterpret_cast<uintptr_t>(dZ)) & 15u) == 0 &&
                   lddc % 8 == 0 && ldc % 8 == 0 && lddz % 8 == 0;
  if (vec) {
    // x: the 16-byte chunks of a row plus one thread for its last N mod 8 columns
    const dim3 grid(static_cast<unsigned>(cdiv(N / 8 + 1, 256)),
                    static_cast<unsigned>(std::min<int64_t>(cdiv(M, kMaskRows), 65535)));
    tg_relu_backward_vec_kernel<<<grid, 256, 0, st_>>>(
        static_cast<const uint16_t*>(dC), lddc, static_cast<const uint16_t*>(C), ldc,
        static_cast<uint16_t*>(dZ), lddz, M, N);
  } else {
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>(cdiv(N, 256), 32)),
                    static_cast<unsigned>(std::min<int64_t>(M, 65535)));
    tg_relu_backward_kernel<<<grid, 256, 0, st_>>>(
        static_cast<const uint16_t*>(dC), lddc, static_cast<const uint16_t*>(C), ldc,
        static_cast<uint16_t*>(dZ), lddz, M, N);
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

tg_status tg_plan_query(const void* A, const void* B, const void* C, int64_t M, int64_t N,
                        int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int num_sms,
                        const tg_options* opt, tg_plan* out) {
  if (out == nullptr) return TG_ERR_INVALID_ARG;
  tg_status st = validate(A, B, C, M, N, K, lda, ldb, ldc, TG_EPILOGUE_RELU);
  if (st != TG_OK) return st;
  Plan pl;
  st = make_plan(reinterpret_cast<uintptr_t>(A), reinterpret_cast<uintptr_t>(B),
                 reinterpret_cast<uintptr_t>(C), M, N, K, lda, ldb, ldc, num_sms, 0, opt, &pl);
  if (st == TG_OK) *out = pl.pub;
  return st;
}

tg_status tg_gemm_relu_f16_host(const void* hA, const void* hB, void* hC, int64_t M, int64_t N,
                                int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                int epilogue_flag, tg_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  tg_status st = validate(hA, hB, hC, M, N, K, lda, ldb, ldc, epilogue_flag);
  if (st != TG_OK) return st;
  if (M == 0 || N == 0) return TG_OK;
  DeviceState* ds = nullptr;
  if ((st = current_device(&ds)) != TG_OK) return st;
  HostPipe* hp = nullptr;
  if ((st = host_pipe(&hp)) != TG_OK) return st;
  std::lock_guard<std::mutex> lock(hp->mu);  // the pipeline's streams and events are shared

  // device copies with 16-byte aligned rows, so the direct (TMA) path applies
  const int64_t lda_d = round_up(std::max<int64_t>(K, 1), 8);
  const int64_t ldb_d = round_up(N, 8);
  const int64_t ldc_d = round_up(N, 8);
  const int64_t bytes_a = round_up(M * lda_d * 2, 256);
  const int64_t bytes_b = round_up(std::max<int64_t>(K, 1) * ldb_d * 2, 256);
  const int64_t bytes_c = round_up(M * ldc_d * 2, 256);
  uint8_t* buf = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf),
                                          size_t(bytes_a + bytes_b + bytes_c), ds->pool, stream);
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    return TG_ERR_NO_WORKSPACE;
  }
  uint8_t* dA = buf;
  uint8_t* dB = buf + bytes_a;
  uint8_t* dC = buf + bytes_a + bytes_b;

  // Row panels: B goes first on the host-to-device stream, then A panel by panel; each
  // panel's GEMM runs on `stream` as soon as its rows have landed, and its C rows go back on
  // the device-to-host stream as soon as it finishes, so copies in both directions overlap
  // the GEMMs of other panels.
  int64_t panels = std::min<int64_t>(kMaxPanels, std::max<int64_t>(1, M / 1024));
  if (K == 0) panels = 1;
  const int64_t rows = round_up(cdiv(M, panels), 256);
  panels = cdiv(M, rows);
  const tg_epilogue epi = epilogue_from_flag(epilogue_flag);
  st = TG_OK;
  if ((e = cudaEventRecord(hp->start, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->h2d, hp->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->d2h, hp->start, 0)) != cudaSuccess)
    st = cuda_fail(e);
  if (st == TG_OK && K > 0 &&
      (e = copy_rows(dB, ldb_d * 2, hB, ldb * 2, N * 2, K, cudaMemcpyHostToDevice, hp->h2d)) !=
          cudaSuccess)
    st = cuda_fail(e);
  for (int64_t pnl = 0; pnl < panels && st == TG_OK; ++pnl) {
    const int64_t r0 = pnl * rows, mr = std::min(rows, M - r0);
    const uint16_t* srcA = static_cast<const uint16_t*>(hA) + r0 * lda;
    if (K > 0 && (e = copy_rows(dA + r0 * lda_d * 2, lda_d * 2, srcA, lda * 2, K * 2, mr,
                                cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess) {
      st = cuda_fail(e);
      break;
    }
    if ((e = cudaEventRecord(hp->a_ready[pnl], hp->h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, hp->a_ready[pnl], 0)) != cudaSuccess) {
      st = cuda_fail(e);
      break;
    }
    st = run_gemm(dA + r0 * lda_d * 2, dB, dC + r0 * ldc_d * 2, mr, N, K, lda_d, ldb_d, ldc_d,
                  epi, nullptr, stream);
    if (st != TG_OK) break;
    uint16_t* dstC = static_cast<uint16_t*>(hC) + r0 * ldc;
    if ((e = cudaEventRecord(hp->c_ready[pnl], stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->d2h, hp->c_ready[pnl], 0)) != cudaSuccess ||
        (e = copy_rows(dstC, ldc * 2, dC + r0 * ldc_d * 2, ldc_d * 2, N * 2, mr,
                       cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess) {
      st = cuda_fail(e);
      break;
    }
  }
  // whatever was queued, the side streams drain before the scratch goes back to the pool
  if ((e = cudaEventRecord(hp->done_h2d, hp->h2d)) == cudaSuccess &&
      (e = cudaEventRecord(hp->done_d2h, hp->d2h)) == cudaSuccess &&
      (e = cudaStreamWaitEvent(stream, hp->done_h2d, 0)) == cudaSuccess)
    e = cudaStreamWaitEvent(stream, hp->done_d2h, 0);
  if (e != cudaSuccess) {
    if (st == TG_OK) st = cuda_fail(e);
    cudaStreamSynchronize(hp->h2d);
    cudaStreamSynchronize(hp->d2h);
  }
  cudaFreeAsync(buf, stream);
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess && st == TG_OK) st = cuda_fail(e);
  if (st == TG_OK) {
    unsigned int word = 0;
    if ((e = cudaMemcpyFromSymbol(&word, g_tg_error_word, sizeof(word))) != cudaSuccess)
      st = cuda_fail(e);
    else if (word != 0)
      st = TG_ERR_TIMEOUT;
  }
  return st;
}

tg_status tg_device_error_check(unsigned* out_word, int clear) {
  DeviceState* ds = nullptr;
  tg_status st = current_device(&ds);
  if (st != TG_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0;
  if ((e = cudaMemcpyFromSymbol(&word, g_tg_error_word, sizeof(word))) != cudaSuccess)
    return cuda_fail(e);
  if (clear) {
    const unsigned int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_tg_error_word, &zero, sizeof(zero))) != cudaSuccess)
      return cuda_fail(e);
  }
  if (out_word) *out_word = word;
  return word ? TG_ERR_TIMEOUT : TG_OK;
}

const char* tg_status_string(tg_status s) {
  switch (s) {
    case TG_OK: return "ok";
    case TG_ERR_INVALID_ARG: return "invalid argument";
    case TG_ERR_MISALIGNED: return "pointer not 2-byte aligned";
    case TG_ERR_UNSUPPORTED_DEVICE: return "unsupported device (compute capability 10.3 required)";
    case TG_ERR_CUDA: return "CUDA error (see tg_last_cuda_error)";
    case TG_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case TG_ERR_NO_WORKSPACE: return "scratch memory unavailable";
  }
  return "unknown status";
}

tg_status tg_last_cuda_error(int* cuda_err) {
  if (cuda_err == nullptr) return TG_ERR_INVALID_ARG;
  *cuda_err = t_last_cuda_error;
  return TG_OK;
}

tg_status tg_release_workspace(void) {
  DeviceState* ds = nullptr;
  tg_status st = current_device(&ds);
  if (st != TG_OK) return st;
  cudaError_t e = cudaMemPoolTrimTo(ds->pool, 0);
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

int tg_version(void) { return 300; }

}  // extern "C"
