// tg_gemm_kernel.cuh — persistent, warp-specialised tcgen05 kernel for C = epi(A·B), sm_103a.
//
// The method is the matmul_relu tile program of the TileLang paper-reading page (section 2):
// per output tile, clear a float32 accumulator, loop over K in pipelined stages that copy an
// A tile and a B tile into shared memory and accumulate their product, then apply max(x, 0)
// elementwise and copy the tile out as fp16.  Section 4 of the same page adds the L2-friendly
// tile order (T.use_swizzle).  The pages' design targets register-file accumulators on
// sm_80/sm_90; this one is written for Blackwell:
//
//   warp 0   producer: one thread issues TMA loads (128B-swizzled boxes) into an S-stage
//            shared-memory ring; full[s]/empty[s] mbarriers hand stages to the MMA thread.
//   warp 1   MMA issuer: allocates tensor memory (TMEM), one thread issues
//            tcgen05.mma.cta_group::1.kind::f16 (128 x BN x 16 per instruction, fp16 in,
//            fp32 accumulate) and tcgen05.commit to release stages; two TMEM accumulators
//            let the epilogue of tile t overlap the main loop of tile t+1.
//   warps 2-5 epilogue: tcgen05.ld the accumulator (each warp owns a 32-lane quarter of
//            TMEM = 32 rows), apply relu (or nothing), round to fp16 (or keep fp32 for a
//            split-K partial), stage the rows in 128B-swizzled shared memory and write them
//            with TMA stores, which clip the M/N tails.
//
// The grid is persistent: CTA b processes work units b, b + gridDim.x, ...  A unit is one
// (split, tile) pair; tiles are ordered in panels of panel_m M-tiles so that CTAs running at
// the same time share A and B panels in L2.
//
// Every mbarrier wait is bounded (p.timeout_ns, measured on %globaltimer); when one runs out
// the thread records the role in *p.err, raises a CTA-wide abort flag and every role drains
// what it has in flight (TMA loads, MMAs, TMA stores) before TMEM is freed and the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tg {

constexpr int kBM = 128;          // UMMA M (TMEM lanes)
constexpr int kBK = 64;           // K per stage: 64 fp16 = 128 bytes = one 128B swizzle row
constexpr int kUmmaK = 16;        // K per tcgen05.mma.kind::f16
constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiWarps = 4;
constexpr int kStagingBuf = 32 * 128;  // one epilogue warp's 32 rows x 128 bytes
constexpr int kSmemLimit = 232448;     // 227 KB opt-in dynamic shared memory per block
constexpr int kSmemReserve = 1024 + 256;

constexpr int kARowClasses = 16;  // row classes of an A read without repacking (AClassMaps)

enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3 };
enum : int { kDebugDropFirstStage = 1 };

struct GemmParams {
  int tiles_m, tiles_n;
  int num_kb;          // ceil(K / kBK)
  int kb_per_split;
  int splits;
  int units;           // work units of this launch: tiles_m * tiles_n * splits, or the
                       // tiles of one split when a plan launches its splits one by one
  int unit_base;       // unit number of this launch's first unit (0, or split * tiles)
  int panel_m;
  int act;             // epilogue activation: kActNone, kActRelu, kActGelu, kActGeluTanh
  int a_mn;            // 1: A is stored K x M (M contiguous): MN-major tiles, two 64-wide boxes
  int b_k;             // 1: B is stored N x K (K contiguous): K-major tiles, one {64, rows} box
  int group_kb;        // int4-weight kernel only: k-blocks per scale group
  // tail split (pair kernel with fp16 output, swapped int4 kernel): units [0, n_full) are
  // whole tiles; each of the remaining tiles is two units, one per K half, that meet through
  // tail_ws / tail_cnt
  int tail;
  int n_full;
  float* tail_ws;      // float32 partials; pair kernel: [slot][half][part = rank*4 + quarter]
                       // [32 rows][256]; swapped int4 kernel: [slot][half][quarter][BMT][32]
  int* tail_cnt;       // [slot][part] arrival counters, zero before the launch
  int debug_flags;
  unsigned long long timeout_ns;
  unsigned int* err;
  // fp16 output only: C itself, for the ragged column tail [n_tma, N) that the TMA store
  // cannot write (a tile store covers whole 16-byte chunks of a row; the tensor map covers
  // columns [0, n_tma) with n_tma = N rounded down to a multiple of 8)
  __half* c;
  long long ldc;
  int M, N, n_tma;
  // optional fused epilogue operands (fp16 output only): bias[j] added to column j before the
  // activation, residual[i*ldr + j] added after it
  const __half* bias;
  const __half* residual;
  long long ldr;
  // A read by row classes (CTA-pair kernel, float32 output; see AClassMaps): M tile m holds
  // rows 16 j + r of class r = m / cls_tiles, j from (m % cls_tiles) * 256; class r's rows
  // start cls_shift[r] elements past a 32-byte boundary, so its K windows (and the matching B
  // rows) start that many elements before each multiple of 64
  int cls_tiles;
  unsigned char cls_shift[kARowClasses];
};

enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2, kActGeluTanh = 3 };

// The activations of the fused epilogue, in float32:
//   relu(x)      = x > 0 ? x : +0                      (-0 and NaN give +0)
//   gelu(x)      = x/2 * (1 + erf(x / sqrt 2))          (Hendrycks & Gimpel, 2016)
//   gelu_tanh(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))   (same paper)
__device__ __forceinline__ float activation(float x, int act) {
  switch (act) {
    case kActRelu: return x > 0.0f ? x : 0.0f;
    case kActGelu: return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
    case kActGeluTanh: {
      const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
      return 0.5f * x * (1.0f + tanhf(u));
    }
    default: return x;
  }
}

// Full epilogue of one float32 sum at (row, col): (sum + bias) -> activation -> + residual.
__device__ __forceinline__ float epilogue_value(float x, int row, int col, const GemmParams& p) {
  if (p.bias) x += __half2float(p.bias[col]);
  x = activation(x, p.act);
  if (p.residual) x += __half2float(p.residual[static_cast<long long>(row) * p.ldr + col]);
  return x;
}

template <int BN>
struct TileCfg {
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64..256 in steps of 64");
  static constexpr int kAStage = kBM * kBK * 2;                 // 16 KB
  static constexpr int kBBox = kBK * 64 * 2;                    // one 64(N) x 64(K) box, 8 KB
  static constexpr int kBStage = kBK * BN * 2;
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kStagingBytes = kEpiWarps * 2 * kStagingBuf;
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve - kStagingBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kAccStride = BN <= 128 ? 128 : 256;      // TMEM columns per accumulator
  static constexpr int kTmemCols = 2 * kAccStride;              // power of two >= 32
  static constexpr int kSmemBytes = kSmemReserve + kStages * kStageBytes + kStagingBytes;
  static_assert(kStages >= 2, "not enough shared memory for a pipeline");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget exceeded");
};

// ---------------------------------------------------------------------------------------
// PTX wrappers (PTX ISA: mbarrier, cp.async.bulk.tensor, tcgen05)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- clusters of two CTAs (the CTA pair of tcgen05 cta_group::2) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// every thread of both CTAs; release/acquire orders shared-memory work across the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an mbarrier that
// may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   holder_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 256 x N x 16 MMA over the CTA pair: A rows 0-127 from this CTA's shared memory and 128-255
// from the peer's (same offset), B columns split in halves the same way; D lanes in each
// CTA's TMEM hold that CTA's 128 rows.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at this shared-memory offset in every CTA of `mask` when the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   holder_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; accumulate == 0 overwrites D (the cleared
// accumulator of the tile program).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: thread l of the warp gets lane (base + l).
// tcgen05.ld is a .sync.aligned instruction: the whole warp must execute it together, so the
// warp is reconverged first (call sites follow lane-dependent branches such as ragged-edge
// stores, after which independent thread scheduling does not promise reconvergence).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's outstanding tcgen05.ld; the registers are threaded through the asm
// so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ---------------------------------------------------------------------------------------
// Descriptors (PTX ISA, tcgen05 "matrix descriptor" and "instruction descriptor")
// ---------------------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle:
//   [0,14) start address >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
//   offset >> 4, [46,49) fixed 0b001, [49,52) base offset (0: atoms are 1024-byte aligned),
//   [52] LBO mode (0), [61,64) layout: 2 = SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// K-major tile (A stored M x K, or B stored N x K): 128 (or BN) rows x 64 K, K contiguous;
// row r at r*128 bytes, 16-byte chunks XOR-swizzled by r%8.  Canonical K-major SW128: 8-row
// groups 1024 bytes apart (SBO); LBO is unused for swizzled K-major layouts (encoded as 16
// bytes).  The k-th 16-wide K slice starts 32*k bytes into the rows.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }

// MN-major tile (B stored K x N, or A stored K x M): 64 K rows x 128 or BN columns, stored
// as boxes of 64 (N or M) x 64 (K), each 8 KB with K row r at r*128 bytes.  Canonical MN-major
// SW128: consecutive 64-wide chunks are LBO = 8 KB apart, consecutive groups of 8 K rows are
// SBO = 1024 bytes apart.  The k-th 16-deep K slice starts 16*128*k = 2048*k bytes in.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) { return sw128_desc(saddr, 8192, 1024); }

// Instruction descriptor for kind::f16: D f32 (bits 4-5 = 1), A f16 (7-9 = 0), B f16
// (10-12 = 0), A major at bit 15 and B major at bit 16 (0: K-major, 1: MN-major), N>>3 at
// 17-22, M>>4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, int a_mn = 0, int b_mn = 1) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Operand tile descriptor and its per-16-K advance (in 16-byte units) for either major:
// K-major tiles advance 32 bytes along the 128-byte row, MN-major tiles advance 16 rows.
__device__ __forceinline__ uint64_t desc_operand(uint32_t saddr, int mn_major) {
  return mn_major ? desc_mnmajor(saddr) : desc_kmajor(saddr);
}
__device__ __forceinline__ uint64_t desc_k_step(int mn_major) { return mn_major ? 128u : 2u; }

// ---------------------------------------------------------------------------------------
// Work decomposition
// ---------------------------------------------------------------------------------------
struct Unit {
  int m_blk, n_blk, split, kb_begin, kb_end;
  int tail_slot;  // -1, or the index of a tail-split tile (split = its K half)
};

// Unit u -> (split, tile); splits are the outer index so that co-running CTAs share a K range.
// Tiles walk panels of panel_m M-tiles, M-tile fastest inside a panel (T.use_swizzle-style
// rasterisation, TileLang paper-reading page, section 4).
// With p.tail, units past n_full are K halves of the last tiles (tile n_full + slot).
__device__ __forceinline__ Unit unit_of(const GemmParams& p, int u) {
  Unit w;
  u += p.unit_base;
  const int tiles = p.tiles_m * p.tiles_n;
  int t;
  w.tail_slot = -1;
  if (p.tail && u >= p.n_full) {
    const int v = u - p.n_full;
    w.tail_slot = v >> 1;
    w.split = v & 1;
    t = p.n_full + w.tail_slot;
  } else {
    w.split = u / tiles;
    t = u - w.split * tiles;
  }
  const int group = p.panel_m * p.tiles_n;
  const int g = t / group;
  const int r = t - g * group;
  const int first_m = g * p.panel_m;
  const int rows = min(p.panel_m, p.tiles_m - first_m);
  w.m_blk = first_m + r % rows;
  w.n_blk = r / rows;
  if (w.tail_slot >= 0) {
    const int half = (p.num_kb + 1) >> 1;
    w.kb_begin = w.split ? half : 0;
    w.kb_end = w.split ? p.num_kb : half;
  } else {
    w.kb_begin = w.split * p.kb_per_split;
    w.kb_end = min(w.kb_begin + p.kb_per_split, p.num_kb);
  }
  return w;
}

// Bounded wait.  Returns false when the CTA is aborting or this wait ran out (then it raises
// the abort flag and records the role in *p.err).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile uint32_t* abort_flag, const GemmParams& p,
                                           uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1u;
        __threadfence_block();
        atomicOr(p.err, 1u | (role << 8));
        return false;
      }
    }
  }
}

// Bounded wait for roles that wait long and gain nothing from waking early (an epilogue
// waiting for a whole tile's main loop): sleeps between polls so that the waiting warp does
// not take issue slots from the warps doing the stage work.
__device__ __forceinline__ bool wait_phase_sleepy(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag,
                                                  const GemmParams& p, uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(256);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1u;
        __threadfence_block();
        atomicOr(p.err, 1u | (role << 8));
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used while draining work already in flight.
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity,
                                                 const GemmParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > p.timeout_ns) return false;
  }
}

__device__ __forceinline__ uint32_t relu_pack_h2(uint32_t a, uint32_t b, int relu) {
  float x = __uint_as_float(a);
  float y = __uint_as_float(b);
  if (relu) {
    x = (x > 0.0f) ? x : 0.0f;  // -0 and NaN become +0
    y = (y > 0.0f) ? y : 0.0f;
  }
  __half2 h = __floats2half2_rn(x, y);  // round to nearest even; x in the low half
  return *reinterpret_cast<uint32_t*>(&h);
}

// Loads 32 fp16 values v[0..31] = src[col .. col+31] (zeros past n): four 16-byte loads when
// the address is 16-byte aligned and all 32 are in range, else guarded 2-byte loads.
__device__ __forceinline__ void load_half32(const __half* src, int col, int n, float (&v)[32]) {
  const __half* q = src + col;
  if (col + 32 <= n && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(q) + j);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[e]));
        v[8 * j + 2 * e] = f.x;
        v[8 * j + 2 * e + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (col + i < n) ? __half2float(q[i]) : 0.0f;
  }
}

// General fused epilogue of 32 consecutive columns of one row: x = acc + bias, activation,
// + residual, then fp16 pairs into pk[0..15].
__device__ __forceinline__ void epilogue_general_32(const uint32_t (&acc)[32], int row, int col,
                                                    const GemmParams& p, uint32_t* pk) {
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(acc[i]);
  if (p.bias) {
    float b[32];
    load_half32(p.bias, col, p.N, b);  // the same 64 bytes for every lane: broadcast
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] += b[i];
  }
  switch (p.act) {
    case kActRelu:
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = activation(x[i], kActRelu);
      break;
    case kActGelu:
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = activation(x[i], kActGelu);
      break;
    case kActGeluTanh:
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = activation(x[i], kActGeluTanh);
      break;
    default:
      break;
  }
  if (p.residual && row < p.M) {
    float r[32];
    load_half32(p.residual + static_cast<long long>(row) * p.ldr, col, p.N, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] += r[i];
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
    pk[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// 64 columns of one row per lane (float32 bits in r0 = columns 0..31, r1 = 32..63): epilogue,
// fp16 pack, 128B-swizzled staging and TMA store of the warp's 32 x 64 block; columns in
// [n_tma, N) are written with plain stores.
__device__ __forceinline__ void store_chunk_f16(const CUtensorMap* tmOut, const GemmParams& p,
                                                const uint32_t (&r0)[32],
                                                const uint32_t (&r1)[32], int row0, int col0,
                                                uint8_t* stg, int& sb, int lane) {
  uint32_t pk[32];
  if (p.bias == nullptr && p.residual == nullptr && p.act <= kActRelu) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      pk[i] = relu_pack_h2(r0[2 * i], r0[2 * i + 1], p.act);
      pk[16 + i] = relu_pack_h2(r1[2 * i], r1[2 * i + 1], p.act);
    }
  } else {
    // general fused epilogue, 32 columns at a time; columns past N and rows past M are
    // computed but never stored
    epilogue_general_32(r0, row0 + lane, col0, p, pk);
    epilogue_general_32(r1, row0 + lane, col0 + 32, p, pk + 16);
  }
  if (col0 < p.n_tma) {
    uint8_t* st = stg + sb * kStagingBuf;
    if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4 v = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      *reinterpret_cast<uint4*>(st + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmOut, smem_u32(st), col0, row0);
      bulk_commit();
    }
    sb ^= 1;
  }
  if (col0 + 64 > p.n_tma && col0 < p.N && row0 + lane < p.M) {
    // ragged tail columns [n_tma, N): plain 2-byte stores of this thread's row
    const int jb = max(p.n_tma, col0) - col0;
    const int je = min(p.N, col0 + 64) - col0;
    unsigned short* dst = reinterpret_cast<unsigned short*>(p.c) +
                          static_cast<long long>(row0 + lane) * p.ldc + col0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (2 * i >= jb && 2 * i < je) dst[2 * i] = static_cast<unsigned short>(pk[i] & 0xFFFFu);
      if (2 * i + 1 >= jb && 2 * i + 1 < je) dst[2 * i + 1] = static_cast<unsigned short>(pk[i] >> 16);
    }
  }
}

// One output tile's epilogue for one warp: TMEM lane quarter at `tl` (32 rows starting at
// row0, BN columns starting at col_base) -> registers -> epilogue -> 128B-swizzled staging ->
// TMA store.  After the last tcgen05.ld the warp releases the accumulator by arriving on
// `release_bar` (a CTA-local barrier, or with `remote` a shared::cluster address of the
// barrier in another CTA of the cluster).
// Within each group of 8 columns, a tile whose B columns were stored in the order
// 0,4,1,5,2,6,3,7 (PERM8) holds output column q at position 2 (q mod 4) + q div 4; this puts
// 32 such columns back in output order (a register reorder, no instructions).
__device__ __forceinline__ void unperm8(uint32_t (&r)[32]) {
  uint32_t t[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) t[i] = r[i];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
#pragma unroll
    for (int q = 0; q < 8; ++q) r[8 * g + q] = t[8 * g + ((q & 3) << 1) + (q >> 2)];
  }
}

template <int BN, bool OUT_F32, bool PERM8 = false>
__device__ __forceinline__ void epilogue_tile(const CUtensorMap* tmOut, const GemmParams& p,
                                              uint32_t tl, int row0, int col_base, int split,
                                              uint8_t* stg, int& sb, uint32_t release_bar,
                                              bool remote, int lane) {
  auto release = [&]() {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (remote)
        mbar_arrive_cluster(release_bar);
      else
        mbar_arrive(release_bar);
    }
  };
  if (row0 >= p.M) {  // none of this warp's 32 rows is in C (e.g. M = 64 under a 128-row tile)
    release();
    return;
  }
  if constexpr (!OUT_F32) {
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      uint32_t r0[32], r1[32];
      tmem_ld_x32(tl + c * 64, r0);
      tmem_wait_ld(r0);
      tmem_ld_x32(tl + c * 64 + 32, r1);
      tmem_wait_ld(r1);
      if (c == BN / 64 - 1) release();
      if constexpr (PERM8) {
        unperm8(r0);
        unperm8(r1);
      }
      store_chunk_f16(tmOut, p, r0, r1, row0, col_base + c * 64, stg, sb, lane);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_x32(tl + c * 32, r);
      tmem_wait_ld(r);
      if (c == BN / 32 - 1) release();
      uint8_t* st = stg + sb * kStagingBuf;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 v = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        *reinterpret_cast<uint4*>(st + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmOut, smem_u32(st), col_base + c * 32, row0, split);
        bulk_commit();
      }
      sb ^= 1;
    }
  }
}

// ---------------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------------
// tmA:   fp16 A, dims {K, M}, box {64, 128}, 128B swizzle   (p.a_mn: dims {M, K}, box {64, 64})
// tmB:   fp16 B, dims {N, K}, box {64, 64}, 128B swizzle    (p.b_k: dims {K, N}, box {64, BN})
// tmOut: OUT_F32 == false: fp16 C, dims {n_tma, M}, box {64, 32}, 128B swizzle (columns
//        [n_tma, N) are written with plain stores through p.c)
//        OUT_F32 == true:  f32 workspace, dims {N, M, splits}, box {32, 32, 1}, 128B swizzle
// GENERAL == false: A K-major and B MN-major fixed at compile time (p.a_mn and p.b_k must be
// 0); the single producer and MMA threads then build descriptors and TMA boxes from constants,
// which keeps their per-k-block instruction count inside the MMA time.  GENERAL == true reads
// the layouts from p.a_mn and p.b_k (the transposed-operand GEMMs of the backward pass).
template <int BN, bool OUT_F32, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1)
    tg_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using Cfg = TileCfg<BN>;
  constexpr int S = Cfg::kStages;
  const int a_mn = GENERAL ? p.a_mn : 0;
  const int b_k = GENERAL ? p.b_k : 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kAStage;
  uint8_t* sStg = sB + S * Cfg::kBStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStagingBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool dropped = false;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const Unit w = unit_of(p, u);
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p, kRoleProducer))
            goto producer_done;
          if ((p.debug_flags & kDebugDropFirstStage) && blockIdx.x == 0 && !dropped) {
            dropped = true;  // injected fault: this stage is never filled
          } else {
            const uint32_t fb = smem_u32(&full[stage]);
            mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
            const uint32_t a_dst = smem_u32(sA + stage * Cfg::kAStage);
            const uint32_t b_dst = smem_u32(sB + stage * Cfg::kBStage);
            if (!a_mn) {
              tma_load_2d(a_dst, &tmA, fb, kb * kBK, w.m_blk * kBM);
            } else {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_2d(a_dst + j * 8192, &tmA, fb, w.m_blk * kBM + j * 64, kb * kBK);
            }
            if (!b_k) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(b_dst + j * Cfg::kBBox, &tmB, fb, w.n_blk * BN + j * 64, kb * kBK);
            } else {
              tma_load_2d(b_dst, &tmB, fb, kb * kBK, w.n_blk * BN);
            }
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:
      // no TMA load may still be writing shared memory when the CTA exits
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) wait_phase_drain(smem_u32(&full[s]), (armed_parity >> s) & 1u, p);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kBM, BN, a_mn, !b_k);
      const uint64_t a_step = desc_k_step(a_mn), b_step = desc_k_step(!b_k);
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
        const Unit w = unit_of(p, u);
        const int buf = t & 1;
        const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
        if (!wait_phase(smem_u32(&tempty[buf]), use ^ 1u, abort_flag, p, kRoleMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        bool ok = true;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&full[stage]), phase, abort_flag, p, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_operand(smem_u32(sA + stage * Cfg::kAStage), a_mn);
          const uint64_t bd = desc_operand(smem_u32(sB + stage * Cfg::kBStage), !b_k);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_f16(d_tmem, ad + a_step * k, bd + b_step * k, idesc,
                     (kb > w.kb_begin || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[buf]));
      }
      // every MMA issued by this thread has finished before TMEM can be released
      umma_commit(smem_u32(drain));
      wait_phase_drain(smem_u32(drain), 0u, p);
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    const int ew = warp - 2;      // staging slot
    uint8_t* stg = sStg + ew * 2 * kStagingBuf;
    int sb = 0;
    int t = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
      const Unit w = unit_of(p, u);
      const int buf = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
      int ok = 0;
      if (lane == 0) ok = wait_phase(smem_u32(&tfull[buf]), use, abort_flag, p, kRoleEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * Cfg::kAccStride);
      epilogue_tile<BN, OUT_F32>(&tmOut, p, tl, w.m_blk * kBM + q * 32, w.n_blk * BN, w.split,
                                 stg, sb, smem_u32(&tempty[buf]), false, lane);
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Epilogue of one K half of a tail-split tile (fp16 output), for one warp of the pair kernel:
// store this half's float32 rows to tail_ws, then count arrivals on the tile's (rank, quarter)
// counter.  The warp that arrives second adds the two halves (a + b == b + a in IEEE
// arithmetic, so the sum does not depend on which half finished last), runs the normal
// epilogue and resets the counter.  No warp waits for another CTA.
template <int BN>
__device__ __forceinline__ void epilogue_tail(const CUtensorMap* tmOut, const GemmParams& p,
                                              uint32_t tl, int row0, int col_base, int slot,
                                              int half, int part, uint8_t* stg, int& sb,
                                              uint32_t release_bar, int lane) {
  // [column][row] within the part: for each column the warp's 32 rows are 128 contiguous
  // bytes, so every store and load below is one coalesced line per warp
  if (row0 >= p.M) {  // none of this warp's rows is in C; the other half skips them too
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(release_bar);
    return;
  }
  const long long per_part = 32LL * BN;
  float* mine = p.tail_ws + ((static_cast<long long>(slot) * 2 + half) * 8 + part) * per_part +
                lane;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_x32(tl + c * 32, r);
    tmem_wait_ld(r);
    if (c == BN / 32 - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(release_bar);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) mine[(c * 32 + j) * 32] = __uint_as_float(r[j]);
  }
  __threadfence();
  __syncwarp();
  int arrived = 0;
  if (lane == 0) arrived = atomicAdd(p.tail_cnt + slot * 8 + part, 1);
  arrived = __shfl_sync(0xffffffffu, arrived, 0);
  if (arrived == 0) return;  // the other half completes this block
  __threadfence();
  const float* other = p.tail_ws + ((static_cast<long long>(slot) * 2 + (half ^ 1)) * 8 + part) *
                                       per_part + lane;
#pragma unroll 1
  for (int c = 0; c < BN / 64; ++c) {
    uint32_t r0[32], r1[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      r0[j] = __float_as_uint(mine[(c * 64 + j) * 32] + __ldcg(other + (c * 64 + j) * 32));
      r1[j] = __float_as_uint(mine[(c * 64 + 32 + j) * 32] +
                              __ldcg(other + (c * 64 + 32 + j) * 32));
    }
    store_chunk_f16(tmOut, p, r0, r1, row0, col_base + c * 64, stg, sb, lane);
  }
  if (lane == 0) p.tail_cnt[slot * 8 + part] = 0;  // ready for the next launch
}

// ---------------------------------------------------------------------------------------
// The CTA-pair kernel: 256 x 256 output tiles computed by a cluster of two CTAs with
// tcgen05.mma.cta_group::2.  CTA r of the pair loads A rows [256m + 128r, +128) and B
// columns [256n + 128r, +128) of each k-block into its own shared memory; both CTAs' TMA
// loads signal the leader's (r = 0) full barrier; the leader alone issues the MMAs, which
// read both CTAs' tiles and accumulate rows [128r, +128) of the 256 x 256 tile into CTA r's
// TMEM.  The leader's tcgen05.commit multicasts to both CTAs' empty (stage free) and
// tmem-full barriers; both CTAs' epilogue warps release an accumulator by arriving on the
// leader's tmem-empty barrier.  Per SM and k-block this moves 32 KB (16 KB A + 16 KB B)
// from L2 instead of the 48 KB of the single-CTA 128 x 256 tile, for the same MMA work.
// ---------------------------------------------------------------------------------------
// KB k-blocks of kBK per pipeline stage.  The forward instance uses KB = 2: its single
// producer and MMA threads then pay one barrier wait, one expect_tx and one commit per 128 k
// instead of per 64 k, which keeps both under the MMA time of a stage (measured per 64 k with
// KB = 1: ~585 cycles in each thread against ~515 cycles of tensor work).
template <int KB>
struct PairCfgT {
  static constexpr int kKB = KB;
  static constexpr int kBN = 256;                       // N of the pair tile
  static constexpr int kHalfN = 128;                    // B columns in each CTA
  static constexpr int kAAtom = kBM * kBK * 2;          // 16 KB: 128 rows x 64 k, K-major
  static constexpr int kAStage = KB * kAAtom;
  static constexpr int kMNBox = KB * kBK * 64 * 2;      // 64 rows or columns x KB*64 k, MN-major
  static constexpr int kBBox = kMNBox;
  static constexpr int kBStage = 2 * kBBox;             // the CTA's 128 columns
  static constexpr int kStageBytes = kAStage + kBStage; // KB x 32 KB per CTA
  static constexpr int kStagingBytes = kEpiWarps * 2 * kStagingBuf;
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve - kStagingBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kAccStride = 256;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemBytes = kSmemReserve + kStages * kStageBytes + kStagingBytes;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget exceeded");
};
using PairCfgFwd = PairCfgT<2>;

// A with a leading dimension that TMA cannot describe (lda * 2 not a multiple of 16), read in
// place through row classes instead of being copied into aligned scratch.  Rows i = 16 j + r
// (class r) lie 32 * lda bytes apart, a multiple of 32, so every row of a class starts at the
// same offset from a 32-byte boundary: e_r elements past it.  Map cls[r] starts at that
// boundary before row r (A itself 32-byte aligned), so element (16 j + r, k) sits at x = k + e_r
// of row j: the box at x = 64 kb holds k in [64 kb - e_r, 64 kb - e_r + 64), every row of the
// class the same window, and the B tile is loaded from K row 64 kb - e_r to match (B's K
// coordinate has no alignment rule; rows before 0 or past K read as zero).  The first window
// would hold e_r elements before the row's start, so it comes from `first`: a small copy of
// each row's window [-e_r, 64 - e_r) with zeros before k = 0, in class-major row order.
struct AClassMaps {
  CUtensorMap cls[kARowClasses];  // fp16, dims {K + e_r, rows of class r}, row stride 32 lda bytes,
                                  // box {64, 128}, 128B swizzle
  CUtensorMap first;              // fp16, dims {64, 16 * class rows}, box {64, 128}, 128B swizzle
};

// Same maps as tg_gemm_tc_kernel, with the operand layouts fixed at compile time (A_MN: A stored
// K x M; B_K: B stored N x K) and 128-k stages: MN-major operands come as {64, 128 K} boxes,
// K-major ones as one {64 K, 128} box per 64-k block.  tiles_m/tiles_n in p count 256 x 256
// pair tiles.  With A_CLS (float32 output, forward layout) A comes through `cls` (tmA unused)
// and M tiles index class-major rows.
template <bool OUT_F32, bool A_MN, bool B_K, bool A_CLS>
__device__ __forceinline__ void pair_gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                               const CUtensorMap& tmOut, const GemmParams& p,
                                               const AClassMaps* cls) {
  static_assert(!A_CLS || (OUT_F32 && !A_MN && !B_K), "row classes: float32 output, forward layout");
  using Cfg = PairCfgFwd;
  constexpr int S = Cfg::kStages;
  constexpr int KB = Cfg::kKB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kAStage;
  uint8_t* sStg = sB + S * Cfg::kBStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStagingBytes);
  uint64_t* full = bars;        // used in the leader
  uint64_t* empty = bars + S;   // in both CTAs
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2; // used in the leader
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if constexpr (A_CLS) {
      prefetch_tmap(&cls->first);
    } else {
      prefetch_tmap(&tmA);
    }
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------ TMA producer (both CTAs) ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool dropped = false;
      for (int u = cluster; u < p.units; u += nclusters) {
        const Unit w = unit_of(p, u);
        const int arow = w.m_blk * 2 * kBM + static_cast<int>(rank) * kBM;
        const int bcol = w.n_blk * Cfg::kBN + static_cast<int>(rank) * Cfg::kHalfN;
        int a_class = 0, a_crow = 0, k_shift = 0;  // A_CLS: the tile's class, its row in it
        if constexpr (A_CLS) {
          a_class = w.m_blk / p.cls_tiles;
          a_crow = (w.m_blk - a_class * p.cls_tiles) * 2 * kBM + static_cast<int>(rank) * kBM;
          k_shift = p.cls_shift[a_class];
        }
        for (int kb = w.kb_begin; kb < w.kb_end; kb += KB) {
          if (!wait_phase(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p, kRoleProducer))
            goto pair_producer_done;
          if ((p.debug_flags & kDebugDropFirstStage) && cluster == 0 && rank == 0 && !dropped) {
            dropped = true;  // injected fault: the leader never arms this stage
          } else {
            const uint32_t fb_local = smem_u32(&full[stage]);
            const uint32_t fb = mapa_shared(fb_local, 0);
            if (rank == 0) {
              mbar_arrive_expect_tx(fb_local, 2 * Cfg::kStageBytes);
              armed |= 1u << stage;
              armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
            const uint32_t a_dst = smem_u32(sA + stage * Cfg::kAStage);
            const uint32_t b_dst = smem_u32(sB + stage * Cfg::kBStage);
            // both k-blocks always load (a second one past the unit's range is never used by
            // the MMA; past K it is zero fill), so the stage's byte count is fixed
            if constexpr (A_CLS) {
#pragma unroll
              for (int h = 0; h < KB; ++h) {
                if (kb + h == 0)  // the first window, zeros before k = 0
                  tma_load_2d_pair(a_dst + h * Cfg::kAAtom, &cls->first, fb, 0, arow);
                else
                  tma_load_2d_pair(a_dst + h * Cfg::kAAtom, &cls->cls[a_class], fb,
                                   (kb + h) * kBK, a_crow);
              }
            } else if constexpr (!A_MN) {
#pragma unroll
              for (int h = 0; h < KB; ++h)
                tma_load_2d_pair(a_dst + h * Cfg::kAAtom, &tmA, fb, (kb + h) * kBK, arow);
            } else {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_2d_pair(a_dst + j * Cfg::kMNBox, &tmA, fb, arow + j * 64, kb * kBK);
            }
            if constexpr (!B_K) {
#pragma unroll
              for (int j = 0; j < Cfg::kHalfN / 64; ++j)
                tma_load_2d_pair(b_dst + j * Cfg::kMNBox, &tmB, fb, bcol + j * 64,
                                 kb * kBK - k_shift);
            } else {
#pragma unroll
              for (int h = 0; h < KB; ++h)
                tma_load_2d_pair(b_dst + h * Cfg::kAAtom, &tmB, fb, (kb + h) * kBK, bcol);
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    pair_producer_done:
      // the leader's full barriers count both CTAs' bytes: once they completed, no load of
      // either CTA is still writing shared memory
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) wait_phase_drain(smem_u32(&full[s]), (armed_parity >> s) & 1u, p);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer (leader) ------------------------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(2 * kBM, Cfg::kBN, A_MN, !B_K);
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      for (int u = cluster; u < p.units; u += nclusters, ++t) {
        const Unit w = unit_of(p, u);
        const int buf = t & 1;
        const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
        if (!wait_phase(smem_u32(&tempty[buf]), use ^ 1u, abort_flag, p, kRoleMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        bool ok = true;
        for (int kb = w.kb_begin; kb < w.kb_end; kb += KB) {
          if (!wait_phase(smem_u32(&full[stage]), phase, abort_flag, p, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K-major operand: KB atoms kAAtom apart, 32 bytes per 16 k inside an atom;
          // MN-major operand: 128 k rows per 64-wide box (boxes kMNBox apart: the leading byte
          // offset), 2048 bytes per 16 k
          const uint32_t a_addr = smem_u32(sA + stage * Cfg::kAStage);
          const uint32_t b_addr = smem_u32(sB + stage * Cfg::kBStage);
          const uint64_t ad = A_MN ? sw128_desc(a_addr, Cfg::kMNBox, 1024) : desc_kmajor(a_addr);
          const uint64_t bd = B_K ? desc_kmajor(b_addr) : sw128_desc(b_addr, Cfg::kMNBox, 1024);
          const int nk = (w.kb_end - kb >= KB ? KB : w.kb_end - kb) * (kBK / kUmmaK);
#pragma unroll
          for (int k = 0; k < KB * (kBK / kUmmaK); ++k) {
            const uint64_t koff_k = static_cast<uint64_t>((k >> 2) * (Cfg::kAAtom >> 4) + 2 * (k & 3));
            const uint64_t koff_mn = static_cast<uint64_t>(128 * k);
            if (k < nk)
              umma_f16_pair(d_tmem, ad + (A_MN ? koff_mn : koff_k), bd + (B_K ? koff_k : koff_mn),
                            idesc, (kb > w.kb_begin || k > 0) ? 1u : 0u);
          }
          umma_commit_pair_mc(smem_u32(&empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(smem_u32(&tfull[buf]), 0x3);
      }
      umma_commit_pair(smem_u32(drain));
      wait_phase_drain(smem_u32(drain), 0u, p);
    }
  } else {
    // ------------------------------ epilogue (both CTAs) ------------------------------
    const int q = warp & 3;
    const int ew = warp - 2;
    uint8_t* stg = sStg + ew * 2 * kStagingBuf;
    int sb = 0;
    int t = 0;
    for (int u = cluster; u < p.units; u += nclusters, ++t) {
      const Unit w = unit_of(p, u);
      const int buf = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
      int ok = 0;
      if (lane == 0) ok = wait_phase(smem_u32(&tfull[buf]), use, abort_flag, p, kRoleEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * Cfg::kAccStride);
      const int row0 = w.m_blk * 2 * kBM + static_cast<int>(rank) * kBM + q * 32;
      const uint32_t release_bar = mapa_shared(smem_u32(&tempty[buf]), 0);
      if (!OUT_F32 && w.tail_slot >= 0)
        epilogue_tail<Cfg::kBN>(&tmOut, p, tl, row0, w.n_blk * Cfg::kBN, w.tail_slot, w.split,
                                static_cast<int>(rank) * 4 + q, stg, sb, release_bar, lane);
      else
        epilogue_tile<Cfg::kBN, OUT_F32>(&tmOut, p, tl, row0, w.n_blk * Cfg::kBN, w.split, stg,
                                         sb, release_bar, true, lane);
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  }

  // After an abort the follower cannot observe its own loads (they complete on the leader's
  // barriers): give any that are still in flight time to land before the CTA can exit.
  if (rank != 0 && *abort_flag && threadIdx.x == 0) __nanosleep(200000);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // all MMAs into either CTA's TMEM and all remote arrivals are done
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

template <bool OUT_F32, bool A_MN, bool B_K>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tg_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut,
                        const __grid_constant__ GemmParams p) {
  pair_gemm_body<OUT_F32, A_MN, B_K, false>(tmA, tmB, tmOut, p, nullptr);
}

// The CTA-pair kernel with A read through row classes (float32 partials, forward layout).
// CLASSES is always kARowClasses (a template so that every unit including this header shares
// one definition).
template <int CLASSES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tg_gemm_pair_cls_kernel(const __grid_constant__ AClassMaps tmAc,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmOut,
                            const __grid_constant__ GemmParams p) {
  static_assert(CLASSES == kARowClasses, "one class count");
  pair_gemm_body<true, false, false, true>(tmAc.first, tmB, tmOut, p, &tmAc);
}

}  // namespace tg
