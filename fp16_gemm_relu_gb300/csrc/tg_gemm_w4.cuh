// tg_gemm_w4.cuh — C = epilogue(A · dequant(Wq)) with fp16 activations A (M x K) and 4-bit
// integer weights (the W_INT4 / A_FP16 dequantising GEMM of the TileLang paper-reading page,
// section 5), on the same tcgen05 main loop as tg_gemm_tc_kernel.
//
// Weight format: Wq is K rows of ceil(N/8) uint32 words; word (k, c) carries columns
// 8c..8c+7, column 8c+e in bits [4e, 4e+4), unsigned q in [0, 15] with zero point 8.  scales
// is ceil(K/G) rows of N fp16 values, G a multiple of 64.  w[k][n] = fp16((q - 8) * s[k/G][n]),
// the product rounded once (fp16 subtract of 1032 from the exact 1024 + q, then an fp16
// multiply: both IEEE round-to-nearest-even).
//
// Warp roles (448 threads):
//   warp 0     TMA: per stage the A tile, the packed Wq tile (64 rows x BN/8 words) and the
//              group's scale row (BN fp16), all on one load_full barrier.
//   warp 1     tcgen05.mma issuer; waits for load_full (A) and deq_full (decoded B).
//   warps 2-5  epilogue (shared with the fp16 kernels).
//   warps 6-13 dequantisers: read packed words and scales from shared memory, decode eight
//              weights per word in registers and store them as the 128B-swizzled MN-major B
//              tile the MMA expects; then fence.proxy.async and arrive on deq_full.
// TMA zero fill makes the tails safe: scales past N or past the last group are 0, so those
// weights decode to 0 whatever their nibbles.
//
// Every kernel here is a template over the weight format FMT: kFmtInt4 above, or kFmtNf4, the
// W_NF4 / A_FP16 case of the same page: the same packing, with each nibble indexing the 16
// NF4 code values of QLoRA (Dettmers et al., NeurIPS 2023, Appendix E) held in fp16,
// w[k][n] = fp16(code16[q] * s[k/G][n]), one rounding of the exact fp16 x fp16 product.
#pragma once

#include "tg_gemm_kernel.cuh"

namespace tg {

constexpr int kDeqWarps = 8;  // two per scheduler (see kW4TDeqWarps)
constexpr int kW4Threads = (2 + 4 + kDeqWarps) * 32;

template <int BN>
struct W4Cfg {
  static constexpr int kAStage = kBM * kBK * 2;   // 16 KB fp16 A
  static constexpr int kBStage = kBK * BN * 2;    // decoded fp16 B tile
  static constexpr int kQStage = kBK * BN / 2;    // packed int4 tile
  static constexpr int kSStage = 1024;            // one scale row (BN fp16), padded
  static constexpr int kStageBytes = kAStage + kBStage + kQStage + kSStage;
  static constexpr int kTxBytes = kAStage + kQStage + BN * 2;
  static constexpr int kStagingBytes = kEpiWarps * 2 * kStagingBuf;
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve - kStagingBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kAccStride = BN <= 128 ? 128 : 256;
  static constexpr int kTmemCols = 2 * kAccStride;
  static constexpr int kSmemBytes = kSmemReserve + kStages * kStageBytes + kStagingBytes;
  static_assert(kStages >= 2, "not enough shared memory");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget exceeded");
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

// ---- tensor-memory operand path of the swapped kernel (TDEC) ----
// D[tmem] (+)= A[tmem] * B[smem desc]: A (M = 128 rows in TMEM lanes, 16 k as eight 32-bit
// columns of fp16 pairs, k even in the low half) read from tensor memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns from registers: thread l writes lane
// (base + l).  Like tcgen05.ld, a .sync.aligned instruction: the warp is reconverged first.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Wait until this thread's tcgen05.st have written tensor memory.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


enum : int { kFmtInt4 = 0, kFmtNf4 = 1 };

// PTX prmt.b32 in its default mode: result byte i is byte (c >> 4i) & 7 of {b, a} (a holds
// bytes 0-3); when bit 3 of that selector nibble is set, the byte's sign bit is replicated
// into all eight bits instead.
__device__ __forceinline__ uint32_t prmt_ptx(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The 16 NF4 code values (QLoRA, Appendix E) rounded to fp16, split into their low and high
// bytes: byte e of kNf4Lo<j> is the low byte of code 4j + e.  Codes in order:
// -1, -0.6962, -0.5251, -0.3949, -0.2844, -0.1848, -0.09105, 0, 0.07958, 0.1609, 0.2461,
// 0.3379, 0.4407, 0.5626, 0.7230, 1 = fp16 0xbc00 0xb992 0xb833 0xb652 0xb48d 0xb1ea 0xadd4
// 0x0000 0x2d18 0x3126 0x33e0 0x3568 0x370d 0x3880 0x39c9 0x3c00.
constexpr uint32_t kNf4Lo0 = 0x52339200u, kNf4Lo1 = 0x00d4ea8du;
constexpr uint32_t kNf4Lo2 = 0x68e02618u, kNf4Lo3 = 0x00c9800du;
constexpr uint32_t kNf4Hi0 = 0xb6b8b9bcu, kNf4Hi1 = 0x00adb1b4u;
constexpr uint32_t kNf4Hi2 = 0x3533312du, kNf4Hi3 = 0x3c393837u;

// Four 16-entry byte lookups at once: byte i of the result is byte q_i of the table
// {t0, t1, t2, t3}, with sel holding (q_i & 7) in nibble i and hi8 0xFF in byte i where q_i >= 8.
__device__ __forceinline__ uint32_t lut16x4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3,
                                            uint32_t sel, uint32_t hi8) {
  const uint32_t lo = prmt_ptx(t0, t1, sel);
  const uint32_t hi = prmt_ptx(t2, t3, sel);
  return (lo & ~hi8) | (hi & hi8);
}

// Eight NF4 weights of one packed word, in column order: pr[j] holds columns (2j, 2j+1);
// sv holds the eight columns' fp16 scales in the same order.
__device__ __forceinline__ uint4 dequant8_nf4(uint32_t w, const uint4& sv) {
  const uint32_t sel_lo = w & 0x7777u;          // q0..q3 (low 3 bits)
  const uint32_t sel_hi = (w >> 16) & 0x7777u;  // q4..q7
  // byte i of hi8_lo is 0xFF when bit 3 of q_i is set: bits 3, 11 sit at the sign bits of
  // the bytes of w << 4, bits 7, 15 at those of w (likewise bits 19..31 for q4..q7)
  const uint32_t w4 = w << 4;
  const uint32_t hi8_lo = prmt_ptx(w4, w, 0xD9C8u);
  const uint32_t hi8_hi = prmt_ptx(w4, w, 0xFBEAu);
  const uint32_t l03 = lut16x4(kNf4Lo0, kNf4Lo1, kNf4Lo2, kNf4Lo3, sel_lo, hi8_lo);
  const uint32_t h03 = lut16x4(kNf4Hi0, kNf4Hi1, kNf4Hi2, kNf4Hi3, sel_lo, hi8_lo);
  const uint32_t l47 = lut16x4(kNf4Lo0, kNf4Lo1, kNf4Lo2, kNf4Lo3, sel_hi, hi8_hi);
  const uint32_t h47 = lut16x4(kNf4Hi0, kNf4Hi1, kNf4Hi2, kNf4Hi3, sel_hi, hi8_hi);
  uint32_t c[4] = {prmt_ptx(l03, h03, 0x5140u), prmt_ptx(l03, h03, 0x7362u),
                   prmt_ptx(l47, h47, 0x5140u), prmt_ptx(l47, h47, 0x7362u)};
  const uint32_t s[4] = {sv.x, sv.y, sv.z, sv.w};
  uint32_t pr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&c[j]),
                        *reinterpret_cast<const __half2*>(&s[j]));  // one rounding
    pr[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(pr[0], pr[1], pr[2], pr[3]);
}

// Eight weights of one packed word; sp[e] holds the scales of columns (e, e+4).  Returns the
// fp16 weights in the column order 0,4,1,5,2,6,3,7, two per 32-bit word: the order in which
// the nibble pairs come out.  The kernels store the decoded tile in that order and undo it in
// their epilogues (a register reorder, or the lane's output column), which saves the four
// byte permutes per word that column order would cost.
__device__ __forceinline__ uint4 dequant8(uint32_t w, const uint32_t (&sp)[4]) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  uint32_t pr[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t x = ((w >> (4 * e)) & 0x000F000Fu) | 0x64006400u;  // (1024+q_e, 1024+q_e+4)
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), k1032);  // q - 8, exact
    h = __hmul2(h, *reinterpret_cast<const __half2*>(&sp[e]));        // one rounding
    pr[e] = *reinterpret_cast<uint32_t*>(&h);                          // columns (e, e+4)
  }
  return make_uint4(pr[0], pr[1], pr[2], pr[3]);
}

// Output column held at position l of a decoded tile (see dequant8).
__device__ __forceinline__ int perm8_column(int l) {
  return (l & ~7) + ((l & 1) << 2) + ((l & 7) >> 1);
}

// The decoded tile of format FMT stores its columns permuted (int4) or in order (NF4).
template <int FMT>
__device__ __forceinline__ int decoded_column(int l) {
  return FMT == kFmtInt4 ? perm8_column(l) : l;
}

// Per-stage scale operands of a dequantiser thread from its eight columns' scales sv.
template <int FMT>
__device__ __forceinline__ void scale_pairs(const uint4& sv, uint32_t (&sp)[4]) {
  if constexpr (FMT == kFmtInt4) {
    sp[0] = prmt(sv.x, sv.z, 0x5410);  // columns (0, 4), as dequant8 pairs them
    sp[1] = prmt(sv.x, sv.z, 0x7632);
    sp[2] = prmt(sv.y, sv.w, 0x5410);
    sp[3] = prmt(sv.y, sv.w, 0x7632);
  } else {
    sp[0] = sv.x;
    sp[1] = sv.y;
    sp[2] = sv.z;
    sp[3] = sv.w;
  }
}

// Two weights of one column in consecutive K rows, t0 and t1 holding each row's nibble in
// bits 0-3 (higher bits are ignored), scaled by s2 = (s, s): fp16 pair (row k low, k + 1 high).
template <int FMT>
__device__ __forceinline__ uint32_t decode_pair(uint32_t t0, uint32_t t1, uint32_t s2) {
  uint32_t c;
  if constexpr (FMT == kFmtInt4) {
    // (1024 + q0, 1024 + q1) as fp16, minus 1032: q - 8 exactly
    const uint32_t x = (prmt_ptx(t0, t1, 0x5410u) & 0x000F000Fu) | 0x64006400u;
    const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), k1032);
    c = *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const uint32_t v = prmt_ptx(t0, t1, 0x0040u);          // byte 0: t0's, byte 1: t1's low byte
    const uint32_t sel = (v & 0x7u) | ((v >> 4) & 0x70u);  // nibbles q0 & 7, q1 & 7
    const uint32_t hi8 = prmt_ptx(v << 4, 0u, 0x0098u);    // byte i: 0xFF where q_i >= 8
    const uint32_t lo = lut16x4(kNf4Lo0, kNf4Lo1, kNf4Lo2, kNf4Lo3, sel, hi8);
    const uint32_t hi = lut16x4(kNf4Hi0, kNf4Hi1, kNf4Hi2, kNf4Hi3, sel, hi8);
    c = prmt_ptx(lo, hi, 0x5140u);                         // (code q0, code q1)
  }
  const __half2 w = __hmul2(*reinterpret_cast<const __half2*>(&c),
                            *reinterpret_cast<const __half2*>(&s2));  // one rounding
  return *reinterpret_cast<const uint32_t*>(&w);
}

template <int FMT>
__device__ __forceinline__ uint4 decode8(uint32_t w, const uint32_t (&sp)[4]) {
  if constexpr (FMT == kFmtInt4) {
    return dequant8(w, sp);
  } else {
    return dequant8_nf4(w, make_uint4(sp[0], sp[1], sp[2], sp[3]));
  }
}

// Eight int4 weights of one packed word in column order: pr[j] holds columns (2j, 2j+1), sv the
// eight columns' fp16 scales in the same order.  The arithmetic of dequant8 per weight:
// (1024 + q) - 1032 = q - 8 exactly, then one rounding in the product with the scale.
__device__ __forceinline__ uint4 dequant8_in_order(uint32_t w, const uint4& sv) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const uint32_t s[4] = {sv.x, sv.y, sv.z, sv.w};
  uint32_t pr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = w >> (8 * j);  // columns 2j and 2j+1 in bits [0, 4) and [4, 8)
    const uint32_t x = (t & 0xFu) | ((t & 0xF0u) << 12) | 0x64006400u;
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), k1032);
    h = __hmul2(h, *reinterpret_cast<const __half2*>(&s[j]));
    pr[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(pr[0], pr[1], pr[2], pr[3]);
}

// The whole weight matrix decoded to fp16, for the decode-first plan of large M: w16[k][n] is
// the weight of row k, column n (K rows of ldw >= N rounded up to 8 values), the same values
// the fused kernels feed their MMAs; the columns of the last word past N are written as +0.
// Thread x of block (bx, by) takes word column c = bx * 256 + x of the row chunks by,
// by + gridDim.y, ... of kDequantRows rows each.  A chunk's loads are all issued before its
// first store, so each thread keeps that many DRAM reads in flight (one row per thread left
// the pass latency-bound: 43.5 us, 3.9 TB/s, on 8192 x 8192).  A chunk starts at a multiple of
// kDequantRows and the group size is a multiple of 64, so a chunk's rows share one scale row.
constexpr int kDequantRows = 8;

template <int FMT>
__global__ void __launch_bounds__(256)
    tg_dequant_kernel(const uint32_t* __restrict__ wq, int64_t ldq,
                      const uint16_t* __restrict__ scales, int64_t lds, int group_size,
                      int64_t K, int64_t N, uint16_t* __restrict__ w16, int64_t ldw) {
  constexpr int R = kDequantRows;
  const int64_t words = (N + 7) / 8;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= words) return;
  const bool whole = 8 * c + 8 <= N;
  for (int64_t k0 = static_cast<int64_t>(blockIdx.y) * R; k0 < K;
       k0 += static_cast<int64_t>(gridDim.y) * R) {
    uint32_t w[R];
#pragma unroll
    for (int j = 0; j < R; ++j) w[j] = k0 + j < K ? __ldg(wq + (k0 + j) * ldq + c) : 0u;
    const uint16_t* srow = scales + (k0 / group_size) * lds + 8 * c;
    uint4 sv;
    if (whole) {
      sv = __ldg(reinterpret_cast<const uint4*>(srow));
    } else {
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = 8 * c + 2 * j < N ? __ldg(srow + 2 * j) : 0u;
        const uint32_t hi = 8 * c + 2 * j + 1 < N ? __ldg(srow + 2 * j + 1) : 0u;
        h[j] = lo | (hi << 16);
      }
      sv = make_uint4(h[0], h[1], h[2], h[3]);
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (k0 + j < K) {
        uint4 v = FMT == kFmtInt4 ? dequant8_in_order(w[j], sv) : dequant8_nf4(w[j], sv);
        if (!whole) {  // columns past N: +0
          uint32_t o[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (8 * c + 2 * q >= N) o[q] &= 0xFFFF0000u;
            if (8 * c + 2 * q + 1 >= N) o[q] &= 0x0000FFFFu;
          }
          v = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(w16 + (k0 + j) * ldw + 8 * c) = v;
      }
    }
  }
}

// tmA: fp16 A {K, M} box {64, 128} SW128; tmQ: uint32 Wq {ceil(N/8), K} box {BN/8, 64};
// tmS: fp16 scales {N, ceil(K/G)} box {BN, 1}; tmOut: fp16 C {n_tma, M} box {64, 32} SW128.
// p.splits must be 1; p.kb_per_split = p.num_kb; p.group_kb = G / 64.
template <int BN, int FMT>
__global__ void __launch_bounds__(kW4Threads, 1)
    tg_gemm_w4_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmS,
                      const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using Cfg = W4Cfg<BN>;
  constexpr int S = Cfg::kStages;
  constexpr int W = BN / 8;  // packed words per row

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kAStage;
  uint8_t* sQ = sB + S * Cfg::kBStage;
  uint8_t* sS = sQ + S * Cfg::kQStage;
  uint8_t* sStg = sS + S * Cfg::kSStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStagingBytes);
  uint64_t* load_full = bars;
  uint64_t* deq_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* tfull = bars + 3 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&load_full[s]), 1);
      mbar_init(smem_u32(&deq_full[s]), kDeqWarps);
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
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmS);
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
        // scale row of k-block kb: g = kb / group_kb, advanced with a counter (one division
        // per tile instead of one per stage on the single producer thread)
        int g = w.kb_begin / p.group_kb;
        int g_rem = w.kb_begin - g * p.group_kb;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p, kRoleProducer))
            goto w4_producer_done;
          if ((p.debug_flags & kDebugDropFirstStage) && blockIdx.x == 0 && !dropped) {
            dropped = true;  // injected fault: this stage is never filled
          } else {
            const uint32_t fb = smem_u32(&load_full[stage]);
            mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
            tma_load_2d(smem_u32(sA + stage * Cfg::kAStage), &tmA, fb, kb * kBK, w.m_blk * kBM);
            tma_load_2d(smem_u32(sQ + stage * Cfg::kQStage), &tmQ, fb, w.n_blk * W, kb * kBK);
            tma_load_2d(smem_u32(sS + stage * Cfg::kSStage), &tmS, fb, w.n_blk * BN, g);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++g_rem == p.group_kb) {
            g_rem = 0;
            ++g;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    w4_producer_done:
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) wait_phase_drain(smem_u32(&load_full[s]), (armed_parity >> s) & 1u, p);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kBM, BN, 0, 1);
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
          if (!wait_phase(smem_u32(&load_full[stage]), phase, abort_flag, p, kRoleMma) ||
              !wait_phase(smem_u32(&deq_full[stage]), phase, abort_flag, p, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_kmajor(smem_u32(sA + stage * Cfg::kAStage));
          const uint64_t bd = desc_mnmajor(smem_u32(sB + stage * Cfg::kBStage));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_f16(d_tmem, ad + 2u * k, bd + 128u * k, idesc, (kb > w.kb_begin || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[buf]));
      }
      umma_commit(smem_u32(drain));
      wait_phase_drain(smem_u32(drain), 0u, p);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const int ew = warp - 2;
    uint8_t* stg = sStg + ew * 2 * kStagingBuf;
    int sb = 0;
    int t = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
      const Unit w = unit_of(p, u);
      const int buf = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
      int ok = 0;
      if (lane == 0)
        ok = wait_phase_sleepy(smem_u32(&tfull[buf]), use, abort_flag, p, kRoleEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * Cfg::kAccStride);
      epilogue_tile<BN, false, FMT == kFmtInt4>(&tmOut, p, tl, w.m_blk * kBM + q * 32,
                                                w.n_blk * BN, 0, stg, sb,
                                                smem_u32(&tempty[buf]), false, lane);
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  } else {
    // ------------------------------ dequantisers ------------------------------
    const int dt = threadIdx.x - (2 + kEpiWarps) * 32;  // 0 .. 32 * kDeqWarps - 1
    const int cw = dt % W;                               // packed word column
    const int row_first = dt / W;
    constexpr int kRowStep = 32 * kDeqWarps / W;
    const int box = cw / 8, chunk = cw % 8;
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit w = unit_of(p, u);
      bool ok = true;
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
        int ready = 0;
        if (lane == 0)
          ready = wait_phase(smem_u32(&load_full[stage]), phase, abort_flag, p, kRoleProducer);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (!ready) {
          ok = false;
          break;
        }
        // the eight scales of this thread's columns, paired (e, e+4) like dequant8's halves
        const uint4 sv = *reinterpret_cast<const uint4*>(sS + stage * Cfg::kSStage + cw * 16);
        uint32_t sp[4];
        scale_pairs<FMT>(sv, sp);
        const uint32_t* q = reinterpret_cast<const uint32_t*>(sQ + stage * Cfg::kQStage);
        uint8_t* bdst = sB + stage * Cfg::kBStage + box * 8192;
        // all of this thread's words first, then independent decodes: the rows give the
        // scheduler 64/kRowStep independent chains to interleave
        constexpr int kRows = 64 / kRowStep;
        uint32_t words[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) words[i] = q[(row_first + i * kRowStep) * W + cw];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const int r = row_first + i * kRowStep;
          const uint4 v = decode8<FMT>(words[i], sp);
          *reinterpret_cast<uint4*>(bdst + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&deq_full[stage]));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// CTA-pair variant for many rows of A: 256 x 256 output tiles on a cluster of two CTAs
// (tcgen05 cta_group::2), as tg_gemm_pair_kernel.  CTA r holds A rows [256m + 128r, +128)
// and decodes B columns [256n + 128r, +128) into its own shared memory; one MMA of 256 x 256
// x 16 uses both CTAs' halves, so every decoded weight serves 256 rows of A and each CTA
// decodes half the tile that tg_gemm_w4_kernel<256> decodes.  Per stage and CTA, shared
// memory carries A 16 KB (TMA), the packed words 4 KB, the decoded tile 16 KB (written, then
// read by the MMA) and A again 16 KB (read by the MMA): ~72 KB per 512 tensor cycles, against
// ~112 KB for the single-CTA kernel.
//
// Barriers: full[s] (leader; both CTAs' A bytes via the pair TMA), qfull[s] (each CTA: its
// packed words and scales), deq_full[s] (leader; its own dequantiser warps plus one arrival
// forwarded from the follower), fdeq[s] (follower; its dequantiser warps), empty[s] (each
// CTA; the leader's commit multicasts), tfull/tempty as tg_gemm_pair_kernel.  A remote
// arrive with cluster-scope release costs ~1000 cycles of the arriving thread; one such
// arrive per dequantiser warp and stage made the decode period ~1.6x longer, hence the local
// fdeq barrier and a few forwarding threads that each carry every kForwarders-th stage.
// ---------------------------------------------------------------------------------------
struct W4PairCfg {
  static constexpr int kBN = 256;                        // N of the pair tile
  static constexpr int kHalfN = 128;                     // columns decoded by each CTA
  static constexpr int kAStage = kBM * kBK * 2;          // 16 KB
  static constexpr int kBStage = kBK * kHalfN * 2;       // 16 KB decoded, MN-major
  static constexpr int kQStage = kBK * kHalfN / 2;       // 4 KB packed
  static constexpr int kSStage = 1024;                   // one scale row (256 B), padded
  static constexpr int kQTx = kQStage + kHalfN * 2;
  static constexpr int kStageBytes = kAStage + kBStage + kQStage + kSStage;
  static constexpr int kStagingBytes = kEpiWarps * 2 * kStagingBuf;
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve - kStagingBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kAccStride = 256;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemBytes = kSmemReserve + kStages * kStageBytes + kStagingBytes;
  // Forwarding of the follower's dequantiser arrivals to the leader: kForwarders threads take
  // the stages in turn (the MMA warp's lane 0 in the follower plus lane 0 of kFwdWarps extra
  // warps), so that the ~1000-cycle latency of cluster-scope arrivals overlaps.
  static constexpr int kFwdWarps = 2;
  static constexpr int kForwarders = 1 + kFwdWarps;
  static constexpr int kThreads = kW4Threads + 32 * kFwdWarps;
  static_assert(kStages >= 2, "not enough shared memory");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget exceeded");
  static_assert((5 * kStages + 5) * 8 + 8 <= kSmemReserve - 1024, "barriers exceed the reserve");
};

// tmA: fp16 A {K, M} box {64, 128} SW128; tmQ: uint32 Wq {ceil(N/8), K} box {16, 64};
// tmS: fp16 scales {N, ceil(K/G)} box {128, 1}; tmOut: fp16 C {n_tma, M} box {64, 32} SW128.
// p.tiles_m / p.tiles_n count 256 x 256 pair tiles; p.splits == 1; p.group_kb = G / 64.
template <int FMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(W4PairCfg::kThreads, 1)
    tg_gemm_w4_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmS,
                           const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using Cfg = W4PairCfg;
  constexpr int S = Cfg::kStages;
  constexpr int W = Cfg::kHalfN / 8;  // packed words per row of a CTA's columns

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kAStage;
  uint8_t* sQ = sB + S * Cfg::kBStage;
  uint8_t* sS = sQ + S * Cfg::kQStage;
  uint8_t* sStg = sS + S * Cfg::kSStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStagingBytes);
  uint64_t* full = bars;          // leader
  uint64_t* qfull = bars + S;     // each CTA
  uint64_t* deq_full = bars + 2 * S;  // leader
  uint64_t* empty = bars + 3 * S; // each CTA
  uint64_t* tfull = bars + 4 * S;
  uint64_t* tempty = tfull + 2;   // leader
  uint64_t* drain = tempty + 2;
  uint64_t* fdeq = drain + 1;     // follower
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fdeq + S);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&qfull[s]), 1);
      mbar_init(smem_u32(&deq_full[s]), kDeqWarps + 1);
      mbar_init(smem_u32(&fdeq[s]), kDeqWarps);
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
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmS);
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

  // Follower only: forwarder f carries stages f, f + kForwarders, ... of the CTA's sequence.
  auto forward = [&](int f) {
    const uint32_t deq0_leader = mapa_shared(smem_u32(&deq_full[0]), 0);
    int stage = 0;
    uint32_t phase = 0;
    int seq = 0;
    for (int u = cluster; u < p.units; u += nclusters) {
      const Unit w = unit_of(p, u);
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++seq) {
        if (seq % Cfg::kForwarders == f) {
          if (!wait_phase(smem_u32(&fdeq[stage]), phase, abort_flag, p, kRoleProducer)) return;
          mbar_arrive_cluster(deq0_leader + 8u * stage);
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  };

  if (warp == 0) {
    // ------------------------------ TMA producer (both CTAs) ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;      // the leader's full barriers
      uint32_t qarmed = 0, qarmed_parity = 0;    // this CTA's qfull barriers
      bool dropped = false;
      const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), 0);
      for (int u = cluster; u < p.units; u += nclusters) {
        const Unit w = unit_of(p, u);
        const int arow = w.m_blk * 2 * kBM + static_cast<int>(rank) * kBM;
        const int bcol = w.n_blk * Cfg::kBN + static_cast<int>(rank) * Cfg::kHalfN;
        int g = w.kb_begin / p.group_kb;
        int g_rem = w.kb_begin - g * p.group_kb;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p, kRoleProducer))
            goto w4pair_producer_done;
          if ((p.debug_flags & kDebugDropFirstStage) && cluster == 0 && rank == 0 && !dropped) {
            dropped = true;  // injected fault: the leader neither arms nor fills this stage
          } else {
            if (rank == 0) {
              mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * Cfg::kAStage);
              armed |= 1u << stage;
              armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
            tma_load_2d_pair(smem_u32(sA + stage * Cfg::kAStage), &tmA,
                             full0_leader + 8u * stage, kb * kBK, arow);
            const uint32_t qb = smem_u32(&qfull[stage]);
            mbar_arrive_expect_tx(qb, Cfg::kQTx);
            tma_load_2d(smem_u32(sQ + stage * Cfg::kQStage), &tmQ, qb, bcol / 8, kb * kBK);
            tma_load_2d(smem_u32(sS + stage * Cfg::kSStage), &tmS, qb, bcol, g);
            qarmed |= 1u << stage;
            qarmed_parity = (qarmed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++g_rem == p.group_kb) {
            g_rem = 0;
            ++g;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    w4pair_producer_done:
      for (int s = 0; s < S; ++s) {
        if (armed & (1u << s)) wait_phase_drain(smem_u32(&full[s]), (armed_parity >> s) & 1u, p);
        if (qarmed & (1u << s)) wait_phase_drain(smem_u32(&qfull[s]), (qarmed_parity >> s) & 1u, p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer (leader) ------------------------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(2 * kBM, Cfg::kBN, 0, 1);
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
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&full[stage]), phase, abort_flag, p, kRoleMma) ||
              !wait_phase(smem_u32(&deq_full[stage]), phase, abort_flag, p, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_kmajor(smem_u32(sA + stage * Cfg::kAStage));
          const uint64_t bd = desc_mnmajor(smem_u32(sB + stage * Cfg::kBStage));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_f16_pair(d_tmem, ad + 2u * k, bd + 128u * k, idesc,
                          (kb > w.kb_begin || k > 0) ? 1u : 0u);
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
    } else if (lane == 0 && rank == 1) {
      forward(0);
    }
  } else if (warp >= 2 + kEpiWarps + kDeqWarps) {
    // ------------------------------ forwarders (follower) ------------------------------
    if (lane == 0 && rank == 1) forward(warp - (2 + kEpiWarps + kDeqWarps) + 1);
  } else if (warp < 2 + kEpiWarps) {
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
      if (lane == 0)
        ok = wait_phase_sleepy(smem_u32(&tfull[buf]), use, abort_flag, p, kRoleEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * Cfg::kAccStride);
      const int row0 = w.m_blk * 2 * kBM + static_cast<int>(rank) * kBM + q * 32;
      const uint32_t release_bar = mapa_shared(smem_u32(&tempty[buf]), 0);
      epilogue_tile<Cfg::kBN, false, FMT == kFmtInt4>(&tmOut, p, tl, row0, w.n_blk * Cfg::kBN,
                                                      0, stg, sb, release_bar, true, lane);
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  } else {
    // ------------------------------ dequantisers (both CTAs) ------------------------------
    const int dt = threadIdx.x - (2 + kEpiWarps) * 32;  // 0 .. 32 * kDeqWarps - 1
    const int cw = dt % W;                               // packed word column
    const int row_first = dt / W;
    constexpr int kRowStep = 32 * kDeqWarps / W;
    const int box = cw / 8, chunk = cw % 8;
    uint64_t* deq_done = rank == 0 ? deq_full : fdeq;
    int stage = 0;
    uint32_t phase = 0;
    for (int u = cluster; u < p.units; u += nclusters) {
      const Unit w = unit_of(p, u);
      bool ok = true;
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
        int ready = 0;
        if (lane == 0)
          ready = wait_phase(smem_u32(&qfull[stage]), phase, abort_flag, p, kRoleProducer);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (!ready) {
          ok = false;
          break;
        }
        const uint4 sv = *reinterpret_cast<const uint4*>(sS + stage * Cfg::kSStage + cw * 16);
        uint32_t sp[4];
        scale_pairs<FMT>(sv, sp);
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(sQ + stage * Cfg::kQStage);
        uint8_t* bdst = sB + stage * Cfg::kBStage + box * 8192;
        constexpr int kRows = 64 / kRowStep;
        uint32_t words[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) words[i] = qw[(row_first + i * kRowStep) * W + cw];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const int r = row_first + i * kRowStep;
          const uint4 v = decode8<FMT>(words[i], sp);
          *reinterpret_cast<uint4*>(bdst + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&deq_done[stage]));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  // After an abort the follower cannot observe its A loads (they complete on the leader's
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

// ---------------------------------------------------------------------------------------
// Swapped-operand variant for few rows of A (decode-like shapes): C^T = W^T · A^T.  The
// decoded weight tile is the MMA's M side (128 output columns n, MN-major, decoded exactly as
// in tg_gemm_w4_kernel with BN = 128) and the activations are the N side (BM rows m of A,
// K-major), so an M = 64 problem wastes no MMA work.  TMEM holds C^T: lane = column n,
// TMEM column = row m; the epilogue writes C[m][n] with plain stores, coalesced across lanes.
// ---------------------------------------------------------------------------------------
// Per-stage costs are paid by single threads (a barrier wait, an MMA issue or a commit each
// costs its thread ~90-170 cycles), so the work of consecutive stages is dealt to parallel
// threads: two MMA issuers take alternate k-blocks of a unit into two TMEM accumulators that
// the epilogue adds (accumulator 0 + accumulator 1, a fixed order), and kW4TDeqGroups groups
// of four dequantiser warps (one warp per scheduler each) take the stages in turn.  With one
// issuer the MMA thread was busy the whole ~1030-cycle stage; now the decode sets the pace.
constexpr int kW4TGroupWarps = 4;
constexpr int kW4TDeqGroups = 2;
constexpr int kW4TDeqWarps = kW4TDeqGroups * kW4TGroupWarps;
constexpr int kW4TMma2Warp = 2 + kEpiWarps + kW4TDeqWarps;  // second MMA issuer
constexpr int kW4TThreads = (3 + kEpiWarps + kW4TDeqWarps) * 32;

// activation(x, act) kept out of line, for the GELU forms in unrolled epilogue loops.
__device__ __noinline__ float activation_outlined(float x, int act) { return activation(x, act); }

// TDEC: the dequantisers write the decoded tile into tensor memory instead of shared memory,
// and the MMA reads its A operand (the decoded weights) from there.  Each dequantiser thread
// owns one TMEM lane = one output column of the tile and writes that column's 64 weights of a
// stage as 32 columns of fp16 pairs (k even in the low half).  A stage's slot sits after the
// accumulators; the slots form the same ring as the shared-memory stages.
template <int BMT, bool TDEC = false>
struct W4TCfg {
  static constexpr int kNTile = 128;                  // output columns per tile (MMA M)
  static constexpr int kActStage = BMT * kBK * 2;     // activations, K-major
  static constexpr int kDecStage = TDEC ? 0 : kBK * kNTile * 2;  // decoded weights, MN-major
  static constexpr int kQStage = kBK * kNTile / 2;
  static constexpr int kSStage = 1024;
  static constexpr int kStageBytes = kActStage + kDecStage + kQStage + kSStage;
  static constexpr int kTxBytes = kActStage + kQStage + kNTile * 2;
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kAccStride = BMT;              // TMEM columns per accumulator
  // two TMEM buffers x two accumulators (even and odd k-blocks of a unit)
  static constexpr int kAccCols = 4 * BMT < 32 ? 32 : 4 * BMT;
  static constexpr int kDecCols = kBK / 2;            // TMEM columns of one decoded stage
  static constexpr int kTmemCols = TDEC ? 512 : kAccCols;
  static constexpr int kSmemBytes = kSmemReserve + kStages * kStageBytes;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget exceeded");
  static_assert(!TDEC || kAccCols + kStages * kDecCols <= 512, "TMEM ring exceeds 512 columns");
};

// tmA: fp16 A {K, M} box {64, BMT} SW128 (K-major operand of the transposed product);
// tmQ / tmS as tg_gemm_w4_kernel with BN = 128.  Tiles: p.tiles_m counts BMT-row blocks of A,
// p.tiles_n counts 128-column blocks of C.  p.splits == 1.  With p.tail, units [0, n_full)
// are whole tiles and each later tile is two units, one per K half (see unit_of); tail_ws
// holds 2 x 4 x 32 x BMT floats per split tile and tail_cnt 4 zeroed counters per split tile.
template <int BMT, int FMT, bool TDEC>
__global__ void __launch_bounds__(kW4TThreads, 1)
    tg_gemm_w4t_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmS, const GemmParams p) {
  using Cfg = W4TCfg<BMT, TDEC>;
  constexpr int S = Cfg::kStages;
  constexpr int W = Cfg::kNTile / 8;  // 16 packed words per row

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sDec = smem;
  uint8_t* sAct = sDec + S * Cfg::kDecStage;
  uint8_t* sQ = sAct + S * Cfg::kActStage;
  uint8_t* sS = sQ + S * Cfg::kQStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + S * Cfg::kSStage);
  uint64_t* load_full = bars;
  uint64_t* deq_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* tfull = bars + 3 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&load_full[s]), 1);
      mbar_init(smem_u32(&deq_full[s]), kW4TGroupWarps);  // one group of dequantisers
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 2);  // both MMA issuers
      mbar_init(smem_u32(&tempty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 2);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmS);
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
        // scale row of k-block kb: g = kb / group_kb, advanced with a counter (one division
        // per tile instead of one per stage on the single producer thread)
        int g = w.kb_begin / p.group_kb;
        int g_rem = w.kb_begin - g * p.group_kb;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!wait_phase(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p, kRoleProducer))
            goto w4t_producer_done;
          if ((p.debug_flags & kDebugDropFirstStage) && blockIdx.x == 0 && !dropped) {
            dropped = true;  // injected fault: this stage is never filled
          } else {
            const uint32_t fb = smem_u32(&load_full[stage]);
            mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
            tma_load_2d(smem_u32(sAct + stage * Cfg::kActStage), &tmA, fb, kb * kBK,
                        w.m_blk * BMT);
            tma_load_2d(smem_u32(sQ + stage * Cfg::kQStage), &tmQ, fb, w.n_blk * W, kb * kBK);
            tma_load_2d(smem_u32(sS + stage * Cfg::kSStage), &tmS, fb, w.n_blk * Cfg::kNTile, g);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++g_rem == p.group_kb) {
            g_rem = 0;
            ++g;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    w4t_producer_done:
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) wait_phase_drain(smem_u32(&load_full[s]), (armed_parity >> s) & 1u, p);
    }
  } else if (warp == 1 || warp == kW4TMma2Warp) {
    // ------------------------------ MMA issuers ------------------------------
    // Issuer j (0: warp 1, 1: the extra warp) takes the k-blocks kb_begin + j, + j + 2, ...
    // of each unit into accumulator j of the unit's TMEM buffer; the epilogue adds the two.
    if (lane == 0) {
      const int j = warp == 1 ? 0 : 1;
      // D (128 n x BMT m) += Wdec (128 n x 16 k, MN-major in shared memory, or K-major in
      // tensor memory) * A^T (16 k x BMT m, K-major)
      const uint32_t idesc = idesc_f16_f32(Cfg::kNTile, BMT, TDEC ? 0 : 1, 0);
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
        const Unit w = unit_of(p, u);
        const int buf = t & 1;
        const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
        if (!wait_phase(smem_u32(&tempty[buf]), use ^ 1u, abort_flag, p, kRoleMma)) break;
        tc_fence_after();
        const uint32_t d_tmem =
            tmem_base + static_cast<uint32_t>((buf * 2 + j) * Cfg::kAccStride);
        bool ok = true;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (((kb - w.kb_begin) & 1) != j) {
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!wait_phase(smem_u32(&load_full[stage]), phase, abort_flag, p, kRoleMma) ||
              !wait_phase(smem_u32(&deq_full[stage]), phase, abort_flag, p, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = desc_kmajor(smem_u32(sAct + stage * Cfg::kActStage));
          if constexpr (TDEC) {
            // the stage's decoded slot: 16 k = 8 columns per MMA
            const uint32_t a_tmem =
                tmem_base + static_cast<uint32_t>(Cfg::kAccCols + stage * Cfg::kDecCols);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              umma_f16_ts(d_tmem, a_tmem + 8u * k, bd + 2u * k, idesc,
                          (kb - w.kb_begin > 1 || k > 0) ? 1u : 0u);
          } else {
            const uint64_t ad = desc_mnmajor(smem_u32(sDec + stage * Cfg::kDecStage));
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              umma_f16(d_tmem, ad + 128u * k, bd + 2u * k, idesc,
                       (kb - w.kb_begin > 1 || k > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[buf]));
      }
      umma_commit(smem_u32(drain));
      wait_phase_drain(smem_u32(drain), 0u, p);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------ epilogue: C[m][n] from TMEM lane n, column m ------------
    const int q = warp & 3;
    int t = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
      const Unit w = unit_of(p, u);
      const int buf = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1) & 1u;
      int ok = 0;
      if (lane == 0)
        ok = wait_phase_sleepy(smem_u32(&tfull[buf]), use, abort_flag, p, kRoleEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * 2 * Cfg::kAccStride);
      const bool two = w.kb_end - w.kb_begin >= 2;  // accumulator 1 holds the odd k-blocks
      // float32 sums of rows c*32 .. c*32 + 31: accumulator 0 + accumulator 1, in that order
      auto load_sums = [&](int c, uint32_t (&r)[32]) {
        tmem_ld_x32(tl + c * 32, r);
        if (two) {
          uint32_t r1[32];
          tmem_ld_x32(tl + Cfg::kAccStride + c * 32, r1);
          tmem_wait_ld(r);
          tmem_wait_ld(r1);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r1[i]));
        } else {
          tmem_wait_ld(r);
        }
      };
      // TMEM lane -> output column (a TMEM-decoded tile keeps the columns in order)
      const int n = w.n_blk * Cfg::kNTile + (TDEC ? q * 32 + lane : decoded_column<FMT>(q * 32 + lane));
      const int m_base = w.m_blk * BMT;
      const bool n_ok = n < p.N;
      const float bias = (n_ok && p.bias) ? __half2float(p.bias[n]) : 0.0f;
      unsigned short* cp = reinterpret_cast<unsigned short*>(p.c);
      // rows m0 .. m0 + 31 of column n, from 32 float32 sums.  The GELU forms go through one
      // out-of-line copy of the activation: with the activation switch inlined in all 32
      // unrolled rows, the kernel's end (its TMEM release) took ~5 us longer on the
      // decode-like shapes, though those paths never ran.
      auto store_rows = [&](const uint32_t (&r)[32], int m0) {
        if (!n_ok) return;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int m = m0 + j;
          if (m < p.M) {
            float x = __uint_as_float(r[j]) + bias;
            if (p.act == kActRelu)
              x = x > 0.0f ? x : 0.0f;  // as activation(x, kActRelu)
            else if (p.act != kActNone)
              x = activation_outlined(x, p.act);
            if (p.residual) x += __half2float(p.residual[static_cast<long long>(m) * p.ldr + n]);
            cp[static_cast<long long>(m) * p.ldc + n] = __half_as_ushort(__float2half_rn(x));
          }
        }
      };
      if (w.tail_slot < 0) {
#pragma unroll 1
        for (int c = 0; c < BMT / 32; ++c) {
          uint32_t r[32];
          load_sums(c, r);
          if (c == BMT / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
          }
          store_rows(r, m_base + c * 32);
        }
        continue;
      }
      // One K half of a split tile: park this half's float32 sums in tail_ws ([slot][half]
      // [quarter][m][lane]), then count arrivals on the (slot, quarter) counter.  The warp
      // that arrives second adds the two halves (a + b == b + a in IEEE arithmetic, so the
      // result does not depend on which half finished last), finishes the rows and resets the
      // counter.  No warp waits for another CTA.
      const long long per_part = 32LL * BMT;
      float* mine = p.tail_ws + ((static_cast<long long>(w.tail_slot) * 2 + w.split) * 4 + q) *
                                    per_part + lane;
#pragma unroll 1
      for (int c = 0; c < BMT / 32; ++c) {
        uint32_t r[32];
        load_sums(c, r);
        if (c == BMT / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) mine[(c * 32 + j) * 32] = __uint_as_float(r[j]);
      }
      __threadfence();
      __syncwarp();
      int arrived = 0;
      if (lane == 0) arrived = atomicAdd(p.tail_cnt + w.tail_slot * 4 + q, 1);
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived == 0) continue;  // the other half finishes these rows
      __threadfence();
      const float* other = p.tail_ws +
                           ((static_cast<long long>(w.tail_slot) * 2 + (w.split ^ 1)) * 4 + q) *
                               per_part + lane;
#pragma unroll 1
      for (int c = 0; c < BMT / 32; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          r[j] = __float_as_uint(mine[(c * 32 + j) * 32] + __ldcg(other + (c * 32 + j) * 32));
        store_rows(r, m_base + c * 32);
      }
      if (lane == 0) p.tail_cnt[w.tail_slot * 4 + q] = 0;
    }
  } else {
    // ------------------------------ dequantisers (as tg_gemm_w4_kernel, BN = 128) ------------
    // group grp decodes stages grp, grp + kW4TDeqGroups, ... of the CTA's k-block sequence
    const int grp = (warp - (2 + kEpiWarps)) / kW4TGroupWarps;
    const int dt = threadIdx.x - (2 + kEpiWarps + grp * kW4TGroupWarps) * 32;  // 0 .. 127
    const int cw = dt % W;
    const int row_first = dt / W;
    constexpr int kRowStep = 32 * kW4TGroupWarps / W;
    int seq = 0;
    const int box = cw / 8, chunk = cw % 8;
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit w = unit_of(p, u);
      bool ok = true;
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++seq) {
        if (seq % kW4TDeqGroups != grp) {
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        int ready = 0;
        if (lane == 0)
          ready = wait_phase(smem_u32(&load_full[stage]), phase, abort_flag, p, kRoleProducer);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (!ready) {
          ok = false;
          break;
        }
        if constexpr (TDEC) {
          // this thread's TMEM lane is tile column nl: its nibble of word column nl / 8 in each
          // of the stage's 64 rows, decoded in k pairs and written as 32 TMEM columns
          const int nl = (warp & 3) * 32 + lane;
          const uint32_t sh = 4u * static_cast<uint32_t>(nl & 7);
          const uint32_t sb =
              reinterpret_cast<const uint16_t*>(sS + stage * Cfg::kSStage)[nl];
          const uint32_t s2 = sb | (sb << 16);
          const uint32_t* col =
              reinterpret_cast<const uint32_t*>(sQ + stage * Cfg::kQStage) + (nl >> 3);
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            r[j] = decode_pair<FMT>(col[(2 * j) * W] >> sh, col[(2 * j + 1) * W] >> sh, s2);
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                                 static_cast<uint32_t>(Cfg::kAccCols + stage * Cfg::kDecCols);
          tmem_st_x32(taddr, r);
          tmem_wait_st();
          tc_fence_before();  // the MMA thread reads these columns after the barrier
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&deq_full[stage]));
        } else {
          const uint4 sv = *reinterpret_cast<const uint4*>(sS + stage * Cfg::kSStage + cw * 16);
          uint32_t sp[4];
          scale_pairs<FMT>(sv, sp);
          const uint32_t* qw = reinterpret_cast<const uint32_t*>(sQ + stage * Cfg::kQStage);
          uint8_t* ddst = sDec + stage * Cfg::kDecStage + box * 8192;
          constexpr int kRows = 64 / kRowStep;
          uint32_t words[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) words[i] = qw[(row_first + i * kRowStep) * W + cw];
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int r = row_first + i * kRowStep;
            const uint4 v = decode8<FMT>(words[i], sp);
            *reinterpret_cast<uint4*>(ddst + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&deq_full[stage]));
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace tg
