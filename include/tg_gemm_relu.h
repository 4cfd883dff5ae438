/*
 * tg_gemm_relu.h — C ABI of the GB300 (sm_103a) relu(A·B) library.
 *
 * The operation (TileLang paper-reading page, section 2, the matmul_relu example; the
 * practitioner page, section 3.2, on the float32 accumulator):
 *
 *     C[i,j] = fp16( epilogue( sum_{k<K} A[i,k] * B[k,j] ) )    0 <= i < M, 0 <= j < N
 *
 * A is M x K and B is K x N, both row-major IEEE binary16 ("fp16"); the sum is accumulated in
 * binary32 on the tensor cores; epilogue is relu(x) = (x > 0 ? x : +0) or the identity; the
 * result is rounded to fp16 with round-to-nearest-even and written to the row-major M x N C.
 * The summation order inside the sum is the kernel's blocked order (not specified); for a
 * given plan it is fixed, so results are bitwise reproducible run to run, split-K included.
 *
 * Conventions shared by every entry point:
 *  - Leading dimensions are in elements: element (i,k) of A is A[i*lda + k], and so on.
 *    lda >= max(1,K), ldb >= max(1,N), ldc >= max(1,N).
 *  - Pointers must be 2-byte aligned (TG_ERR_MISALIGNED otherwise). 16-byte aligned pointers
 *    with leading dimensions that are multiples of 8 take the direct path; anything else is
 *    handled too (operands are first repacked into aligned scratch, C goes through a float32
 *    scratch and a final conversion pass).
 *  - M == 0 or N == 0 is a no-op. K == 0 writes +0 to every element of C.
 *  - C must not overlap A or B (not checked).
 *  - Errors are detected on the host before anything is launched; a call that returns an
 *    error has launched nothing and written nothing.
 *  - Device support: compute capability 10.3 (GB300) only (TG_ERR_UNSUPPORTED_DEVICE).
 *  - Thread safety: every entry point may be called from several host threads at once.
 *  - CUDA graphs: the asynchronous device-pointer entry points (tg_gemm_relu_f16, _ex,
 *    tg_gemm_f16_epilogue, tg_gemm_f16_t, tg_relu_backward_f16, tg_gemm_w4a16_f16,
 *    tg_gemm_nf4a16_f16) may be
 *    captured by stream capture once the calling thread has made one eager call on the device
 *    (that first call sets up library state); scratch is taken stream-ordered from the
 *    library's pool and becomes graph allocation nodes.  tg_gemm_relu_f16_host synchronises
 *    and cannot be captured.
 */
#ifndef TG_GEMM_RELU_H
#define TG_GEMM_RELU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* tg_stream_t;

typedef enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1,        /* negative size, short leading dimension, NULL, bad flag */
  TG_ERR_MISALIGNED = 2,         /* a pointer that is not 2-byte aligned */
  TG_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  TG_ERR_CUDA = 4,               /* a CUDA call failed; see tg_last_cuda_error */
  TG_ERR_TIMEOUT = 5,            /* a kernel gave up waiting on a pipeline barrier */
  TG_ERR_NO_WORKSPACE = 6        /* scratch memory could not be obtained */
} tg_status;

enum { TG_EPILOGUE_NONE = 0, TG_EPILOGUE_RELU = 1 };

/* Activations of the fused epilogue (tg_gemm_f16_epilogue).  The first two equal the
 * TG_EPILOGUE_* flags.  GELU is x/2 * (1 + erf(x/sqrt 2)); GELU_TANH is the tanh form
 * x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))) (Hendrycks & Gimpel, 2016). */
enum { TG_ACT_NONE = 0, TG_ACT_RELU = 1, TG_ACT_GELU = 2, TG_ACT_GELU_TANH = 3 };

/* Fused epilogue: C = fp16( act( A·B + bias ) + residual ), every step in float32 and one
 * rounding to fp16 at the end. */
typedef struct {
  int activation;         /* TG_ACT_* */
  const void* bias;       /* NULL, or device fp16[N]: bias[j] is added to column j */
  const void* residual;   /* NULL, or device fp16 M x N (leading dimension ldr) added after the
                             activation; it may be C itself (same pointer, ldr == ldc), and
                             must not otherwise overlap C */
  int64_t ldr;
} tg_epilogue;

/*
 * C = fp16(relu(A·B)) (epilogue_flag = TG_EPILOGUE_RELU) or C = fp16(A·B) (TG_EPILOGUE_NONE).
 * A, B, C: device pointers to fp16 data, owned by the caller.  Asynchronous on `stream`:
 * returns once the work is queued; the caller synchronises.  Scratch memory, when a plan
 * needs it, comes from a library-owned stream-ordered pool on the current device and is
 * released back to the pool in stream order (see tg_release_workspace).
 */
tg_status tg_gemm_relu_f16(const void* A, const void* B, void* C, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int epilogue_flag,
                           tg_stream_t stream);

/* Plan overrides, for tests and tuning.  Zero-initialise; every zero field means "choose". */
typedef struct {
  int block_n;          /* 0, or the N extent of an output tile: 128, 192 or 256 */
  int split_k;          /* 0, or the number of K splits (>= 1) */
  int force_repack;     /* 1: copy A and B into aligned scratch even when not needed */
  int force_workspace;  /* 1: write C through the float32 scratch and conversion pass */
  int panel_m;          /* 0, or the L2 panel height in M tiles for the tile order */
  int max_ctas;         /* 0 (one per SM), or a cap on the persistent grid */
  int debug_flags;      /* TG_DEBUG_* below; 0 in normal use */
  int timeout_ms;       /* 0 (default 2000 ms), or the per-wait limit of the pipeline */
  int pair;             /* 0: choose; 1: use the two-CTA 256x256 tile; -1: never use it */
  int tail;             /* run the last partial wave's tiles as two K halves that meet through
                           a float32 workspace.  CTA-pair plans without split-K, with 0 or 1:
                           when at least one full wave precedes a last wave that holds at most
                           half the clusters.  The int4 GEMM's swapped kernel: with 0 when the
                           last wave holds at most half a grid, with 1 whenever it is partial.
                           -1: never */
  int swap_ab;          /* int4 GEMM only: 0 choose (swapped for M <= 128), 1 compute C^T =
                           W^T A^T with the decoded weights as the 128-row MMA side, -1 never */
  int a_in_place;       /* 1: an A whose leading dimension is not a multiple of 8 is read in
                           place through 16 row classes (tg_plan.a_row_classes) instead of being
                           copied into aligned scratch, when A is 32-byte aligned and the plan
                           uses CTA pairs.  Saves the copy's M * K * 2 bytes of scratch; on GB300
                           the copy is faster (4095 x 3073 x 65537: 1.35 against 1.47 ms),
                           because a class's rows start mid-line in L2.  0: copy */
  int repack_overlap;   /* 0: choose (tg_plan.repack_overlap); -1: never overlap the operand
                           copies with the GEMM */
  int tmem_decode;      /* int4 / NF4 GEMM, swapped kernel with M <= 64: 1 decode the weights
                           into tensor memory, where the MMA reads them (each thread gathers
                           its column's nibbles row by row: slower than the default on every
                           shape measured, e.g. 64 x 28672 x 8192 int4 111 against 93 us);
                           0 decode into shared memory */
  int dequant_first;    /* int4 / NF4 GEMM: 1 decode the whole weight matrix once into fp16
                           scratch (K x N rounded up to 8, 2 bytes each, from the library's
                           pool) and run the fp16 GEMM on it; -1 never; 0 choose: decode first
                           when M is large enough (see tg_gemm_w4a16_f16) and no other
                           int4-kernel override (swap_ab, pair, block_n, tmem_decode) is set */
} tg_options;

/* Fault injection: the first producer of the grid drops its first stage (no load, no
 * arrival), so the consumer's wait on that stage runs out; the kernel records the timeout,
 * drains and returns.  Honoured by every GEMM kernel (fp16, int4 and NF4 weights).  Only for
 * the error-path test. */
#define TG_DEBUG_DROP_FIRST_STAGE 1

/* What a call will do; filled by tg_plan_query (host only, no device needed). */
typedef struct {
  int block_m, block_n, block_k;  /* output tile and the k-block unit of kblocks */
  int stages;                      /* pipeline stages; a forward CTA-pair stage holds two
                                      k-blocks, every other stage one */
  int split_k;                 /* K splits actually used */
  int64_t kblocks;             /* ceil(K / block_k) */
  int64_t kblocks_per_split;
  int64_t tiles_m, tiles_n;
  int64_t units;               /* tiles_m * tiles_n * split_k work units */
  int grid;                    /* persistent CTAs */
  int panel_m;
  int repack_a, repack_b;      /* operand copied into aligned scratch first */
  int workspace_epilogue;      /* C produced by the float32 scratch + conversion pass */
  int64_t workspace_bytes;     /* scratch needed per call */
  int kernels;                 /* kernel launches per call */
  int cta_pair;                /* 1: 256x256 tiles on clusters of two CTAs (tcgen05 cta_group::2) */
  int64_t tail_tiles;          /* tiles of the last partial wave computed as two K halves (the
                                  units count both halves); 0 when not used */
  int a_row_classes;           /* 16: A (leading dimension not a multiple of 8) read in place in
                                  16 row classes, each tile's rows from one class, instead of
                                  being repacked (tg_options.a_in_place); 0 otherwise */
  int repack_overlap;          /* 1: with split-K and operand copies, the copies are made split
                                  by split on a library stream, each split's GEMM launched (on
                                  two more library streams, in turn) as soon as its slice is
                                  copied, so copies overlap the GEMMs of earlier splits; all
                                  streams join the caller's stream before the reduction.  A
                                  call made under stream capture runs the copies first instead.
                                  0: copies first, then one GEMM launch */
} tg_plan;

/*
 * Same as tg_gemm_relu_f16 with plan overrides (opt may be NULL).  An override that the
 * shape cannot honour (for example split_k larger than the number of K blocks) is clamped.
 */
tg_status tg_gemm_relu_f16_ex(const void* A, const void* B, void* C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              int epilogue_flag, const tg_options* opt, tg_stream_t stream);

/*
 * GEMM with the fused bias / activation / residual epilogue.  The pages motivate fusing the
 * epilogue into the GEMM (the practitioner page, section 2: fusion keeps intermediates on chip)
 * and use relu as their example (TileLang paper-reading page, section 2).  epi == NULL is
 * the identity epilogue.  Other arguments, layouts and errors as tg_gemm_relu_f16_ex; bias and
 * residual need 2-byte alignment; ldr >= max(1, N) when residual is given.
 */
tg_status tg_gemm_f16_epilogue(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                               const tg_epilogue* epi, const tg_options* opt,
                               tg_stream_t stream);

/*
 * C = fp16(epilogue(op(A)·op(B))) with op(A) M x K and op(B) K x N, for the backward pass of
 * relu(A·B) (the practitioner page, section 3.3: the kernel behind torch.autograd.Function
 * needs its own backward kernels).
 *   trans_a = 0: A stored M x K row-major (lda >= K);  1: A stored K x M row-major (lda >= M)
 *   trans_b = 0: B stored K x N row-major (ldb >= N);  1: B stored N x K row-major (ldb >= K)
 * Everything else as tg_gemm_f16_epilogue (epi may be NULL for the identity epilogue).
 */
tg_status tg_gemm_f16_t(int trans_a, int trans_b, const void* A, const void* B, void* C,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        const tg_epilogue* epi, const tg_options* opt, tg_stream_t stream);

/*
 * Backward of the relu epilogue on its fp16 output C: dZ[i,j] = C[i,j] > 0 ? dC[i,j] : +0
 * (M x N, each with its own leading dimension).  Device pointers, 2-byte aligned;
 * asynchronous on `stream`.  With dZ, dA = dZ·B^T (tg_gemm_f16_t(0, 1, ...)) and
 * dB = A^T·dZ (tg_gemm_f16_t(1, 0, ...)).
 */
tg_status tg_relu_backward_f16(const void* dC, const void* C, void* dZ, int64_t M, int64_t N,
                               int64_t lddc, int64_t ldc, int64_t lddz, tg_stream_t stream);

/*
 * Dequantising GEMM with 4-bit integer weights and fp16 activations (the W_INT4 / A_FP16
 * case of the TileLang paper-reading page, section 5):
 *     C = fp16( epilogue( A · W ) ),   W[k][n] = fp16( (q[k][n] - 8) * scales[k / G][n] )
 * A: device fp16 M x K row-major, 16-byte aligned, lda a multiple of 8.
 * Wq: device uint32, K rows of ldq words (ldq >= ceil(N/8), multiple of 4, 16-byte aligned);
 *     word (k, c) holds columns 8c..8c+7, column 8c+e in bits [4e, 4e+4), q unsigned 0..15.
 * scales: device fp16, ceil(K/G) rows of lds values (lds >= N, multiple of 8, 16-byte
 *     aligned).  group_size G: a multiple of 64.
 * C: device fp16 M x N, 16-byte aligned, ldc a multiple of 8.  epi as tg_gemm_f16_epilogue.
 * Plans: by default for M >= 512 (int4; NF4: M >= 384) with no int4-kernel override
 * (opt->dequant_first), the whole weight matrix is decoded once into fp16 scratch from the
 * library's pool (K x N rounded up to 8, 2 bytes each; released in stream order), the same
 * values the fused kernels use, and the
 * fp16 GEMM (tg_gemm_f16_epilogue) runs on it; without scratch the plan falls back to a fused
 * kernel (TG_ERR_NO_WORKSPACE only when dequant_first = 1 forces it).  Otherwise the weights are
 * decoded inside the GEMM kernel (never written to memory).  Fused kernels: for
 * M <= 128 the swapped-operand kernel (C^T = W^T A^T; opt->swap_ab); otherwise, by default for
 * M >= 256 when the 256 x 256 tiles fill at least half of the clusters of two CTAs that fit at
 * once, 256 x 256 tiles on CTA pairs, each CTA decoding half of the weight tile (opt->pair:
 * 1 force, -1 never); else single-CTA 128 x block_n tiles (opt->block_n 128 or 256, which
 * also selects this kernel).  opt may also set max_ctas (a pair counts as two CTAs), tail
 * (swapped kernel: the last partial wave's tiles as two K halves), tmem_decode, panel_m,
 * timeout_ms and debug_flags.
 * A split tail takes stream-ordered scratch from the library's pool (TG_ERR_NO_WORKSPACE if
 * unavailable).  Misaligned arguments return TG_ERR_MISALIGNED; asynchronous on `stream`.
 */
tg_status tg_gemm_w4a16_f16(const void* A, const void* Wq, const void* scales, void* C,
                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldq,
                            int64_t lds, int64_t ldc, int group_size, const tg_epilogue* epi,
                            const tg_options* opt, tg_stream_t stream);

/*
 * Dequantising GEMM with 4-bit NormalFloat (NF4) weights and fp16 activations (the W_NF4 /
 * A_FP16 case of the TileLang paper-reading page, section 5):
 *     C = fp16( epilogue( A · W ) ),   W[k][n] = fp16( code16[q[k][n]] * scales[k / G][n] )
 * code16[q] is the NF4 code value q of QLoRA (Dettmers et al., NeurIPS 2023, Appendix E:
 * sixteen quantiles of a standard normal scaled to [-1, 1], with an exact 0 at q = 7) rounded
 * to fp16; the product of two fp16 values is rounded to fp16 once.  Packing of Wq, the
 * scales, every other argument, the kernels chosen, the options, alignment and errors are
 * those of tg_gemm_w4a16_f16.
 */
tg_status tg_gemm_nf4a16_f16(const void* A, const void* Wq, const void* scales, void* C,
                             int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldq,
                             int64_t lds, int64_t ldc, int group_size, const tg_epilogue* epi,
                             const tg_options* opt, tg_stream_t stream);

/*
 * The plan tg_gemm_relu_f16_ex would use for these arguments on a device with num_sms SMs.
 * The pointers are used only for their alignment.  Pure host function.
 */
tg_status tg_plan_query(const void* A, const void* B, const void* C, int64_t M, int64_t N,
                        int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int num_sms,
                        const tg_options* opt, tg_plan* out);

/*
 * End-to-end call on HOST buffers: copies A and B (host, row-major with lda/ldb) to the
 * current device, runs the GEMM on `stream`, copies C back into the host buffer (ldc) and
 * synchronises `stream` before returning.  Page-locked host memory gives the fastest copies.
 * Device buffers come from the library pool.  Also reports a kernel timeout
 * (TG_ERR_TIMEOUT), which the asynchronous entry points cannot.
 */
tg_status tg_gemm_relu_f16_host(const void* hA, const void* hB, void* hC, int64_t M,
                                int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                int epilogue_flag, tg_stream_t stream);

/*
 * Reads the current device's error word that the kernels set when a pipeline wait runs out
 * (bit 0: timeout; bits 8..15: the role that gave up: 1 producer, 2 MMA, 3 epilogue).
 * Synchronises the device.  clear != 0 resets the word.  Returns TG_ERR_TIMEOUT if set.
 */
tg_status tg_device_error_check(unsigned* out_word, int clear);

/* Static text for a status code (never NULL). */
const char* tg_status_string(tg_status status);

/* The cudaError_t value behind the calling thread's last TG_ERR_CUDA (0 if none). */
tg_status tg_last_cuda_error(int* cuda_err);

/* Returns the library pool's unused scratch memory on the current device to the system. */
tg_status tg_release_workspace(void);

/*
 * Split-K relu(A·B) that allocates no memory at all.  The paper has no counterpart to it: it
 * exists for callers that cannot call cudaMalloc, cudaMallocAsync or any other allocator
 * while they run a GEMM, for example code running inside an allocator that must not be
 * re-entered, a runtime that has handed all device memory to its own arena, or
 * latency-critical work where an allocation could block or fail.
 *
 * It always takes the split-K path: the K range is cut into S_eff splits, each split writes a
 * float32 partial tile into a fixed workspace, and a second kernel adds the splits in order,
 * applies the epilogue and writes fp16 C.  The workspace is one array of
 * TG_STATIC_WORKSPACE_BYTES bytes of device memory that is part of the library itself: every
 * GPU on which the library is used holds it until the process exits.
 *
 *  - The effective split count: with kb = ceil(K / 64) K blocks and S = split_k (0 means 2)
 *    clamped to 1..kb, each split takes ceil(kb / S) K blocks and S_eff = ceil(kb / ceil(kb /
 *    S)) <= S splits are non-empty (for example kb = 10, S = 6 gives S_eff = 5).
 *  - Needs S_eff * M * (N rounded up to 4) * 4 bytes <= TG_STATIC_WORKSPACE_BYTES (sizing
 *    with split_k in place of S_eff is always enough); a larger need returns
 *    TG_ERR_NO_WORKSPACE before anything is launched.  K == 0 needs no workspace (C = +0).
 *  - A and B must be 16-byte aligned with lda and ldb multiples of 8 (TG_ERR_MISALIGNED
 *    otherwise); C only needs 2-byte alignment.  Other arguments as for tg_gemm_relu_f16.
 *  - The first call on each device does a one-time set-up with that device current (it
 *    looks up the workspace's device address and the device's properties); make that first
 *    call before any stream capture.
 *  - All calls share the one workspace, and it keeps whatever the last call left there.
 *    Nothing in it needs to start at zero (each split overwrites its whole slice before the
 *    reduction reads it), but calls whose work overlaps on the GPU race on it: issue them
 *    on one stream, or order them with events.
 */
#define TG_STATIC_WORKSPACE_BYTES (64ull << 20)
tg_status tg_gemm_relu_f16_splitk_noalloc(const void* A, const void* B, void* C, int64_t M,
                                          int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                          int64_t ldc, int epilogue_flag, int split_k,
                                          tg_stream_t stream);

/* Library version as major*10000 + minor*100 + patch.  300: tg_options gained dequant_first
 * (callers must be built against this header). */
int tg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_RELU_H */
