/*
 * fp8blk -- block-scaled FP8 linear layer for GB300 (sm_103a), C ABI.
 *
 * The layer computes, with FP32 accumulation and a bf16 result,
 *
 *     C[m, n] = sum_kb ( sum_{k in kb} A[m, k] * B[n, k] ) * As[kb, m] * Bs[n/128, kb]
 *
 * where kb runs over 128-wide blocks of K, B holds e4m3 weights with one fp32
 * scale per 128x128 block, and A holds e4m3 activations with one fp32 scale
 * per token per 128 values of K ("Blockwise FP8 on Ada GPUs, part 2",
 * "The starting point" and "The fix").  The weight-only variant keeps the
 * activations in bf16 ("perf(ArcKernels): blockwise-FP8 GEMM on tensor cores,
 * scale promoted per 128-K", "What this adds"), and a second weight format
 * stores one power-of-two UE8M0 scale per 32x32 block ("SM70 FP8 block-32
 * kernels (PLI Labs)", "How it works").
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never frees them and keeps no reference after the call.
 *  - Matrices are row-major with an explicit leading dimension counted in
 *    ELEMENTS (ld >= number of columns).
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream) and return after the launch.  Argument errors are found on the
 *    host before anything is launched; nothing is written in that case.
 *  - No entry point allocates device memory on the compute path.  The only
 *    host state is a small cache of TMA descriptors and per-device facts.
 *  - e4m3 is the finite-only variant: 0x7F / 0xFF are NaN codes, max 448.
 *  - Kernels never trap.  A pipeline wait that exceeds about one second
 *    makes the kernel record FP8BLK_ERR_TIMEOUT in a per-device error word
 *    and return; fp8blk_device_error() reads (and optionally clears) it.
 *  - Every entry point is thread-safe with respect to the host cache.
 *  - The library refuses to run on any device that is not compute
 *    capability 10.3 (FP8BLK_ERR_ARCH).  There is no CPU fallback.
 */
#ifndef FP8BLK_H_
#define FP8BLK_H_

#include <stdint.h>

#if defined(__GNUC__)
#define FP8BLK_API __attribute__((visibility("default")))
#else
#define FP8BLK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* fp8blk_stream_t;

typedef enum {
  FP8BLK_OK = 0,
  FP8BLK_ERR_INVALID_ARG = 1,       /* null pointer, negative size, ld < cols, lds < M */
  FP8BLK_ERR_UNSUPPORTED_SHAPE = 2, /* N or K not a multiple of the scale block, M above a limit */
  FP8BLK_ERR_MISALIGNED = 3,        /* pointer or row pitch not 16-byte aligned */
  FP8BLK_ERR_ARCH = 4,              /* current device is not sm_103 */
  FP8BLK_ERR_CUDA = 5,              /* a CUDA runtime/driver call or launch failed */
  FP8BLK_ERR_NAN_CODE = 6,          /* fp8blk_validate_weights: an e4m3 NaN code was found */
  FP8BLK_ERR_SCALE_WINDOW = 7,      /* fp8blk_validate_weights: a scale is out of range */
  FP8BLK_ERR_TIMEOUT = 8            /* a kernel gave up on a pipeline wait (device error word) */
} fp8blk_status;

typedef enum {
  /* fp32 scale per 128x128 weight block, array [N/128][K/128] row-major. */
  FP8BLK_SCALE_F32_128x128 = 0,
  /* one byte per 32x32 weight block, array [N/32][K/32] row-major; the byte
   * holds 127 + e and the block's scale is 2^e, e in [-14, 7]. */
  FP8BLK_SCALE_UE8M0_32x32 = 1
} fp8blk_scale_fmt;

/* Compile-time facts of the kernels, exported so that callers never
 * duplicate them ("perf(ArcKernels) ...", "Correctness guards": eligibility
 * is read from the kernel, not restated by the caller). */
typedef struct {
  int32_t abi_version;        /* FP8BLK_ABI_VERSION */
  int32_t scale_block_k;      /* 128: K width of one fp32 scale block */
  int32_t scale_block_n;      /* 128: N height of one fp32 weight scale block */
  int32_t ue8m0_block;        /* 32: side of one UE8M0 block */
  int32_t w8a8_tile_m;        /* rows of C per W8A8 tile */
  int32_t w8a8_tile_n;        /* columns of C per W8A8 tile */
  int32_t w8a16_tile_n;       /* weight rows per W8A16 tile */
  int32_t w8a16_max_tile_m;   /* largest token tile of the W8A16 kernel */
  int32_t gemv_max_m;         /* largest M accepted by fp8blk_gemv_w8a16 (16) */
  int32_t ptr_align_bytes;    /* 16: required alignment of every tensor pointer */
  int32_t row_align_bytes;    /* 16: required alignment of every row pitch */
  int32_t lds_multiple;       /* 4: lds must be a multiple of this */
  int32_t max_split_k;        /* largest split-K cluster the kernels use */
} fp8blk_constraints;

#define FP8BLK_ABI_VERSION 3

/*
 * Launch flags of the three GEMM entry points (bitwise OR; 0 = none).
 *
 * FP8BLK_FLAG_PDL  programmatic dependent launch.  The call's kernel may
 *   start while kernels queued before it on the stream are still running:
 *   it sets up, then reads the weights (b_e4m3) and their scales (b_scales)
 *   at once, and reads the activations and their scales, and writes the
 *   output, only after those kernels have finished and their writes are
 *   visible.  This hides the launch and the first weight fetch behind the
 *   previous kernel's tail, which matters when one call streams only a few
 *   megabytes (decode).  Set it only when no kernel that may still be
 *   running at that point writes the weights or their scales (the usual
 *   case: weights prepared once, long before).  Without the flag every
 *   call waits for the previous work on the stream as usual.
 */
#define FP8BLK_FLAG_PDL 1u

/*
 * FP8BLK_FLAG_OUT_F32  C is float32 instead of bf16: the FP32 accumulator
 *   is stored as it is, with no rounding to bf16, for outputs that are summed
 *   further in FP32 (the K-sharded, row-parallel form of the layer, whose
 *   partial outputs are reduced across devices before the final rounding;
 *   "SM70 FP8 block-32 kernels", which keeps row-parallel outputs in FP32).
 *   ldc then counts float32 elements and ldc*4 % 16 == 0.  The accumulation
 *   is the same as for bf16 output: rounding the float32 result to bf16
 *   (nearest even) gives exactly the bf16 result of the same call.
 */
#define FP8BLK_FLAG_OUT_F32 2u

/* ------------------------------------------------------------------------ */
/* Hot path                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Per-token 1x128 activation quantisation to e4m3
 * ("Blockwise FP8 on Ada GPUs, part 2", "The starting point";
 *  "perf(ArcKernels) ...", "Route-2 handover", finding 2).
 *
 * For every row m and every group g of 128 consecutive K values:
 *     amax = max |x[m, 128g .. 128g+127]|
 *     s    = amax / 448 (IEEE float32 division); s = 1 when amax == 0
 *     a[m, k] = e4m3(x[m, k] / s), round to nearest even, saturating to +-448
 *     a_scales[g * lds + m] = s
 *
 *  x_bf16    [M, K] bf16, row pitch ldx elements (ldx*2 % 16 == 0).
 *  a_e4m3    [M, K] e4m3 bytes out, row pitch lda bytes (lda % 16 == 0).
 *  a_scales  [K/128][lds] float32 out; M is the contiguous axis
 *            (the reading of "[M, ceil(K/128)], M-major"); lds >= M,
 *            lds % 4 == 0.
 *  K % 128 == 0.  M == 0 is a no-op.
 *  Non-finite inputs are outside the contract.
 */
FP8BLK_API fp8blk_status fp8blk_quant_act(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                               void* a_e4m3, int64_t lda, float* a_scales, int64_t lds,
                               fp8blk_stream_t stream);

/*
 * W8A8 block-scaled GEMM ("Blockwise FP8 on Ada GPUs, part 2", "The fix").
 * For each 128-wide K block the kernel forms an FP32 partial on the tensor
 * cores from e4m3 operands only, then promotes it once into the FP32
 * accumulator, multiplied by As[kb, m] * Bs[n/128, kb].  C = bf16(acc),
 * round to nearest even.
 *
 *  a_e4m3    [M, K] e4m3, row pitch lda bytes (lda % 16 == 0).
 *  a_scales  [K/128][lds] float32 (as written by fp8blk_quant_act).
 *  b_e4m3    [N, K] e4m3 weights, K contiguous, row pitch ldb bytes.
 *  b_scales  [N/128][K/128] float32, row-major, packed.
 *  c_bf16    [M, N] bf16 out, row pitch ldc elements (ldc*2 % 16 == 0);
 *            float32 with FP8BLK_FLAG_OUT_F32 (ldc*4 % 16 == 0).
 *  N % 128 == 0, K % 128 == 0, M >= 0 (M == 0 is a no-op).
 *  Weights are assumed finite (see fp8blk_validate_weights).
 *  flags     FP8BLK_FLAG_* (unknown bits: FP8BLK_ERR_INVALID_ARG).
 */
FP8BLK_API fp8blk_status fp8blk_gemm_w8a8(const void* a_e4m3, int64_t lda,
                               const float* a_scales, int64_t lds,
                               const void* b_e4m3, int64_t ldb,
                               const float* b_scales,
                               void* c_bf16, int64_t ldc,
                               int64_t M, int64_t N, int64_t K,
                               uint32_t flags, fp8blk_stream_t stream);

/*
 * Decode-size W8A8 linear layer in one launch: per-token 1x128 quantisation
 * of x fused into the block-scaled GEMM ("Blockwise FP8 on Ada GPUs, part 2",
 * "The starting point" counts the activation quantisation inside the layer's
 * time).  The kernel's producer loads the bf16 rows of each 128-wide K block
 * and quantiser warps compute the codes and scales in shared memory with the
 * same arithmetic as fp8blk_quant_act, so the result is bit for bit the
 * result of fp8blk_quant_act followed by fp8blk_gemm_w8a8 on the same shape,
 * without the intermediate e4m3 tensor in HBM and without a second launch.
 *
 *  x_bf16    [M, K] bf16, row pitch ldx elements (ldx*2 % 16 == 0).
 *  b_e4m3, ldb, b_scales, c_bf16, ldc, N, K, flags   as fp8blk_gemm_w8a8
 *            (FP8BLK_FLAG_PDL, FP8BLK_FLAG_OUT_F32).
 *  1 <= M <= 32 (larger M: FP8BLK_ERR_UNSUPPORTED_SHAPE; call
 *  fp8blk_quant_act and fp8blk_gemm_w8a8 with caller-owned buffers, where the
 *  quantisation pass runs once instead of once per weight tile).  M == 0 is
 *  a no-op.
 */
FP8BLK_API fp8blk_status fp8blk_linear_w8a8(const void* x_bf16, int64_t ldx,
                               const void* b_e4m3, int64_t ldb,
                               const float* b_scales,
                               void* c_bf16, int64_t ldc,
                               int64_t M, int64_t N, int64_t K,
                               uint32_t flags, fp8blk_stream_t stream);

/*
 * Grouped (mixture-of-experts) W8A8 GEMM: the same block-scaled product as
 * fp8blk_gemm_w8a8, but row m of A is multiplied by the weights of group
 * row_group[m] (one expert per row).  The rows of each group are stored
 * contiguously in whole 128-row tiles (the token rows routed to one expert,
 * padded to a multiple of 128), so the group is constant over every aligned
 * 128-row block of A and C; a block whose group is negative is padding and
 * is skipped (its C rows are not written).
 *
 *  a_e4m3, a_scales, lda, lds   as fp8blk_gemm_w8a8, for all M rows.
 *  b_e4m3     [G][N][K] e4m3: group g's weights are rows g*N .. g*N+N-1 of a
 *             [G*N, K] matrix with row pitch ldb bytes.
 *  b_scales   [G][N/128][K/128] float32, packed.
 *  row_group  device int32 [M]; row_group[m] in [0, G) or negative (padding),
 *             constant within each aligned 128-row block.  A block naming a
 *             group >= G is skipped and reported through the device error word.
 *  c_bf16     [M, N] out as fp8blk_gemm_w8a8 (FP8BLK_FLAG_OUT_F32 allowed).
 *  M % 128 == 0, N % 128 == 0, K % 128 == 0, G >= 1.  K == 0 zero-fills all
 *  M rows of C.
 *  flags      FP8BLK_FLAG_PDL (the weights are then read only after the
 *             previous kernel, since row_group decides which) and
 *             FP8BLK_FLAG_OUT_F32.
 */
FP8BLK_API fp8blk_status fp8blk_gemm_w8a8_grouped(const void* a_e4m3, int64_t lda,
                               const float* a_scales, int64_t lds,
                               const void* b_e4m3, int64_t ldb,
                               const float* b_scales,
                               const int32_t* row_group, int64_t G,
                               void* c_bf16, int64_t ldc,
                               int64_t M, int64_t N, int64_t K,
                               uint32_t flags, fp8blk_stream_t stream);

/*
 * UE8M0 scale operands of the W8A8 product are stored in the tiled layout
 * the tensor cores' block scaling reads (one exponent byte, 127 + e, per row
 * -- token or weight column -- per 32 values of K).  For each 128-row block
 * and each 128-wide K block, 512 bytes [r][q][j] with row = 32 q + r and
 * slice j of the K block; byte (row, g) of a rows x K array is at
 *
 *   ((row / 128) * (K / 128) + g / 4) * 512 + (row % 32) * 16
 *     + ((row / 32) % 4) * 4 + g % 4.
 *
 * The pages fix the exponents, not this byte order; it is the one the
 * product's scale copies take without rearranging.
 * fp8blk_ue8m0_sf_bytes: size of such an array for `rows` rows (padded to
 * 128) and K; -1 when rows < 0, K < 0, K % 128 != 0 or the size overflows.
 */
FP8BLK_API int64_t fp8blk_ue8m0_sf_bytes(int64_t rows, int64_t K);

/*
 * Per-token activation quantisation for W8A8 in the 32x32 UE8M0 weight
 * format: one power-of-two scale per token per 32 values of K, so that each
 * 1x32 activation slice meets one 32x32 weight block ("SM70 FP8 block-32
 * kernels (PLI Labs)", "How it works": power-of-two scales per 32x32 block).
 * For each group of 32: e = the smallest integer with 448 * 2^e >= max|x|
 * (no code saturates), clamped to [-127, 126]; max|x| == 0 gives -127;
 * q = e4m3(x * 2^-e), round to nearest even (x * 2^-e is exact).  The pages
 * do not state how activation exponents are chosen; this is the reading.
 *
 *  x_bf16   [M, K] bf16, row pitch ldx elements (ldx*2 % 16 == 0).
 *  a_e4m3   [M, K] e4m3 out, row pitch lda bytes (lda % 16 == 0).
 *  a_sf     fp8blk_ue8m0_sf_bytes(M, K) bytes out, the tiled scale layout;
 *           rows M .. 128*ceil(M/128)-1 get 127 (scale 1).
 *  K % 128 == 0 (the product consumes 128-wide K blocks), M >= 0 (0: no-op).
 *  All pointers 16-byte aligned.  Asynchronous on stream.
 */
FP8BLK_API fp8blk_status fp8blk_quant_act_ue8m0(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                               void* a_e4m3, int64_t lda, uint8_t* a_sf,
                               fp8blk_stream_t stream);

/*
 * Offline weight preparation for fp8blk_gemm_w8a8_ue8m0: the 32x32 block
 * exponents b_exps [N/32][K/32] (the UE8M0 weight format of
 * fp8blk_gemm_w8a16, packed) written as per-column scales in the tiled
 * layout (each block's byte for its 32 columns), fp8blk_ue8m0_sf_bytes(N, K)
 * bytes into b_sf.  N % 128 == 0, K % 128 == 0; 16-byte aligned pointers.
 * Asynchronous on stream.
 */
FP8BLK_API fp8blk_status fp8blk_ue8m0_weight_sf(const uint8_t* b_exps, int64_t N, int64_t K, uint8_t* b_sf,
                               fp8blk_stream_t stream);

/*
 * W8A8 GEMM in the 32x32 UE8M0 format on the tensor cores' block scaling
 * (tcgen05.mma kind::mxf8f6f4 with one UE8M0 scale per 32 values of K on
 * each side; "perf(ArcKernels) ...", "Cheap checks done first" names these
 * VEC32_UE8M0 modes): every K = 32 slice's product is scaled by
 * 2^(ea - 127) * 2^(eb - 127) inside the MMA and accumulated in FP32, with
 * no software promotion.
 *
 *   C[m, n] = sum_k A[m, k] 2^(ea[m, k/32] - 127) * B[n, k] 2^(eb[n/32, k/32] - 127)
 *
 *  a_e4m3, lda, a_sf   as written by fp8blk_quant_act_ue8m0.
 *  b_e4m3   [N, K] e4m3 weights, K contiguous, row pitch ldb bytes.
 *  b_sf     the weight exponents as written by fp8blk_ue8m0_weight_sf.
 *  c        [M, N] bf16 out (round to nearest even), row pitch ldc
 *           elements; float32 with FP8BLK_FLAG_OUT_F32.
 *  N % 128 == 0, K % 128 == 0, M >= 0 (0: no-op), K == 0 zero-fills C.
 *  flags    FP8BLK_FLAG_PDL, FP8BLK_FLAG_OUT_F32.
 *  Weight codes are assumed finite and exponent bytes below 255 (the UE8M0
 *  NaN); fp8blk_validate_weights checks the stricter [-14, 7] window.
 */
FP8BLK_API fp8blk_status fp8blk_gemm_w8a8_ue8m0(const void* a_e4m3, int64_t lda, const uint8_t* a_sf,
                               const void* b_e4m3, int64_t ldb, const uint8_t* b_sf,
                               void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                               uint32_t flags, fp8blk_stream_t stream);

/*
 * W8A16 GEMM: bf16 activations, e4m3 weights decoded to bf16 in registers by
 * integer operations, bf16 tensor-core products with FP32 accumulation
 * ("FP8 / NVFP4 weight-only inference on the RTX 3090 loses nothing",
 *  sections 2 and 4.1; "perf(ArcKernels) ...", "What this adds").
 *
 *  fmt == FP8BLK_SCALE_F32_128x128:
 *     C[m, n] = sum_kb Bs[n/128, kb] * sum_{k in kb} x[m, k] * w[n, k],
 *     one FP32 partial per 128-wide K block promoted with Bs.
 *     b_scales: float32 [N/128][K/128].  N % 128 == 0, K % 128 == 0.
 *  fmt == FP8BLK_SCALE_UE8M0_32x32 ("SM70 FP8 block-32 kernels", "Exactness"):
 *     C[m, n] = sum_k x[m, k] * w[n, k] * 2^e[n/32, k/32],
 *     the power of two is folded exactly into the decoded bf16 weight.
 *     b_scales: uint8 [N/32][K/32] holding 127 + e.  N % 128 == 0, K % 128 == 0.
 *
 *  x_bf16  [M, K] bf16, row pitch ldx elements (ldx*2 % 16 == 0).
 *  b_e4m3  [N, K] e4m3, row pitch ldb bytes (ldb % 16 == 0).
 *  c_bf16  [M, N] bf16 out, row pitch ldc elements (ldc*2 % 16 == 0);
 *          float32 with FP8BLK_FLAG_OUT_F32 (ldc*4 % 16 == 0).
 *  M == 0 is a no-op.  Scales outside [-14, 7] are outside the contract.
 *  flags   FP8BLK_FLAG_* (unknown bits: FP8BLK_ERR_INVALID_ARG).
 *  M <= 32 runs the decode-size kernel (weight stream split over clusters of
 *  CTAs); larger M the token-tiled kernel.
 */
FP8BLK_API fp8blk_status fp8blk_gemm_w8a16(const void* x_bf16, int64_t ldx,
                                const void* b_e4m3, int64_t ldb,
                                const void* b_scales, fp8blk_scale_fmt fmt,
                                void* c_bf16, int64_t ldc,
                                int64_t M, int64_t N, int64_t K,
                                uint32_t flags, fp8blk_stream_t stream);

/*
 * Decode-size W8A16 product (M <= 16), same contract as fp8blk_gemm_w8a16
 * (it runs the same decode-size kernel as fp8blk_gemm_w8a16 at M <= 16).
 * The weights are streamed once from HBM ("FP8 / NVFP4 weight-only
 * inference ...", section 4.3: at small M the time is set by DRAM
 * bandwidth).  M > 16 returns FP8BLK_ERR_UNSUPPORTED_SHAPE.
 */
FP8BLK_API fp8blk_status fp8blk_gemv_w8a16(const void* x_bf16, int64_t ldx,
                                const void* b_e4m3, int64_t ldb,
                                const void* b_scales, fp8blk_scale_fmt fmt,
                                void* c_bf16, int64_t ldc,
                                int64_t M, int64_t N, int64_t K,
                                uint32_t flags, fp8blk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Off the hot path                                                          */
/* ------------------------------------------------------------------------ */

/*
 * 128x128 block weight quantisation ("Blockwise FP8 on Ada GPUs, part 2",
 * "The starting point"): the same rule as fp8blk_quant_act applied to each
 * 128x128 block of w (amax over the block, s = amax / 448).
 *
 *  w_bf16    [N, K] bf16, row pitch ldw elements.
 *  b_e4m3    [N, K] e4m3 out, row pitch ldb bytes.
 *  b_scales  [N/128][K/128] float32 out, packed.
 *  N % 128 == 0, K % 128 == 0.
 */
FP8BLK_API fp8blk_status fp8blk_quant_weight(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                                  void* b_e4m3, int64_t ldb, float* b_scales,
                                  fp8blk_stream_t stream);

/*
 * Load-time weight check ("SM70 FP8 block-32 kernels", "Exactness": the
 * packer refuses NaN codes and scales outside the window).
 * Counts, on the device, into dev_counts[0] the e4m3 NaN codes of b and
 * into dev_counts[1] the bad scales: for FP8BLK_SCALE_F32_128x128 a scale
 * that is not finite or not > 0; for FP8BLK_SCALE_UE8M0_32x32 a byte whose
 * exponent is outside [-14, 7].  dev_counts is a caller-owned device int32[2];
 * it is overwritten.  Asynchronous: read dev_counts after the stream.
 */
FP8BLK_API fp8blk_status fp8blk_validate_weights(const void* b_e4m3, int64_t ldb,
                                      const void* b_scales, fp8blk_scale_fmt fmt,
                                      int64_t N, int64_t K, int32_t* dev_counts,
                                      fp8blk_stream_t stream);

/*
 * Diagnostic: runs the W8A16 kernels' e4m3 -> bf16 integer decode on n codes
 * and writes the bf16 bit patterns of dec(code) * 2^e, e = exp_shift in
 * [-14, 7] (0 for the fp32-scale format).  codes: device uint8[n];
 * out_bf16: device uint16[n].  n % 4 == 0.
 */
FP8BLK_API fp8blk_status fp8blk_debug_decode_e4m3(const void* codes, int64_t n, int32_t exp_shift,
                                       void* out_bf16, fp8blk_stream_t stream);

/*
 * Diagnostic: runs the activation quantisers' scale arithmetic on n group
 * maxima (finite, >= 0): s_out[i] = the group scale amax / 448 (1 for a zero
 * maximum), divisor_out[i] = s scaled by an exact power of two into
 * [2^-60, 2^64], recip_out[i] = the reciprocal the quotients use.  All device
 * float32 arrays of n elements, 4-byte aligned.
 */
FP8BLK_API fp8blk_status fp8blk_debug_group_scale(const float* amax, int64_t n, float* s_out,
                                       float* divisor_out, float* recip_out,
                                       fp8blk_stream_t stream);

/*
 * Diagnostic: the device's rate for a plain read-only stream, the bound on
 * what any kernel that reads a weight set once can reach (no counterpart in
 * the pages; it frames the decode-size rooflines).  Reads `bytes` bytes at p
 * with 16-byte loads (eight in flight per thread, a grid-stride loop over
 * four 512-thread CTAs per SM, streaming cache hint) and XORs every 32-bit
 * word into *sink (*sink ^= w0 ^ w1 ^ ...; the caller sets its initial
 * value).  p: device, 16-byte aligned; bytes % 16 == 0 (else
 * FP8BLK_ERR_MISALIGNED / FP8BLK_ERR_INVALID_ARG before any device work);
 * sink: device uint32, 4-byte aligned.  Asynchronous on stream.
 */
FP8BLK_API fp8blk_status fp8blk_debug_stream_read(const void* p, int64_t bytes, uint32_t* sink,
                                       fp8blk_stream_t stream);

/*
 * Failure-detection check of the bounded waits (no counterpart in the pages;
 * it exercises the library's own error path).  Launches one warp that
 * initialises an mbarrier nobody arrives on and waits for it with the same
 * bounded-wait loop the GEMM kernels use, but with a limit of limit_ns
 * nanoseconds of %globaltimer instead of one second.  When the limit passes
 * the kernel writes FP8BLK_DIAG_TIMEOUT_CODE into the device error word (if
 * it is still 0) and returns normally, so the CUDA context stays usable; the
 * caller then sees FP8BLK_ERR_TIMEOUT from fp8blk_device_error().
 * limit_ns must lie in [1000, 100000000] (1 us .. 100 ms), else
 * FP8BLK_ERR_INVALID_ARG before any device work.  Asynchronous on stream.
 */
#define FP8BLK_DIAG_TIMEOUT_CODE 0x4F01
FP8BLK_API fp8blk_status fp8blk_debug_wait_timeout(int64_t limit_ns, fp8blk_stream_t stream);

/* Fills *out with the kernels' compile-time constraints.  No device needed. */
FP8BLK_API fp8blk_status fp8blk_query_constraints(fp8blk_constraints* out);

/* Static English text for a status code.  Never NULL. */
FP8BLK_API const char* fp8blk_status_string(fp8blk_status status);

/*
 * Reads the current device's error word.  It first waits for all work on
 * the device to finish (cudaDeviceSynchronize: every stream, non-blocking
 * ones included), so a kernel that gave up on a wait is always seen, and a
 * clear cannot race a kernel that records a timeout later.
 * *out_code receives the raw word (0 = no error; otherwise an internal code
 * naming the wait that expired).  Returns FP8BLK_ERR_TIMEOUT when the word
 * is set, FP8BLK_OK when clear, FP8BLK_ERR_CUDA when the synchronisation or
 * the read fails.  clear != 0 resets the word to 0.
 */
FP8BLK_API fp8blk_status fp8blk_device_error(int32_t* out_code, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* FP8BLK_H_ */
