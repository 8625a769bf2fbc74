// W8A8 in the 32x32 UE8M0 format on hardware block scaling, sm_103a.
//
//   C[m, n] = sum_k A[m, k] 2^(ea[m, k/32] - 127) * B[n, k] 2^(eb[n/32, k/32] - 127)
//
// The weight format is one power-of-two scale per 32x32 block ("SM70 FP8
// block-32 kernels (PLI Labs)", "How it works"); the activations get one
// power of two per token per 32 values of K, so that every 1x32 slice of a
// K block carries one scale on each side: exactly what the tensor cores'
// block-scaled MMA multiplies in ("perf(ArcKernels) ...", "Cheap checks done
// first": the VEC32_UE8M0 scale modes of Blackwell).  The product therefore
// needs no software promotion at all: tcgen05.mma kind::mxf8f6f4
// block_scale scale_vec::1X applies the two scales to each K = 32 slice and
// accumulates the whole K range in TMEM.
//
// Scale operands are kept in the tiled layout the MMA consumes (one byte per
// row -- token or weight column -- per 32 values of K): for 128 rows and one
// 128-wide K block, 512 bytes [r][q][j] with row = 32 q + r and slice j of the
// block, so byte (row, g) sits at
//   ((row / 128) * (K / 128) + g / 4) * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4 + g % 4.
// One such 512-byte block, copied into TMEM by tcgen05.cp 32x128b.warpx4
// (row r into lanes r, 32 + r, 64 + r, 96 + r, four columns), puts row
// 32 q + r's four slice bytes at lane 32 q + r, column q: where the MMA reads
// an A row's scale (lane m, column m / 32) and, for the B side, column n's
// scale (lane 32 (m / 32) + n % 32, column n / 32; layout measured with
// one-hot operands and distinct exponents per lane, column and byte).  The
// 32x32 weight exponents become this layout once per weight, each block's
// byte repeated for its 32 columns.
//
// quant_act_ue8m0_kernel: bf16 x -> e4m3 codes + tiled exponent bytes, one
// thread per 32-value group: e is the smallest integer with 448 * 2^e >= amax
// (from amax's exponent and whether its mantissa exceeds 1.75 = 448 / 2^8),
// clamped to [-127, 126] (bf16 inputs never pass 120), and q =
// e4m3(x * 2^-e), exact before the rounding, never saturating.  Rows past M
// in the last 128-row block get the byte 127 (scale 1).
//
// ue8m0_weight_sf_kernel: [N/32][K/32] weight exponent bytes -> the tiled
// per-column layout.
//
// w8a8_mx_kernel: persistent, one CTA per SM over 128 x 256 output tiles.
//   warp 0      TMA producer: per 128-K block A [128 rows x 128 B], B
//               [256 rows x 128 B] and the three 512-byte scale blocks (A;
//               B columns 0..127 and 128..255) into a 4-stage ring, one
//               barrier per stage.
//   warp 1      TMEM allocation (512 columns: the 256-column accumulator and
//               four scale slots of 12 columns).
//   warps 1, 2  one thread each takes alternate K blocks: it copies the
//               stage's scale blocks into the block's TMEM slot with
//               tcgen05.cp and issues the four K = 32 MMAs (scale byte j for
//               slice j); the two take turns through a barrier pair, so the
//               blocks reach the accumulator in order, and each commits its
//               own stages.
//   warps 4..7  epilogue: the accumulator rows of their lane quarter into
//               registers (bf16), the accumulator released for the next tile,
//               then TMA tensor stores from a swizzled staging box while the
//               next tile's MMAs run.
// Shapes whose tiles would leave at least half of the SMs idle split K over
// a cluster of 2, 4 or 8 CTAs per tile instead (no global workspace): each
// rank accumulates its K range in TMEM, writes the fp32 partial tile to its
// shared memory, and after a cluster barrier sums 1 / split of the tile's
// rows over all ranks (distributed shared memory, rank order) and stores it.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fp8blk {
namespace {

// ------------------------------------------------------------------ quantiser

__device__ __forceinline__ int act_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int E = int((bits >> 23) & 0xFFu);
  if (E == 0) return -127;                                   // zero or subnormal: the clamp
  const int e = (E - 127) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 126 ? 126 : e);
}

// Byte offset of (row, slice g) in the tiled scale layout (kb_count = K / 128).
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t row, int64_t g, int64_t kb_count) {
  return ((row >> 7) * kb_count + (g >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (g & 3);
}

__global__ void __launch_bounds__(256) quant_act_ue8m0_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                                              int64_t K, int64_t ldx, uint8_t* __restrict__ a,
                                                              int64_t lda, uint8_t* __restrict__ sf) {
  griddep_launch_dependents();
  const int64_t groups = K / 32;
  const int64_t kb_count = K / 128;
  const int64_t total = (M + 127) / 128 * 128 * groups;   // rows padded to the 128-row block
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t m = i / groups, g = i % groups;
    if (m >= M) {
      sf[sf_offset(m, g, kb_count)] = 127;
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + m * ldx + g * 32);
    float f[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) bf16x8_to_f32(ld_nc_v4(src + j), f + 8 * j);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(f[j]));
    const int e = act_exponent(amax);
    const float inv = __uint_as_float(uint32_t(127 - e) << 23);   // 2^-e, exact (e <= 126)
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = e4m3x4(f[4 * j] * inv, f[4 * j + 1] * inv, f[4 * j + 2] * inv, f[4 * j + 3] * inv);
    uint4* dst = reinterpret_cast<uint4*>(a + m * lda + g * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sf[sf_offset(m, g, kb_count)] = uint8_t(e + 127);
  }
}

// One thread per 4-byte word of the tiled layout: the word of (128-column
// block nb, K block kb, row r, column group c) holds the four slice bytes of
// 32-column block 4 nb + c, the same for every r.
__global__ void __launch_bounds__(256) ue8m0_weight_sf_kernel(const uint8_t* __restrict__ eb, int64_t N, int64_t K,
                                                              uint32_t* __restrict__ sf) {
  const int64_t kb_count = K / 128;
  const int64_t kw = K / 32;
  const int64_t words = N / 128 * kb_count * 128;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t w = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; w < words; w += stride) {
    const int64_t chunk = w >> 7;
    const int64_t c = w & 3;
    const int64_t nb = chunk / kb_count, kb = chunk % kb_count;
    sf[w] = *reinterpret_cast<const uint32_t*>(eb + (nb * 4 + c) * kw + 4 * kb);
  }
}

// ------------------------------------------------------------------ GEMM

constexpr int BM = 128;               // rows of A / C per tile
constexpr int BN = 256;               // rows of B (columns of C) per tile
constexpr int BK = 128;               // K per stage: four K = 32 MMAs, one scale word
constexpr int kStages = 4;            // operand stages; also the ring of TMEM scale slots
constexpr int kStageA = BM * BK;
constexpr int kStageB = BN * BK;
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kSfCols = 4 + BN / 32;  // A: one column per lane quarter; B: one per 32 columns
constexpr uint32_t kAccCols = BN;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 256;         // warps 0..3 control, 4..7 epilogue
constexpr int kSfBytes = 3 * 512;     // per stage: the A scale block, then B's for columns 0..127 and 128..255
constexpr int kStageC = 32 * 128;     // a warp's 32-row x 128-byte output box
constexpr int kCBufs = 1;             // output boxes in flight per epilogue warp
constexpr size_t kSfOff = size_t(kStages) * kStageBytes;
constexpr size_t kCOff = kSfOff + size_t(kStages) * kSfBytes;
constexpr size_t kBarOff = kCOff + size_t(4 * kCBufs) * kStageC;
constexpr size_t kSmemBytes = kBarOff + 256 + 1024;
static_assert(kAccCols + kStages * kSfCols <= kTmemCols, "TMEM budget");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0 && kCOff % 1024 == 0, "swizzle atoms");
static_assert(kSfOff % 128 == 0 && kSfBytes % 128 == 0, "scale blocks: 16-byte aligned copies");
// Split-K: each rank's fp32 partial tile in its own shared memory (in the
// operand stages), rows padded by 16 bytes so that the row-per-lane stores
// spread over the banks.
constexpr int kRedPitch = BN + 4;
static_assert(size_t(BM) * kRedPitch * 4 <= kSfOff, "partial tile fits in the operand stages");
constexpr int kMaxSplit = 8;

// kind::mxf8f6f4 instruction descriptor: B scale byte [4,6), e4m3 A and B
// (format 0), both K-major, N >> 3 at [17,23), scale type UE8M0 (bit 23),
// M >> 4 at [24,29), A scale byte [29,31).
__host__ __device__ constexpr uint32_t mx_idesc(int m, int n, uint32_t sf_id) {
  return (sf_id << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(m >> 4) << 24) |
         (sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "setp.ne.b32 P, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], P;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}

// Shared-memory descriptor of a 32-row x 16-byte block without swizzle: rows
// of 16 bytes, 8-row core matrices 128 bytes apart (both offset fields 128 B;
// there is one core matrix along the 16 bytes), descriptor version 1.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(128 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Copies 32 rows x 128 bits of shared memory into TMEM columns [taddr,
// taddr + 4), the same rows into each of the four lane quarters (row r to
// lanes r, 32 + r, 64 + r, 96 + r).  Issued by the MMA thread, so it is
// ordered with the MMAs that read the columns.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// Waits until at most kCBufs - 1 of the thread's committed bulk stores are
// still reading shared memory (the oldest staging buffer is free).
__device__ __forceinline__ void wait_staging() {
  if constexpr (kCBufs == 1)
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  else
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
static_assert(kCBufs == 1 || kCBufs == 2, "staging buffers");

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A8Mx | site);
}

// Tile t of the row-major tile grid (columns fastest).
__device__ __forceinline__ void mx_tile(int t, int n_tiles, int& m0, int& n0) {
  const int mt = t / n_tiles;
  m0 = mt * BM;
  n0 = (t - mt * n_tiles) * BN;
}

// One persistent CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Per K block ("it" counts K blocks over all of the CTA's tiles; stage and
// scale slot are it % kStages):
//   warp 0 (producer)  waits empty[s], loads A, B and the three scale blocks
//                      into stage s (one barrier, full[s], with all the bytes);
//   warp 1 (issuer)    waits full[s], copies the scale blocks into TMEM slot s,
//                      issues the four K = 32 MMAs and commits empty[s]; after
//                      a tile's last block it commits acc_full, and before a
//                      tile's first block it waits for acc_empty;
//   warps 4..7         wait acc_full, read the 32 x 256 accumulator rows of
//                      their lane quarter into registers, release the
//                      accumulator (acc_empty) and only then store the tile,
//                      so the next tile's MMAs overlap the stores.
// A scale slot is rewritten only after empty[s] (the MMAs that read it have
// completed) and the next full[s].
template <bool F32>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const uint8_t* __restrict__ a_sf,
                   const uint8_t* __restrict__ b_sf, void* __restrict__ C, int64_t ldc, int M, int N, int K,
                   int split, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* turn = drain + 1;   // [2]: issuer w may issue its next K block
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(turn + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (N + BN - 1) / BN;
  const int num_tiles = ((M + BM - 1) / BM) * n_tiles;
  const int kblocks = K / BK;
  // With split > 1 the grid is one cluster of `split` CTAs per tile, and
  // rank r accumulates K blocks [kb0, kb1) of it; otherwise CTAs walk the
  // tiles persistently over the whole K range.
  const int rank = split > 1 ? int(cluster_ctarank()) : 0;
  const int tile0 = int(blockIdx.x) / split;
  const int tile_step = int(gridDim.x) / split;
  const int kb0 = kblocks * rank / split;
  const int kb1 = kblocks * (rank + 1) / split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);    // producer, with the bytes
      mbar_init(&empty[s], 1);   // MMA commit
    }
    mbar_init(acc_full, 2);      // both issuers' commits
    mbar_init(acc_empty, 4);     // the four epilogue warps
    mbar_init(drain, 2);
    mbar_init(&turn[0], 1);
    mbar_init(&turn[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sf_base = tmem + kAccCols;

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      griddep_wait();   // A and its scales may be the previous kernel's output
      uint32_t it = 0;
      bool ok = true;
      for (int t = tile0; t < num_tiles && ok; t += tile_step) {
        int m0, n0;
        mx_tile(t, n_tiles, m0, n0);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = int(it % kStages);
          if (!mbar_wait(&empty[s], ((it / kStages) & 1u) ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(s) * kStageBytes;
          uint8_t* sf = smem + kSfOff + size_t(s) * kSfBytes;
          // B columns past N (a 128-column last tile): the first half's scales
          // again, so that every slot holds finite scales (B is zero there).
          const uint8_t* sfb0 = b_sf + (int64_t(n0 / 128) * kblocks + kb) * 512;
          const uint8_t* sfb1 = n0 + 128 < N ? sfb0 + int64_t(kblocks) * 512 : sfb0;
          mbar_arrive_expect_tx(&full[s], kStageBytes + kSfBytes);
          tma_load_2d(sa, &tmA, &full[s], kb * BK, m0);
          tma_load_2d(sa + kStageA, &tmB, &full[s], kb * BK, n0);
          tma_load_2d(sa + kStageA + kStageB / 2, &tmB, &full[s], kb * BK, n0 + BN / 2);
          bulk_copy_g2s(sf, a_sf + (int64_t(m0 / 128) * kblocks + kb) * 512, 512, &full[s]);
          bulk_copy_g2s(sf + 512, sfb0, 512, &full[s]);
          bulk_copy_g2s(sf + 1024, sfb1, 512, &full[s]);
        }
      }
      if (!ok) {
        // Copies still in flight complete on full[]: wait for their bytes
        // (bounded) before the CTA can exit.
        const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1u, nullptr);
      }
    } else if ((warp == 1 || warp == 2) && lane == 0) {
      // ---------------------------------------------------------- MMA issuers
      // Issuer w (warps 1 and 2) takes the K blocks `it` with it % 2 == w.
      // One issuing thread alone leaves the tensor pipe idle while it waits
      // on its barrier and commits (the pipe takes an MMA only as the
      // previous one finishes); two issuers hide that.  They take turns
      // through turn[]: block it is issued only after block it - 1 (the
      // fences order the other thread's MMAs before this thread's), so the
      // accumulator sees the blocks in order.
      const uint32_t w = uint32_t(warp - 1);
      uint32_t it = 0;
      bool ok = true;
      int i = 0;
      for (int t = tile0; t < num_tiles && ok; t += tile_step, ++i) {
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if ((it & 1u) != w) continue;
          const int s = int(it % kStages);
          if (kb == kb0 && !mbar_wait(acc_empty, (uint32_t(i) & 1u) ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAccEmpty);
            ok = false;
            break;
          }
          if (!mbar_wait(&full[s], (it / kStages) & 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + size_t(s) * kStageBytes);
          const uint32_t b0 = a0 + kStageA;
          const uint32_t sfa = sf_base + uint32_t(s * kSfCols);
          const uint32_t sfb = sfa + 4u;
          const uint32_t sfs = smem_u32(smem + kSfOff + size_t(s) * kSfBytes);
          tmem_cp_sf(sfa, sf_desc(sfs));
          tmem_cp_sf(sfb, sf_desc(sfs + 512u));
          tmem_cp_sf(sfb + 4u, sf_desc(sfs + 1024u));
          // Turn: issuer 0's k-th block waits for the k-th arrival of issuer
          // 1 (none for its first), issuer 1's k-th for the (k + 1)-th.
          const uint32_t k = it >> 1;
          if ((w == 1u || k > 0u) && !mbar_wait(&turn[w], w == 0u ? ((k - 1u) & 1u) : (k & 1u), abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < BK / 32; ++j)
            mma_mx(tmem, desc_sw128_kmajor(a0 + 32u * j), desc_sw128_kmajor(b0 + 32u * j),
                   mx_idesc(BM, BN, uint32_t(j)), sfa, sfb, (kb > kb0 || j > 0) ? 1u : 0u);
          tc_fence_before();
          mbar_arrive(&turn[w ^ 1u]);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(acc_full);   // each issuer's share of the tile
      }
      // TMEM is released only after every MMA issued above has completed.
      mma_commit(drain);
      if (!mbar_wait(drain, 0, nullptr)) raise_error(err, abort_flag, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    uint8_t* stg = smem + kCOff + size_t(q) * kCBufs * kStageC;
    int i = 0;
    uint32_t boxes = 0;   // output boxes this warp has stored (picks the staging buffer)
    for (int t = tile0; t < num_tiles; t += tile_step, ++i) {
      int m0, n0;
      mx_tile(t, n_tiles, m0, n0);
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full, uint32_t(i) & 1u, abort_flag))) {
        raise_error(err, abort_flag, kSiteEpilogueFull);
        break;
      }
      tc_fence_after();
      const bool rows = m0 + 32 * q < M;
      if (split > 1) {
        // This rank's partial tile into its shared memory, one row per
        // thread, for the cluster reduction below.
        float* red = reinterpret_cast<float*>(smem) + size_t(32 * q + lane) * kRedPitch;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_base + uint32_t(c), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(red + c + 4 * j) = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      } else if constexpr (!F32) {
        // The whole 32 x 256 block: TMEM -> bf16 pairs in registers, then the
        // accumulator is released and the stores follow.
        uint32_t packed[BN / 2];
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          uint32_t v[64];
          tmem_ld_x32(tmem + lane_base + uint32_t(c), v);
          tmem_ld_x32(tmem + lane_base + uint32_t(c + 32), v + 32);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            packed[c / 2 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
#pragma unroll
        for (int b = 0; b < BN / 64; ++b) {
          if (rows && n0 + 64 * b < N) {
            uint8_t* box = stg + size_t(boxes % kCBufs) * kStageC;
            if (lane == 0) wait_staging();   // the box stored kCBufs boxes ago has left this buffer
            __syncwarp();
            uint8_t* dst = box + lane * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(dst + ((ch ^ (lane & 7)) << 4)) =
                  make_uint4(packed[32 * b + 4 * ch], packed[32 * b + 4 * ch + 1], packed[32 * b + 4 * ch + 2],
                             packed[32 * b + 4 * ch + 3]);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, box, n0 + 64 * b, m0 + 32 * q);
              bulk_commit_group();
            }
            ++boxes;
          }
        }
      } else {
        // float32 output: 32-column boxes straight from TMEM; the accumulator
        // is released after the last read.
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_base + uint32_t(c), v);
          tmem_ld_wait();
          if (c + 32 == BN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
          }
          if (rows && n0 + c < N) {
            uint8_t* box = stg + size_t(boxes % kCBufs) * kStageC;
            if (lane == 0) wait_staging();
            __syncwarp();
            uint8_t* dst = box + lane * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(dst + ((ch ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, box, n0 + c, m0 + 32 * q);
              bulk_commit_group();
            }
            ++boxes;
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
  }

  __syncwarp();
  if (split > 1) {
    // Reduce-scatter over the cluster: rank r sums rows [r, r + 1) * BM /
    // split of the tile over all ranks' shared memory, in rank order, and
    // stores them.  Every thread of every CTA reaches both cluster barriers,
    // also after an abort.  (Pushing each row to its owner with st.async
    // instead measured slower: 15.3 against 13.2 us at M = 128, N = 2048,
    // K = 7168.)
    cluster_sync();
    if (!*abort_flag) {
      int m0, n0;
      mx_tile(tile0, n_tiles, m0, n0);
      const int rows_per_rank = BM / split;
      const int total = rows_per_rank * (BN / 4);   // float4 items of this rank's rows
      uint32_t peer[kMaxSplit];
#pragma unroll
      for (int p = 0; p < kMaxSplit; ++p) peer[p] = map_shared_rank(smem_u32(smem), uint32_t(p < split ? p : 0));
      // Two items per thread per pass, every peer's load issued before the
      // sums, so up to 2 * split remote loads are in flight together.
      for (int idx0 = int(threadIdx.x); idx0 < total; idx0 += 2 * kThreads) {
        float4 v[2][kMaxSplit];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int idx = idx0 + h * kThreads;
          const int rr = rank * rows_per_rank + idx / (BN / 4);
          const uint32_t off = uint32_t((rr * kRedPitch + 4 * (idx % (BN / 4))) * 4);
#pragma unroll
          for (int p = 0; p < kMaxSplit; ++p)
            if (idx < total && p < split) v[h][p] = ld_shared_cluster_f4(peer[p] + off);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int idx = idx0 + h * kThreads;
          const int m = m0 + rank * rows_per_rank + idx / (BN / 4);
          const int n = n0 + 4 * (idx % (BN / 4));
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int p = 0; p < kMaxSplit; ++p) {
            if (p < split) {   // rank order
              acc.x += v[h][p].x;
              acc.y += v[h][p].y;
              acc.z += v[h][p].z;
              acc.w += v[h][p].w;
            }
          }
          if (idx < total && m < M && n < N) {
            if constexpr (F32) {
              *reinterpret_cast<float4*>(static_cast<float*>(C) + int64_t(m) * ldc + n) = acc;
            } else {
              *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(C) + int64_t(m) * ldc + n) =
                  make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            }
          }
        }
      }
    }
    cluster_sync();   // the peers have finished reading this CTA's shared memory
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ CTA pairs
// w8a8_mx_pair_kernel: the same product on CTA pairs (tcgen05 .cta_group::2),
// 256 x 256 output tiles, for problems with enough tiles to keep most pairs
// busy.  Each CTA loads its 128 rows of A and its 128 rows of B (N) per K
// block, so per SM the operand bytes per FLOP are two thirds of the 128 x 256
// single-CTA tile's; one thread of the even CTA copies the scale blocks into
// TMEM (tcgen05.cp.cta_group::2: each CTA's own shared memory into its own
// TMEM) and issues M = 256, N = 256 block-scaled MMAs.  A CTA's scale area
// holds its own 128 rows' activation scales and the weight scales of all 256
// columns (both CTAs' MMA halves read every column's scale), loaded with 2-D
// tensor maps so that blocks past M or N arrive zero-filled.
//   warp 0      TMA producer (both CTAs; the bytes complete on the even CTA's
//               stage barrier, whose producer announces the pair's bytes);
//   warp 1      TMEM allocation with the peer;
//   warps 1, 2  in the even CTA, one thread each issues the copies and MMAs of
//               alternate K blocks, taking turns, and multicasts its commits;
//   warps 4..7  epilogue of the CTA's 128 rows, releasing the accumulator to
//               the even CTA's issuer before the stores.
constexpr int PTM = 128;                    // A rows per CTA (256 per pair)
constexpr int PBN = 256;                    // C columns per pair tile (MMA N)
constexpr int PHN = PBN / 2;                // B rows per CTA
constexpr int kPStages = 6;
constexpr int kPStageA = PTM * BK;
constexpr int kPStageB = PHN * BK;
constexpr int kPStageBytes = kPStageA + kPStageB;
constexpr size_t kPSfOff = size_t(kPStages) * kPStageBytes;
constexpr size_t kPCOff = kPSfOff + size_t(kPStages) * kSfBytes;
constexpr size_t kPBarOff = kPCOff + size_t(4) * kStageC;
constexpr size_t kPSmemBytes = kPBarOff + 256 + 1024;
static_assert(kSfCols * kPStages + PBN <= int(kTmemCols), "TMEM budget (pair)");
static_assert(kPSmemBytes <= 232448, "shared memory per CTA (pair)");
static_assert(kPStageA % 1024 == 0 && kPStageB % 1024 == 0 && kPCOff % 1024 == 0, "swizzle atoms (pair)");

__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "setp.ne.b32 P, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], P;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}

__device__ __forceinline__ void tmem_cp_sf_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

template <bool F32>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSfa,
                        const __grid_constant__ CUtensorMap tmSfb, int M, int N, int K, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPBarOff);
  uint64_t* empty = full + kPStages;
  uint64_t* acc_full = empty + kPStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* turn = drain + 1;   // [2] (even CTA): issuer w may issue its next K block
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(turn + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = int(cluster_ctarank());
  const int pair = int(blockIdx.x) >> 1;
  const int num_pairs = int(gridDim.x) >> 1;
  const int n_tiles = (N + PBN - 1) / PBN;
  const int num_tiles = ((M + 2 * PTM - 1) / (2 * PTM)) * n_tiles;
  const int kblocks = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);    // the even CTA's producer, with both CTAs' bytes
      mbar_init(&empty[s], 1);   // MMA commit (multicast to both CTAs)
    }
    mbar_init(acc_full, 2);      // both issuers' commits (multicast)
    mbar_init(acc_empty, 8);     // both CTAs' epilogue warps (used in the even CTA)
    mbar_init(drain, 2);
    mbar_init(&turn[0], 1);
    mbar_init(&turn[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmSfa);
    tma_prefetch_desc(&tmSfb);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any commit or arrive reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sf_base = tmem + kAccCols;

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      griddep_wait();   // A and its scales may be the previous kernel's output
      const uint32_t full0 = map_shared_rank(smem_u32(full), 0);
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs) {
        const int mt = t / n_tiles, nt = t - (t / n_tiles) * n_tiles;
        const int m0 = mt * 2 * PTM + rank * PTM;   // this CTA's A rows
        const int n0 = nt * PBN;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = int(it % kPStages);
          if (!mbar_wait(&empty[s], ((it / kPStages) & 1u) ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(s) * kPStageBytes;
          uint8_t* sf = smem + kPSfOff + size_t(s) * kSfBytes;
          const uint32_t bar = full0 + uint32_t(s) * 8u;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (kPStageBytes + kSfBytes));
          tma_load_2d_pair(sa, &tmA, bar, kb * BK, m0);
          tma_load_2d_pair(sa + kPStageA, &tmB, bar, kb * BK, n0 + rank * PHN);
          // Scale blocks: 512-byte rows of the tiled arrays (128 words each).
          tma_load_2d_pair(sf, &tmSfa, bar, 0, (m0 / 128) * kblocks + kb);
          tma_load_2d_pair(sf + 512, &tmSfb, bar, 0, (n0 / 128) * kblocks + kb);
          tma_load_2d_pair(sf + 1024, &tmSfb, bar, 0, (n0 / 128 + 1) * kblocks + kb);
        }
      }
      if (!ok && rank == 0) {
        const uint32_t first = it > uint32_t(kPStages) ? it - kPStages : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % kPStages], (j / kPStages) & 1u, nullptr);
      }
    } else if ((warp == 1 || warp == 2) && lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuers (even CTA)
      // Two issuers taking turns, as in the single-CTA kernel.
      const uint32_t w = uint32_t(warp - 1);
      uint32_t it = 0;
      bool ok = true;
      int i = 0;
      for (int t = pair; t < num_tiles && ok; t += num_pairs, ++i) {
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          if ((it & 1u) != w) continue;
          const int s = int(it % kPStages);
          if (kb == 0 && !mbar_wait_acq_cluster(acc_empty, (uint32_t(i) & 1u) ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAccEmpty);
            ok = false;
            break;
          }
          if (!mbar_wait_acq_cluster(&full[s], (it / kPStages) & 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + size_t(s) * kPStageBytes);
          const uint32_t b0 = a0 + kPStageA;
          const uint32_t sfa = sf_base + uint32_t(s * kSfCols);
          const uint32_t sfb = sfa + 4u;
          const uint32_t sfs = smem_u32(smem + kPSfOff + size_t(s) * kSfBytes);
          tmem_cp_sf_pair(sfa, sf_desc(sfs));
          tmem_cp_sf_pair(sfb, sf_desc(sfs + 512u));
          tmem_cp_sf_pair(sfb + 4u, sf_desc(sfs + 1024u));
          const uint32_t k = it >> 1;
          if ((w == 1u || k > 0u) && !mbar_wait(&turn[w], w == 0u ? ((k - 1u) & 1u) : (k & 1u), abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < BK / 32; ++j)
            mma_mx_pair(tmem, desc_sw128_kmajor(a0 + 32u * j), desc_sw128_kmajor(b0 + 32u * j),
                        mx_idesc(2 * PTM, PBN, uint32_t(j)), sfa, sfb, (kb > 0 || j > 0) ? 1u : 0u);
          tc_fence_before();
          mbar_arrive(&turn[w ^ 1u]);
          mma_commit_pair_mc(&empty[s], 0x3);
        }
        if (ok) mma_commit_pair_mc(acc_full, 0x3);   // each issuer's share of the tile
      }
      mma_commit_pair_mc(drain, 0x1);
      if (!mbar_wait(drain, 0, nullptr)) raise_error(err, abort_flag, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const uint32_t acc_empty0 = map_shared_rank(smem_u32(acc_empty), 0);
    uint8_t* box = smem + kPCOff + size_t(q) * kStageC;
    int i = 0;
    for (int t = pair; t < num_tiles; t += num_pairs, ++i) {
      const int mt = t / n_tiles, nt = t - (t / n_tiles) * n_tiles;
      const int y = mt * 2 * PTM + rank * PTM + 32 * q;   // this warp's first output row
      const int n0 = nt * PBN;
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full, uint32_t(i) & 1u, abort_flag))) {
        raise_error(err, abort_flag, kSiteEpilogueFull);
        break;
      }
      tc_fence_after();
      const bool rows = y < M;
      if constexpr (!F32) {
        uint32_t packed[PBN / 2];
#pragma unroll
        for (int c = 0; c < PBN; c += 64) {
          uint32_t v[64];
          tmem_ld_x32(tmem + lane_base + uint32_t(c), v);
          tmem_ld_x32(tmem + lane_base + uint32_t(c + 32), v + 32);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            packed[c / 2 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0);
#pragma unroll
        for (int b = 0; b < PBN / 64; ++b) {
          if (rows && n0 + 64 * b < N) {
            if (lane == 0) wait_staging();
            __syncwarp();
            uint8_t* dst = box + lane * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(dst + ((ch ^ (lane & 7)) << 4)) =
                  make_uint4(packed[32 * b + 4 * ch], packed[32 * b + 4 * ch + 1], packed[32 * b + 4 * ch + 2],
                             packed[32 * b + 4 * ch + 3]);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, box, n0 + 64 * b, y);
              bulk_commit_group();
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < PBN; c += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_base + uint32_t(c), v);
          tmem_ld_wait();
          if (c + 32 == PBN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0);
          }
          if (rows && n0 + c < N) {
            if (lane == 0) wait_staging();
            __syncwarp();
            uint8_t* dst = box + lane * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(dst + ((ch ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, box, n0 + c, y);
              bulk_commit_group();
            }
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA leaves while the other may still reach its shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_quant_act_ue8m0(const QuantActUe8m0Args& p, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t total = (p.M + 127) / 128 * 128 * (p.K / 32);
  const int64_t want = (total + 255) / 256;
  const int64_t cap = int64_t(dev.num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? want : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, quant_act_ue8m0_kernel, static_cast<const __nv_bfloat16*>(p.x), p.M, p.K, p.ldx,
                            static_cast<uint8_t*>(p.a), p.lda, p.sf);
}

cudaError_t launch_ue8m0_weight_sf(const uint8_t* eb, int64_t N, int64_t K, uint8_t* sf, const DeviceInfo& dev,
                                   cudaStream_t s) {
  const int64_t words = N / 128 * (K / 128) * 128;
  const int64_t want = (words + 255) / 256;
  const int64_t cap = int64_t(dev.num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? want : cap);
  ue8m0_weight_sf_kernel<<<grid, 256, 0, s>>>(eb, N, K, reinterpret_cast<uint32_t*>(sf));
  return cudaGetLastError();
}

namespace {
// K is split over a cluster of 2, 4 or 8 CTAs when the tiles alone would
// leave at least half of the SMs idle, as far as the tiles x split CTAs fit
// on the GPU and every rank keeps at least two K blocks.  Eight-CTA clusters
// only for up to eight tiles: sixteen of them (M = 16, N = K = 4096) took
// 21.5 us against 12.3 us as sixteen four-CTA clusters, while eight (M = 128,
// N = 2048, K = 7168) took 13.1 us against 14.6 us with four.
int mx_split(int64_t tiles, int kblocks, int num_sms) {
  if (tiles * 2 > num_sms) return 1;
  for (int s = kMaxSplit; s >= 2; s >>= 1)
    if (tiles * s <= num_sms && kblocks >= 2 * s && (s < 8 || tiles <= 8)) return s;
  return 1;
}

template <bool F32>
cudaError_t launch_mx(const GemmW8A8MxArgs& p, const DeviceInfo& dev, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(w8a8_mx_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int64_t tiles = int64_t((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int split = mx_split(tiles, p.K / BK, dev.num_sms);
  const int64_t grid = split > 1 ? tiles * split : (tiles < dev.num_sms ? tiles : dev.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (split > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = unsigned(split);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(na);
  return cudaLaunchKernelEx(&cfg, w8a8_mx_kernel<F32>, p.tmA, p.tmB, p.tmC, p.a_sf, p.b_sf, p.C, p.ldc, p.M, p.N,
                            p.K, split, p.err);
}
}  // namespace

namespace {
template <bool F32>
cudaError_t launch_mx_pair(const GemmW8A8MxArgs& p, const DeviceInfo& dev, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(w8a8_mx_pair_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int tiles = mx_pair_tiles(p.M, p.N);
  const int max_pairs = dev.num_sms / 2;
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w8a8_mx_pair_kernel<F32>, p.tmA, p.tmB, p.tmC, p.tmSfa, p.tmSfb, p.M, p.N, p.K,
                            p.err);
}
}  // namespace

int mx_pair_tiles(int M, int N) { return ((M + 2 * PTM - 1) / (2 * PTM)) * ((N + PBN - 1) / PBN); }

cudaError_t launch_gemm_w8a8_mx(const GemmW8A8MxArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  // Enough 256 x 256 tiles to keep at least half of the CTA pairs busy: the
  // pair kernel; otherwise the single-CTA kernel (K split over a cluster
  // when its tiles leave most SMs idle).
  if (p.M > PTM && 2 * mx_pair_tiles(p.M, p.N) >= dev.num_sms / 2)
    return p.out_f32 ? launch_mx_pair<true>(p, dev, s) : launch_mx_pair<false>(p, dev, s);
  return p.out_f32 ? launch_mx<true>(p, dev, s) : launch_mx<false>(p, dev, s);
}

}  // namespace fp8blk
