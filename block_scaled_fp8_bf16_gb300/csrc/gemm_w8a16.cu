// W8A16 GEMM for sm_103a: bf16 activations x e4m3 weights, FP32 accumulate.
//
// There is no bf16 x e4m3 tensor-core instruction, so the weights are decoded
// to bf16 and the product runs as bf16 x bf16 MMA ("FP8 / NVFP4 weight-only
// inference on the RTX 3090 loses nothing", section 2; the Blackwell kernel
// it quotes decodes to BF16 and issues BF16 tcgen05 MMA).
//
// The problem is computed transposed, C^T[n, m] = sum_k W[n, k] X[m, k]: a
// 128-row weight tile is the MMA's M side and a token tile of TM = 16..256
// rows is the MMA's N side, so decode-size batches still fill the 128-row
// tensor-core operand, and at large M one decoded weight block feeds 256
// tokens (UE8M0 scales only: the fp32 format needs two partial buffers per
// tile, which do not fit in TMEM next to a 256-column accumulator).  The decoded weights go straight from registers into
// tensor memory (tcgen05.st) and feed the MMA as its TMEM-resident A operand,
// so shared memory only carries the raw e4m3 tile and the activation tile:
//
//   warp 0      TMA producer: e4m3 weight tile [128 n x 128 k] (16 KB) and
//               bf16 activation tile [TM x 128 k] per 128-K block.
//   warp 1      TMEM allocation.
//   warps 1, 2  one thread each issues the eight tcgen05.mma kind::f16
//               (K = 16) of alternate K blocks, A from TMEM, B from smem (the
//               tensor pipe takes an MMA only as the previous one finishes, so
//               one thread alone would leave it idle while it waits and
//               commits); with UE8M0 scales, whose blocks share one
//               accumulator, the two take turns through a barrier pair.
//   warps 3..   decode: thread = weight row; reads its 128 codes, decodes them
//               exactly to bf16 (integer ops + one packed multiply, see
//               decode.cuh) and stores them to one of four TMEM A buffers.
//   then        epilogue: thread = weight row n, TM accumulators (tokens);
//               at TM = 256 streamed from TMEM to C in 32-column chunks.
//
// Scale formats:
//   fp32 128x128: one FP32 partial per 128-K block in TMEM (double buffered),
//     promoted once per block as acc += partial * Bs[n/128, kb]
//     ("perf(ArcKernels) ...", "What this adds": promote at every scale-block
//     boundary along K).
//   UE8M0 32x32: the power of two 2^e of each 32x32 block is folded exactly
//     into the decode multiplier, so the whole K range accumulates in TMEM
//     and the epilogue only converts ("SM70 FP8 block-32 kernels (PLI Labs)",
//     "Exactness").
//
// Tiles run persistently; when the tile count cannot fill the GPU, K is split
// over a 2..4-CTA cluster and the FP32 partial tiles are summed in rank order
// through distributed shared memory by rank 0.
#include <cuda_bf16.h>

#include "decode.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8blk {
namespace {

constexpr int BN = kW8A16TileN;   // weight rows per tile (MMA M)
constexpr int BK = 128;           // K per block (one fp32 scale block)
constexpr int kStageW = BN * BK;  // 16 KB of e4m3
constexpr int kACols = BK / 2;    // TMEM columns of one decoded A block (2 bf16 per column)
constexpr int kABufs = 4;         // decoded A blocks in flight in TMEM
constexpr int kGroupN = 8;
constexpr int kBarrierBytes = 512;
constexpr int kCtlWarps = 3;      // producer, two MMA issuers; the decode warps follow

// F32: float output (the 256-token tile then keeps eight decode warps: with
// four, its float epilogue does not fit in the registers left).
template <int TM, bool F32 = false>
struct Cfg {
  // Epilogue warps: 4 (one per TMEM lane quarter), or 8 / 16 for the 128- /
  // 256-token tiles, where two / four warps share a lane quarter and split
  // the columns.
  static constexpr int kEpiWarps = TM == 256 ? 16 : (TM == 128 ? 8 : 4);
  static constexpr int kEpiCols = TM / (kEpiWarps / 4);
  // Decode warps: two per TMEM lane quarter (each decodes half of the K
  // block), except at TM = 64 and 256, where one per quarter keeps up with
  // the MMAs (at TM = 128 with two MMA issuers, eight decode warps measured
  // 3-4 % faster than four; at TM = 256 a decoded block feeds twice the MMA
  // work, and four warps leave registers for the epilogue).
  static constexpr int kDecWarps = (TM == 64 || (TM == 256 && !F32)) ? 4 : 8;
  static constexpr int kDecChunks = 8 / (kDecWarps / 4);   // 16-byte chunks of a row per decode warp
  static constexpr int kThreads = 32 * kCtlWarps + (kDecWarps + kEpiWarps) * 32;
  static constexpr int kStageX = TM * BK * 2;                  // bf16 activation tile
  // TM = 256: the weight codes and the activations come through separate
  // rings, the activations in half-K-block stages of 32 KB, so that within
  // the same shared memory the activations are requested two K blocks ahead
  // of the MMAs (whole 80 KB stages left room for one block of lookahead).
  static constexpr bool kSplitRing = TM == 256;
  static constexpr int kStageBytes = kSplitRing ? kStageW : kStageW + kStageX;
  static constexpr int kXHalf = TM * 64 * 2;                   // activation half block (split ring)
  static constexpr int kXStages = kSplitRing ? 5 : 1;
  // One CTA per SM (registers are allocated per 4-warp group, so a second
  // 10..14-warp CTA would not fit); the ring is as deep as shared memory allows.
  static constexpr int kStages = TM == 16 ? 8 : (TM == 32 ? 7 : (TM == 64 ? 5 : (TM == 128 ? 4 : 2)));
  static constexpr size_t kXOffset = size_t(kStages) * kStageBytes;   // activation ring (split ring)
  static constexpr size_t kRingBytes = kXOffset + (kSplitRing ? size_t(kXStages) * kXHalf : 0);
  // A 32 x 32 bf16 transpose buffer per epilogue warp (bf16 output).
  static constexpr size_t kOutStage = size_t(kEpiWarps) * 32 * 32 * 2;
  // FP32 partial buffers: as many as fit next to the A blocks (the promotion
  // round trip per K block is long compared with a narrow tile's MMA time).
  // TM = 256 (UE8M0 only) has one accumulator: the tensor pipe waits while
  // the epilogue drains it.
  static constexpr int kDBufs = TM <= 32 ? 8 : (TM == 64 ? 4 : (TM == 128 ? 2 : 1));
  static constexpr uint32_t kTmemUsed = kABufs * kACols + kDBufs * TM;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static constexpr uint32_t kIdesc = make_idesc(1 /* bf16 */, BN, TM);
  static constexpr size_t kSmemBytes = kRingBytes + kOutStage + kBarrierBytes + 1024;
  static constexpr int kMinBlocks = 1;
  static_assert(TM % 16 == 0 && TM >= 16 && TM <= 256, "tcgen05 N for M = 128");
  static_assert(kStageX % 1024 == 0, "activation tile must keep 1024-B swizzle alignment");
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kRingBytes >= size_t(TM) * BN * 4, "reduction buffer fits in the stages");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kMinBlocks == 1 || 2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM must fit");
};

__device__ __forceinline__ void tile_coords(int t, int n_tiles, int m_tiles, int& nt, int& mt) {
  const int per_group = kGroupN * m_tiles;
  const int g = t / per_group;
  const int first = g * kGroupN;
  const int gsz = min(n_tiles - first, kGroupN);
  const int r = t - g * per_group;
  nt = first + r % gsz;
  mt = r / gsz;
}

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A16 | site);
}

__device__ __forceinline__ float to_out(float v, float*) { return v; }

template <int COLS, class OutT>
__device__ __forceinline__ void store_col(OutT* __restrict__ C, int64_t ldc, int M, int m0, int n, const float* acc) {
#pragma unroll
  for (int j = 0; j < COLS; ++j) {
    if (m0 + j < M) C[size_t(m0 + j) * ldc + n] = to_out(acc[j], C);
  }
}

// Stores 32 tokens of C for the warp's 32 weight rows: lane l holds v[j] =
// C[m0 + j][n0 + l].  The values go through the warp's 32 x 32 transpose
// buffer in shared memory, so C is written in 16-byte pieces of its rows
// (eight tokens per pass, four lanes per token) instead of one 2-byte store
// per lane and token.
__device__ __forceinline__ void store_rows32_bf16(__nv_bfloat16* __restrict__ C, int64_t ldc, int M, int m0, int n0,
                                                  const float* v, __nv_bfloat16* tr, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j) tr[j * 32 + lane] = __float2bfloat16_rn(v[j]);
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = q * 8 + (lane >> 2);
    const uint4 val = *reinterpret_cast<const uint4*>(tr + r * 32 + (lane & 3) * 8);
    if (m0 + r < M) *reinterpret_cast<uint4*>(C + size_t(m0 + r) * ldc + n0 + (lane & 3) * 8) = val;
  }
  __syncwarp();
}

// OutT: __nv_bfloat16 (rounded to nearest even) or float (the accumulator as is).
template <int TM, class OutT>
__global__ void __launch_bounds__(Cfg<TM, sizeof(OutT) == 4>::kThreads, Cfg<TM, sizeof(OutT) == 4>::kMinBlocks)
    w8a16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const void* __restrict__ scales, int fmt, OutT* __restrict__ C, int64_t ldc, int M,
                 int N, int K, int split, int* __restrict__ err) {
  using Q = Cfg<TM, sizeof(OutT) == 4>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Q::kRingBytes + Q::kOutStage);
  uint64_t* empty = full + Q::kStages;
  uint64_t* xfull = empty + Q::kStages;       // split ring: activation half blocks
  uint64_t* xempty = xfull + Q::kXStages;
  uint64_t* afull = xempty + Q::kXStages;
  uint64_t* aempty = afull + kABufs;
  uint64_t* dfull = aempty + kABufs;
  uint64_t* dempty = dfull + Q::kDBufs;
  uint64_t* drain = dempty + Q::kDBufs;
  uint64_t* turn = drain + 1;   // [2], UE8M0: issuer w may issue its next K block
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(turn + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  griddep_launch_dependents();   // the next kernel may start its prologue; it gets an SM when this CTA leaves

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = N / BN;
  const int m_tiles = (M + TM - 1) / TM;
  const int num_tiles = n_tiles * m_tiles;
  const int kblocks = K / BK;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster_id = blockIdx.x / split;
  const int num_clusters = gridDim.x / split;
  const int kb_begin = (kblocks * rank) / split;
  const int kb_end = (kblocks * (rank + 1)) / split;
  const bool ue8m0 = fmt != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Q::kStages; ++s) {
      mbar_init(&full[s], 1);
      // decoders done with W (and, with one ring, the MMA done with X)
      mbar_init(&empty[s], Q::kDecWarps + (Q::kSplitRing ? 0 : 1));
    }
    for (int s = 0; s < Q::kXStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int i = 0; i < kABufs; ++i) {
      mbar_init(&afull[i], Q::kDecWarps);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < Q::kDBufs; ++i) {
      mbar_init(&dfull[i], ue8m0 ? 2 : 1);   // UE8M0: both issuers' commits at the end of a tile
      mbar_init(&dempty[i], Q::kEpiWarps);
    }
    mbar_init(drain, 2);
    mbar_init(&turn[0], 1);
    mbar_init(&turn[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Q::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tmem_a = tmem;                 // 2 x 64 columns of decoded weights
  const uint32_t tmem_d = tmem + kABufs * kACols;   // kDBufs x TM columns of FP32 accumulators

  constexpr int EC = Q::kEpiCols;
  float acc[TM == 256 ? 1 : EC];   // TM = 256 streams the accumulator instead
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;          // weight row within the tile (TMEM lane)
  // first token column of this epilogue warp (warps sharing a lane quarter split the columns)
  const int col0 = TM == 256 ? (warp >= kCtlWarps + Q::kDecWarps ? ((warp - kCtlWarps - Q::kDecWarps) >> 2) * EC : 0)
                             : (warp >= kCtlWarps + Q::kDecWarps + 4 ? EC : 0);
  int last_nt = 0, last_mt = 0;   // the epilogue's last tile (one per cluster when K is split)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();   // activations may come from the previous kernel (programmatic dependent launch)
      uint32_t it = 0, w_issued = 0, x_issued = 0;
      bool ok = true;
      const uint64_t pol_w = m_tiles > 1 ? policy_evict_last() : policy_evict_first();
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
        int nt, mt;
        tile_coords(t, n_tiles, m_tiles, nt, mt);
        for (int kb = kb_begin; kb < kb_end && ok; ++kb, ++it) {
          const int s = it % Q::kStages;
          const uint32_t ph = (it / Q::kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          uint8_t* sw = smem + size_t(s) * Q::kStageBytes;
          if constexpr (Q::kSplitRing) {
            mbar_arrive_expect_tx(&full[s], kStageW);
            tma_load_2d_hint(sw, &tmW, &full[s], kb * BK, nt * BN, pol_w);
            ++w_issued;
            for (int h = 0; h < 2; ++h) {
              const uint32_t xs = x_issued % uint32_t(Q::kXStages);
              if (!mbar_wait(&xempty[xs], ((x_issued / Q::kXStages) & 1u) ^ 1u, abort_flag)) {
                raise_error(err, abort_flag, kSiteProducerEmpty);
                ok = false;
                break;
              }
              uint8_t* sx = smem + Q::kXOffset + size_t(xs) * Q::kXHalf;
              mbar_arrive_expect_tx(&xfull[xs], Q::kXHalf);
              tma_load_2d(sx, &tmX, &xfull[xs], kb * BK + 64 * h, mt * TM);
              ++x_issued;
            }
          } else {
            uint8_t* sx = sw + kStageW;
            mbar_arrive_expect_tx(&full[s], Q::kStageBytes);
            tma_load_2d_hint(sw, &tmW, &full[s], kb * BK, nt * BN, pol_w);
            tma_load_2d(sx, &tmX, &full[s], kb * BK, mt * TM);
            tma_load_2d(sx + TM * 128, &tmX, &full[s], kb * BK + 64, mt * TM);
            ++w_issued;
          }
        }
      }
      if (!ok) {
        // wait for the copies still in flight before the CTA exits
        const uint32_t first = w_issued > uint32_t(Q::kStages) ? w_issued - Q::kStages : 0u;
        for (uint32_t j = first; j < w_issued; ++j) mbar_wait(&full[j % Q::kStages], (j / Q::kStages) & 1u, nullptr);
        const uint32_t xfirst = x_issued > uint32_t(Q::kXStages) ? x_issued - Q::kXStages : 0u;
        for (uint32_t j = xfirst; j < x_issued; ++j)
          mbar_wait(&xfull[j % Q::kXStages], (j / Q::kXStages) & 1u, nullptr);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer w takes the K blocks `it` with it % 2 == w, so its stages, A
    // buffers and (fp32 format) partial buffers are those of its parity; the
    // stage's own barrier is not re-tested: "A block decoded" implies the
    // stage landed, because every decode warp waits for the stage before it
    // decodes.  (With the split ring the activation half blocks have their
    // own barriers, waited here; their stages pass between the issuers, which
    // is unambiguous because the turns order every block after the previous
    // one, whose half blocks had landed.)  UE8M0 blocks accumulate into one buffer per tile, so the
    // issuers take turns there: block it after block it - 1 (the fences
    // order the other thread's MMAs before this thread's).
    if (lane == 0) {
      const uint32_t w = uint32_t(warp - 1);
      uint32_t it = 0;
      bool ok = true;
      int i = 0;
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters, ++i) {
        for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
          if ((it & 1u) != w) continue;
          const bool first_kb = kb == kb_begin;
          // fp32 format: one accumulator buffer per K block; UE8M0: per tile.
          const bool new_acc = !ue8m0 || first_kb;
          const uint32_t acc_it = ue8m0 ? uint32_t(i) : it;
          const uint32_t d = acc_it % uint32_t(Q::kDBufs);
          const uint32_t dph = (acc_it / uint32_t(Q::kDBufs)) & 1u;
          const uint32_t s = it % uint32_t(Q::kStages);
          const uint32_t a = it % uint32_t(kABufs);
          const uint32_t aph = (it / uint32_t(kABufs)) & 1u;
          if (new_acc && !mbar_wait(&dempty[d], dph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAccEmpty);
            ok = false;
            break;
          }
          if (!mbar_wait(&afull[a], aph, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAFull);
            ok = false;
            break;
          }
          if (ue8m0) {
            // issuer 0's k-th block waits for the k-th arrival of issuer 1
            // (none for its first), issuer 1's k-th for the (k + 1)-th
            const uint32_t k = it >> 1;
            if ((w == 1u || k > 0u) && !mbar_wait(&turn[w], w == 0u ? ((k - 1u) & 1u) : (k & 1u), abort_flag)) {
              raise_error(err, abort_flag, kSiteMmaAFull);
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_d + d * uint32_t(TM);
          const uint32_t a_tmem = tmem_a + a * uint32_t(kACols);
          if constexpr (Q::kSplitRing) {
            // the activation half blocks of this K block, 2 it and 2 it + 1
            for (uint32_t h = 0; h < 2u; ++h) {
              const uint32_t xi = 2u * it + h;
              const uint32_t xs = xi % uint32_t(Q::kXStages);
              if (!mbar_wait(&xfull[xs], (xi / Q::kXStages) & 1u, abort_flag)) {
                raise_error(err, abort_flag, kSiteMmaAFull);
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t xdesc = desc_sw128_kmajor(smem_u32(smem + Q::kXOffset + size_t(xs) * Q::kXHalf));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_bf16_ts(d_tmem, a_tmem + uint32_t((h * 4 + j) * 8), xdesc + uint64_t((j * 32) >> 4), Q::kIdesc,
                            (h > 0 || j > 0 || !new_acc) ? 1u : 0u);
              mma_commit(&xempty[xs]);
            }
            if (!ok) break;
          } else {
            const uint64_t xdesc = desc_sw128_kmajor(smem_u32(smem + size_t(s) * Q::kStageBytes + kStageW));
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              // advance the start-address field (16-byte units) to k-step j
              const uint64_t xd = xdesc + uint64_t(((j >> 2) * TM * 128 + (j & 3) * 32) >> 4);
              mma_bf16_ts(d_tmem, a_tmem + uint32_t(j * 8), xd, Q::kIdesc, (j > 0 || !new_acc) ? 1u : 0u);
            }
          }
          if (ue8m0) {
            tc_fence_before();
            mbar_arrive(&turn[w ^ 1u]);
          }
          if constexpr (!Q::kSplitRing) mma_commit(&empty[s]);
          mma_commit(&aempty[a]);
          if (!ue8m0) mma_commit(&dfull[d]);
        }
        // UE8M0: each issuer's share of the tile's accumulator (count 2).
        if (ok && ue8m0) mma_commit(&dfull[uint32_t(i) % uint32_t(Q::kDBufs)]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < kCtlWarps + Q::kDecWarps) {
    // ------------------------------------------------------------ decode
    // First 16-byte chunk of the row this warp decodes (second warp of a
    // lane quarter takes the upper half of the K block).
    const int c_first = ((warp - kCtlWarps) / 4) * Q::kDecChunks;
    uint32_t it = 0;
    bool ok = true;
    const float* bs32 = static_cast<const float*>(scales);
    const uint8_t* ue = static_cast<const uint8_t*>(scales);
    (void)bs32;
    for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
      int nt, mt;
      tile_coords(t, n_tiles, m_tiles, nt, mt);
      const int n = nt * BN + row;
      // The warp's 32 rows share one UE8M0 scale row (n / 32): its four bytes
      // per K block are loaded 32 K blocks at a time, one K block per lane,
      // and handed out by shuffles, so no global load waits on the decode.
      const uint32_t* ue_row = reinterpret_cast<const uint32_t*>(ue + size_t(n / 32) * (K / 32));
      uint32_t e4_win = 0;
      for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
        const int s = it % Q::kStages;
        const uint32_t ph = (it / Q::kStages) & 1u;
        const int a = it % kABufs;
        const uint32_t aph = (it / kABufs) & 1u;
        // multipliers for the four 32-wide K groups of this block
        uint32_t mul[4];
        if (ue8m0) {
          const int wi = (kb - kb_begin) & 31;
          if (wi == 0) e4_win = kb + lane < kb_end ? __ldg(ue_row + kb + lane) : 0u;
          const uint32_t e4 = __shfl_sync(0xffffffffu, e4_win, wi);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int e = int((e4 >> (8 * g)) & 0xFFu) - 127;
            mul[g] = decode_multiplier_bf16x2(e);
          }
        } else {
#pragma unroll
          for (int g = 0; g < 4; ++g) mul[g] = decode_multiplier_bf16x2(0);
        }
        const bool got_w = __all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_flag));
        if (!got_w) {
          raise_error(err, abort_flag, kSiteDecodeFull);
          ok = false;
          break;
        }
        // This warp's codes of the row (all 128, or one 64-wide half), 16 per
        // 16-byte chunk; chunk c sits at position c ^ (row & 7) of the
        // 128-byte swizzled row.
        const uint8_t* wrow = smem + size_t(s) * Q::kStageBytes + row * 128;
        uint4 raw[Q::kDecChunks];
#pragma unroll
        for (int c = 0; c < Q::kDecChunks; ++c)
          raw[c] = *reinterpret_cast<const uint4*>(wrow + (((c + c_first) ^ (row & 7)) << 4));
        // The codes were read through the generic proxy and the stage is
        // refilled by TMA (async proxy): without this fence the refill can
        // overtake the reads (seen as wrong weight rows in whole tiles).
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const bool got_a = __all_sync(0xffffffffu, mbar_wait(&aempty[a], aph ^ 1u, abort_flag));
        if (!got_a) {
          raise_error(err, abort_flag, kSiteDecodeAEmpty);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_a + (uint32_t(quarter * 32) << 16) + uint32_t(a * kACols + c_first * 8);
#pragma unroll
        for (int h = 0; h < Q::kDecChunks / 2; ++h) {   // 32 codes -> 16 TMEM columns
          uint32_t words[16];
          // group of 32 codes: h (first half or whole block) or h + 2 (second half)
          const uint32_t m = c_first == 0 ? mul[h] : mul[(h + 2) & 3];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const uint4 v = raw[2 * h + c2];
            decode4_e4m3_bf16(v.x, m, words[8 * c2 + 0], words[8 * c2 + 1]);
            decode4_e4m3_bf16(v.y, m, words[8 * c2 + 2], words[8 * c2 + 3]);
            decode4_e4m3_bf16(v.z, m, words[8 * c2 + 4], words[8 * c2 + 5]);
            decode4_e4m3_bf16(v.w, m, words[8 * c2 + 6], words[8 * c2 + 7]);
          }
          tmem_st_x16(taddr + uint32_t(h * 16), words);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[a]);
      }
    }
  } else if constexpr (TM == 256) {
    // ------------------------------------------------------------ epilogue, UE8M0
    // The whole K range is in the one accumulator, and the tensor pipe waits
    // while it drains.  With bf16 output this warp reads all of its 64 token
    // columns at once, releases the buffer, so that the next tile's MMAs
    // overlap the stores, and then stores them through its transpose buffer
    // (a 2-byte store per thread and token took most of the time).  Float
    // output (64 more registers would spill) is read and stored 32 columns at
    // a time and released after the stores.
    griddep_wait();   // the output may still be read or written by the previous kernel
    __nv_bfloat16* tr = reinterpret_cast<__nv_bfloat16*>(smem + Q::kRingBytes) +
                        (warp - kCtlWarps - Q::kDecWarps) * (32 * 32);
    uint32_t i = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++i) {
      int nt, mt;
      tile_coords(t, n_tiles, m_tiles, nt, mt);
      const bool got = __all_sync(0xffffffffu, mbar_wait(&dfull[0], i & 1u, abort_flag));
      if (!got) {
        raise_error(err, abort_flag, kSiteEpilogueFull);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_d + (uint32_t(quarter * 32) << 16) + uint32_t(col0);
      const int m0 = mt * TM + col0;
      const int n = nt * BN + row;
      static_assert(EC == 64, "two 32-column chunks per epilogue warp");
      if constexpr (sizeof(OutT) == 2) {
        uint32_t p[64];
        tmem_ld_x32(taddr, p);
        tmem_ld_x32(taddr + 32u, p + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[0]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(p[c * 32 + j]);
          store_rows32_bf16(C, ldc, M, m0 + c * 32, nt * BN + quarter * 32, v, tr, lane);
        }
      } else {
        (void)tr;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t p[32];
          tmem_ld_x32(taddr + uint32_t(c * 32), p);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(p[j]);
          store_col<32>(C, ldc, M, m0 + c * 32, n, v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[0]);
      }
    }
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    griddep_wait();   // the output may still be read or written by the previous kernel
    __nv_bfloat16* tr = reinterpret_cast<__nv_bfloat16*>(smem + Q::kRingBytes) +
                        (warp - kCtlWarps - Q::kDecWarps) * (32 * 32);
    uint32_t acc_it = 0;
    bool ok = true;
    const float* bs32 = static_cast<const float*>(scales);
    for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
      int nt, mt;
      tile_coords(t, n_tiles, m_tiles, nt, mt);
      last_nt = nt;
      last_mt = mt;
#pragma unroll
      for (int j = 0; j < EC; ++j) acc[j] = 0.f;
      const int kb_stop = ue8m0 ? kb_begin + 1 : kb_end;   // UE8M0: one drain per tile
      for (int kb = kb_begin; kb < kb_stop; ++kb, ++acc_it) {
        const int d = acc_it % Q::kDBufs;
        const uint32_t dph = (acc_it / Q::kDBufs) & 1u;
        // (issued before the wait for the partial, which takes longer)
        const float sc = ue8m0 ? 1.f : __ldg(bs32 + size_t(nt) * kblocks + kb);
        const bool got = __all_sync(0xffffffffu, mbar_wait(&dfull[d], dph, abort_flag));
        if (!got) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_d + (uint32_t(quarter * 32) << 16) + uint32_t(d * TM + col0);
#pragma unroll
        for (int c = 0; c < EC / 16; ++c) {
          uint32_t p[16];
          tmem_ld_x16(taddr + uint32_t(c * 16), p);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c * 16 + j] = fmaf(__uint_as_float(p[j]), sc, acc[c * 16 + j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[d]);
      }
      if (ok && split == 1) {
        if constexpr (sizeof(OutT) == 2) {
#pragma unroll
          for (int c = 0; c < EC / 32; ++c)
            store_rows32_bf16(C, ldc, M, mt * TM + col0 + c * 32, nt * BN + quarter * 32, acc + c * 32, tr, lane);
        } else {
          store_col<EC>(C, ldc, M, mt * TM + col0, nt * BN + row, acc);
        }
      }
    }
  }

  __syncwarp();   // single-lane roles rejoin their warp before the aligned barriers below
  if constexpr (TM != 256) {
  if (split > 1) {
    // Every rank publishes its partial tile [TM tokens][BN rows] in its own
    // shared memory; then rank r sums the token rows
    // [r * TM / split, (r + 1) * TM / split) over all ranks, in rank order,
    // and stores them.  Consecutive threads take consecutive weight rows, so
    // the remote reads and the stores are coalesced and every rank shares
    // the reduction.
    const bool epi = warp >= kCtlWarps + Q::kDecWarps;
    float* red = reinterpret_cast<float*>(smem);   // [TM][BN] floats, reuses the stages
    if (epi) {
#pragma unroll
      for (int j = 0; j < EC; ++j) red[(col0 + j) * BN + row] = acc[j];
    }
    cluster_sync();
    // With bf16 output every thread of the CTA takes part (the decode and
    // control warps are idle by now; with the epilogue warps alone the sum
    // took 6-15 % longer on split shapes), each item being four weight rows
    // of one token: 16-byte remote loads, 8-byte stores.  Float output keeps
    // it on the epilogue warps, one value per thread (with all threads taking
    // part, that instantiation no longer fits in its registers).
    constexpr bool kAll = sizeof(OutT) == 2;
    if constexpr (kAll) {
      if (!*abort_flag) {
        const int et = int(threadIdx.x);
        int rnt, rmt;
        tile_coords(cluster_id, n_tiles, m_tiles, rnt, rmt);   // one tile per cluster when K is split
        const int m0 = rmt * TM;
        const int n0 = rnt * BN;
        const int t_begin = (TM * rank) / split;
        const int items = ((TM * (rank + 1)) / split - t_begin) * (BN / 4);
        const uint32_t red_addr = smem_u32(red);
        for (int idx = et; idx < items; idx += Q::kThreads) {
          const int t = t_begin + idx / (BN / 4);
          const int r4 = 4 * (idx % (BN / 4));
          if (m0 + t >= M) break;   // idx grows with t
          const uint32_t off = red_addr + uint32_t(t * BN + r4) * 4u;
          float4 v[kMaxSplitK];
#pragma unroll
          for (int r = 0; r < kMaxSplitK; ++r)
            if (r < split) v[r] = ld_shared_cluster_f4(map_shared_rank(off, uint32_t(r)));
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r = 0; r < kMaxSplitK; ++r) {
            if (r < split) {   // rank order
              sum.x += v[r].x;
              sum.y += v[r].y;
              sum.z += v[r].z;
              sum.w += v[r].w;
            }
          }
          const __nv_bfloat162 lo = __floats2bfloat162_rn(sum.x, sum.y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(sum.z, sum.w);
          uint2 packed;
          packed.x = *reinterpret_cast<const uint32_t*>(&lo);
          packed.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(C + size_t(m0 + t) * ldc + n0 + r4) = packed;
        }
      }
    } else if (epi && !*abort_flag) {
      const int et = (warp - kCtlWarps - Q::kDecWarps) * 32 + lane;   // 0 .. 32 * kEpiWarps - 1
      constexpr int kTStep = 32 * Q::kEpiWarps / BN;          // token rows handled per pass
      static_assert(32 * Q::kEpiWarps % BN == 0, "whole token rows per pass");
      const int r_row = et % BN;
      const int t_end = (TM * (rank + 1)) / split;
      const int m0 = last_mt * TM;
      const int n0 = last_nt * BN;
      uint32_t base[kMaxSplitK];
#pragma unroll
      for (int r = 0; r < kMaxSplitK; ++r)
        if (r < split) base[r] = map_shared_rank(smem_u32(red), uint32_t(r)) + uint32_t(r_row) * 4u;
      for (int t = (TM * rank) / split + et / BN; t < t_end && m0 + t < M; t += kTStep) {
        const uint32_t off = uint32_t(t * BN) * 4u;
        float v[kMaxSplitK];
#pragma unroll
        for (int r = 0; r < kMaxSplitK; ++r)
          if (r < split) v[r] = ld_dsmem_f32(base[r] + off);
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxSplitK; ++r)
          if (r < split) sum += v[r];
        C[size_t(m0 + t) * ldc + n0 + r_row] = to_out(sum, C);
      }
    }
    cluster_sync();
  }
  }   // TM != 256 (no K split)

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Q::kTmemCols);
  }
}

template <int TM, class OutT>
cudaError_t launch_tm(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  using Q = Cfg<TM, sizeof(OutT) == 4>;
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(w8a16_kernel<TM, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(Q::kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int n_tiles = p.N / BN;
  const int m_tiles = (p.M + TM - 1) / TM;
  const int tiles = n_tiles * m_tiles;
  const int kblocks = p.K / BK;
  const int slots = dev.num_sms * Q::kMinBlocks;
  // K is split over at most 4 CTAs: with 16 tiles of K = 7168 at M = 64 or
  // 128, 8-way splits took 20-21 us against 16 us for 4-way (the 8-rank
  // reduction of 64 KB partial tiles costs more than the K blocks it saves).
  constexpr int kSplitCap = 4;
  int split = 1;
  if (TM != 256 && tiles * 2 <= slots) {
    for (int s = kSplitCap; s >= 2; s >>= 1) {
      if (tiles * s <= slots && kblocks >= 2 * s) {
        split = s;
        break;
      }
    }
  }
  const int clusters = split > 1 ? tiles : (tiles < slots ? tiles : slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(clusters * split), 1, 1);
  cfg.blockDim = dim3(Q::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Q::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w8a16_kernel<TM, OutT>, p.tmW, p.tmX, p.scales, p.fmt, static_cast<OutT*>(p.C),
                            p.ldc, p.M, p.N, p.K, split, p.err);
}

}  // namespace

int w8a16_pick_tile_m(int64_t M, int64_t N, int fmt, int num_sms) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  // UE8M0: 256-token tiles when they take fewer rounds of the SMs, counting
  // a 256-token tile as 1.41 rounds of 128-token tiles (measured: 16.4 against
  // 11.6 us per tile at K = 2048; 1.45 at K = 7168).  Few tiles stay at 128,
  // which can also split K over a cluster.
  if (fmt == 1) {
    const int64_t n_tiles = N / BN;
    const int64_t r128 = (n_tiles * ((M + 127) / 128) + num_sms - 1) / num_sms;
    const int64_t r256 = (n_tiles * ((M + 255) / 256) + num_sms - 1) / num_sms;
    if (100 * r128 > 141 * r256) return 256;
  }
  return 128;
}

cudaError_t launch_gemm_w8a16(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  if (p.tile_m == 256 && p.fmt != 1) return cudaErrorInvalidValue;   // one accumulator: UE8M0 only
  if (p.out_f32) {
    switch (p.tile_m) {
      case 64: return launch_tm<64, float>(p, dev, stream);
      case 128: return launch_tm<128, float>(p, dev, stream);
      case 256: return launch_tm<256, float>(p, dev, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.tile_m) {
    case 64: return launch_tm<64, __nv_bfloat16>(p, dev, stream);
    case 128: return launch_tm<128, __nv_bfloat16>(p, dev, stream);
    case 256: return launch_tm<256, __nv_bfloat16>(p, dev, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp8blk
