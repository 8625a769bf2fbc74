// W8A8 block-scaled FP8 GEMM for sm_103a.
//
//   C[m, n] = bf16( sum_kb P[m, n, kb] * As[kb, m] * Bs[n/128, kb] ),
//   P[m, n, kb] = sum_{k in kb} A[m, k] * B[n, k]       (e4m3 x e4m3, fp32)
//
// Structure ("Blockwise FP8 on Ada GPUs, part 2", "The fix"): the tensor
// cores form one FP32 partial per 128-wide K block with no scaling inside the
// block, and the partial is promoted once into the FP32 accumulator with
// As * Bs.  On sm_103a the partial lives in tensor memory (TMEM), so the
// per-slice fragments that spilled registers on Ada never exist here:
//
//   warp 0      TMA producer: A tile [128 x 128 B], B tile [128 x 128 B] and
//               the tile rows' activation scales As[kb, m0..m0+127] per 128-K
//               block into a 6-stage shared-memory ring.
//   warp 1      allocates all 512 TMEM columns.
//   warps 1, 2  MMA issuers (one in the fused form): one thread each issues
//               the four tcgen05.mma kind::f8f6f4 (K = 32 each) of alternate
//               K blocks into one of four 128-column partial buffers, so the
//               tensor cores run up to three K blocks ahead of the promotion.
//   next 8      promotion + epilogue: each thread owns one row and 64
//               columns of the 128x128 tile; per K block it reads its partial
//               with tcgen05.ld, releases the buffer, and does
//               acc = fma(partial, As[kb, m] * Bs[n/128, kb], acc).
//               Activation scales come from shared memory (loaded by TMA with
//               the operands), weight scales from a per-lane register window
//               handed out by shuffle, so no global load sits on this path.
//               At the end of the tile it rounds to bf16 and stores C.
//
// The weight scale is looked up per 128-wide N slice of the tile, never once
// per CTA ("Blockwise FP8 on Ada GPUs, part 2", "The fix": the latent bug was
// a single weight scale per thread block).  With 128-wide N tiles each tile
// is exactly one slice.
//
// Large problems run persistently, one CTA per SM, over tiles in a grouped
// raster order so that concurrently running tiles share A and B panels in L2
// ("Blockwise FP8 on Ada GPUs, part 2", "One tile doesn't fit all M": the
// launch-order swizzle).  Problems with too few tiles to fill the GPU split K
// over a thread-block cluster of 2..4 CTAs; the partial accumulators are
// summed through distributed shared memory in rank order (no global
// workspace), and rank 0 writes C.
//
// Grouped (mixture-of-experts) form: with row_group != nullptr the rows of A
// and C are split into groups (experts) stored contiguously in 128-row tiles,
// row_group[m] naming the group of row m (the same for the 128 rows of a
// tile; negative for a padding tile, which is skipped and left untouched).
// Tile (mt, nt) then multiplies with rows g*N + nt*128 of the stacked
// weights [G*N, K] and scales Bs[g][nt][kb]; every role reads the tile's
// group from row_group and skips the same tiles.  Grouped problems whose
// groups average at least 256 rows run on the CTA-pair kernel instead
// (gemm_w8a8_pair.cu).
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fp8blk {
namespace {

constexpr int BM = kW8A8TileM;   // 128 rows of A / C per tile
constexpr int BN = kW8A8TileN;   // 128 rows of B (columns of C) per tile
constexpr int BK = 128;          // one scale block of K, 128 bytes of e4m3
constexpr int kStages = 6;
constexpr int kStageA = BM * BK;
constexpr int kStageB = BN * BK;
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kStageAs = BM * 4;          // fp32 activation scales of the tile's rows for one K block
constexpr int kEpiWarps = 8;
constexpr int kColsPerThread = BN / 2;   // two epilogue warps share a TMEM lane quarter
constexpr int kAccBufs = 4;              // FP32 partials in flight in TMEM
constexpr uint32_t kTmemCols = kAccBufs * BN;
constexpr uint32_t kIdesc = make_idesc(0 /* e4m3 */, BM, BN);
constexpr int kGroupM = 8;
constexpr int kBarrierBytes = 512;

static_assert(BK == 128, "one MMA K block must be exactly one scale block");
static_assert(kTmemCols <= 512, "TMEM budget");
static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 N for M = 128");
static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "128B-swizzle atoms need 1024-B alignment");
static_assert(2 * kStageBytes >= BM * BN * 4, "split-K reduction buffer reuses two stages");
// Configuration of the kernel.  FUSED quantises the activations itself: the
// producer loads bf16 token rows (at most kFusedMaxM, one 32-row tile) and
// the quantiser warps turn each 128-wide K block into e4m3 codes and a scale
// per row, with the arithmetic of the stand-alone quantiser (quant.cuh), into
// the stage's A tile and scale slot (two quantiser warps).
// Otherwise A and As arrive by TMA.
constexpr int kFusedMaxM = kW8A8FusedMaxM;
template <bool FUSED>
struct W8A8Cfg {
  static constexpr int kStages = FUSED ? 5 : fp8blk::kStages;
  static constexpr int kQuantWarps = FUSED ? 2 : 0;   // 12 warps: 168 registers per thread
  // MMA-issuing threads: two on alternate K blocks (the tensor pipe takes an
  // MMA only as the previous one finishes, so one thread alone leaves it idle
  // while it waits on its barriers and commits); the fused form keeps one,
  // since its odd stage count would give one stage to both issuers.
  static constexpr int kIssuers = FUSED ? 1 : 2;
  static constexpr int kCtlWarps = 1 + kIssuers;     // producer, issuers; the epilogue warps follow
  static constexpr int kThreads = 32 * kCtlWarps + (kEpiWarps + kQuantWarps) * 32;
  static constexpr int kStageX = FUSED ? kFusedMaxM * BK * 2 : 0;   // bf16 [32][128] as two 64-column boxes
  static constexpr size_t kAsOff = size_t(kStages) * kStageBytes;
  static constexpr size_t kXOff = (kAsOff + size_t(kStages) * kStageAs + 1023) / 1024 * 1024;
  static constexpr size_t kBarOff = kXOff + size_t(kStages) * kStageX;
  static constexpr size_t kSmemBytes = kBarOff + kBarrierBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert((3 * kStages + 2 * kAccBufs + 1) * 8 + 8 <= kBarrierBytes, "barrier area");
  static_assert(kFusedMaxM % (4 * (FUSED ? kQuantWarps : 1)) == 0, "whole passes of four rows per quantiser warp");
  static_assert(kIssuers == 1 || (kStages % 2 == 0 && kAccBufs % 2 == 0),
                "each stage and partial buffer belongs to one issuer");
};
static_assert(W8A8Cfg<false>::kBarOff == size_t(kStages) * (kStageBytes + kStageAs), "unfused layout unchanged");

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int& mt, int& nt) {
  const int per_group = kGroupM * n_tiles;
  const int g = t / per_group;
  const int first = g * kGroupM;
  const int gsz = min(m_tiles - first, kGroupM);
  const int r = t - g * per_group;
  mt = first + r % gsz;
  nt = r / gsz;
}

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A8 | site);
}

__device__ __forceinline__ void store_row64(float* dst, const float* acc) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < kColsPerThread / 4; ++i) d[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
}

__device__ __forceinline__ void store_row64(__nv_bfloat16* dst, const float* acc) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < kColsPerThread / 8; ++i) {
    uint4 v;
    v.x = pack_bf16x2(acc[8 * i + 0], acc[8 * i + 1]);
    v.y = pack_bf16x2(acc[8 * i + 2], acc[8 * i + 3]);
    v.z = pack_bf16x2(acc[8 * i + 4], acc[8 * i + 5]);
    v.w = pack_bf16x2(acc[8 * i + 6], acc[8 * i + 7]);
    d[i] = v;
  }
}

// OutT: __nv_bfloat16 (rounded to nearest even) or float (the accumulator as is).
template <class OutT, bool FUSED>
__global__ void __launch_bounds__(W8A8Cfg<FUSED>::kThreads, 1)
    w8a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmX,
                const float* __restrict__ Bs,
                OutT* __restrict__ C, int64_t ldc, int M, int N, int K, int split,
                const int* __restrict__ row_group, int G, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  using Q = W8A8Cfg<FUSED>;
  constexpr int kStages = Q::kStages;
  float* as_stage = reinterpret_cast<float*>(smem + Q::kAsOff);   // [kStages][BM]
  uint8_t* x_stage = smem + Q::kXOff;                            // [kStages][kStageX] (FUSED)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Q::kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* dfull = empty + kStages;
  uint64_t* dempty = dfull + kAccBufs;
  uint64_t* drain = dempty + kAccBufs;
  // FUSED: the weight tile and the bf16 token rows of a stage complete on
  // xfull[s]; full[s] then completes when the quantiser warps have written
  // the codes and scales.
  uint64_t* xfull = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(xfull + kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  griddep_launch_dependents();   // the next kernel may start its prologue; it gets an SM when this CTA leaves

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kblocks = K / BK;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster_id = blockIdx.x / split;
  const int num_clusters = gridDim.x / split;
  const int kb_begin = (kblocks * rank) / split;
  const int kb_end = (kblocks * (rank + 1)) / split;
  // Group of row tile mt (0 when ungrouped); outside [0, G) the tile is skipped.
  auto group_of = [&](int mt) -> int { return row_group != nullptr ? __ldg(row_group + size_t(mt) * BM) : 0; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], FUSED ? Q::kQuantWarps : 1);
      mbar_init(&xfull[s], 1);
      mbar_init(&empty[s], 1 + kEpiWarps);   // MMA done with A/B, epilogue done with the scales
    }
    for (int d = 0; d < kAccBufs; ++d) {
      mbar_init(&dfull[d], 1);
      mbar_init(&dempty[d], kEpiWarps);
    }
    mbar_init(drain, Q::kIssuers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    if constexpr (FUSED) {
      tma_prefetch_desc(&tmX);
    } else {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmAs);
    }
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Accumulator of the epilogue threads; kept live across the split-K
  // reduction after the tile loop.
  float acc[kColsPerThread];
  const int quarter = warp & 3;
  const int half = (warp - Q::kCtlWarps) >> 2;
  const int row_in_tile = quarter * 32 + lane;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !FUSED && row_group != nullptr) {
      // Grouped: the tile's group (an activation-side input) decides which
      // weight rows to load, so nothing is requested before the previous
      // kernel has finished.
      griddep_wait();
      const uint64_t pol_b = policy_evict_last();
      int it = 0;
      bool ok = true;
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
        int mt, nt;
        tile_coords(t, m_tiles, n_tiles, mt, nt);
        const int g = group_of(mt);
        if (g < 0 || g >= G) continue;
        for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (uint32_t(it) / kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(s) * kStageBytes;
          mbar_arrive_expect_tx(&full[s], kStageBytes + kStageAs);
          tma_load_2d(sa, &tmA, &full[s], kb * BK, mt * BM);
          tma_load_2d_hint(sa + kStageA, &tmB, &full[s], kb * BK, g * N + nt * BN, pol_b);
          tma_load_2d(as_stage + s * BM, &tmAs, &full[s], mt * BM, kb);
        }
      }
      if (!ok) {
        const int first = it > kStages ? it - kStages : 0;
        for (int j = first; j < it; ++j) mbar_wait(&full[j % kStages], (uint32_t(j) / kStages) & 1u, nullptr);
      }
    } else if (lane == 0) {
      // Items are this CTA's (tile, K block) pairs in order.
      const int nkb = kb_end - kb_begin;
      const int my_tiles = cluster_id < num_tiles ? (num_tiles - cluster_id + num_clusters - 1) / num_clusters : 0;
      const int n_items = my_tiles * nkb;
      // Weights are re-read by every row tile when there are several; with a
      // single row tile they stream through once.
      const uint64_t pol_b = m_tiles > 1 ? policy_evict_last() : policy_evict_first();
      // Under programmatic dependent launch the weight tiles of the first
      // stages are requested before the previous kernel has finished; the
      // activations and their scales only after it.
      // The barrier the stage's copies complete on, and their bytes.
      uint64_t* const cbar = FUSED ? xfull : full;
      constexpr uint32_t kTx = FUSED ? uint32_t(kStageB + Q::kStageX) : uint32_t(kStageBytes + kStageAs);
      // Activation-side copies of item it into stage s: A + As, or the bf16
      // token rows (two 64-column boxes) that the quantiser warps consume.
      auto load_act = [&](int s, int mt, int kb) {
        if constexpr (FUSED) {
          tma_load_2d(x_stage + size_t(s) * Q::kStageX, &tmX, &xfull[s], kb * BK, 0);
          tma_load_2d(x_stage + size_t(s) * Q::kStageX + Q::kStageX / 2, &tmX, &xfull[s], kb * BK + 64, 0);
        } else {
          tma_load_2d(smem + size_t(s) * kStageBytes, &tmA, &full[s], kb * BK, mt * BM);
          tma_load_2d(as_stage + s * BM, &tmAs, &full[s], mt * BM, kb);
        }
      };
      const int pre = n_items < kStages ? n_items : kStages;
      for (int it = 0; it < pre; ++it) {
        int mt, nt;
        tile_coords(cluster_id + (it / nkb) * num_clusters, m_tiles, n_tiles, mt, nt);
        const int kb = kb_begin + it % nkb;
        mbar_arrive_expect_tx(&cbar[it], kTx);
        tma_load_2d_hint(smem + size_t(it) * kStageBytes + kStageA, &tmB, &cbar[it], kb * BK, nt * BN, pol_b);
      }
      griddep_wait();
      for (int it = 0; it < pre; ++it) {
        int mt, nt;
        tile_coords(cluster_id + (it / nkb) * num_clusters, m_tiles, n_tiles, mt, nt);
        load_act(it, mt, kb_begin + it % nkb);
      }
      int it = pre;
      for (; it < n_items; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (uint32_t(it) / kStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteProducerEmpty);
          break;
        }
        int mt, nt;
        tile_coords(cluster_id + (it / nkb) * num_clusters, m_tiles, n_tiles, mt, nt);
        const int kb = kb_begin + it % nkb;
        mbar_arrive_expect_tx(&cbar[s], kTx);
        load_act(s, mt, kb);
        tma_load_2d_hint(smem + size_t(s) * kStageBytes + kStageA, &tmB, &cbar[s], kb * BK, nt * BN, pol_b);
      }
      if (it < n_items) {
        // Let every copy this thread issued land before the CTA can exit.
        const int first = it > kStages ? it - kStages : 0;
        for (int j = first; j < it; ++j) mbar_wait(&cbar[j % kStages], (uint32_t(j) / kStages) & 1u, nullptr);
      }
    }
  } else if (warp >= 1 && warp <= Q::kIssuers) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer w takes the K blocks with it % kIssuers == w, whose stages and
    // partial buffers are those of its parity.
    if (lane == 0) {
      const uint32_t w = uint32_t(warp - 1);
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
        if (row_group != nullptr) {
          int mt, nt;
          tile_coords(t, m_tiles, n_tiles, mt, nt);
          const int g = group_of(mt);
          if (g < 0 || g >= G) continue;
        }
        for (int kb = kb_begin; kb < kb_end; ++kb, ++it, ++acc_it) {
          if (it % uint32_t(Q::kIssuers) != w) continue;
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const int d = acc_it % kAccBufs;
          const uint32_t dph = (acc_it / kAccBufs) & 1u;
          if (!mbar_wait(&dempty[d], dph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAccEmpty);
            ok = false;
            break;
          }
          if (!mbar_wait(&full[s], ph, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + size_t(s) * kStageBytes);
          const uint32_t b0 = a0 + kStageA;
          const uint32_t d_tmem = tmem + uint32_t(d * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            mma_f8_ss(d_tmem, desc_sw128_kmajor(a0 + 32u * k), desc_sw128_kmajor(b0 + 32u * k), kIdesc,
                      k > 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          mma_commit(&dfull[d]);
        }
      }
      // No MMA may still be running when TMEM is released.
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < Q::kCtlWarps + kEpiWarps) {
    // ------------------------------------------------------------ promotion + epilogue
    griddep_wait();        // the output may still be read or written by the previous kernel
    uint32_t it = 0;       // stage counter, in step with the producer and the MMA issuer
    bool ok = true;
    for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
      int mt, nt;
      tile_coords(t, m_tiles, n_tiles, mt, nt);
      const int g = group_of(mt);
      if (g < 0 || g >= G) {
        // Padding tile, or a group index past the weights: skipped by every
        // role; the latter is also reported in the error word.
        if (g >= G && threadIdx.x == 32 * Q::kCtlWarps) atomicCAS(err, 0, kDevErrW8A8 | kSiteBadGroup);
        continue;
      }
      const int m = mt * BM + row_in_tile;
      const bool row_ok = m < M;
#pragma unroll
      for (int j = 0; j < kColsPerThread; ++j) acc[j] = 0.f;
      // Weight scales of this tile: lane j holds Bs[nt, kb0 + j] for a window
      // of 32 K blocks, handed out by shuffle (one load per 32 blocks).
      const float* bs_row = Bs + (size_t(g) * n_tiles + nt) * kblocks;
      float bs_win = 0.f;
      for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
        const int rel = kb - kb_begin;
        if ((rel & 31) == 0) bs_win = (kb + lane < kb_end) ? __ldg(bs_row + kb + lane) : 0.f;
        const float sb = __shfl_sync(0xffffffffu, bs_win, rel & 31);
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        const int d = it % kAccBufs;
        const uint32_t dph = (it / kAccBufs) & 1u;
        // Activation scales of this K block arrived with the A/B tiles.
        const bool got_s = __all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_flag));
        if (!got_s) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          break;
        }
        const float sa = as_stage[s * BM + row_in_tile];
        fence_async_shared();   // generic-proxy read of the stage before its TMA (async-proxy) refill
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        // The decision must be warp-uniform: tcgen05.ld below is .sync.aligned.
        const bool got = __all_sync(0xffffffffu, mbar_wait(&dfull[d], dph, abort_flag));
        if (!got) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(d * BN + half * kColsPerThread);
        const float sc = sa * sb;
        if constexpr (FUSED) {
          // 128 registers per thread in this configuration: one 32-column
          // load at a time.
#pragma unroll
          for (int h = 0; h < kColsPerThread / 32; ++h) {
            uint32_t p[32];
            tmem_ld_x32(taddr + uint32_t(32 * h), p);
            tmem_ld_wait();
            if (h + 1 == kColsPerThread / 32) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&dempty[d]);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[32 * h + j] = fmaf(__uint_as_float(p[j]), sc, acc[32 * h + j]);
          }
        } else {
          uint32_t p[kColsPerThread];
          tmem_ld_x32(taddr, p);
          tmem_ld_x32(taddr + 32, p + 32);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dempty[d]);
#pragma unroll
          for (int j = 0; j < kColsPerThread; ++j) acc[j] = fmaf(__uint_as_float(p[j]), sc, acc[j]);
        }
      }
      if (ok && split == 1 && row_ok) {
        store_row64(C + size_t(m) * ldc + size_t(nt) * BN + half * kColsPerThread, acc);
      }
    }
  } else if constexpr (FUSED) {
    // ------------------------------------------------------------ activation quantisers
    // Eight lanes share a token row (16 columns each, the row's amax from
    // three xor shuffles inside the group), a warp covers four rows per
    // pass, and the warps interleave: pass j of warp q takes rows
    // 8j + 4q .. 8j + 4q + 3, so both warps work from the fifth row on.  Codes go to the 128-byte-swizzled A tile the MMA
    // reads, one 16-byte chunk per lane and row.
    const int qw = warp - Q::kCtlWarps - kEpiWarps;
    const int sub = lane & 7;              // 16-column slice of the row
    const int rg = lane >> 3;              // row within the pass
    constexpr int kPasses = kFusedMaxM / (4 * Q::kQuantWarps);
    constexpr int kNarrowM = 4;            // up to this many rows: one warp per row
    static_assert(kPasses % 2 == 0, "passes run in pairs");
    uint32_t it = 0;
    bool ok = true;
    for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
      for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&xfull[s], ph, abort_flag))) {
          raise_error(err, abort_flag, kSiteDecodeFull);
          ok = false;
          break;
        }
        // Columns 16 sub .. 16 sub + 15 are chunks 2 (sub & 3), +1 of box sub / 4.
        const uint8_t* xs = x_stage + size_t(s) * Q::kStageX + (sub >> 2) * (Q::kStageX / 2);
        uint8_t* a_tile = smem + size_t(s) * kStageBytes;
        if (M <= kNarrowM) {
          // Few rows: a whole warp per row (four columns per lane, amax from
          // five xor shuffles), warp q taking rows q, q + 2, ..., two at a
          // time as independent chains.
#pragma unroll
          for (int i0 = 0; i0 < kNarrowM / Q::kQuantWarps; i0 += 2) {
            if (qw + Q::kQuantWarps * i0 >= M) break;   // warp-uniform
            float f[2][4];
            int r[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              r[u] = qw + Q::kQuantWarps * (i0 + u);
              const uint2 v = *reinterpret_cast<const uint2*>(
                  x_stage + size_t(s) * Q::kStageX + (lane >> 4) * (Q::kStageX / 2) + r[u] * 128 +
                  ((((lane & 15) >> 1) ^ (r[u] & 7)) << 4) + (lane & 1) * 8);
              f[u][0] = __uint_as_float(v.x << 16);
              f[u][1] = __uint_as_float(v.x & 0xFFFF0000u);
              f[u][2] = __uint_as_float(v.y << 16);
              f[u][3] = __uint_as_float(v.y & 0xFFFF0000u);
            }
            float amax[2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
              amax[u] = fmaxf(fmaxf(fabsf(f[u][0]), fabsf(f[u][1])), fmaxf(fabsf(f[u][2]), fabsf(f[u][3])));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
              amax[0] = fmaxf(amax[0], __shfl_xor_sync(0xffffffffu, amax[0], o));
              amax[1] = fmaxf(amax[1], __shfl_xor_sync(0xffffffffu, amax[1], o));
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float sc = group_scale(amax[u]);
              const Divisor dv = make_divisor(sc);
              const uint32_t codes =
                  e4m3x4(quotient(f[u][0], dv), quotient(f[u][1], dv), quotient(f[u][2], dv), quotient(f[u][3], dv));
              if (r[u] < M) {
                *reinterpret_cast<uint32_t*>(a_tile + r[u] * 128 + (((lane >> 2) ^ (r[u] & 7)) << 4) + (lane & 3) * 4) =
                    codes;
                if (lane == 0) as_stage[s * BM + r[u]] = sc;
              }
            }
          }
        } else {
        // Passes run two at a time as independent chains (loads, amax,
        // scale, quotients), so one pass's latency hides the other's.
#pragma unroll
        for (int j0 = 0; j0 < kPasses; j0 += 2) {
          if (4 * Q::kQuantWarps * j0 + 4 * qw >= M) break;   // warp-uniform
          float f[2][16];
          int r[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            r[u] = 4 * Q::kQuantWarps * (j0 + u) + 4 * qw + rg;
            const int rr = r[u] < kFusedMaxM ? r[u] : kFusedMaxM - 1;
            const int c0 = 2 * (sub & 3);
            const uint4 v0 = *reinterpret_cast<const uint4*>(xs + rr * 128 + (((c0 + 0) ^ (rr & 7)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(xs + rr * 128 + (((c0 + 1) ^ (rr & 7)) << 4));
            bf16x8_to_f32(v0, f[u]);
            bf16x8_to_f32(v1, f[u] + 8);
          }
          float amax[2] = {0.f, 0.f};
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 16; ++i) amax[u] = fmaxf(amax[u], fabsf(f[u][i]));
#pragma unroll
          for (int o = 4; o >= 1; o >>= 1) {
            amax[0] = fmaxf(amax[0], __shfl_xor_sync(0xffffffffu, amax[0], o));
            amax[1] = fmaxf(amax[1], __shfl_xor_sync(0xffffffffu, amax[1], o));
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float sc = group_scale(amax[u]);
            const Divisor dv = make_divisor(sc);
            uint4 codes;
            codes.x = e4m3x4(quotient(f[u][0], dv), quotient(f[u][1], dv), quotient(f[u][2], dv), quotient(f[u][3], dv));
            codes.y = e4m3x4(quotient(f[u][4], dv), quotient(f[u][5], dv), quotient(f[u][6], dv), quotient(f[u][7], dv));
            codes.z =
                e4m3x4(quotient(f[u][8], dv), quotient(f[u][9], dv), quotient(f[u][10], dv), quotient(f[u][11], dv));
            codes.w =
                e4m3x4(quotient(f[u][12], dv), quotient(f[u][13], dv), quotient(f[u][14], dv), quotient(f[u][15], dv));
            if (r[u] < M) {
              *reinterpret_cast<uint4*>(a_tile + r[u] * 128 + ((sub ^ (r[u] & 7)) << 4)) = codes;
              if (sub == 0) as_stage[s * BM + r[u]] = sc;
            }
          }
        }
        }
        fence_async_shared();   // the codes are read by the tensor cores (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
  }

  __syncwarp();   // single-lane roles rejoin their warp before the aligned barriers below
  if (split > 1) {
    // One tile per cluster: every rank writes the valid rows (m < M) of its
    // accumulator tile to its shared memory; after a cluster barrier each
    // rank sums its share of those rows (split evenly) over all ranks' tiles
    // through distributed shared memory, in rank order (so the result is the
    // rank-0-first sum), and stores them.
    // All of a CTA's threads take part, consecutive threads on consecutive
    // rows of one 4-column group (contiguous 16-byte reads).  Every thread of
    // every CTA reaches both cluster barriers, also after an abort.
    const bool epi = warp >= Q::kCtlWarps && warp < Q::kCtlWarps + kEpiWarps;
    float4* red = reinterpret_cast<float4*>(smem);   // [BN/4][BM] float4, reuses stages 0-1
    // Split K runs one tile per cluster: every thread can name it.
    int tile_mt, tile_nt;
    tile_coords(cluster_id, m_tiles, n_tiles, tile_mt, tile_nt);
    const int valid = min(BM, M - tile_mt * BM);   // rows of the tile below M
    if (epi && row_in_tile < valid) {
#pragma unroll
      for (int j4 = 0; j4 < kColsPerThread / 4; ++j4)
        red[(half * (kColsPerThread / 4) + j4) * BM + row_in_tile] =
            make_float4(acc[4 * j4], acc[4 * j4 + 1], acc[4 * j4 + 2], acc[4 * j4 + 3]);
    }
    cluster_sync();
    if (!*abort_flag) {
      const int per = (valid + split - 1) / split;
      const int r0 = min(valid, rank * per);
      const int rows = min(valid, r0 + per) - r0;    // rows this rank sums
      const int items = rows * (BN / 4);             // float4 items of those rows
      uint32_t peer[kMaxSplitK];
#pragma unroll
      for (int p = 0; p < kMaxSplitK; ++p) peer[p] = map_shared_rank(smem_u32(red), uint32_t(p < split ? p : 0));
      for (int idx = int(threadIdx.x); idx < items; idx += int(blockDim.x)) {
        const int r = r0 + idx % rows;               // row within the tile
        const int c4 = idx / rows;                   // 4-column group
        const int m = tile_mt * BM + r;
        const uint32_t off = uint32_t((c4 * BM + r) * 16);
        float4 v[kMaxSplitK];
#pragma unroll
        for (int p = 0; p < kMaxSplitK; ++p)
          if (p < split) v[p] = ld_shared_cluster_f4(peer[p] + off);
        float4 sum = v[0];
#pragma unroll
        for (int p = 1; p < kMaxSplitK; ++p) {
          if (p < split) {
            sum.x += v[p].x;
            sum.y += v[p].y;
            sum.z += v[p].z;
            sum.w += v[p].w;
          }
        }
        {
          OutT* dst = C + size_t(m) * ldc + size_t(tile_nt) * BN + size_t(4 * c4);
          if constexpr (std::is_same<OutT, float>::value) {
            *reinterpret_cast<float4*>(dst) = sum;
          } else {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
          }
        }
      }
    }
    cluster_sync();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <class OutT, bool FUSED>
cudaError_t launch_single(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  using Q = W8A8Cfg<FUSED>;
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(w8a8_kernel<OutT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(Q::kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int m_tiles = (p.M + BM - 1) / BM;
  const int n_tiles = p.N / BN;
  const int tiles = m_tiles * n_tiles;
  const int kblocks = p.K / BK;
  // K is split over at most 4 CTAs: with 16 tiles of K = 7168 at M = 16 or
  // 128, 8-way splits took 17.6 and 19.8 us against 12.4 and 13.9 us for
  // 4-way, also with the reduce-scatter (eight-CTA clusters of full-SM CTAs
  // are the cost, not the sum).
  constexpr int kSplitCap = 4;
  int split = 1;
  if (tiles * 2 <= dev.num_sms && p.row_group == nullptr) {
    for (int s = kSplitCap; s >= 2; s >>= 1) {
      if (tiles * s <= dev.num_sms && kblocks >= 2 * s) {
        split = s;
        break;
      }
    }
  }
  const int clusters = split > 1 ? tiles : (tiles < dev.num_sms ? tiles : dev.num_sms);

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
  return cudaLaunchKernelEx(&cfg, w8a8_kernel<OutT, FUSED>, p.tmA, p.tmB, p.tmAs, p.tmX, p.Bs,
                            static_cast<OutT*>(p.C), p.ldc, p.M, p.N, p.K, split, p.row_group, p.groups, p.err);
}

}  // namespace

cudaError_t launch_gemm_w8a8(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  // Enough 256x256 tiles to keep most CTA pairs busy: the pair kernel.
  // Grouped problems go there too when the groups average at least 256 rows:
  // it runs a pair tile once per group among its two 128-row halves, so
  // 128-row groups would double its work (measured: G = 8 x 512 rows, N = K =
  // 4096: 72 against 113 us single-CTA; G = 32 x 256 rows: 128 against 187 us;
  // G = 64 x 128 rows: 225 against 217 us).
  if (p.fused) {
    if (p.M > kFusedMaxM || p.row_group != nullptr) return cudaErrorInvalidValue;
    return p.out_f32 ? launch_single<float, true>(p, dev, stream) : launch_single<__nv_bfloat16, true>(p, dev, stream);
  }
  const bool pair_groups = p.row_group == nullptr || int64_t(p.M) >= 256 * int64_t(p.groups);
  const int pair_tiles = w8a8_pair_tiles(p.M, p.N);
  const bool pair_whole = 2 * pair_tiles >= dev.num_sms / 2;
  // Few pair tiles, but more 128 x 128 tiles than the single-CTA kernel can
  // split over K (M = 256, N = 7168: 112 tiles): the pair kernel runs every
  // tile as two 256 x 128 halves, whose MMAs do twice the single-CTA work per
  // SM and cycle (measured: M = 256, N = 7168, K = 18432: 80.7 us single-CTA).
  const int single_tiles = (p.M + kW8A8TileM - 1) / kW8A8TileM * (p.N / kW8A8TileN);
  const bool pair_halves = p.row_group == nullptr && 4 * pair_tiles <= dev.num_sms && 2 * single_tiles > dev.num_sms;
  if (pair_groups && p.M > kW8A8TileM && (pair_whole || pair_halves)) return launch_gemm_w8a8_pair(p, dev, stream);
  return p.out_f32 ? launch_single<float, false>(p, dev, stream) : launch_single<__nv_bfloat16, false>(p, dev, stream);
}

}  // namespace fp8blk
