// W8A16 for decode-size token counts (M <= 32) on sm_103a.
//
// Same arithmetic as the general W8A16 kernel: the e4m3 weights are decoded
// exactly to bf16 in registers, the product runs as bf16 tcgen05 MMA with the
// decoded 128-row weight tile as the TMEM-resident A operand and the token
// tile (TM = 16 or 32 rows, zero-filled past M) as B, and every 128-wide K
// block gets its own FP32 partial, which the epilogue promotes with the
// block's scale ("perf(ArcKernels) ...", "What this adds"; "FP8 / NVFP4
// weight-only inference on the RTX 3090 loses nothing", section 4.3: at
// small M the time is set by how fast the weights stream from DRAM).
//
// At these sizes one MMA is a few cycles of tensor work, so what limits the
// weight stream is the cost of issuing MMAs and of the barriers around them.
// This kernel is laid out for that:
//   * two MMA-issuing warps take alternate K blocks (one thread issues an
//     MMA about every 50 cycles; two issue nearly twice as many);
//   * weight tiles and token tiles travel in separate rings: a weight stage
//     is handed back as soon as the decode warps hold its codes in
//     registers, so nearly the whole weight ring is in flight from DRAM
//     (at full load DRAM answers in about 3 us, and the bytes in flight per
//     SM set the bandwidth);
//   * one MMA-completion barrier per K block (mdone ring) replaces separate
//     "token tile free", "decoded block free" and "partial ready" commits:
//     each role waits on the completion of the K block whose buffer it
//     reuses;
//   * weight scales (fp32 per 128x128 block or the UE8M0 exponents of the
//     32x32 blocks) are loaded as one 32-block window per warp and handed
//     out by shuffles, so no per-K-block global load sits on the path;
//   * K is split over a cluster of 2..8 CTAs chosen from the number of
//     clusters that can be co-resident, tiles run persistently, and the
//     ranks' FP32 partial tiles are summed per tile through distributed
//     shared memory, each rank reducing and storing a 128/split-row slice;
//   * the kernel is ready for programmatic dependent launch: weights and
//     scales are read before griddepcontrol.wait, activations and the output
//     only after it.
//
// Warp roles (16 warps):
//   warp 0        TMA producer of the e4m3 weight tiles [128 n x 128 k] (16 KB);
//                 its first loads go out before the CTA-wide setup barrier.
//   warp 1        TMA producer of the bf16 token tiles [TM x 128 k].
//   warps 2, 3    MMA issuers (lane 0); warp 2 also owns the TMEM allocation.
//   decode warps  8, in two groups of four (one warp per TMEM lane quarter);
//                 group g decodes whole rows of every other K block into a
//                 TMEM A buffer, the blocks MMA issuer g multiplies.
//   4 warps       promotion + epilogue: thread = weight row, TM accumulators.
#include <cuda_bf16.h>

#include "decode.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8blk {
namespace {

constexpr int BN = kW8A16TileN;   // weight rows per tile (MMA M)
constexpr int BK = 128;           // K per block
constexpr int kStageW = BN * BK;  // 16 KB of e4m3
constexpr int kACols = BK / 2;    // TMEM columns of one decoded A block
constexpr int kIssuers = 2;
constexpr int kEpiWarps = 4;
constexpr int kWarpXProducer = 1;
constexpr int kWarpIssuer0 = 2;
constexpr int kWarpDec0 = kWarpIssuer0 + kIssuers;
constexpr int kABufs = 4;         // decoded A blocks in TMEM
constexpr int kDBufs = 8;         // FP32 partials in TMEM
constexpr int kRing = 16;         // MMA-completion barriers, indexed by K-block count
constexpr int kBarrierBytes = 1024;
constexpr int kEarlyW = 4;        // weight stages requested before the setup barrier

template <int TM>
struct DecCfg {
  // Decode warps form kIssuers groups of four (one per TMEM lane quarter);
  // group g decodes whole rows of the K blocks it with it % kIssuers == g,
  // the blocks issuer g multiplies.
  static constexpr int kDecWarps = 4 * kIssuers;
  static constexpr int kWarpEpi0 = kWarpDec0 + kDecWarps;
  static constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;
  static constexpr int kStageX = TM * BK * 2;
  // Token tiles are refilled only after the MMA that read them has
  // completed, and while the weights stream at full rate an L2 refill takes
  // a few thousand cycles, so the token ring is deep (16 or 8 tiles = 64 KB).
  // Eight weight stages (128 KB per SM, ~19 MB over the GPU) already keep
  // HBM saturated.
  static constexpr int kXStages = TM == 16 ? 16 : 8;
  static constexpr int kWStages = 8;
  static constexpr int kRedFloats = BN * TM;                   // one partial tile, token-major [TM][BN]
  static constexpr size_t kXOff = size_t(kWStages) * kStageW;
  static constexpr size_t kRedOff = kXOff + size_t(kXStages) * kStageX;
  static constexpr size_t kBarOff = kRedOff + 2 * kRedFloats * sizeof(float);
  static constexpr size_t kSmemBytes = kBarOff + kBarrierBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdesc = make_idesc(1 /* bf16 */, BN, TM);
  static_assert(TM == 16 || TM == 32, "decode token tiles");
  static_assert(kStageX % 1024 == 0, "token tile must keep 1024-B swizzle alignment");
  static_assert(kABufs * kACols + kDBufs * TM <= int(kTmemCols), "TMEM budget");
  // A waiter on mdone slot (x % kRing) must know that use x - kRing has
  // completed and that use x + kRing cannot have: the token-tile producer
  // reuses a slot kXStages blocks later, the decoders an A buffer kABufs
  // later, and the MMA runs at most kDBufs blocks ahead of the epilogue.
  static_assert(kRing >= kXStages && kRing >= kABufs && kRing >= kDBufs, "completion ring too short");
  static_assert(kABufs % kIssuers == 0 && kDBufs % kIssuers == 0 && kXStages % kIssuers == 0,
                "each issuer owns fixed buffers");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert((2 * kWStages + kXStages + kABufs + kRing + kDBufs + 5) * 8 + 8 <= kBarrierBytes, "barrier area");
  static_assert(kXOff % 1024 == 0 && kRedOff % 1024 == 0, "swizzled tiles need 1024-B alignment");
  static_assert(kWarpDec0 % 4 == 0 && kDecWarps % 4 == 0, "warp w may only reach TMEM lanes 32*(w%4)..+31");
  // Each decode group consumes every use of the stages it owns (those with
  // s % kIssuers == g), so its parity waits are never two phases behind.
  static_assert(kWStages % kIssuers == 0, "weight stages split evenly between the decode groups");
};

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A16Decode | site);
}

// Whole-warp bounded wait: every lane polls, the result is agreed by vote.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait_sleep(bar, parity, abort_flag));
}

__device__ __forceinline__ __nv_bfloat16 to_out(float v, __nv_bfloat16*) { return __float2bfloat16_rn(v); }
__device__ __forceinline__ float to_out(float v, float*) { return v; }

// Four consecutive outputs of one row (the address is 8-byte aligned for bf16, 16-byte for float).
__device__ __forceinline__ void store4(__nv_bfloat16* dst, const float4& v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&lo);
  packed.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = packed;
}
__device__ __forceinline__ void store4(float* dst, const float4& v) { *reinterpret_cast<float4*>(dst) = v; }

// OutT: __nv_bfloat16 (rounded to nearest even) or float (the accumulator as is).
template <int TM, class OutT>
__global__ void __launch_bounds__(DecCfg<TM>::kThreads, 1)
    w8a16_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const void* __restrict__ scales, int fmt, OutT* __restrict__ C, int64_t ldc,
                        int M, int N, int K, int split, int* __restrict__ err) {
  using Q = DecCfg<TM>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float* red = reinterpret_cast<float*>(smem + Q::kRedOff);
  uint8_t* xring = smem + Q::kXOff;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + Q::kBarOff);
  uint64_t* wempty = wfull + Q::kWStages;
  uint64_t* xfull = wempty + Q::kWStages;
  uint64_t* afull = xfull + Q::kXStages;
  uint64_t* mdone = afull + kABufs;
  uint64_t* dempty = mdone + kRing;
  uint64_t* red_full = dempty + kDBufs;
  uint64_t* red_empty = red_full + 2;
  uint64_t* drain = red_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  // The next kernel of the stream may begin its own prologue now; it cannot
  // take this CTA's SM before this CTA exits.
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = N / BN;
  const int kblocks = K / BK;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster_id = blockIdx.x / split;
  const int num_clusters = gridDim.x / split;
  const int kb_begin = (kblocks * rank) / split;
  const int kb_end = (kblocks * (rank + 1)) / split;
  const int nkb = kb_end - kb_begin;
  const int my_tiles = cluster_id < n_tiles ? (n_tiles - cluster_id + num_clusters - 1) / num_clusters : 0;
  const int n_items = my_tiles * nkb;
  const bool ue8m0 = fmt != 0;

  // Weight loads of the first ring stages: issued by the weight producer
  // (thread 0) right after it has set up the barriers, so that the first
  // DRAM round trip overlaps the TMEM allocation and the setup barrier.
  // One thread issues a box about every 300 cycles, so only a few go out
  // before the barrier; the producer loop issues the rest.
  const uint64_t pol_w = policy_evict_first();
  const int pre = n_items < kEarlyW ? n_items : kEarlyW;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Q::kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 4);   // the four warps of one decode group
    }
    for (int j = 0; j < Q::kXStages; ++j) mbar_init(&xfull[j], 1);
    for (int i = 0; i < kABufs; ++i) mbar_init(&afull[i], 4);
    for (int i = 0; i < kRing; ++i) mbar_init(&mdone[i], 1);
    for (int i = 0; i < kDBufs; ++i) mbar_init(&dempty[i], kEpiWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], uint32_t(split * kEpiWarps));
      mbar_init(&red_empty[i], uint32_t(split * kEpiWarps));
    }
    mbar_init(drain, kIssuers);
    *abort_flag = 0;
    fence_mbar_init();
    fence_async_shared();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    int nt = cluster_id, kb = kb_begin;
    for (int it = 0; it < pre; ++it) {
      mbar_arrive_expect_tx(&wfull[it], kStageW);
      tma_load_2d_hint(smem + size_t(it) * kStageW, &tmW, &wfull[it], kb * BK, nt * BN, pol_w);
      if (++kb == kb_end) {
        kb = kb_begin;
        nt += num_clusters;
      }
    }
  }
  if (warp == kWarpIssuer0) {
    tmem_alloc(tmem_holder, Q::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (split > 1) {
    // Peers' barriers are initialised before any remote arrive reaches them.
    cluster_arrive_relaxed();
    cluster_wait();
  }
  const uint32_t tmem = *tmem_holder;
  const uint32_t tmem_a = tmem;                               // kABufs x 64 columns of decoded weights
  const uint32_t tmem_d = tmem + uint32_t(kABufs * kACols);   // kDBufs x TM columns of FP32 partials
  const int quarter = warp & 3;                               // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;                        // weight row within the tile

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    // Weights never depend on the previous kernel: no griddepcontrol.wait.
    if (lane == 0) {
      // Ring position and (tile, K block) of item `it`, advanced without
      // divisions.  Stage s is reused from item kWStages on, after its
      // previous contents were released (wempty phase (it / kWStages - 1)).
      int it = pre, s = pre, nt = cluster_id + (pre / nkb) * num_clusters, kb = kb_begin + pre % nkb;
      uint32_t ph = 1;   // parity of the release to wait for, once the ring wraps
      for (; it < n_items; ++it) {
        if (it >= Q::kWStages && !mbar_wait_sleep(&wempty[s], ph, abort_flag)) {
          raise_error(err, abort_flag, kSiteProducerEmpty);
          break;
        }
        mbar_arrive_expect_tx(&wfull[s], kStageW);
        tma_load_2d_hint(smem + size_t(s) * kStageW, &tmW, &wfull[s], kb * BK, nt * BN, pol_w);
        if (++s == Q::kWStages) {
          s = 0;
          ph ^= 1u;
        }
        if (++kb == kb_end) {
          kb = kb_begin;
          nt += num_clusters;
        }
      }
      if (it < n_items) {
        // Gave up: let the copies already issued land before the CTA exits.
        const int first = it > Q::kWStages ? it - Q::kWStages : 0;
        for (int j = first; j < it; ++j) mbar_wait(&wfull[j % Q::kWStages], uint32_t(j / Q::kWStages) & 1u, nullptr);
      }
    }
  } else if (warp == kWarpXProducer) {
    // ------------------------------------------------------------ token-tile producer
    if (lane == 0) {
      griddep_wait();   // activations may come from the previous kernel
      int it = 0;
      for (; it < n_items; ++it) {
        const int j = it % Q::kXStages;
        const int prev = it - Q::kXStages;   // K block whose MMA last read this slot
        if (prev >= 0 && !mbar_wait_sleep(&mdone[prev % kRing], uint32_t(prev / kRing) & 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteProducerEmpty);
          break;
        }
        const int kb = kb_begin + it % nkb;
        uint8_t* sx = xring + size_t(j) * Q::kStageX;
        mbar_arrive_expect_tx(&xfull[j], Q::kStageX);
        tma_load_2d(sx, &tmX, &xfull[j], kb * BK, 0);
        tma_load_2d(sx + TM * 128, &tmX, &xfull[j], kb * BK + 64, 0);
      }
      if (it < n_items) {
        const int first = it > Q::kXStages ? it - Q::kXStages : 0;
        for (int j = first; j < it; ++j) mbar_wait(&xfull[j % Q::kXStages], uint32_t(j / Q::kXStages) & 1u, nullptr);
      }
    }
  } else if (warp < kWarpDec0) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const int w = warp - kWarpIssuer0;
      for (int it = w; it < n_items; it += kIssuers) {
        const int d = it % kDBufs;
        const int a = it % kABufs;
        const int j = it % Q::kXStages;
        if (it >= kDBufs && !mbar_wait_sleep(&dempty[d], (uint32_t(it / kDBufs) & 1u) ^ 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteMmaAccEmpty);
          break;
        }
        if (!mbar_wait_sleep(&afull[a], uint32_t(it / kABufs) & 1u, abort_flag) ||
            !mbar_wait_sleep(&xfull[j], uint32_t(it / Q::kXStages) & 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteMmaAFull);
          break;
        }
        tc_fence_after();
        const uint64_t xdesc = desc_sw128_kmajor(smem_u32(xring + size_t(j) * Q::kStageX));
        const uint32_t d_tmem = tmem_d + uint32_t(d * TM);
        const uint32_t a_tmem = tmem_a + uint32_t(a * kACols);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // start-address field (16-byte units) of k-step k: 64-wide box k/4, 32 bytes per step
          const uint64_t xd = xdesc + uint64_t(((k >> 2) * TM * 128 + (k & 3) * 32) >> 4);
          mma_bf16_ts(d_tmem, a_tmem + uint32_t(k * 8), xd, Q::kIdesc, k > 0 ? 1u : 0u);
        }
        mma_commit(&mdone[it % kRing]);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < Q::kWarpEpi0) {
    // ------------------------------------------------------------ decode
    // Group g decodes the K blocks it = g, g + kIssuers, ...: whole 128-code
    // rows, one block per loop, so the two groups of a lane quarter run out
    // of step with each other and each block pays one set of waits.
    const int g = (warp - kWarpDec0) / 4;
    const uint32_t* ue32 = static_cast<const uint32_t*>(scales);
    uint32_t ewin = 0;   // lane l: exponent bytes of K block (win + l) of this tile, for this warp's 32 rows
    int win = -32;
    int s = g, j = g, nt = cluster_id;
    while (j >= nkb) {
      j -= nkb;
      nt += num_clusters;
    }
    uint32_t ph = 0;
    for (int it = g; it < n_items; it += kIssuers) {
      const int a = it % kABufs;
      uint32_t mul[4];   // multipliers of the four 32-wide K groups of the block
      if (ue8m0) {
        if (j < win || j >= win + 32) {
          win = j;
          const int kb = kb_begin + j + lane;
          ewin = kb < kb_end ? __ldg(ue32 + size_t(nt * 4 + quarter) * kblocks + kb) : 0u;
        }
        const uint32_t e4 = __shfl_sync(0xffffffffu, ewin, j - win);
#pragma unroll
        for (int q = 0; q < 4; ++q) mul[q] = decode_multiplier_bf16x2(int((e4 >> (8 * q)) & 0xFFu) - 127);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) mul[q] = decode_multiplier_bf16x2(0);
      }
      if (!warp_wait(&wfull[s], ph, abort_flag)) {
        raise_error(err, abort_flag, kSiteDecodeFull);
        break;
      }
      // Chunk c of the 128-byte swizzled row sits at position c ^ (row & 7).
      const uint8_t* wrow = smem + size_t(s) * kStageW + row * 128;
      uint4 raw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4*>(wrow + ((c ^ (row & 7)) << 4));
      fence_async_shared();   // generic-proxy reads of the stage come before its TMA (async-proxy) refill
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[s]);   // the codes are in registers: the stage can refill
      s += kIssuers;
      if (s >= Q::kWStages) {
        s -= Q::kWStages;
        ph ^= 1u;
      }
      j += kIssuers;
      while (j >= nkb) {
        j -= nkb;
        nt += num_clusters;
        win = -32;
      }
      if (it >= kABufs) {
        const int prev = it - kABufs;   // K block whose MMA last read this A buffer
        if (!warp_wait(&mdone[prev % kRing], uint32_t(prev / kRing) & 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteDecodeAEmpty);
          break;
        }
      }
      tc_fence_after();
      const uint32_t taddr = tmem_a + (uint32_t(quarter * 32) << 16) + uint32_t(a * kACols);
#pragma unroll
      for (int h = 0; h < 4; ++h) {   // 32 codes -> 16 TMEM columns
        uint32_t words[16];
        const uint32_t m = mul[h];
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
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    griddep_wait();   // the output may still be read or written by the previous kernel
    const float* bs32 = static_cast<const float*>(scales);
    const int et = (warp - Q::kWarpEpi0) * 32 + lane;   // 0..127, work index in the cluster reduction
    // Sums rows [rank * rows, (rank + 1) * rows) of tile q's partials over the
    // cluster's ranks once all of them have published it, stores them, and
    // hands the buffers back; false if a wait gave up.
    auto reduce_tile = [&](int q) -> bool {
      const int b = q & 1;
      const float* rb = red + b * Q::kRedFloats;
      if (!__all_sync(0xffffffffu, mbar_wait_acq_cluster(&red_full[b], uint32_t(q >> 1) & 1u, abort_flag))) {
        raise_error(err, abort_flag, kSiteReduceFull);
        return false;
      }
      // Items of four consecutive weight rows of one token: 16-byte remote
      // loads and one 8-byte (bf16) or 16-byte (float) store each.
      const int rows = BN / split;
      const int quads = rows / 4;
      const int n_base = (cluster_id + q * num_clusters) * BN + rank * rows;
      for (int idx = et; idx < M * quads; idx += 32 * kEpiWarps) {
        const int m = idx / quads;
        const int r4 = 4 * (idx % quads);
        const uint32_t local = smem_u32(rb + m * BN + rank * rows + r4);
        float4 v[kMaxSplitK];
#pragma unroll
        for (int r = 0; r < kMaxSplitK; ++r)
          if (r < split) v[r] = ld_shared_cluster_f4(map_shared_rank(local, uint32_t(r)));
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
        store4(C + size_t(m) * ldc + n_base + r4, sum);
      }
      __syncwarp();
      if (lane == 0) {
        for (int r = 0; r < split; ++r) mbar_arrive_cluster_relaxed(map_shared_rank(smem_u32(&red_empty[b]), r));
      }
      return true;
    };
    bool ok = true;
    for (int q = 0; q < my_tiles && ok; ++q) {
      const int nt = cluster_id + q * num_clusters;
      float acc[TM];
#pragma unroll
      for (int j = 0; j < TM; ++j) acc[j] = 0.f;
      float swin = 0.f;   // lane l: scale of K block (window base + l)
      for (int j = 0; j < nkb; ++j) {
        const int it = q * nkb + j;
        float sc = 1.f;
        if (!ue8m0) {
          if ((j & 31) == 0) {
            const int kb = kb_begin + j + lane;
            swin = kb < kb_end ? __ldg(bs32 + size_t(nt) * kblocks + kb) : 0.f;
          }
          sc = __shfl_sync(0xffffffffu, swin, j & 31);
        }
        if (!warp_wait(&mdone[it % kRing], uint32_t(it / kRing) & 1u, abort_flag)) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_d + (uint32_t(quarter * 32) << 16) + uint32_t((it % kDBufs) * TM);
        uint32_t p[TM];
        if constexpr (TM == 16) {
          tmem_ld_x16(taddr, p);
        } else {
          tmem_ld_x32(taddr, p);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[it % kDBufs]);
#pragma unroll
        for (int c = 0; c < TM; ++c) acc[c] = fmaf(__uint_as_float(p[c]), sc, acc[c]);
      }
      if (!ok) break;
      if (split == 1) {
        const int n = nt * BN + row;
#pragma unroll
        for (int m = 0; m < TM; ++m)
          if (m < M) C[size_t(m) * ldc + n] = to_out(acc[m], C);
        continue;
      }
      // ---- cluster reduction: every rank publishes its partial of tile q in
      // its own shared memory now, and sums one 128/split-row slice of tile
      // q - 1 over all ranks (in rank order) afterwards, so a peer that runs
      // behind does not hold up this rank's accumulation of the next tile.
      const int b = q & 1;
      float* rb = red + b * Q::kRedFloats;   // [TM][BN]
      if (q >= 2 && !warp_wait(&red_empty[b], (uint32_t(q >> 1) & 1u) ^ 1u, abort_flag)) {
        raise_error(err, abort_flag, kSiteReduceEmpty);
        break;
      }
#pragma unroll
      for (int m = 0; m < TM; ++m)
        if (m < M) rb[m * BN + row] = acc[m];
      __syncwarp();
      if (lane == 0) {
        fence_acq_rel_cluster();   // this warp's partial is visible before the arrivals below
        for (int r = 0; r < split; ++r) mbar_arrive_cluster_relaxed(map_shared_rank(smem_u32(&red_full[b]), r));
      }
      if (q >= 1 && !reduce_tile(q - 1)) {
        ok = false;
        break;
      }
    }
    if (ok && split > 1 && my_tiles > 0) reduce_tile(my_tiles - 1);
  }

  __syncwarp();   // single-lane roles rejoin their warp before the aligned barriers below
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIssuer0) {
    tc_fence_after();
    tmem_dealloc(tmem, Q::kTmemCols);
  }
  if (split > 1) cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

// Largest number of clusters of `split` CTAs that can be resident at once
// (both output types use the same resources).
template <int TM>
int max_active_clusters(int split, const DeviceInfo& dev) {
  using Q = DecCfg<TM>;
  static int cache[64][kMaxSplitK + 1] = {};
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device >= 64) return dev.num_sms / split;
  int& slot = cache[device][split];
  if (slot == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(split * (dev.num_sms / split)), 1, 1);
    cfg.blockDim = dim3(Q::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Q::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w8a16_decode_kernel<TM, __nv_bfloat16>, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = dev.num_sms / split;
    }
    slot = n;
  }
  return slot;
}

template <int TM, class OutT>
cudaError_t launch_decode_tm(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  using Q = DecCfg<TM>;
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(w8a16_decode_kernel<TM, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(Q::kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const W8A16DecodePlan plan = w8a16_decode_plan(p.N, p.K, dev.num_sms, [&](int s) {
    return s == 1 ? dev.num_sms : max_active_clusters<TM>(s, dev);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(plan.clusters * plan.split), 1, 1);
  cfg.blockDim = dim3(Q::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Q::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w8a16_decode_kernel<TM, OutT>, p.tmW, p.tmX, p.scales, p.fmt,
                            static_cast<OutT*>(p.C), p.ldc, p.M, p.N, p.K, plan.split, p.err);
}

}  // namespace

cudaError_t launch_w8a16_decode(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  if (p.M > p.tile_m) return cudaErrorInvalidValue;
  switch (p.tile_m) {
    case 16: return p.out_f32 ? launch_decode_tm<16, float>(p, dev, stream)
                              : launch_decode_tm<16, __nv_bfloat16>(p, dev, stream);
    case 32: return p.out_f32 ? launch_decode_tm<32, float>(p, dev, stream)
                              : launch_decode_tm<32, __nv_bfloat16>(p, dev, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp8blk
