// W8A8 block-scaled FP8 GEMM on CTA pairs (tcgen05 .cta_group::2), sm_103a.
//
// Same arithmetic as the single-CTA kernel in gemm_w8a8.cu: one FP32 partial
// per 128-wide K block from e4m3 operands only, promoted once with
// As[kb, m] * Bs[n/128, kb] ("Blockwise FP8 on Ada GPUs, part 2", "The fix").
// Here two CTAs of a cluster form one 256 x 256 output tile: each CTA loads
// its 128 rows of A and its 128 rows of B (N) per K block, and one thread of
// the even CTA issues M = 256, N = 256, K = 32 MMAs that read both CTAs'
// shared memory and write each CTA's 128 rows of the partial into its own
// TMEM.  Per SM this halves the operand bytes fetched from L2 and read from
// shared memory per FLOP compared with a 128 x 128 single-CTA tile, which is
// what bounds the single-CTA kernel on large problems.
//
// Roles per CTA (three warpgroups; registers are rebalanced with setmaxnreg
// from 168 per thread at launch to 40 for warpgroup 0 and 232 for the two
// epilogue warpgroups: 40*128 + 232*256 = 168*384, which the build checks):
//   warps 0, 2   TMA producers: this CTA's A rows + activation scales (warp 0,
//                the scales eight K blocks per copy) and B rows (warp 2).
//   warp 1       TMEM allocation (with the peer, 512 columns = two 256-column
//                partials).
//   warps 1, 3   in the even CTA, one thread each issues the MMAs of every
//                other K block (the block's partial buffer is fixed by its
//                parity) and commits to both CTAs' barriers.  A single thread
//                needs longer to issue a K block's four pair MMAs than the
//                tensor cores need to run them, so two issue in turn.  Both
//                CTAs' operand copies complete on the even CTA's stage
//                barrier (.cta_group::2 TMA), so an issuer waits on one
//                barrier per stage.
//   warps 4..11  promotion + epilogue, 8 warps: TMEM lane quarter = warp % 4,
//                128 of the 256 columns each; acc = fma(partial, As*Bs, acc).
//                At the end of a tile each warp writes its 32 x 128 bf16
//                block to shared memory in the 128-byte swizzled layout and
//                one lane stores it with two TMA tensor stores (coalesced,
//                asynchronous; rows past M are clipped by the tensor map).
// Tiles of the pair run persistently in grouped raster order ("Blockwise FP8
// on Ada GPUs, part 2", "One tile doesn't fit all M": launch-order swizzle).
// A last round that would leave at most half of the pairs busy runs its
// tiles as 256 x 128 halves instead (MMA N = 128), so that it takes about
// half as long.
//
// Split K (ksplit = 2), for dense problems whose tiles fit on half of the
// pairs and whose K range is long: a cluster of 4 CTAs (two pairs) per tile,
// pair p accumulating K blocks [p, p + 1) * kblocks / 2.  At the end the
// promotion warps of the half of the columns a pair does not keep write
// their accumulators to shared memory, and after a cluster barrier the
// keeping warps (pair 0: columns 0..127 of the tile, pair 1: 128..255) add
// the other pair's values through distributed shared memory and store them.
//
// Grouped (mixture-of-experts) form, row_group != nullptr: the rows of A and
// C come in 128-row tiles of one group each (row_group[m] names row m's
// group, negative for padding), and the weights are stacked [G*N, K] with
// scales [G][N/128][K/128].  Both CTAs of a pair share one B tile, so a pair
// tile runs once per distinct group among its two 128-row halves: pass 0
// with the first half's group, pass 1 with the second half's when it
// differs; a CTA stores its rows only in the pass of its own group, and
// padding halves are never stored.  The pass-0 items of all tiles come
// before the pass-1 items, so that the pairs share the real work evenly.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fp8blk {
namespace {

constexpr int TM = 128;              // A rows per CTA (256 per pair)
constexpr int PN = 256;              // C columns per pair tile (MMA N)
constexpr int HN = PN / 2;           // B rows per CTA
constexpr int BK = 128;              // one scale block of K
// An even number of stages keeps every stage with one issuer (stage s holds
// the K blocks of parity s & 1), so each issuer waits on every phase of its
// stages in order and a parity wait can never mistake an old phase for a new one.
constexpr int kStages = 4;
constexpr int kStageA = TM * BK;
constexpr int kStageB = HN * BK;
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kAsGroup = 8;          // K blocks of activation scales per scale stage
constexpr int kStageAs = kAsGroup * TM * 4;   // [kAsGroup][TM] fp32
constexpr int kAsStages = 4;         // 32 K blocks of scales in flight: the ring never gates the operands
constexpr int kEpiWarps = 8;
constexpr int kIssuers = 2;                     // MMA-issuing threads (even CTA)
constexpr int kStageC = 32 * 64 * 2;            // one 32-row x 64-column bf16 box, 128-byte swizzled
constexpr int kBoxesPerWarp = 2;                // a warp's 32 x 128 output block
constexpr int kThreads = 128 + kEpiWarps * 32;   // 384: three warpgroups
constexpr int kCols = PN / (kEpiWarps / 4);      // 128 columns per epilogue thread
constexpr int kChunk = 32;                       // columns per tcgen05.ld
constexpr int kRegsLaunch = 168;                 // registers per thread at launch (checked at build time)
constexpr int kRegsWg0 = 40;
constexpr int kRegsEpi = 232;
static_assert(kRegsWg0 * 128 + kRegsEpi * 256 <= kRegsLaunch * kThreads, "register split");
constexpr int kAccBufs = 2;
constexpr uint32_t kTmemCols = kAccBufs * PN;
constexpr uint32_t kIdesc = make_idesc(0 /* e4m3 */, 2 * TM, PN);
constexpr uint32_t kIdescHalf = make_idesc(0 /* e4m3 */, 2 * TM, HN);   // a 256 x 128 half tile
constexpr int kGroupM = 8;
constexpr int kBarrierBytes = 1024;
// Split K over two pairs from K = 12288: M = 256, N = 7168 took 23.1 / 31.8 /
// 52.7 us split against 17.8 / 29.9 / 59.9 us as halves at K = 4096 / 8192 /
// 18432 (the exchange and the four-CTA clusters cost ~6 us up front).
constexpr int kSplitMinKBlocks = 96;
constexpr size_t kAsOff = size_t(kStages) * kStageBytes;
constexpr size_t kCOff = kAsOff + size_t(kAsStages) * kStageAs;   // kEpiWarps staging boxes
constexpr size_t kBarOff = kCOff + size_t(kEpiWarps) * kBoxesPerWarp * kStageC;
constexpr size_t kSmemBytes = kBarOff + kBarrierBytes + 1024;
static_assert(kCOff % 1024 == 0 && kStageC % 1024 == 0, "swizzled staging boxes need 1024-byte alignment");
static_assert(kAccBufs == kIssuers, "each issuer owns one partial buffer");
static_assert(kStages % kIssuers == 0, "each stage belongs to one issuer");

static_assert(kTmemCols == 512, "two 256-column partials fill TMEM");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "swizzle atoms");

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int& mt, int& nt) {
  const int per_group = kGroupM * n_tiles;
  const int g = t / per_group;
  const int first = g * kGroupM;
  const int gsz = min(m_tiles - first, kGroupM);
  const int r = t - g * per_group;
  mt = first + r % gsz;
  nt = r / gsz;
}

// Work items of the persistent loop (dense problems).  When the tiles leave a
// last round that would keep at most half of the pairs busy, each of those
// last tiles runs as two 256 x 128 halves on two pairs (MMA N = 128), which
// halves the length of that round; when all tiles fit on half of the pairs
// (the launch then gives two pairs per tile), every tile runs as two halves.
// Items [0, full_items) are whole tiles; item full_items + 2u + h is half h
// of tile full_items + u.  half = -1 marks a whole tile.  Grouped problems
// add, from item pass1 on, a second pass over every tile (whole), for the
// group of its second 128-row half when that differs from the first's; the
// first passes are scheduled like a dense problem (halves in a last round
// that would fill at most half of the pairs).
struct Items {
  int full_items, num_items, pass1;
};
__device__ __forceinline__ Items make_items(int num_tiles, int num_pairs, bool grouped) {
  Items it;
  if (2 * num_tiles <= num_pairs) {
    it.full_items = 0;
    it.num_items = 2 * num_tiles;
  } else {
    const int rem = num_tiles % num_pairs;
    const int split = (num_tiles > num_pairs && rem > 0 && 2 * rem <= num_pairs) ? rem : 0;
    it.full_items = num_tiles - split;
    it.num_items = num_tiles + split;
  }
  it.pass1 = it.num_items;
  if (grouped) it.num_items += num_tiles;
  return it;
}
__device__ __forceinline__ void item_coords(int t, const Items& items, int m_tiles, int n_tiles, int& mt, int& nt,
                                            int& half) {
  if (t >= items.pass1) {
    tile_coords(t - items.pass1, m_tiles, n_tiles, mt, nt);   // grouped second pass, whole tile
    half = -1;
  } else if (t < items.full_items) {
    tile_coords(t, m_tiles, n_tiles, mt, nt);
    half = -1;
  } else {
    const int u = t - items.full_items;
    tile_coords(items.full_items + (u >> 1), m_tiles, n_tiles, mt, nt);
    half = u & 1;
  }
}

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A8 | 0x80 | site);
}

// Group of the 128 rows starting at row r (-1 past M: padding).
__device__ __forceinline__ int half_group(const int* row_group, int r, int M) {
  return r < M ? __ldg(row_group + r) : -1;
}

// Grouped: the group that item t's pass multiplies with (the first pass,
// items before pass1, takes the group of the pair tile row's first half, the
// second pass that of its second half), or -1 when the pass has no rows to
// compute (padding, a second half of the same group, or a group past the
// weights).  Dense problems: 0.
__device__ __forceinline__ int item_group(const int* row_group, int G, int M, int t, int pass1, int mt) {
  if (row_group == nullptr) return 0;
  const int g0 = half_group(row_group, mt * 2 * TM, M);
  const int g1 = half_group(row_group, mt * 2 * TM + TM, M);
  const int g = t < pass1 ? g0 : (g1 != g0 ? g1 : -1);
  return g < G ? g : -1;
}

// try_wait with cluster-scope acquire, for phases completed by the peer CTA.
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// 16 bytes of output row r, chunk c of 128-byte box b of a warp's 128
// columns: eight bf16 (acc pairs 32b + 4c ..) or four float32 (16b + 2c ..).
template <bool F32>
__device__ __forceinline__ uint4 out_chunk(const float2* acc, int b, int c) {
  uint4 v;
  if constexpr (F32) {
    const float2 p = acc[b * 16 + 2 * c], q = acc[b * 16 + 2 * c + 1];
    v = make_uint4(__float_as_uint(p.x), __float_as_uint(p.y), __float_as_uint(q.x), __float_as_uint(q.y));
  } else {
    const float2* a = acc + b * 32 + 4 * c;
    v.x = pack_bf16x2(a[0].x, a[0].y);
    v.y = pack_bf16x2(a[1].x, a[1].y);
    v.z = pack_bf16x2(a[2].x, a[2].y);
    v.w = pack_bf16x2(a[3].x, a[3].y);
  }
  return v;
}

template <bool F32, int ksplit>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmAsG, const __grid_constant__ CUtensorMap tmC,
                     const float* __restrict__ Bs, const int* __restrict__ row_group, int G, int M, int N, int K,
                     int* __restrict__ err) {
  static_assert(ksplit == 1 || ksplit == 2, "one or two pairs per tile");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float* as_stage = reinterpret_cast<float*>(smem + kAsOff);   // [kAsStages][kAsGroup][TM]
  uint8_t* c_stage = smem + kCOff;                              // [kEpiWarps][kBoxesPerWarp][kStageC]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* as_full = empty + kStages;
  uint64_t* as_empty = as_full + kAsStages;
  uint64_t* dfull = as_empty + kAsStages;
  uint64_t* dempty = dfull + kAccBufs;
  uint64_t* drain = dempty + kAccBufs;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // The epilogue re-reads the item counts from here at each tile instead of
  // keeping them in registers across its K loop.
  volatile int* items_sh = abort_flag + 1;   // full_items, num_items, pass1

  griddep_launch_dependents();   // the next kernel may start its prologue; it gets an SM when this CTA leaves

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = static_cast<int>(cluster_ctarank());
  const int rank = crank & 1;                            // position in the CTA pair
  const int even = ksplit == 1 ? 0 : (crank & ~1);       // cluster rank of the pair's even CTA
  const int kslice = ksplit == 1 ? 0 : (crank >> 1);     // split K: the pair's half of the K blocks
  const uint16_t pair_mask = uint16_t(0x3u << even);
  // One slot per pair, or per two pairs with split K (one tile each);
  // ksplit is 1 or 2, so 2 * ksplit = 1 << ksplit (shifts, not divisions).
  const int pair = int(blockIdx.x) >> ksplit;
  const int num_pairs = int(gridDim.x) >> ksplit;
  const int m_tiles = (M + 2 * TM - 1) / (2 * TM);
  const int n_tiles = (N + PN - 1) / PN;
  const int num_tiles = m_tiles * n_tiles;
  const Items items = make_items(num_tiles, num_pairs, row_group != nullptr);
  const int kblocks = K / BK;
  const int kb0 = kslice * (kblocks >> 1);                  // 0 unless K is split
  const int kb1 = kslice + 1 == ksplit ? kblocks : (kblocks >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);                // A and B producers of the even CTA; both CTAs' bytes
      mbar_init(&empty[s], 1);               // MMA done with A/B
    }
    for (int j = 0; j < kAsStages; ++j) {
      mbar_init(&as_full[j], 1);
      mbar_init(&as_empty[j], kEpiWarps);    // this CTA's epilogue done with the scales
    }
    for (int d = 0; d < kAccBufs; ++d) {
      mbar_init(&dfull[d], 1);
      mbar_init(&dempty[d], 2 * kEpiWarps);   // both CTAs' epilogues (used in the even CTA)
    }
    mbar_init(drain, kIssuers);
    *abort_flag = 0;
    items_sh[0] = items.full_items;
    items_sh[1] = items.num_items;
    items_sh[2] = items.pass1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmAsG);
    tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any commit or arrive reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWg0));
    if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    // Two issuing threads (A + scales from warp 0, B from warp 2): one thread
    // alone cannot issue strided 128-byte-row tiles at the rate the MMAs use.
    const bool a_side = warp == 0;
    const uint32_t full0_base = map_shared_rank(smem_u32(full), uint32_t(even));
    if (lane == 0) {
      // Under programmatic dependent launch the weights stream in at once;
      // the activations and their scales wait for the previous kernel.
      if (a_side) griddep_wait();
      uint32_t it = 0, gi = 0;   // operand items and scale groups issued
      bool ok = true;
      for (int t = pair; t < items.num_items && ok; t += num_pairs) {
        int mt, nt, half;
        item_coords(t, items, m_tiles, n_tiles, mt, nt, half);
        const int g = item_group(row_group, G, M, t, items.pass1, mt);
        if (g < 0) continue;
        const int m0 = mt * 2 * TM + rank * TM;
        // A half tile's MMA reads the first 64 of this CTA's B rows: rows
        // 128 half + 64 rank of the tile (the box's other 64 rows go unused).
        // Grouped: group g's weights are rows g*N .. g*N + N - 1.
        const int n0 = g * N + (half < 0 ? nt * PN + rank * HN : nt * PN + half * HN + rank * (HN / 2));
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (a_side && (kb - kb0) % kAsGroup == 0) {
            // Scales of K blocks kb .. kb + kAsGroup - 1 in one box (rows
            // past K / 128 arrive zero-filled and are never read).
            const int j = gi % kAsStages;
            if (!mbar_wait(&as_empty[j], ((gi / kAsStages) & 1u) ^ 1u, abort_flag)) {
              raise_error(err, abort_flag, kSiteProducerEmpty);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&as_full[j], kStageAs);
            tma_load_2d(as_stage + j * (kAsGroup * TM), &tmAsG, &as_full[j], m0, kb);
            ++gi;
          }
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(s) * kStageBytes;
          // Operand tiles of both CTAs complete on the even CTA's full[s]:
          // its producers announce the pair's bytes, the odd CTA's loads
          // only deliver them.
          const uint32_t full0 = full0_base + uint32_t(s) * 8u;
          if (a_side) {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kStageA);
            tma_load_2d_pair(sa, &tmA, full0, kb * BK, m0);
          } else {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kStageB);
            tma_load_2d_pair(sa + kStageA, &tmB, full0, kb * BK, n0);
          }
        }
      }
      if (!ok) {
        // Let issued copies land before the CTA can exit (the odd CTA's
        // operand copies complete on the even CTA's barrier; they finish
        // within microseconds, long before any bounded wait gives up).
        const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0u;
        if (rank == 0)
          for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1u, nullptr);
        const uint32_t first_as = gi > uint32_t(kAsStages) ? gi - kAsStages : 0u;
        if (a_side)
          for (uint32_t j = first_as; j < gi; ++j) mbar_wait(&as_full[j % kAsStages], (j / kAsStages) & 1u, nullptr);
      }
    }
  } else {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuers (even CTA, warps 1 and 3)
      // Issuer w takes the K blocks with item parity w; they accumulate into
      // partial buffer w, so the two issuers' MMAs never touch the same
      // TMEM columns or operand stage.
      const uint32_t w = warp == 1 ? 0u : 1u;
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; t < items.num_items && ok; t += num_pairs) {
        if (row_group != nullptr) {
          int mt, nt, half;
          item_coords(t, items, m_tiles, n_tiles, mt, nt, half);
          if (item_group(row_group, G, M, t, items.pass1, mt) < 0) continue;
        }
        const uint32_t idesc = (t < items.full_items || t >= items.pass1) ? kIdesc : kIdescHalf;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if ((it & 1u) != w) continue;
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t dph = (it / kAccBufs) & 1u;
          if (!mbar_wait_cluster(&dempty[w], dph ^ 1u, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaAccEmpty);
            ok = false;
            break;
          }
          if (!mbar_wait_cluster(&full[s], ph, abort_flag)) {
            raise_error(err, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + size_t(s) * kStageBytes);
          const uint32_t b0 = a0 + kStageA;
          const uint32_t d_tmem = tmem + w * uint32_t(PN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            mma_f8_ss_pair(d_tmem, desc_sw128_kmajor(a0 + 32u * k), desc_sw128_kmajor(b0 + 32u * k), idesc,
                           k > 0 ? 1u : 0u);
          }
          mma_commit_pair_mc(&empty[s], pair_mask);
          mma_commit_pair_mc(&dfull[w], pair_mask);
        }
      }
      mma_commit_pair_mc(drain, uint16_t(1u << even));
      mbar_wait(drain, 0, nullptr);
    }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t dempty0 = map_shared_rank(smem_u32(dempty), uint32_t(even));
    uint8_t* stg = c_stage + size_t(e) * kBoxesPerWarp * kStageC;
    griddep_wait();   // the output may still be read or written by the previous kernel
    float2 acc[kCols / 2];
    uint32_t it = 0, gi = 0;   // K blocks and scale groups consumed
    bool ok = true;
    // One tile (NC = 128: half of a whole tile's 256 partial columns) or one
    // half tile (NC = 64 of its 128); instantiated for both so that the
    // whole-tile path keeps its column offsets as constants.
    // y: first row of this warp's 32-row block; n_item: first output column
    // of the tile or half tile.
    // The warp's 32 x NC block of acc leaves as 128-byte-wide boxes (64 bf16
    // or 32 float32 columns), at most kBoxesPerWarp at a time through the
    // staging boxes; chunk c (16 bytes) of row r sits at 16-byte position
    // c ^ (r & 7) of the row (128-byte swizzle).  n: first column.
    auto store_block = [&](auto nc_tag, int y, int n) {
      constexpr int NC = decltype(nc_tag)::value;
      constexpr int kBoxCols = F32 ? 32 : 64;
      constexpr int kBoxes = NC / kBoxCols;
      constexpr int kPer = kBoxes < kBoxesPerWarp ? kBoxes : kBoxesPerWarp;
#pragma unroll
      for (int r = 0; r < kBoxes / kPer; ++r) {
        if (lane == 0) bulk_wait_group_read0();   // earlier stores have left the staging boxes
        __syncwarp();
#pragma unroll
        for (int h = 0; h < kPer; ++h) {
          uint8_t* dst = stg + h * kStageC + lane * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(dst + ((c ^ (lane & 7)) << 4)) = out_chunk<F32>(acc, r * kPer + h, c);
        }
        fence_async_shared();   // generic-proxy writes become visible to the TMA engine
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < kPer; ++h) tma_store_2d(&tmC, stg + h * kStageC, n + (r * kPer + h) * kBoxCols, y);
          bulk_commit_group();
        }
      }
    };
    auto promote = [&](auto nc_tag, int y, int n_item, int g, bool store) {
      constexpr int NC = decltype(nc_tag)::value;
      const int col0 = (e >> 2) * NC;
      const int n = n_item + col0;
      const bool col_ok = n < N;
#pragma unroll
      for (int j = 0; j < NC / 2; ++j) acc[j] = make_float2(0.f, 0.f);
      // kr: K block within this pair's range [kb0, kb1) (the whole range
      // unless K is split); bs_row starts at the range's first K block.
      const float* bs_row = Bs + (size_t(g) * (N / 128) + size_t(col_ok ? n / 128 : 0)) * kblocks + kb0;
      const int nkb = kb1 - kb0;
      float bs_win = 0.f;
      for (int kr = 0; kr < nkb; ++kr, ++it) {
        if ((kr & 31) == 0) bs_win = (col_ok && kr + lane < nkb) ? __ldg(bs_row + kr + lane) : 0.f;
        const float sb = __shfl_sync(0xffffffffu, bs_win, kr & 31);
        const int j = gi % kAsStages;
        const int d = it % kAccBufs;
        const uint32_t dph = (it / kAccBufs) & 1u;
        if (kr % kAsGroup == 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&as_full[j], (gi / kAsStages) & 1u, abort_flag))) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          return;
        }
        const float sa = as_stage[(j * kAsGroup + kr % kAsGroup) * TM + row];
        if (kr % kAsGroup == kAsGroup - 1 || kr == nkb - 1) {
          fence_async_shared();   // generic-proxy reads of the scale stage before its TMA (async-proxy) refill
          __syncwarp();
          if (lane == 0) mbar_arrive(&as_empty[j]);
          ++gi;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&dfull[d], dph, abort_flag))) {
          raise_error(err, abort_flag, kSiteEpilogueFull);
          ok = false;
          return;
        }
        tc_fence_after();
        const float sc = sa * sb;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(d * PN + col0);
        // Two 32-column loads per wait; the buffer is handed back as soon as
        // the last columns are in registers.
#pragma unroll
        for (int c = 0; c < NC / kChunk; c += 2) {
          uint32_t p[2 * kChunk];
          tmem_ld_x32(taddr + uint32_t(c * kChunk), p);
          tmem_ld_x32(taddr + uint32_t((c + 1) * kChunk), p + kChunk);
          tmem_ld_wait();
          if (c + 2 == NC / kChunk) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(dempty0 + uint32_t(d) * 8u);
          }
#pragma unroll
          for (int j = 0; j < 2 * kChunk; j += 2) {
            const int i = (c * kChunk + j) / 2;
            acc[i].x = fmaf(__uint_as_float(p[j]), sc, acc[i].x);
            acc[i].y = fmaf(__uint_as_float(p[j + 1]), sc, acc[i].y);
          }
        }
      }
      if (y < M && col_ok && store) store_block(nc_tag, y, n);
    };
    for (int t = pair; ok; t += num_pairs) {
      const Items it_sh{items_sh[0], items_sh[1], items_sh[2]};
      if (t >= it_sh.num_items) break;
      int mt, nt, half;
      item_coords(t, it_sh, m_tiles, n_tiles, mt, nt, half);
      const int g = item_group(row_group, G, M, t, it_sh.pass1, mt);
      if (g < 0) {
        // A group index past the weights in this CTA's rows: skipped and
        // reported (by one thread).
        if (row_group != nullptr && threadIdx.x == 128) {
          const int own = half_group(row_group, mt * 2 * TM + rank * TM, M);
          if (own >= G) atomicCAS(err, 0, kDevErrW8A8 | kSiteBadGroup);
        }
        continue;
      }
      // Grouped: this CTA's rows are stored in the pass of their own group;
      // split K: after the exchange below.
      const bool store = ksplit == 1 && (row_group == nullptr || half_group(row_group, mt * 2 * TM + rank * TM, M) == g);
      const int y = mt * 2 * TM + rank * TM + quarter * 32;
      if (half < 0)
        promote(std::integral_constant<int, kCols>{}, y, nt * PN, g, store);
      else
        promote(std::integral_constant<int, kCols / 2>{}, y, nt * PN + half * HN, g, store);
    }
    if (ksplit > 1) {
      // Split K: exchange the column halves between the two pairs (the
      // control warps take part in the cluster barrier at the end of their
      // branch).  This CTA's stages are free: every MMA of its pair has
      // completed, and every copy into them has been consumed.  (The cluster
      // rank is read again here rather than kept live across the K loop.)
      const int xrank = int(cluster_ctarank());   // ksplit == 2 here
      const int xslice = xrank >> 1;
      const bool keep = (e >> 2) == xslice;
      constexpr int kXPitch = kCols + 4;   // floats per row, rows 16 bytes apart in bank terms
      float* xbuf = reinterpret_cast<float*>(smem);   // [TM][kXPitch]: the half this pair gives away
      if (!keep) {
        float4* dst = reinterpret_cast<float4*>(xbuf + size_t(row) * kXPitch);
#pragma unroll
        for (int i = 0; i < kCols / 4; ++i)
          dst[i] = make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y);
      }
      cluster_sync();
      if (keep && ok && !*abort_flag) {
        int mt, nt;
        tile_coords(pair, m_tiles, n_tiles, mt, nt);   // split K: one whole tile per cluster
        const uint32_t peer = map_shared_rank(smem_u32(xbuf + size_t(row) * kXPitch), uint32_t(xrank ^ 2));
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) {
          float4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = ld_shared_cluster_f4(peer + uint32_t((c * 16 + 4 * i) * 4));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2& a0 = acc[c * 8 + 2 * i];
            float2& a1 = acc[c * 8 + 2 * i + 1];
            a0.x += v[i].x;
            a0.y += v[i].y;
            a1.x += v[i].z;
            a1.y += v[i].w;
          }
        }
        const int y = mt * 2 * TM + (xrank & 1) * TM + quarter * 32;
        const int n = nt * PN + xslice * kCols;
        if (y < M && n < N) store_block(std::integral_constant<int, kCols>{}, y, n);
      }
    }
    if (lane == 0) bulk_wait_group0();   // the staging buffer stays valid until the stores are done
  }

  __syncwarp();
  if (ksplit > 1 && (threadIdx.x >> 5) < 4) cluster_sync();   // the exchange barrier of the promotion warps
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves while another may still reach its shared memory
  // Re-read the TMEM address here instead of keeping it live across the role
  // branches, where the register budget is the smaller warpgroup's.
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc_pair(*reinterpret_cast<volatile uint32_t*>(tmem_holder), kTmemCols);
  }
}

}  // namespace

int w8a8_pair_tiles(int M, int N) { return ((M + 2 * TM - 1) / (2 * TM)) * ((N + PN - 1) / PN); }

namespace {

template <bool F32, int ksplit>
cudaError_t launch_pair_k(const GemmW8A8Args& p, int pairs, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    // The setmaxnreg split assumes the launch register count; refuse to run
    // any build where it differs.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, w8a8_pair_kernel<F32, ksplit>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(w8a8_pair_kernel<F32, ksplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * ksplit * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(2 * ksplit);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w8a8_pair_kernel<F32, ksplit>, p.tmA, p.tmB, p.tmAsG, p.tmC, p.Bs, p.row_group,
                            p.groups, p.M, p.N, p.K, p.err);
}

template <bool F32>
cudaError_t launch_pair(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  const int tiles = w8a8_pair_tiles(p.M, p.N);
  const int max_pairs = dev.num_sms / 2;
  // Dense problems whose tiles fit on half of the pairs run each tile on two
  // pairs: split over K when the K range is long (kSplitMinKBlocks blocks or
  // more), otherwise as two 256 x 128 halves (see make_items).
  const bool two_per_tile = p.row_group == nullptr && 2 * tiles <= max_pairs;
  if (two_per_tile && p.K / BK >= kSplitMinKBlocks) return launch_pair_k<F32, 2>(p, tiles, stream);
  const int items = two_per_tile ? 2 * tiles : tiles;
  return launch_pair_k<F32, 1>(p, items < max_pairs ? items : max_pairs, stream);
}

}  // namespace

cudaError_t launch_gemm_w8a8_pair(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t stream) {
  return p.out_f32 ? launch_pair<true>(p, dev, stream) : launch_pair<false>(p, dev, stream);
}

}  // namespace fp8blk
