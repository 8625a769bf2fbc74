// W8A8 in the 32x32 UE8M0 format on hardware block scaling, sm_103a.
//
//   C[m, n] = sum_k A[m, k] 2^(ea[k/32, m] - 127) * B[n, k] 2^(eb[n/32, k/32] - 127)
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
// quant_act_ue8m0_kernel: bf16 x -> e4m3 codes + exponent bytes, one thread
// per 32-value group: e is the smallest integer with 448 * 2^e >= amax
// (from amax's exponent and whether its mantissa exceeds 1.75 = 448 / 2^8),
// clamped to [-127, 126] (bf16 inputs never pass 120), and q =
// e4m3(x * 2^-e), exact before the rounding, never saturating.
//
// w8a8_mx_kernel: one 128 x 256 output tile per CTA.
//   warp 0      TMA producer: A [128 rows x 128 B] and B [256 rows x 128 B]
//               per 128-K block into a 4-stage ring.
//   warp 1      TMEM allocation (512 columns); one thread issues the four
//               K = 32 MMAs of each block (scale-factor byte j of the
//               block's scale words for slice j) into the 256-column
//               accumulator.
//   warps 4..7  scale-factor writers, then the epilogue.  Warp q (lane
//               quarter q) writes, per K block, into a ring of TMEM scale
//               slots: its 32 rows' activation exponent words (four bytes:
//               the block's four slices) at lane m, column q of the A slot,
//               and the tile's eight 32-row weight exponent words at its
//               lanes, columns 0..7 of the B slot.  The MMA reads row m's A
//               scale at (lane m, column m / 32) and column n's B scale at
//               (lane 32 (m / 32) + n % 32, column n / 32): every lane
//               quarter holds the B scales of all 256 columns (layout
//               measured with one-hot operands and distinct exponents per
//               lane, column and byte).  At the end each warp reads its 32
//               accumulator rows, rounds to bf16 (or keeps float32) and
//               stores them with TMA tensor stores from a swizzled staging
//               box.
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

__global__ void __launch_bounds__(256) quant_act_ue8m0_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                                              int64_t K, int64_t ldx, uint8_t* __restrict__ a,
                                                              int64_t lda, uint8_t* __restrict__ ex, int64_t lde) {
  griddep_launch_dependents();
  const int64_t groups = K / 32;
  const int64_t total = M * groups;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t m = i / groups, g = i % groups;
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
    ex[g * lde + m] = uint8_t(e + 127);
  }
}

// ------------------------------------------------------------------ GEMM

constexpr int BM = 128;               // rows of A / C per tile
constexpr int BN = 256;               // rows of B (columns of C) per tile
constexpr int BK = 128;               // K per stage: four K = 32 MMAs, one scale word
constexpr int kStages = 4;
constexpr int kStageA = BM * BK;
constexpr int kStageB = BN * BK;
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kSfSlots = 4;           // K blocks of scale factors in TMEM ahead of the MMA
constexpr int kSfAhead = 4;           // K blocks of scale factors in registers ahead of the TMEM writes
constexpr int kSfCols = 4 + BN / 32;  // A: one column per lane quarter; B: one per 32 columns
constexpr uint32_t kAccCols = BN;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 256;         // warps 0..3 control, 4..7 scale writers + epilogue
constexpr int kStageC = 32 * 128;     // a warp's 32-row x 128-byte output box
constexpr size_t kCOff = size_t(kStages) * kStageBytes;
constexpr size_t kBarOff = kCOff + 4 * size_t(kStageC);
constexpr size_t kSmemBytes = kBarOff + 256 + 1024;
static_assert(kAccCols + kSfSlots * kSfCols <= kTmemCols, "TMEM budget");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "swizzle atoms");

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

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrW8A8Mx | site);
}

template <bool F32>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const uint8_t* __restrict__ ea, int64_t lde,
                   const uint8_t* __restrict__ eb, int M, int N, int K, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* sf_full = empty + kStages;
  uint64_t* sf_empty = sf_full + kSfSlots;
  uint64_t* acc_full = sf_empty + kSfSlots;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (N + BN - 1) / BN;
  const int mt = blockIdx.x / n_tiles;
  const int nt = blockIdx.x % n_tiles;
  const int m0 = mt * BM, n0 = nt * BN;
  const int kblocks = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSfSlots; ++s) {
      mbar_init(&sf_full[s], 4);   // the four scale-writer warps
      mbar_init(&sf_empty[s], 1);  // MMA commit
    }
    mbar_init(acc_full, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();   // A may be the previous kernel's output
      int kb = 0;
      for (; kb < kblocks; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag)) {
          raise_error(err, abort_flag, kSiteProducerEmpty);
          break;
        }
        uint8_t* sa = smem + size_t(s) * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(sa, &tmA, &full[s], kb * BK, m0);
        tma_load_2d(sa + kStageA, &tmB, &full[s], kb * BK, n0);
        tma_load_2d(sa + kStageA + kStageB / 2, &tmB, &full[s], kb * BK, n0 + BN / 2);
      }
      if (kb < kblocks) {
        const int first = kb > kStages ? kb - kStages : 0;
        for (int j = first; j < kb; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % kStages;
        const int ss = kb % kSfSlots;
        if (!mbar_wait(&full[s], (kb / kStages) & 1, abort_flag)) {
          raise_error(err, abort_flag, kSiteMmaFull);
          break;
        }
        if (!mbar_wait(&sf_full[ss], (kb / kSfSlots) & 1, abort_flag)) {
          raise_error(err, abort_flag, kSiteMmaAFull);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smem + size_t(s) * kStageBytes);
        const uint32_t b0 = a0 + kStageA;
        const uint32_t sfa = sf_base + uint32_t(ss * kSfCols);
        const uint32_t sfb = sfa + 4u;
#pragma unroll
        for (int j = 0; j < BK / 32; ++j)
          mma_mx(tmem, desc_sw128_kmajor(a0 + 32u * j), desc_sw128_kmajor(b0 + 32u * j), mx_idesc(BM, BN, uint32_t(j)),
                 sfa, sfb, (kb > 0 || j > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        mma_commit(&sf_empty[ss]);
      }
      mma_commit(acc_full);   // also after an abort: the epilogue and the release of TMEM wait for it
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ scale writers
    const int q = warp & 3;
    const int m = m0 + 32 * q + lane;
    const int kw = K / 32;            // exponent bytes per weight row block
    const int nb0 = n0 / 32;
    griddep_wait();                   // the activation exponents may be the previous kernel's output
    bool ok = true;
    // The exponent words of K block kb are loaded kSfAhead blocks before they
    // are written to TMEM, so the loads' latency overlaps the MMAs of the
    // blocks in between (rows past M and columns past N: scale 1).
    auto load_sf = [&](int kb, uint32_t& wa, uint32_t* wb) {
      wa = 0x7F7F7F7Fu;
      if (m < M) {
        wa = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) wa |= uint32_t(__ldg(ea + int64_t(4 * kb + j) * lde + m)) << (8 * j);
      }
#pragma unroll
      for (int j = 0; j < BN / 32; ++j)
        wb[j] = (nb0 + j) * 32 < N ? __ldg(reinterpret_cast<const uint32_t*>(eb + int64_t(nb0 + j) * kw + 4 * kb))
                                   : 0x7F7F7F7Fu;
    };
    uint32_t qa[kSfAhead], qb[kSfAhead][BN / 32];
#pragma unroll
    for (int i = 0; i < kSfAhead; ++i)
      if (i < kblocks) load_sf(i, qa[i], qb[i]);
    for (int kb = 0; kb < kblocks; ++kb) {
      const int ss = kb % kSfSlots;
      const uint32_t wa = qa[0];
      uint32_t wb[BN / 32];
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) wb[j] = qb[0][j];
#pragma unroll
      for (int i = 0; i + 1 < kSfAhead; ++i) {
        qa[i] = qa[i + 1];
#pragma unroll
        for (int j = 0; j < BN / 32; ++j) qb[i][j] = qb[i + 1][j];
      }
      if (kb + kSfAhead < kblocks) load_sf(kb + kSfAhead, qa[kSfAhead - 1], qb[kSfAhead - 1]);
      if (!__all_sync(0xffffffffu, mbar_wait(&sf_empty[ss], ((kb / kSfSlots) & 1) ^ 1, abort_flag))) {
        raise_error(err, abort_flag, kSiteDecodeAEmpty);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t lane_base = uint32_t(32 * q) << 16;
      const uint32_t sfa = sf_base + uint32_t(ss * kSfCols);
      tmem_st_x1(sfa + lane_base + uint32_t(q), wa);
      tmem_st_x8(sfa + lane_base + 4u, wb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[ss]);
    }
    // ------------------------------------------------------------ epilogue
    if (!__all_sync(0xffffffffu, mbar_wait(acc_full, 0, ok ? abort_flag : nullptr))) {
      raise_error(err, abort_flag, kSiteEpilogueFull);
    } else if (ok && !*abort_flag && m0 + 32 * q < M) {
      tc_fence_after();
      uint8_t* stg = smem + kCOff + size_t(q) * kStageC;
      constexpr int kBoxCols = F32 ? 32 : 64;
#pragma unroll 1
      for (int c = 0; c < BN; c += kBoxCols) {
        if (n0 + c >= N) break;
        uint32_t v[64];
        const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(c);
        tmem_ld_x32(taddr, v);
        if constexpr (!F32) tmem_ld_x32(taddr + 32u, v + 32);
        tmem_ld_wait();
        if (lane == 0) bulk_wait_group_read0();   // the previous box has left the staging buffer
        __syncwarp();
        uint8_t* dst = stg + lane * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 o;
          if constexpr (F32) {
            o = make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
          } else {
            o.x = pack_bf16x2(__uint_as_float(v[8 * ch]), __uint_as_float(v[8 * ch + 1]));
            o.y = pack_bf16x2(__uint_as_float(v[8 * ch + 2]), __uint_as_float(v[8 * ch + 3]));
            o.z = pack_bf16x2(__uint_as_float(v[8 * ch + 4]), __uint_as_float(v[8 * ch + 5]));
            o.w = pack_bf16x2(__uint_as_float(v[8 * ch + 6]), __uint_as_float(v[8 * ch + 7]));
          }
          *reinterpret_cast<uint4*>(dst + ((ch ^ (lane & 7)) << 4)) = o;
        }
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, stg, n0 + c, m0 + 32 * q);
          bulk_commit_group();
        }
      }
      if (lane == 0) bulk_wait_group0();
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_quant_act_ue8m0(const QuantActUe8m0Args& p, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t total = p.M * (p.K / 32);
  const int64_t want = (total + 255) / 256;
  const int64_t cap = int64_t(dev.num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? want : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, quant_act_ue8m0_kernel, static_cast<const __nv_bfloat16*>(p.x), p.M, p.K, p.ldx,
                            static_cast<uint8_t*>(p.a), p.lda, p.ex, p.lde);
}

namespace {
template <bool F32>
cudaError_t launch_mx(const GemmW8A8MxArgs& p, const DeviceInfo&, cudaStream_t stream) {
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(tiles), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, w8a8_mx_kernel<F32>, p.tmA, p.tmB, p.tmC, p.ea, p.lde, p.eb, p.M, p.N, p.K, p.err);
}
}  // namespace

cudaError_t launch_gemm_w8a8_mx(const GemmW8A8MxArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  return p.out_f32 ? launch_mx<true>(p, dev, s) : launch_mx<false>(p, dev, s);
}

}  // namespace fp8blk
