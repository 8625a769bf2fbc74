// One-token products on the CUDA cores (sm_103a): W8A16 (bf16 token), W8A8
// (e4m3 token codes with their 1x128 scales) and the W8A8 linear that
// quantises the bf16 token itself.
//
// With M = 1 every weight byte carries one multiply-add, so the product is a
// stream of the weight matrix past the token: its time is the DRAM time of
// the weights, with most issue slots idle ("FP8 / NVFP4 weight-only inference
// on the RTX 3090 loses nothing", section 4.3 and its M = 1 measurements;
// "SM70 FP8 block-32 kernels (PLI Labs)", "How it works": a GEMV that decodes
// in registers and accumulates in FP32 serves the smallest M).  One token
// fills no tensor-core tile, and on weight sets of up to ~32 MB the MMA
// kernels' setup (TMEM, barriers, split-K reduction) costs more than the
// stream.
//
// Arithmetic (the sums of the tensor-core kernels, in another order):
//   * the token is staged once per CTA in shared memory as f32: bf16 values
//     exactly; e4m3 codes decoded exactly; or, for the quantising form, the
//     codes of the 1x128 quantisation with the stand-alone quantiser's
//     arithmetic (quant.cuh: amax, s = amax / 448, correctly rounded
//     quotient, e4m3 round-to-nearest-even with saturation), decoded;
//   * a weight code pair becomes two f16 values with cvt.rn.f16x2.e4m3x2,
//     exactly (every finite e4m3 value is an f16 normal), then two f32 values;
//   * a lane sums the 16 products of its chunk in f32 (products of e4m3 or
//     bf16 values are exact in f32), multiplies the partial by the weight
//     block's scale -- the fp32 scale of the 128 x 128 block, or 2^(e - 127)
//     for the UE8M0 byte e of the 32 x 32 block -- times, for W8A8, the
//     token's scale of the 128-block, and accumulates ("Blockwise FP8 on Ada
//     GPUs, part 2", "The fix": one promotion per 128-K block);
//   * at the end of a row the 32 lanes' sums are added with shuffles.
// A 16-code chunk never straddles a scale block (16 divides 32 and 128).
//
// Streaming: one CTA per SM owns a contiguous range of rows (the ranges
// differ by at most one row).  16 warps take the rows in turn, a whole row
// per warp, and each warp has its own ring of S shared-memory slots (a slot
// holds a segment of up to 4096 codes of one row; S is as large as shared
// memory allows, up to 6).  A warp feeds its ring itself: one lane requests
// segment c + S with a bulk copy into the slot of segment c as soon as the
// warp has used segment c, so S segments per warp are always on their way
// and no other warp or barrier is involved.  Per segment a warp makes 8
// passes of 512 codes (16 per lane).  The first S segments of every warp are
// requested before griddepcontrol.wait; the token is read and the output
// written after it.
//
// Shared-memory layout: the token as f32 [K] (16-byte unit u stored at unit
// u ^ ((u >> 2) & 7), so that the eight lanes of one 16-byte-load phase,
// whose chunks are 64 bytes apart, fall in eight different bank groups), the
// token's K / 128 scales (W8A8 forms), the slots, then one barrier per slot.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fp8blk {
namespace {

constexpr int kChunk = 16;              // codes per lane per pass
constexpr int kPass = 32 * kChunk;      // codes per warp pass
constexpr int kSeg = 4096;              // codes per slot (8 passes)
constexpr int kPasses = kSeg / kPass;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSlotsPerWarp = 6;
constexpr int kMaxStages = kWarps * kMaxSlotsPerWarp;
constexpr int kBarrierBytes = kMaxStages * 8 + 16;
constexpr int kMinSlotsPerWarp = 2;

// Scales of one segment (4096 codes of a row) are loaded by the lanes
// together and handed out by shuffles: the fp32 format has 32 blocks of 128
// in a segment (lane l holds block l), UE8M0 has 128 blocks of 32 (lane l
// holds blocks l + 32 j).
template <int FMT>
struct SegScales {
  static constexpr int kRegs = FMT == 0 ? 1 : 4;
  static constexpr int kBlock = FMT == 0 ? 128 : 32;
};
static_assert(kSeg == 32 * 128, "a segment spans 32 blocks of 128 codes");

__host__ __device__ constexpr int slot_bytes(int K) { return K < kSeg ? K : kSeg; }

// Bytes of the token area: K f32 values, then K / 128 f32 scales rounded up
// to 128 bytes (the slots after it need 16-byte alignment).
__host__ __device__ constexpr int64_t token_bytes(int64_t K) { return K * 4 + ((K / 128 * 4 + 127) / 128) * 128; }

// Bulk copy of `bytes` (a multiple of 16) global -> shared, completing on bar.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ int x_unit(int u) { return u ^ ((u >> 2) & 7); }

// Two e4m3 codes (the lower byte is the lower k) -> two f32 values, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two_codes)));
  __half2 hh;
  *reinterpret_cast<uint32_t*>(&hh) = h;
  return __half22float2(hh);
}

// Four codes (byte i = element i) -> one float4, exactly.
__device__ __forceinline__ float4 e4m3x4_to_f32x4(uint32_t four_codes) {
  const float2 lo = e4m3x2_to_f32x2(four_codes);
  const float2 hi = e4m3x2_to_f32x2(four_codes >> 16);
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Scale of K block kb (of SegScales<FMT>::kBlock codes) in weight row n.
template <int FMT>
__device__ __forceinline__ float block_scale(const void* scales, int n, int kb, int K) {
  if constexpr (FMT == 0) {
    return __ldg(static_cast<const float*>(scales) + size_t(n >> 7) * (K >> 7) + kb);
  } else {
    const uint32_t e = __ldg(static_cast<const uint8_t*>(scales) + size_t(n >> 5) * (K >> 5) + kb);
    return __uint_as_float(e << 23);   // 2^(e - 127); in-window bytes are normal exponents
  }
}

// Stages the token into shared memory as f32 (and, for the W8A8 forms, its
// K / 128 scales).  All threads of the CTA take part.
template <int ACT>
__device__ __forceinline__ void stage_token(const void* x, const float* a_scales, int64_t lds, int K, float4* xs4,
                                            float* as_sm) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if constexpr (ACT == kGemvActBf16) {
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    for (int i = threadIdx.x; i < K / 8; i += blockDim.x) {
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(xb + 8 * i), f);
      xs4[x_unit(2 * i)] = make_float4(f[0], f[1], f[2], f[3]);
      xs4[x_unit(2 * i + 1)] = make_float4(f[4], f[5], f[6], f[7]);
    }
  } else if constexpr (ACT == kGemvActE4m3) {
    const uint8_t* a = static_cast<const uint8_t*>(x);
    for (int i = threadIdx.x; i < K / 16; i += blockDim.x) {
      const uint4 v = *reinterpret_cast<const uint4*>(a + 16 * i);
      xs4[x_unit(4 * i)] = e4m3x4_to_f32x4(v.x);
      xs4[x_unit(4 * i + 1)] = e4m3x4_to_f32x4(v.y);
      xs4[x_unit(4 * i + 2)] = e4m3x4_to_f32x4(v.z);
      xs4[x_unit(4 * i + 3)] = e4m3x4_to_f32x4(v.w);
    }
    for (int g = threadIdx.x; g < K / 128; g += blockDim.x) as_sm[g] = a_scales[int64_t(g) * lds];
  } else {
    // One warp per 128-group, four values per lane.
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    for (int g = warp; g < K / 128; g += kWarps) {
      const uint2 v = *reinterpret_cast<const uint2*>(xb + g * 128 + 4 * lane);
      const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xFFFF0000u);
      const float f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xFFFF0000u);
      float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = group_scale(amax);
      const Divisor d = make_divisor(s);
      const uint32_t q = e4m3x4(quotient(f0, d), quotient(f1, d), quotient(f2, d), quotient(f3, d));
      xs4[x_unit(g * 32 + lane)] = e4m3x4_to_f32x4(q);
      if (lane == 0) as_sm[g] = s;
    }
  }
}

template <int ACT, class OutT, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const void* __restrict__ x, const float* __restrict__ a_scales, int64_t lds,
                const uint8_t* __restrict__ b, int64_t ldb, const void* __restrict__ scales, OutT* __restrict__ c,
                int N, int K, int slots_per_warp, int* __restrict__ err) {
  static_assert(ACT == kGemvActBf16 || FMT == 0, "W8A8 weights carry fp32 128x128 scales");
  extern __shared__ __align__(128) uint8_t smem[];
  float4* xs4 = reinterpret_cast<float4*>(smem);
  float* as_sm = reinterpret_cast<float*>(smem + size_t(K) * 4);
  const int slot = slot_bytes(K);
  uint8_t* stages = smem + token_bytes(K);
  const int S = slots_per_warp;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + size_t(kWarps) * S * slot);
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = int(int64_t(blockIdx.x) * N / gridDim.x);
  const int rows = int(int64_t(blockIdx.x + 1) * N / gridDim.x) - row0;
  const int nseg = (K + kSeg - 1) / kSeg;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * S; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Segment c of this warp is segment c % nseg of row warp + kWarps *
  // (c / nseg), in slot warp * S + c % S, use c / S of that slot.
  const uint64_t policy = policy_evict_first();
  auto request = [&](int c) {   // one lane
    const int j = warp + kWarps * (c / nseg);
    if (j >= rows) return;
    const int seg = c % nseg;
    const int sl = warp * S + c % S;
    const int bytes = K - seg * kSeg < kSeg ? K - seg * kSeg : kSeg;
    fence_async_shared();   // the warp's reads of the slot come before the copy's writes
    mbar_arrive_expect_tx(&full[sl], uint32_t(bytes));
    bulk_load(stages + size_t(sl) * slot, b + int64_t(row0 + j) * ldb + int64_t(seg) * kSeg, uint32_t(bytes),
              &full[sl], policy);
  };
  if (lane == 0)
    for (int c = 0; c < S; ++c) request(c);

  griddep_wait();   // the token may be the previous kernel's output
  stage_token<ACT>(x, a_scales, lds, K, xs4, as_sm);
  __syncthreads();

  constexpr int kSRegs = SegScales<FMT>::kRegs;
  constexpr int kBlock = SegScales<FMT>::kBlock;
  const int nblocks = K / kBlock;
  for (int j = warp, r = 0; j < rows; j += kWarps, ++r) {
    const int n = row0 + j;
    float acc = 0.f;
    bool ok = true;
    for (int seg = 0; seg < nseg; ++seg) {
      const int cs = r * nseg + seg;   // this warp's stage
      const int s = warp * S + cs % S;
      const int bytes = K - seg * kSeg < kSeg ? K - seg * kSeg : kSeg;
      float sreg[kSRegs];
      const int kb0 = seg * (kSeg / kBlock);
#pragma unroll
      for (int q = 0; q < kSRegs; ++q) {
        const int kb = kb0 + lane + 32 * q;
        sreg[q] = kb < nblocks ? block_scale<FMT>(scales, n, kb, K) : 0.f;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], uint32_t((cs / S) & 1), nullptr))) {
        // Nothing else waits on this warp: it reports and leaves after the
        // copies it requested have landed (each wait bounded).
        if (lane == 0) {
          atomicCAS(err, 0, kDevErrGemv | kSiteDecodeFull);
          for (int c = cs; c < cs + S; ++c)
            if (warp + kWarps * (c / nseg) < rows) mbar_wait(&full[warp * S + c % S], uint32_t((c / S) & 1), nullptr);
        }
        ok = false;
        break;
      }
      const uint8_t* st = stages + size_t(s) * slot;
      uint4 w[kPasses];
#pragma unroll
      for (int u = 0; u < kPasses; ++u) {
        const int k0 = u * kPass + lane * kChunk;
        w[u] = k0 < bytes ? *reinterpret_cast<const uint4*>(st + k0) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kPasses; ++u) {
        const int k0 = u * kPass + lane * kChunk;
        // This chunk's block within the segment: 4u + lane / 8 (fp32 format)
        // or 16u + lane / 2 (UE8M0); every lane takes part in the shuffle.
        const int gb = FMT == 0 ? 4 * u + (lane >> 3) : 16 * u + (lane >> 1);
        float su = __shfl_sync(0xffffffffu, sreg[gb >> 5], gb & 31);
        if (k0 < bytes) {
          if constexpr (ACT != kGemvActBf16) su *= as_sm[seg * (kSeg / 128) + gb];
          const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
          const int ux = (seg * kSeg + k0) / 4;   // first 16-byte unit of the token for this chunk
          // Packed f32x2 multiply-adds: even and odd k in the two halves.
          float2 part = make_float2(0.f, 0.f);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const float2 lo = e4m3x2_to_f32x2(q[jj]);
            const float2 hi = e4m3x2_to_f32x2(q[jj] >> 16);
            const float4 xv = xs4[x_unit(ux + jj)];
            part = ffma2(lo, make_float2(xv.x, xv.y), part);
            part = ffma2(hi, make_float2(xv.z, xv.w), part);
          }
          acc = fmaf(part.x + part.y, su, acc);
        }
      }
      // Every lane's codes have been used: the slot takes segment cs + S.
      __syncwarp();
      if (lane == 0) request(cs + S);
    }
    if (!ok) break;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if constexpr (sizeof(OutT) == 4)
        c[n] = acc;
      else
        c[n] = __float2bfloat16_rn(acc);
    }
  }
}

// Slots per warp that fit next to the staged token (0 if none).
int gemv_slots_per_warp(int64_t K, int smem_optin) {
  const int64_t avail = int64_t(smem_optin) - token_bytes(K) - kBarrierBytes;
  if (avail <= 0) return 0;
  const int64_t n = avail / (int64_t(kWarps) * slot_bytes(int(K < kSeg ? K : kSeg)));
  return int(n < kMaxSlotsPerWarp ? n : kMaxSlotsPerWarp);
}

template <int ACT, class OutT, int FMT>
cudaError_t launch_typed(const GemvArgs& p, const DeviceInfo& dev, cudaStream_t stream) {
  auto kernel = gemv_kernel<ACT, OutT, FMT>;
  const int spw = gemv_slots_per_warp(p.K, dev.max_smem_optin);
  if (spw < kMinSlotsPerWarp) return cudaErrorInvalidValue;
  const size_t smem = size_t(token_bytes(p.K)) + size_t(kWarps) * spw * slot_bytes(p.K) + kBarrierBytes;
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[device]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int grid = p.N < dev.num_sms ? p.N : dev.num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p.x, p.a_scales, p.lds, static_cast<const uint8_t*>(p.b), p.ldb,
                            p.scales, static_cast<OutT*>(p.C), p.N, p.K, spw, p.err);
}

template <int ACT, int FMT>
cudaError_t launch_act(const GemvArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  return p.out_f32 ? launch_typed<ACT, float, FMT>(p, dev, s) : launch_typed<ACT, __nv_bfloat16, FMT>(p, dev, s);
}

}  // namespace

bool gemv_window(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  return M == 1 && K >= kSeg && N * K <= (int64_t(1) << 25) &&
         gemv_slots_per_warp(K, dev.max_smem_optin) >= kMinSlotsPerWarp;
}

cudaError_t launch_gemv(const GemvArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  switch (p.act) {
    case kGemvActBf16:
      return p.fmt == 0 ? launch_act<kGemvActBf16, 0>(p, dev, s) : launch_act<kGemvActBf16, 1>(p, dev, s);
    case kGemvActE4m3:
      return p.fmt == 0 ? launch_act<kGemvActE4m3, 0>(p, dev, s) : cudaErrorInvalidValue;
    case kGemvActQuant:
      return p.fmt == 0 ? launch_act<kGemvActQuant, 0>(p, dev, s) : cudaErrorInvalidValue;
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fp8blk
