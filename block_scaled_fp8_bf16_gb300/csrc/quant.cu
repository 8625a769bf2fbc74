// Quantisers (bf16 -> e4m3 with fp32 block scales), the weight validator and
// the decode and wait-timeout diagnostics.
//
// Per-token activation quantisation ("Blockwise FP8 on Ada GPUs, part 2",
// "The starting point": one scale per token per 128 values of K) follows the
// warp-per-group shape the ArcKernels PR proposes in its "Route-2 handover"
// (finding 3: one warp per 128-block, shuffle max reduction, vectorised
// loads) instead of a 1024-thread block with 32 active threads: here each
// warp takes two adjacent 128-groups of four consecutive rows, sixteen lanes
// per group and eight bf16 per lane (one 16-byte load per row, four in
// flight), reduces |x| with four xor shuffles, and writes eight codes per
// lane (one 8-byte store).  The pass reads 2 bytes and writes 1 + 4/128
// bytes per element and is bound by HBM bandwidth.
//
// The scale is s = amax / 448 with IEEE division; the codes are
// e4m3(x / s) with the correctly rounded quotient, round-to-nearest-even and
// saturation to +-448 (cvt.rn.satfinite); amax == 0 gives s = 1.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "decode.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fp8blk {
namespace {

// Activation quantiser, persistent and fed by TMA.  A tile is 64 token rows
// of one 128-wide group (16 KB of bf16); tile t covers rows 64 (t / G) ..
// and group t % G (G = K / 128).  One producer thread keeps kQStages tiles
// in flight per CTA, three CTAs per SM (12 tiles, 192 KB, in flight per SM:
// more consuming warps per SM than two CTAs of six tiles, for the same bytes
// in flight).  Eight warps consume a tile: warp w takes rows
// 8w .. 8w + 7, four lanes per row and 32 bf16 per lane (four 8-column
// chunks, 32 columns apart, so a row's lanes read consecutive bytes), so the per-group
// work (the row's amax from two xor shuffles, the IEEE scale division and
// the reciprocal behind the correctly rounded quotients, all with the
// arithmetic of quant.cuh) is spread over 32 elements per lane.  Rows past M
// arrive zero-filled and are not stored.
constexpr int kQTileRows = kQuantTileRows;
constexpr int64_t kQuantSmallM = 256;   // up to this many rows the register-fed kernel below runs
constexpr int kQTileBytes = kQTileRows * 128 * 2;
constexpr int kQStages = 4;
constexpr int kQCtasPerSm = 3;
constexpr int kQWarps = 8;
constexpr int kQThreads = (kQWarps + 1) * 32;
constexpr size_t kQSmemBytes = size_t(kQStages) * kQTileBytes + 2 * kQStages * 8 + 1024;

__device__ __forceinline__ void quant_raise(int* err, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(err, 0, kDevErrQuant | site);
}

__global__ void __launch_bounds__(kQThreads, kQCtasPerSm) quant_act_kernel(const __grid_constant__ CUtensorMap tmX, int64_t M,
                                                              int64_t K, uint8_t* __restrict__ a, int64_t lda,
                                                              float* __restrict__ scales, int64_t lds,
                                                              int* __restrict__ err) {
  // A GEMM launched after this kernel with programmatic dependent launch may
  // begin streaming its weights now; it waits for this grid before reading
  // the codes and scales written here.
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(kQStages) * kQTileBytes);
  uint64_t* empty = full + kQStages;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t groups = K / 128;
  const int64_t num_tiles = ((M + kQTileRows - 1) / kQTileRows) * groups;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kQWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      uint32_t it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
        const int s = it % kQStages;
        if (!mbar_wait(&empty[s], ((it / kQStages) & 1u) ^ 1u, abort_flag)) {
          quant_raise(err, abort_flag, kSiteProducerEmpty);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kQTileBytes);
        tma_load_2d(smem + size_t(s) * kQTileBytes, &tmX, &full[s], int32_t((t % groups) * 128),
                    int32_t((t / groups) * kQTileRows));
      }
      if (!ok) {
        const uint32_t first = it > uint32_t(kQStages) ? it - kQStages : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % kQStages], (j / kQStages) & 1u, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ quantisers
    const int sub = lane & 3;          // the row's 8-column chunks sub, sub + 4, sub + 8, sub + 12
    const int row = 8 * warp + (lane >> 2);
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int s = it % kQStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / kQStages) & 1u, abort_flag))) {
        quant_raise(err, abort_flag, kSiteEpilogueFull);
        break;
      }
      const int64_t g = t % groups;
      const int64_t m0 = (t / groups) * kQTileRows;
      // The four lanes of a row read 64 consecutive bytes per load.
      const uint8_t* src = smem + size_t(s) * kQTileBytes + row * 256 + sub * 16;
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4*>(src + j * 64);
      fence_async_shared();   // generic-proxy reads of the stage before its TMA (async-proxy) refill
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);   // the rows are in registers: the stage can refill
      float f[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) bf16x8_to_f32(v[j], f + 8 * j);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      const float sc = group_scale(amax);
      const Divisor dv = make_divisor(sc);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = e4m3x4(quotient(f[4 * i], dv), quotient(f[4 * i + 1], dv), quotient(f[4 * i + 2], dv),
                      quotient(f[4 * i + 3], dv));
      const int64_t m = m0 + row;
      if (m < M) {
        uint8_t* dst = a + m * lda + g * 128 + sub * 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint2*>(dst + 32 * j) = make_uint2(w[2 * j], w[2 * j + 1]);
        if (sub == 0) scales[g * lds + m] = sc;
      }
    }
  }
}

// Few rows (M <= kQuantSmallM): no TMA ring, every warp loads its rows
// straight into registers, which keeps the latency of a small call low.
// Grid: x covers rows (each warp takes kQuantRows consecutive rows per
// step), y covers pairs of 128-groups (lanes 0-15: group 2y, 16-31: 2y+1).
constexpr int kQuantRows = 4;

__global__ void __launch_bounds__(256) quant_act_small_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, uint8_t* __restrict__ a, int64_t lda,
                                                        float* __restrict__ scales, int64_t lds) {
  // A GEMM launched after this kernel with programmatic dependent launch may
  // begin streaming its weights now; it waits for this grid before reading
  // the codes and scales written here.
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;
  const int64_t g = int64_t(blockIdx.y) * 2 + (lane >> 4);
  const bool active = g < K / 128;
  const int64_t col = g * 128 + hl * 8;
  const int64_t step = int64_t(gridDim.x) * (blockDim.x >> 5) * kQuantRows;
  for (int64_t m0 = (int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kQuantRows; m0 < M;
       m0 += step) {
    uint4 v[kQuantRows];
#pragma unroll
    for (int r = 0; r < kQuantRows; ++r) {
      v[r] = make_uint4(0, 0, 0, 0);
      if (active && m0 + r < M) v[r] = ld_nc_v4(x + (m0 + r) * ldx + col);
    }
#pragma unroll
    for (int r = 0; r < kQuantRows; ++r) {
      float f[8];
      bf16x8_to_f32(v[r], f);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = group_scale(amax);
      const Divisor dv = make_divisor(s);
      float q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = quotient(f[i], dv);
      if (active && m0 + r < M) {
        uint2 out;
        out.x = e4m3x4(q[0], q[1], q[2], q[3]);
        out.y = e4m3x4(q[4], q[5], q[6], q[7]);
        *reinterpret_cast<uint2*>(a + (m0 + r) * lda + col) = out;
        if (hl == 0) scales[g * lds + m0 + r] = s;
      }
    }
  }
}

// One CTA = one 128x128 weight block; 256 threads x 8 x (8 bf16).
__global__ void __launch_bounds__(256) quant_weight_kernel(const __nv_bfloat16* __restrict__ w, int64_t N, int64_t K,
                                                           int64_t ldw, uint8_t* __restrict__ b, int64_t ldb,
                                                           float* __restrict__ scales) {
  __shared__ float red[8];
  const int64_t kb_count = K / 128;
  const int64_t nb = blockIdx.x / kb_count;
  const int64_t kb = blockIdx.x % kb_count;
  const int tid = threadIdx.x;
  uint4 v[8];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = tid + 256 * j;      // 16-byte chunk index inside the block
    const int r = i >> 4, c = i & 15;
    v[j] = ld_nc_v4(w + (nb * 128 + r) * ldw + kb * 128 + c * 8);
    float f[8];
    bf16x8_to_f32(v[j], f);
#pragma unroll
    for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(f[t]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = group_scale(amax);
  const Divisor dv = make_divisor(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = tid + 256 * j;
    const int r = i >> 4, c = i & 15;
    float f[8];
    bf16x8_to_f32(v[j], f);
    uint2 out;
    out.x = e4m3x4(quotient(f[0], dv), quotient(f[1], dv), quotient(f[2], dv), quotient(f[3], dv));
    out.y = e4m3x4(quotient(f[4], dv), quotient(f[5], dv), quotient(f[6], dv), quotient(f[7], dv));
    *reinterpret_cast<uint2*>(b + (nb * 128 + r) * ldb + kb * 128 + c * 8) = out;
  }
  if (tid == 0) scales[nb * kb_count + kb] = s;
}

__global__ void validate_kernel(const uint8_t* __restrict__ b, int64_t ldb, const void* __restrict__ sc, int fmt,
                                int64_t N, int64_t K, int32_t* __restrict__ counts) {
  int nan_codes = 0, bad_scales = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t chunks_per_row = K / 16;
  for (int64_t i = tid; i < N * chunks_per_row; i += stride) {
    const int64_t r = i / chunks_per_row, c = i % chunks_per_row;
    const uint4 v = ld_nc_v4(b + r * ldb + c * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int t = 0; t < 4; ++t) nan_codes += ((w[j] >> (8 * t)) & 0x7Fu) == 0x7Fu;
    }
  }
  if (fmt == 0) {
    const float* s = static_cast<const float*>(sc);
    for (int64_t i = tid; i < (N / 128) * (K / 128); i += stride) {
      const float v = s[i];
      bad_scales += !(isfinite(v) && v > 0.f);
    }
  } else {
    const uint8_t* s = static_cast<const uint8_t*>(sc);
    for (int64_t i = tid; i < (N / 32) * (K / 32); i += stride) {
      const int e = int(s[i]) - 127;
      bad_scales += (e < -14 || e > 7);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    nan_codes += __shfl_xor_sync(0xffffffffu, nan_codes, o);
    bad_scales += __shfl_xor_sync(0xffffffffu, bad_scales, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (nan_codes) atomicAdd(&counts[0], nan_codes);
    if (bad_scales) atomicAdd(&counts[1], bad_scales);
  }
}

__global__ void debug_decode_kernel(const uint8_t* __restrict__ codes, int64_t n, int exp_shift,
                                    uint32_t* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;   // one word of 4 codes
  if (i * 4 >= n) return;
  const uint32_t q = *reinterpret_cast<const uint32_t*>(codes + 4 * i);
  uint32_t lo, hi;
  decode4_e4m3_bf16(q, decode_multiplier_bf16x2(exp_shift), lo, hi);
  out[2 * i] = lo;
  out[2 * i + 1] = hi;
}

int grid_for(int64_t items, int per_block, int num_sms, int waves) {
  int64_t g = (items + per_block - 1) / per_block;
  const int64_t cap = int64_t(num_sms) * waves;
  if (g > cap) g = cap;
  return g < 1 ? 1 : int(g);
}

}  // namespace

cudaError_t launch_quant_act(const QuantActArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  if (p.M <= kQuantSmallM) {
    const int64_t pairs = (p.K / 128 + 1) / 2;
    if (pairs > 65535) return cudaErrorInvalidValue;
    const int64_t row_steps = (p.M + kQuantRows - 1) / kQuantRows;     // warps needed along M
    int64_t gx = (row_steps + 7) / 8;
    const int64_t cap = (int64_t(dev.num_sms) * 16 + pairs - 1) / pairs;  // about 16 CTAs per SM in total
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    quant_act_small_kernel<<<dim3(unsigned(gx), unsigned(pairs)), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(p.x), p.M, p.K, p.ldx, static_cast<uint8_t*>(p.a), p.lda, p.scales, p.lds);
    return cudaGetLastError();
  }
  static bool attr_done[64] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 64 && !attr_done[device]) {
    e = cudaFuncSetAttribute(quant_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kQSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[device] = true;
  }
  const int64_t tiles = ((p.M + kQTileRows - 1) / kQTileRows) * (p.K / 128);
  const int64_t slots = int64_t(dev.num_sms) * kQCtasPerSm;
  const unsigned grid = unsigned(tiles < slots ? tiles : slots);
  quant_act_kernel<<<grid, kQThreads, kQSmemBytes, s>>>(p.tmX, p.M, p.K, static_cast<uint8_t*>(p.a), p.lda,
                                                        p.scales, p.lds, p.err);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight(const QuantWeightArgs& p, const DeviceInfo&, cudaStream_t s) {
  const int64_t blocks = (p.N / 128) * (p.K / 128);
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  quant_weight_kernel<<<unsigned(blocks), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.w), p.N, p.K, p.ldw,
                                                       static_cast<uint8_t*>(p.b), p.ldb, p.scales);
  return cudaGetLastError();
}

cudaError_t launch_validate(const ValidateArgs& p, const DeviceInfo& dev, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.counts, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(p.N * (p.K / 16), 256, dev.num_sms, 8);
  validate_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(p.b), p.ldb, p.scales, p.fmt, p.N, p.K,
                                       p.counts);
  return cudaGetLastError();
}

// Waits on an mbarrier that no thread ever arrives on, with the bounded-wait
// loop of the GEMM kernels (try_wait polling, %globaltimer limit), and
// records `code` in the error word when the limit passes.
__global__ void debug_wait_timeout_kernel(int64_t limit_ns, int code, int* __restrict__ err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  bool done = mbar_test(&bar, 0);
  const uint64_t t0 = globaltimer_ns();
  while (!done && globaltimer_ns() - t0 < uint64_t(limit_ns)) done = mbar_test(&bar, 0);
  if (!done && threadIdx.x == 0) atomicCAS(err, 0, code);
}

cudaError_t launch_debug_wait_timeout(int64_t limit_ns, int code, int* err, cudaStream_t s) {
  debug_wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, code, err);
  return cudaGetLastError();
}

// A plain read-only stream: n 16-byte words, eight loads in flight per
// thread (grid-stride), every 32-bit word XORed into *sink (one atomic per
// CTA), so that nothing of the stream can be dropped.
constexpr int kReadThreads = 512;
__global__ void __launch_bounds__(kReadThreads) debug_stream_read_kernel(const uint4* __restrict__ p, int64_t n,
                                                                          uint32_t* __restrict__ sink) {
  constexpr int U = 8;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (U - 1) * stride < n; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n; i += stride) {
    const uint4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t warp_x[kReadThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_x[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kReadThreads / 32; ++w) b ^= warp_x[w];
    atomicXor(sink, b);
  }
}

cudaError_t launch_debug_stream_read(const void* p, int64_t words16, uint32_t* sink, int num_sms, cudaStream_t s) {
  debug_stream_read_kernel<<<4 * num_sms, kReadThreads, 0, s>>>(static_cast<const uint4*>(p), words16, sink);
  return cudaGetLastError();
}

// Runs the quantisers' scale arithmetic on n group maxima: s = group_scale,
// and the divisor make_divisor(s) forms (scaled divisor and its reciprocal).
__global__ void debug_group_scale_kernel(const float* __restrict__ amax, int64_t n, float* __restrict__ s_out,
                                         float* __restrict__ ds_out, float* __restrict__ y_out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float s = group_scale(amax[i]);
  const Divisor d = make_divisor(s);
  s_out[i] = s;
  ds_out[i] = d.s;
  y_out[i] = d.y;
}

cudaError_t launch_debug_group_scale(const float* amax, int64_t n, float* s, float* ds, float* y, cudaStream_t st) {
  const int grid = int((n + 255) / 256);
  debug_group_scale_kernel<<<grid, 256, 0, st>>>(amax, n, s, ds, y);
  return cudaGetLastError();
}

cudaError_t launch_debug_decode(const void* codes, int64_t n, int exp_shift, void* out, cudaStream_t s) {
  const int64_t words = n / 4;
  const int grid = int((words + 255) / 256);
  debug_decode_kernel<<<grid < 1 ? 1 : grid, 256, 0, s>>>(static_cast<const uint8_t*>(codes), n, exp_shift,
                                                         static_cast<uint32_t*>(out));
  return cudaGetLastError();
}

}  // namespace fp8blk
