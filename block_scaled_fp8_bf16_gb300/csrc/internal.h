// Internal interface between the C ABI layer (api.cu) and the kernel
// translation units.  Not installed, not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8blk {

// Values a kernel writes into the per-device error word when a bounded wait
// gives up.  The low byte names the kernel, the next byte the wait site.
enum DeviceErr : int {
  kDevErrNone = 0,
  kDevErrW8A8 = 0x100,
  kDevErrW8A16 = 0x200,
};
enum WaitSite : int {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteEpilogueFull = 4,
  kSiteDecodeFull = 5,
  kSiteDecodeAEmpty = 6,
  kSiteMmaAFull = 7,
  kSiteDrain = 8,
};

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
  int max_smem_optin = 0;
  int* err_word = nullptr;   // device address of the error word
};

// ------------------------------------------------------------------ quant
struct QuantActArgs {
  const void* x;
  int64_t M, K, ldx;
  void* a;
  int64_t lda;
  float* scales;
  int64_t lds;
};
cudaError_t launch_quant_act(const QuantActArgs& p, const DeviceInfo& dev, cudaStream_t s);

struct QuantWeightArgs {
  const void* w;
  int64_t N, K, ldw;
  void* b;
  int64_t ldb;
  float* scales;
};
cudaError_t launch_quant_weight(const QuantWeightArgs& p, const DeviceInfo& dev, cudaStream_t s);

struct ValidateArgs {
  const void* b;
  int64_t ldb;
  const void* scales;
  int fmt;
  int64_t N, K;
  int32_t* counts;
};
cudaError_t launch_validate(const ValidateArgs& p, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_debug_decode(const void* codes, int64_t n, int exp_shift, void* out, cudaStream_t s);

// ------------------------------------------------------------------ W8A8
struct GemmW8A8Args {
  CUtensorMap tmA;    // e4m3 [M, K], box {128 (K), 128 (M)}, 128B swizzle
  CUtensorMap tmB;    // e4m3 [N, K], box {128 (K), kW8A8TileN (N)}, 128B swizzle
  CUtensorMap tmAs;   // fp32 [K/128][lds] read as {M, K/128}, box {128, 1}, no swizzle
  const float* Bs;    // [N/128][K/128]
  void* C;            // bf16 [M, ldc]
  int64_t ldc;
  int M, N, K;
  int* err;
};
constexpr int kW8A8TileM = 128;
constexpr int kW8A8TileN = 128;
constexpr int kMaxSplitK = 8;
cudaError_t launch_gemm_w8a8(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t s);
// CTA-pair kernel (256 x 256 tiles); chosen by launch_gemm_w8a8 for large problems.
int w8a8_pair_tiles(int M, int N);
cudaError_t launch_gemm_w8a8_pair(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t s);

// ------------------------------------------------------------------ W8A16
struct GemmW8A16Args {
  CUtensorMap tmW;    // e4m3 [N, K], box {128 (K), 128 (N)}, 128B swizzle
  CUtensorMap tmX;    // bf16 [M, K], box {64 (K), tile_m (M)}, 128B swizzle
  const void* scales; // fp32 [N/128][K/128] or uint8 [N/32][K/32]
  int fmt;            // 0 = fp32 128x128, 1 = UE8M0 32x32
  void* C;
  int64_t ldc;
  int M, N, K;
  int tile_m;         // token tile (MMA N): 16, 32, 64 or 128
  int* err;
};
constexpr int kW8A16TileN = 128;
constexpr int kW8A16MaxTileM = 128;
int w8a16_pick_tile_m(int64_t M);
cudaError_t launch_gemm_w8a16(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t s);

}  // namespace fp8blk
