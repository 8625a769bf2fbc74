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
  kDevErrW8A16Decode = 0x300,
  kDevErrQuant = 0x400,
  kDevErrGemv = 0x500,
  kDevErrW8A8Mx = 0x600,
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
  kSiteReduceEmpty = 9,
  kSiteReduceFull = 10,
  kSiteBadGroup = 11,   // not a wait: a grouped tile named a group past the weights
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
  CUtensorMap tmX;    // bf16 x [M, K] pitch ldx, box {128 (K), kQuantTileRows (M)}, no swizzle
  const void* x;      // the same tensor, for the few-row kernel
  int64_t ldx;
  int64_t M, K;
  void* a;
  int64_t lda;
  float* scales;
  int64_t lds;
  int* err;
};
constexpr int kQuantTileRows = 64;   // token rows per tile of the activation quantiser (the x box height)
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
cudaError_t launch_debug_group_scale(const float* amax, int64_t n, float* s, float* ds, float* y, cudaStream_t st);
cudaError_t launch_debug_wait_timeout(int64_t limit_ns, int code, int* err, cudaStream_t s);
cudaError_t launch_debug_stream_read(const void* p, int64_t words16, uint32_t* sink, int num_sms, cudaStream_t s);

// ------------------------------------------------------------------ W8A8
struct GemmW8A8Args {
  CUtensorMap tmA;    // e4m3 [M, K], box {128 (K), 128 (M)}, 128B swizzle
  CUtensorMap tmB;    // e4m3 [N, K], box {128 (K), kW8A8TileN (N)}, 128B swizzle
  CUtensorMap tmAs;   // fp32 [K/128][lds] read as {M, K/128}, box {128, 1}, no swizzle
  CUtensorMap tmAsG;  // the same scales, box {128, 8}: eight K blocks per copy (pair kernel)
  CUtensorMap tmC;    // C [M, N] pitch ldc, box {128 bytes of N, 32 (M)}, 128B swizzle (pair kernel's stores)
  CUtensorMap tmX;    // fused form: bf16 x [M, K] pitch ldx, box {64 (K), 32 (M)}, 128B swizzle
  const float* Bs;    // [N/128][K/128]
  void* C;            // bf16 [M, ldc]
  int64_t ldc;
  int M, N, K;
  bool pdl;           // launch with programmatic stream serialisation
  bool out_f32;       // C is float32 (ldc in float32 elements), else bf16
  const int* row_group = nullptr;   // grouped form: group of each row (device), else nullptr
  int groups = 1;                   // G: the weights are [G*N, K], their scales [G][N/128][K/128]
  bool fused = false;               // quantise bf16 x (tmX) in the kernel; M <= kW8A8FusedMaxM
  int* err;
};
constexpr int kW8A8TileM = 128;
constexpr int kW8A8FusedMaxM = 32;   // token rows the activation-quantising form takes
constexpr int kW8A8TileN = 128;
constexpr int kMaxSplitK = 8;
cudaError_t launch_gemm_w8a8(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t s);
// CTA-pair kernel (256 x 256 tiles); chosen by launch_gemm_w8a8 for large problems.
int w8a8_pair_tiles(int M, int N);
cudaError_t launch_gemm_w8a8_pair(const GemmW8A8Args& p, const DeviceInfo& dev, cudaStream_t s);

// ------------------------------------------------------------------ W8A8, 32x32 UE8M0 format
// Activation quantiser with power-of-two 1x32 scales (exponent bytes in the
// tiled scale layout) and the block-scaled tensor-core product.
struct QuantActUe8m0Args {
  const void* x;      // bf16 [M, K] pitch ldx
  int64_t ldx;
  int64_t M, K;
  void* a;            // e4m3 [M, K] pitch lda
  int64_t lda;
  uint8_t* sf;        // exponent bytes in the tiled scale layout, rows padded to 128
};
cudaError_t launch_quant_act_ue8m0(const QuantActUe8m0Args& p, const DeviceInfo& dev, cudaStream_t s);
// [N/32][K/32] weight exponent bytes -> the tiled per-column scale layout.
cudaError_t launch_ue8m0_weight_sf(const uint8_t* eb, int64_t N, int64_t K, uint8_t* sf, const DeviceInfo& dev,
                                   cudaStream_t s);

struct GemmW8A8MxArgs {
  CUtensorMap tmA;    // e4m3 [M, K], box {128 (K), 128 (M)}, 128B swizzle
  CUtensorMap tmB;    // e4m3 [N, K], box {128 (K), 128 (N)}, 128B swizzle
  CUtensorMap tmC;    // C [M, N], box {128 bytes of N, 32 (M)}, 128B swizzle
  CUtensorMap tmSfa;  // the activation scale array as uint32 [blocks][128], box {128, 1} (pair kernel)
  CUtensorMap tmSfb;  // the weight scale array, the same way
  const uint8_t* a_sf;  // activation exponent bytes, tiled scale layout (rows padded to 128)
  const uint8_t* b_sf;  // weight exponent bytes per column, tiled scale layout
  void* C;              // C itself, for the split-K form's direct stores
  int64_t ldc;
  int M, N, K;
  bool pdl;
  bool out_f32;
  int* err;
};
cudaError_t launch_gemm_w8a8_mx(const GemmW8A8MxArgs& p, const DeviceInfo& dev, cudaStream_t s);
int mx_pair_tiles(int M, int N);

// ------------------------------------------------------------------ W8A16
struct GemmW8A16Args {
  CUtensorMap tmW;    // e4m3 [N, K], box {128 (K), 128 (N)}, 128B swizzle
  CUtensorMap tmX;    // bf16 [M, K], box {64 (K), tile_m (M)}, 128B swizzle
  const void* scales; // fp32 [N/128][K/128] or uint8 [N/32][K/32]
  int fmt;            // 0 = fp32 128x128, 1 = UE8M0 32x32
  void* C;
  int64_t ldc;
  int M, N, K;
  int tile_m;         // token tile (MMA N): 16, 32, 64, 128 or 256 (UE8M0 only)
  bool pdl;           // launch with programmatic stream serialisation
  bool out_f32;       // C is float32 (ldc in float32 elements), else bf16
  int* err;
};
constexpr int kW8A16TileN = 128;
constexpr int kW8A16MaxTileM = 256;
int w8a16_pick_tile_m(int64_t M, int64_t N, int fmt, int num_sms);
cudaError_t launch_gemm_w8a16(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t s);

// Decode-size W8A16 (M <= tile_m, tile_m 16 or 32).
constexpr int kW8A16DecodeMaxM = 32;
cudaError_t launch_w8a16_decode(const GemmW8A16Args& p, const DeviceInfo& dev, cudaStream_t s);

// ------------------------------------------------------------------ one token
// CUDA-core GEMV (gemv.cu) streaming the weight rows through per-warp rings
// of shared-memory slots, the token staged as f32 in shared memory.  Chosen
// where the sweep measured it faster than the tensor-core kernels: M = 1,
// K >= 4096 and at most 2^25 weight codes; on larger weight sets the
// tensor-core kernels stream faster, and at M = 2 the decode-size kernel
// costs what it costs at M = 1 while the GEMV's arithmetic doubles.
enum GemvAct : int {
  kGemvActBf16 = 0,    // W8A16: x is a bf16 row
  kGemvActE4m3 = 1,    // W8A8: x is an e4m3 row, its scales a_scales[kb * lds]
  kGemvActQuant = 2,   // W8A8 linear: x is a bf16 row, quantised 1x128 in the kernel
};
struct GemvArgs {
  const void* x;
  const float* a_scales;   // kGemvActE4m3 only
  int64_t lds;
  const void* b;           // e4m3 [N, K] pitch ldb
  int64_t ldb;
  const void* scales;      // fp32 [N/128][K/128] or uint8 [N/32][K/32]
  int fmt;                 // 0 = fp32 128x128, 1 = UE8M0 32x32 (W8A16 only)
  int act;                 // GemvAct
  void* C;                 // bf16 or float32 [N]
  int N, K;
  bool pdl;
  bool out_f32;
  int* err;
};
bool gemv_window(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
cudaError_t launch_gemv(const GemvArgs& p, const DeviceInfo& dev, cudaStream_t s);

// Work split of the decode kernel: K is divided over clusters of `split`
// CTAs (1, 2, 4 or 8) and the 128-row weight tiles run persistently over
// `clusters` clusters.  Chosen to minimise the per-CTA K blocks on the
// critical path, rounds x ceil(K blocks / split), with half a block charged
// per round for the cross-CTA reduction; max_clusters(s) is how many
// clusters of s CTAs can be resident at once.
struct W8A16DecodePlan {
  int split;
  int clusters;
};
template <class MaxClusters>
W8A16DecodePlan w8a16_decode_plan(int N, int K, int num_sms, MaxClusters max_clusters) {
  const int n_tiles = N / kW8A16TileN;
  const int kblocks = K / 128;
  W8A16DecodePlan best{1, n_tiles < num_sms ? n_tiles : num_sms};
  long long best_cost = 2LL * ((n_tiles + num_sms - 1) / num_sms) * kblocks;
  for (int s = 2; s <= kMaxSplitK && s <= kblocks; s *= 2) {
    const int c = max_clusters(s);
    if (c <= 0) continue;
    const long long rounds = (n_tiles + c - 1) / c;
    const long long cost = rounds * (2LL * ((kblocks + s - 1) / s) + 1);
    if (cost < best_cost) {
      best_cost = cost;
      best = W8A16DecodePlan{s, n_tiles < c ? n_tiles : c};
    }
  }
  return best;
}

}  // namespace fp8blk
