// C ABI of the block-scaled FP8 linear layer: argument checks, device facts,
// TMA descriptor cache and dispatch to the kernels.  Every check that can be
// made on the host is made before anything touches the device, so argument
// errors need no GPU and leave every buffer untouched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "fp8blk.h"
#include "internal.h"

namespace fp8blk {
namespace {

// Per-device error word written by kernels whose bounded waits gave up.
__device__ int g_err_word;

constexpr int kMaxDevices = 64;
constexpr int64_t kIntMax = 0x7FFFFFFF;

struct DevState {
  bool init = false;
  fp8blk_status status = FP8BLK_OK;
  DeviceInfo info;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];

fp8blk_status device_info(DeviceInfo& out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return FP8BLK_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& st = g_dev[d];
  if (!st.init) {
    DeviceInfo info;
    if (cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess) {
      return FP8BLK_ERR_CUDA;
    }
    if (info.cc_major != 10 || info.cc_minor != 3) {
      st.status = FP8BLK_ERR_ARCH;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return FP8BLK_ERR_CUDA;
      info.err_word = static_cast<int*>(p);
      st.status = FP8BLK_OK;
    }
    st.info = info;
    st.init = true;
  }
  out = st.info;
  return st.status;
}

// ------------------------------------------------------------------ TMA descriptors

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

struct MapKey {
  int device;
  int dtype;
  const void* ptr;
  uint64_t inner, outer, stride_bytes;
  uint32_t box_inner, box_outer;
  int swizzle;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};

constexpr int kCacheSize = 64;
MapEntry g_cache[kCacheSize];
int g_cache_next = 0;
std::mutex g_cache_mu;

// 2-D tiled map, zero fill outside the tensor; 128-byte swizzle unless told otherwise.
fp8blk_status make_map(CUtensorMap& out, CUtensorMapDataType dtype, const void* ptr, uint64_t inner, uint64_t outer,
                       uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128 = true) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8BLK_ERR_CUDA;
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.device = dev;
  key.dtype = int(dtype);
  key.ptr = ptr;
  key.inner = inner;
  key.outer = outer;
  key.stride_bytes = stride_bytes;
  key.box_inner = box_inner;
  key.box_outer = box_outer;
  key.swizzle = swizzle128 ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    for (int i = 0; i < kCacheSize; ++i) {
      if (g_cache[i].used && g_cache[i].key == key) {
        out = g_cache[i].map;
        return FP8BLK_OK;
      }
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return FP8BLK_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = fn(&m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FP8BLK_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    MapEntry& e = g_cache[g_cache_next];
    g_cache_next = (g_cache_next + 1) % kCacheSize;
    e.key = key;
    e.map = m;
    e.used = true;
  }
  out = m;
  return FP8BLK_OK;
}

// ------------------------------------------------------------------ checks

constexpr uint32_t kKnownFlags = FP8BLK_FLAG_PDL | FP8BLK_FLAG_OUT_F32;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline fp8blk_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8BLK_OK : FP8BLK_ERR_CUDA; }

fp8blk_status check_w8a16_args(const void* x, int64_t ldx, const void* b, int64_t ldb, const void* sc, int fmt,
                               const void* c, int64_t ldc, int64_t M, int64_t N, int64_t K, int64_t c_elem) {
  if (M < 0 || N < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (fmt != FP8BLK_SCALE_F32_128x128 && fmt != FP8BLK_SCALE_UE8M0_32x32) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M > kIntMax || N > kIntMax || K > kIntMax) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!x && K > 0) return FP8BLK_ERR_INVALID_ARG;
  if ((!b || !sc) && K > 0) return FP8BLK_ERR_INVALID_ARG;
  if (!c) return FP8BLK_ERR_INVALID_ARG;
  if (ldx < K || ldb < K || ldc < N) return FP8BLK_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (b && !aligned16(b)) || (sc && !aligned16(sc)) || !aligned16(c))
    return FP8BLK_ERR_MISALIGNED;
  if ((ldx * 2) % 16 != 0 || ldb % 16 != 0 || (ldc * c_elem) % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  return FP8BLK_OK;
}

fp8blk_status zero_output(void* c, int64_t ldc, int64_t M, int64_t N, int64_t elem, cudaStream_t s) {
  return cuda_status(cudaMemset2DAsync(c, size_t(ldc * elem), 0, size_t(N * elem), size_t(M), s));
}

// One-token products on the CUDA-core GEMV (see gemv_window for when).
fp8blk_status run_gemv(int act, const void* x, const float* a_scales, int64_t lds, const void* b, int64_t ldb,
                       const void* sc, int fmt, void* c, int64_t N, int64_t K, uint32_t flags, const DeviceInfo& dev,
                       cudaStream_t s) {
  GemvArgs g;
  g.x = x;
  g.a_scales = a_scales;
  g.lds = lds;
  g.b = b;
  g.ldb = ldb;
  g.scales = sc;
  g.fmt = fmt;
  g.act = act;
  g.C = c;
  g.N = int(N);
  g.K = int(K);
  g.pdl = (flags & FP8BLK_FLAG_PDL) != 0;
  g.out_f32 = (flags & FP8BLK_FLAG_OUT_F32) != 0;
  g.err = dev.err_word;
  return cuda_status(launch_gemv(g, dev, s));
}

fp8blk_status run_w8a16(const void* x, int64_t ldx, const void* b, int64_t ldb, const void* sc, int fmt, void* c,
                        int64_t ldc, int64_t M, int64_t N, int64_t K, uint32_t flags, cudaStream_t s) {
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  const bool f32 = (flags & FP8BLK_FLAG_OUT_F32) != 0;
  if (K == 0) return zero_output(c, ldc, M, N, f32 ? 4 : 2, s);
  if (gemv_window(M, N, K, dev)) return run_gemv(kGemvActBf16, x, nullptr, 0, b, ldb, sc, fmt, c, N, K, flags, dev, s);
  GemmW8A16Args p;
  p.scales = sc;
  p.fmt = fmt;
  p.C = c;
  p.ldc = ldc;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.pdl = (flags & FP8BLK_FLAG_PDL) != 0;
  p.out_f32 = f32;
  p.err = dev.err_word;
  const bool decode = M <= kW8A16DecodeMaxM;
  const int tile_m = decode ? (M <= 16 ? 16 : 32) : w8a16_pick_tile_m(M, N, fmt, dev.num_sms);
  st = make_map(p.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, uint64_t(K), uint64_t(N), uint64_t(ldb), 128, 128);
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, uint64_t(K), uint64_t(M), uint64_t(ldx) * 2, 64,
                uint32_t(tile_m));
  if (st != FP8BLK_OK) return st;
  p.tile_m = tile_m;
  return cuda_status(decode ? launch_w8a16_decode(p, dev, s) : launch_gemm_w8a16(p, dev, s));
}

// Shared by the plain and the grouped W8A8 entry points; G == 0 means plain.
fp8blk_status run_w8a8(const void* a_e4m3, int64_t lda, const float* a_scales, int64_t lds, const void* b_e4m3,
                       int64_t ldb, const float* b_scales, const int32_t* row_group, int64_t G, void* c_bf16,
                       int64_t ldc, int64_t M, int64_t N, int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || G < 0 || (flags & ~kKnownFlags) != 0) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M > kIntMax || N > kIntMax || K > kIntMax || G * N > kIntMax) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (G > 0 && M % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!c_bf16) return FP8BLK_ERR_INVALID_ARG;
  if (K > 0 && (!a_e4m3 || !a_scales || !b_e4m3 || !b_scales)) return FP8BLK_ERR_INVALID_ARG;
  if (G > 0 && K > 0 && !row_group) return FP8BLK_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N || lds < M) return FP8BLK_ERR_INVALID_ARG;
  if ((a_e4m3 && !aligned16(a_e4m3)) || (a_scales && !aligned16(a_scales)) || (b_e4m3 && !aligned16(b_e4m3)) ||
      (b_scales && !aligned16(b_scales)) || !aligned16(c_bf16) ||
      (row_group && (reinterpret_cast<uintptr_t>(row_group) & 3u) != 0))
    return FP8BLK_ERR_MISALIGNED;
  const int64_t c_elem = (flags & FP8BLK_FLAG_OUT_F32) ? 4 : 2;
  if (lda % 16 != 0 || ldb % 16 != 0 || (ldc * c_elem) % 16 != 0 || lds % 4 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool f32 = (flags & FP8BLK_FLAG_OUT_F32) != 0;
  if (K == 0) return zero_output(c_bf16, ldc, M, N, f32 ? 4 : 2, s);
  if (G == 0 && gemv_window(M, N, K, dev))
    return run_gemv(kGemvActE4m3, a_e4m3, a_scales, lds, b_e4m3, ldb, b_scales, 0, c_bf16, N, K, flags, dev, s);
  const int64_t b_rows = G > 0 ? G * N : N;
  GemmW8A8Args p;
  std::memset(&p.tmX, 0, sizeof(p.tmX));     // read only by the fused form
  st = make_map(p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_e4m3, uint64_t(K), uint64_t(M), uint64_t(lda), 128,
                kW8A8TileM);
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_e4m3, uint64_t(K), uint64_t(b_rows), uint64_t(ldb), 128,
                kW8A8TileN);
  if (st != FP8BLK_OK) return st;
  // Scales are read through the full pitch (lds >= M, a multiple of 4, so
  // 16-byte rows); rows past M are never stored.
  st = make_map(p.tmAs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_scales, uint64_t(lds), uint64_t(K / 128),
                uint64_t(lds) * 4, kW8A8TileM, 1, false);
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmAsG, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_scales, uint64_t(lds), uint64_t(K / 128),
                uint64_t(lds) * 4, kW8A8TileM, 8, false);
  if (st != FP8BLK_OK) return st;
  // Output boxes of 32 rows x 128 bytes (64 bf16 or 32 float32 columns).
  if (f32)
    st = make_map(p.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c_bf16, uint64_t(N), uint64_t(M), uint64_t(ldc) * 4, 32, 32);
  else
    st = make_map(p.tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c_bf16, uint64_t(N), uint64_t(M), uint64_t(ldc) * 2, 64, 32);
  if (st != FP8BLK_OK) return st;
  p.Bs = b_scales;
  p.C = c_bf16;
  p.ldc = ldc;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.pdl = (flags & FP8BLK_FLAG_PDL) != 0;
  p.out_f32 = f32;
  p.row_group = G > 0 ? row_group : nullptr;
  p.groups = G > 0 ? int(G) : 1;
  p.err = dev.err_word;
  return cuda_status(launch_gemm_w8a8(p, dev, s));
}

}  // namespace
}  // namespace fp8blk

using namespace fp8blk;

extern "C" {

fp8blk_status fp8blk_quant_act(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* a_e4m3, int64_t lda,
                               float* a_scales, int64_t lds, fp8blk_stream_t stream) {
  if (M < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || K == 0) return FP8BLK_OK;
  if (!x_bf16 || !a_e4m3 || !a_scales) return FP8BLK_ERR_INVALID_ARG;
  if (ldx < K || lda < K || lds < M) return FP8BLK_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(a_e4m3) || !aligned16(a_scales)) return FP8BLK_ERR_MISALIGNED;
  if ((ldx * 2) % 16 != 0 || lda % 16 != 0 || lds % 4 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  QuantActArgs p;
  st = make_map(p.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_bf16, uint64_t(K), uint64_t(M), uint64_t(ldx) * 2, 128,
                kQuantTileRows, false);
  if (st != FP8BLK_OK) return st;
  p.x = x_bf16;
  p.ldx = ldx;
  p.M = M;
  p.K = K;
  p.a = a_e4m3;
  p.lda = lda;
  p.scales = a_scales;
  p.lds = lds;
  p.err = dev.err_word;
  return cuda_status(launch_quant_act(p, dev, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_gemm_w8a8(const void* a_e4m3, int64_t lda, const float* a_scales, int64_t lds,
                               const void* b_e4m3, int64_t ldb, const float* b_scales, void* c_bf16, int64_t ldc,
                               int64_t M, int64_t N, int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  return run_w8a8(a_e4m3, lda, a_scales, lds, b_e4m3, ldb, b_scales, nullptr, 0, c_bf16, ldc, M, N, K, flags,
                  stream);
}

fp8blk_status fp8blk_linear_w8a8(const void* x_bf16, int64_t ldx, const void* b_e4m3, int64_t ldb,
                                 const float* b_scales, void* c_bf16, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 uint32_t flags, fp8blk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || (flags & ~kKnownFlags) != 0) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0 || M > kW8A8FusedMaxM) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (N > kIntMax || K > kIntMax) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!c_bf16) return FP8BLK_ERR_INVALID_ARG;
  if (K > 0 && (!x_bf16 || !b_e4m3 || !b_scales)) return FP8BLK_ERR_INVALID_ARG;
  if (ldx < K || ldb < K || ldc < N) return FP8BLK_ERR_INVALID_ARG;
  if ((x_bf16 && !aligned16(x_bf16)) || (b_e4m3 && !aligned16(b_e4m3)) || (b_scales && !aligned16(b_scales)) ||
      !aligned16(c_bf16))
    return FP8BLK_ERR_MISALIGNED;
  const bool f32 = (flags & FP8BLK_FLAG_OUT_F32) != 0;
  if ((ldx * 2) % 16 != 0 || ldb % 16 != 0 || (ldc * (f32 ? 4 : 2)) % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return zero_output(c_bf16, ldc, M, N, f32 ? 4 : 2, s);
  if (gemv_window(M, N, K, dev))
    return run_gemv(kGemvActQuant, x_bf16, nullptr, 0, b_e4m3, ldb, b_scales, 0, c_bf16, N, K, flags, dev, s);
  GemmW8A8Args p;
  std::memset(&p.tmA, 0, sizeof(p.tmA));     // not read by the fused form
  std::memset(&p.tmAs, 0, sizeof(p.tmAs));
  std::memset(&p.tmAsG, 0, sizeof(p.tmAsG));
  std::memset(&p.tmC, 0, sizeof(p.tmC));
  st = make_map(p.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_bf16, uint64_t(K), uint64_t(M), uint64_t(ldx) * 2, 64,
                uint32_t(kW8A8FusedMaxM));
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_e4m3, uint64_t(K), uint64_t(N), uint64_t(ldb), 128,
                kW8A8TileN);
  if (st != FP8BLK_OK) return st;
  p.Bs = b_scales;
  p.C = c_bf16;
  p.ldc = ldc;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.pdl = (flags & FP8BLK_FLAG_PDL) != 0;
  p.out_f32 = f32;
  p.fused = true;
  p.err = dev.err_word;
  return cuda_status(launch_gemm_w8a8(p, dev, s));
}

int64_t fp8blk_ue8m0_sf_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0 || K % 128 != 0) return -1;
  const int64_t blocks = (rows + 127) / 128;
  if (K > 0 && blocks > INT64_MAX / 512 / (K / 128)) return -1;
  return blocks * (K / 128) * 512;
}

fp8blk_status fp8blk_quant_act_ue8m0(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* a_e4m3,
                                     int64_t lda, uint8_t* a_sf, fp8blk_stream_t stream) {
  if (M < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || K == 0) return FP8BLK_OK;
  if (!x_bf16 || !a_e4m3 || !a_sf) return FP8BLK_ERR_INVALID_ARG;
  if (ldx < K || lda < K) return FP8BLK_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(a_e4m3) || !aligned16(a_sf)) return FP8BLK_ERR_MISALIGNED;
  if ((ldx * 2) % 16 != 0 || lda % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  QuantActUe8m0Args p{x_bf16, ldx, M, K, a_e4m3, lda, a_sf};
  return cuda_status(launch_quant_act_ue8m0(p, dev, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_ue8m0_weight_sf(const uint8_t* b_exps, int64_t N, int64_t K, uint8_t* b_sf,
                                     fp8blk_stream_t stream) {
  if (N < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (N == 0 || K == 0) return FP8BLK_OK;
  if (!b_exps || !b_sf) return FP8BLK_ERR_INVALID_ARG;
  if (!aligned16(b_exps) || !aligned16(b_sf)) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  return cuda_status(launch_ue8m0_weight_sf(b_exps, N, K, b_sf, dev, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_gemm_w8a8_ue8m0(const void* a_e4m3, int64_t lda, const uint8_t* a_sf, const void* b_e4m3,
                                     int64_t ldb, const uint8_t* b_sf, void* c, int64_t ldc, int64_t M, int64_t N,
                                     int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || (flags & ~kKnownFlags) != 0) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M > kIntMax || N > kIntMax || K > kIntMax) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!c) return FP8BLK_ERR_INVALID_ARG;
  if (K > 0 && (!a_e4m3 || !a_sf || !b_e4m3 || !b_sf)) return FP8BLK_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N) return FP8BLK_ERR_INVALID_ARG;
  if ((a_e4m3 && !aligned16(a_e4m3)) || (a_sf && !aligned16(a_sf)) || (b_e4m3 && !aligned16(b_e4m3)) ||
      (b_sf && !aligned16(b_sf)) || !aligned16(c))
    return FP8BLK_ERR_MISALIGNED;
  const bool f32 = (flags & FP8BLK_FLAG_OUT_F32) != 0;
  if (lda % 16 != 0 || ldb % 16 != 0 || (ldc * (f32 ? 4 : 2)) % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return zero_output(c, ldc, M, N, f32 ? 4 : 2, s);
  GemmW8A8MxArgs p;
  st = make_map(p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_e4m3, uint64_t(K), uint64_t(M), uint64_t(lda), 128, 128);
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_e4m3, uint64_t(K), uint64_t(N), uint64_t(ldb), 128, 128);
  if (st != FP8BLK_OK) return st;
  if (f32)
    st = make_map(p.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, uint64_t(N), uint64_t(M), uint64_t(ldc) * 4, 32, 32);
  else
    st = make_map(p.tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c, uint64_t(N), uint64_t(M), uint64_t(ldc) * 2, 64, 32);
  if (st != FP8BLK_OK) return st;
  // The tiled scale arrays as rows of 128 words (one 512-byte block per row).
  st = make_map(p.tmSfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, a_sf, 128, uint64_t((M + 127) / 128) * uint64_t(K / 128),
                512, 128, 1, false);
  if (st != FP8BLK_OK) return st;
  st = make_map(p.tmSfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, b_sf, 128, uint64_t(N / 128) * uint64_t(K / 128), 512, 128,
                1, false);
  if (st != FP8BLK_OK) return st;
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.C = c;
  p.ldc = ldc;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.pdl = (flags & FP8BLK_FLAG_PDL) != 0;
  p.out_f32 = f32;
  p.err = dev.err_word;
  return cuda_status(launch_gemm_w8a8_mx(p, dev, s));
}

fp8blk_status fp8blk_gemm_w8a8_grouped(const void* a_e4m3, int64_t lda, const float* a_scales, int64_t lds,
                                       const void* b_e4m3, int64_t ldb, const float* b_scales,
                                       const int32_t* row_group, int64_t G, void* c_bf16, int64_t ldc, int64_t M,
                                       int64_t N, int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  if (G < 1) return FP8BLK_ERR_INVALID_ARG;
  return run_w8a8(a_e4m3, lda, a_scales, lds, b_e4m3, ldb, b_scales, row_group, G, c_bf16, ldc, M, N, K, flags,
                  stream);
}

fp8blk_status fp8blk_gemm_w8a16(const void* x_bf16, int64_t ldx, const void* b_e4m3, int64_t ldb,
                                const void* b_scales, fp8blk_scale_fmt fmt, void* c_bf16, int64_t ldc, int64_t M,
                                int64_t N, int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  if ((flags & ~kKnownFlags) != 0) return FP8BLK_ERR_INVALID_ARG;
  fp8blk_status st = check_w8a16_args(x_bf16, ldx, b_e4m3, ldb, b_scales, int(fmt), c_bf16, ldc, M, N, K,
                                      (flags & FP8BLK_FLAG_OUT_F32) ? 4 : 2);
  if (st != FP8BLK_OK || M == 0 || N == 0) return st;
  return run_w8a16(x_bf16, ldx, b_e4m3, ldb, b_scales, int(fmt), c_bf16, ldc, M, N, K, flags,
                   reinterpret_cast<cudaStream_t>(stream));
}

fp8blk_status fp8blk_gemv_w8a16(const void* x_bf16, int64_t ldx, const void* b_e4m3, int64_t ldb,
                                const void* b_scales, fp8blk_scale_fmt fmt, void* c_bf16, int64_t ldc, int64_t M,
                                int64_t N, int64_t K, uint32_t flags, fp8blk_stream_t stream) {
  if ((flags & ~kKnownFlags) != 0) return FP8BLK_ERR_INVALID_ARG;
  fp8blk_status st = check_w8a16_args(x_bf16, ldx, b_e4m3, ldb, b_scales, int(fmt), c_bf16, ldc, M, N, K,
                                      (flags & FP8BLK_FLAG_OUT_F32) ? 4 : 2);
  if (st != FP8BLK_OK) return st;
  if (M > 16) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  return run_w8a16(x_bf16, ldx, b_e4m3, ldb, b_scales, int(fmt), c_bf16, ldc, M, N, K, flags,
                   reinterpret_cast<cudaStream_t>(stream));
}

fp8blk_status fp8blk_quant_weight(const void* w_bf16, int64_t N, int64_t K, int64_t ldw, void* b_e4m3, int64_t ldb,
                                  float* b_scales, fp8blk_stream_t stream) {
  if (N < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (N == 0 || K == 0) return FP8BLK_OK;
  if (!w_bf16 || !b_e4m3 || !b_scales) return FP8BLK_ERR_INVALID_ARG;
  if (ldw < K || ldb < K) return FP8BLK_ERR_INVALID_ARG;
  if (!aligned16(w_bf16) || !aligned16(b_e4m3) || !aligned16(b_scales)) return FP8BLK_ERR_MISALIGNED;
  if ((ldw * 2) % 16 != 0 || ldb % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  QuantWeightArgs p{w_bf16, N, K, ldw, b_e4m3, ldb, b_scales};
  return cuda_status(launch_quant_weight(p, dev, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_validate_weights(const void* b_e4m3, int64_t ldb, const void* b_scales, fp8blk_scale_fmt fmt,
                                      int64_t N, int64_t K, int32_t* dev_counts, fp8blk_stream_t stream) {
  if (N < 0 || K < 0) return FP8BLK_ERR_INVALID_ARG;
  if (fmt != FP8BLK_SCALE_F32_128x128 && fmt != FP8BLK_SCALE_UE8M0_32x32) return FP8BLK_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return FP8BLK_ERR_UNSUPPORTED_SHAPE;
  if (!dev_counts) return FP8BLK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_counts) & 3u) != 0) return FP8BLK_ERR_MISALIGNED;
  if ((N > 0 && K > 0) && (!b_e4m3 || !b_scales)) return FP8BLK_ERR_INVALID_ARG;
  if (ldb < K) return FP8BLK_ERR_INVALID_ARG;
  if ((b_e4m3 && !aligned16(b_e4m3)) || ldb % 16 != 0) return FP8BLK_ERR_MISALIGNED;
  if (b_scales && (reinterpret_cast<uintptr_t>(b_scales) & 3u) != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  ValidateArgs p{b_e4m3, ldb, b_scales, int(fmt), N, K, dev_counts};
  return cuda_status(launch_validate(p, dev, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_debug_decode_e4m3(const void* codes, int64_t n, int32_t exp_shift, void* out_bf16,
                                       fp8blk_stream_t stream) {
  if (n < 0 || n % 4 != 0) return FP8BLK_ERR_INVALID_ARG;
  if (exp_shift < -14 || exp_shift > 7) return FP8BLK_ERR_INVALID_ARG;
  if (n == 0) return FP8BLK_OK;
  if (!codes || !out_bf16) return FP8BLK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 3u) != 0 || (reinterpret_cast<uintptr_t>(out_bf16) & 3u) != 0)
    return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  return cuda_status(launch_debug_decode(codes, n, exp_shift, out_bf16, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_debug_group_scale(const float* amax, int64_t n, float* s_out, float* divisor_out,
                                       float* recip_out, fp8blk_stream_t stream) {
  if (n < 0 || n > kIntMax) return FP8BLK_ERR_INVALID_ARG;
  if (n == 0) return FP8BLK_OK;
  if (!amax || !s_out || !divisor_out || !recip_out) return FP8BLK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) != 0 || (reinterpret_cast<uintptr_t>(s_out) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(divisor_out) & 3u) != 0 || (reinterpret_cast<uintptr_t>(recip_out) & 3u) != 0)
    return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  return cuda_status(
      launch_debug_group_scale(amax, n, s_out, divisor_out, recip_out, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_debug_stream_read(const void* p, int64_t bytes, uint32_t* sink, fp8blk_stream_t stream) {
  if (bytes < 0 || bytes % 16 != 0) return FP8BLK_ERR_INVALID_ARG;
  if (bytes == 0) return FP8BLK_OK;
  if (!p || !sink) return FP8BLK_ERR_INVALID_ARG;
  if (!aligned16(p) || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0) return FP8BLK_ERR_MISALIGNED;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  return cuda_status(launch_debug_stream_read(p, bytes / 16, sink, dev.num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_debug_wait_timeout(int64_t limit_ns, fp8blk_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 100000000) return FP8BLK_ERR_INVALID_ARG;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  return cuda_status(launch_debug_wait_timeout(limit_ns, FP8BLK_DIAG_TIMEOUT_CODE, dev.err_word,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

fp8blk_status fp8blk_query_constraints(fp8blk_constraints* out) {
  if (!out) return FP8BLK_ERR_INVALID_ARG;
  out->abi_version = FP8BLK_ABI_VERSION;
  out->scale_block_k = 128;
  out->scale_block_n = 128;
  out->ue8m0_block = 32;
  out->w8a8_tile_m = kW8A8TileM;
  out->w8a8_tile_n = kW8A8TileN;
  out->w8a16_tile_n = kW8A16TileN;
  out->w8a16_max_tile_m = kW8A16MaxTileM;
  out->gemv_max_m = 16;
  out->ptr_align_bytes = 16;
  out->row_align_bytes = 16;
  out->lds_multiple = 4;
  out->max_split_k = kMaxSplitK;
  return FP8BLK_OK;
}

const char* fp8blk_status_string(fp8blk_status s) {
  switch (s) {
    case FP8BLK_OK: return "ok";
    case FP8BLK_ERR_INVALID_ARG: return "invalid argument";
    case FP8BLK_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP8BLK_ERR_MISALIGNED: return "pointer or row pitch not 16-byte aligned";
    case FP8BLK_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case FP8BLK_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FP8BLK_ERR_NAN_CODE: return "e4m3 NaN code in weights";
    case FP8BLK_ERR_SCALE_WINDOW: return "weight scale out of range";
    case FP8BLK_ERR_TIMEOUT: return "kernel gave up on a pipeline wait";
  }
  return "unknown status";
}

fp8blk_status fp8blk_device_error(int32_t* out_code, int32_t clear) {
  if (!out_code) return FP8BLK_ERR_INVALID_ARG;
  DeviceInfo dev;
  fp8blk_status st = device_info(dev);
  if (st != FP8BLK_OK) return st;
  // Every stream of the device, non-blocking ones included, must have
  // finished before the word is read: a kernel still running on such a
  // stream could record a timeout after the read, or after the clear.
  if (cudaDeviceSynchronize() != cudaSuccess) return FP8BLK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(int)) != cudaSuccess) return FP8BLK_ERR_CUDA;
  *out_code = v;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(int)) != cudaSuccess) return FP8BLK_ERR_CUDA;
  }
  return v ? FP8BLK_ERR_TIMEOUT : FP8BLK_OK;
}

}  // extern "C"
