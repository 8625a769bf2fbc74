// Arithmetic of the 1x128 / 128x128 e4m3 quantisation, shared by the
// stand-alone quantisers (quant.cu) and the W8A8 kernel that quantises its
// activation tiles itself (gemm_w8a8.cu), so that both produce the same
// codes and scales bit for bit.
//
// The scale is s = amax / 448 with IEEE division; the codes are
// e4m3(x / s) with the correctly rounded quotient, round-to-nearest-even and
// saturation to +-448 (cvt.rn.satfinite); amax == 0 gives s = 1.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace fp8blk {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

__device__ __forceinline__ float group_scale(float amax) {
  return amax == 0.f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
}

// Correctly rounded float32 quotient x / s from the correctly rounded
// reciprocal y = RN(1/s) by one Markstein correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x*y) is faithful, the
// residual r = x - q0*s is exact with FMA, and RN(q0 + r*y) is RN(x/s) when
// nothing underflows.
//
// The scale is first brought into [2^-60, 2^64] by exact power-of-two factors
// applied to both operands (the quotient is unchanged); there every quotient
// that can decide an e4m3 code (|x/s| >= 2^-11) keeps q0, r and y normal.
// Quotients below that round to a signed zero code either way.
struct Divisor {
  float s;      // scaled divisor
  float y;      // RN(1 / s)
  float m1, m2; // factors applied to the dividend (1 when s needed no scaling)
  bool scaled;
};

__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d{s, 0.f, 1.f, 1.f, false};
  if (d.s < 0x1p-60f) {
    d.s *= 0x1p64f;
    d.m1 = 0x1p64f;
    d.scaled = true;
    if (d.s < 0x1p-60f) {
      d.s *= 0x1p64f;
      d.m2 = 0x1p64f;
    }
  } else if (d.s > 0x1p64f) {
    d.s *= 0x1p-64f;
    d.m1 = 0x1p-64f;
    d.scaled = true;
  }
  d.y = __frcp_rn(d.s);
  return d;
}

__device__ __forceinline__ float quotient(float x, const Divisor& d) {
  if (d.scaled) x = __fmul_rn(__fmul_rn(x, d.m1), d.m2);
  const float q0 = __fmul_rn(x, d.y);
  const float r = __fmaf_rn(-q0, d.s, x);
  // s > 0, so the quotient has the dividend's sign; this also keeps -0 / s = -0,
  // which the correction step would turn into +0.
  return copysignf(__fmaf_rn(r, d.y, q0), x);
}

}  // namespace fp8blk
