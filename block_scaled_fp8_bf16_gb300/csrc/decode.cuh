// e4m3 -> bf16 decode by integer operations.
//
// An e4m3 byte s|EEEE|mmm placed in the top byte of a 16-bit half and moved
// right by four bits, with the sign kept at bit 15, is the bf16 pattern of
// the code's value times 2^-120: the exponent field then holds E with bf16's
// bias 127 instead of e4m3's 7, and an e4m3 subnormal (E = 0) becomes the
// bf16 subnormal with the same significand ("FP8 / NVFP4 weight-only
// inference on the RTX 3090 loses nothing", section 4.1: and/shift/or on four
// codes per 32-bit word, bias gap 2^120 for bf16).  One packed bf16 multiply
// by 2^(120 + e) then gives the exact value times 2^e: every e4m3 value has at
// most 4 significant bits, so the product is representable in bf16 for
// e in [-14, 7] ("SM70 FP8 block-32 kernels (PLI Labs)", "Exactness").  The
// 2^120 is applied here, not folded into a later scale, so the tensor cores
// never see subnormal operands.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace fp8blk {

// bf16x2 pattern of 2^(120 + e) in both halves.
__host__ __device__ constexpr uint32_t decode_multiplier_bf16x2(int e) {
  return (static_cast<uint32_t>(127 + 120 + e) << 7) * 0x00010001u;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Four codes (byte i of q is element k0+i) -> two bf16x2 words:
// lo = {k0, k0+1}, hi = {k0+2, k0+3} (lower k in the lower half).
__device__ __forceinline__ void decode4_e4m3_bf16(uint32_t q, uint32_t mul, uint32_t& lo, uint32_t& hi) {
  // r = [b2, b0, b3, b1] (byte 0 first): then bytes 1/3 carry {b0, b1} and
  // bytes 0/2 carry {b2, b3}, each in the top byte of a 16-bit half.
  const uint32_t r = __byte_perm(q, 0u, 0x1302u);
  const uint32_t u = r << 8;
  const uint32_t w01 = (r & 0x80008000u) | ((r & 0x7F007F00u) >> 4);
  const uint32_t w23 = (u & 0x80008000u) | ((u & 0x7F007F00u) >> 4);
  lo = bf16x2_mul(w01, mul);
  hi = bf16x2_mul(w23, mul);
}

}  // namespace fp8blk
