// e4m3 -> bf16 decode by integer operations.
//
// An e4m3 byte s|EEEE|mmm with its magnitude bits moved to bits 10..4 of a
// 16-bit half and its sign to bit 15 is the bf16 pattern of the code's value
// times 2^-120: the exponent field then holds E with bf16's
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

// Byte permute in the default mode: selector nibble bits 0..2 pick a byte of
// {a, b}; bit 3 set replaces that byte by copies of its most significant bit.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four codes (byte i of q is element k0+i) -> two bf16x2 words:
// lo = {k0, k0+1}, hi = {k0+2, k0+3} (lower k in the lower half).
// Each 16-bit half is first built as [sign-replicated byte : code byte]; the
// mask keeps the replicated sign at bit 11 and the seven magnitude bits at
// 6..0, and the shift by four moves them to bit 15 and bits 10..4.  That is
// one permute, one logic operation and one shift per two codes on the
// integer pipe, and one multiply on the floating-point pipe.
__device__ __forceinline__ void decode4_e4m3_bf16(uint32_t q, uint32_t mul, uint32_t& lo, uint32_t& hi) {
  const uint32_t t01 = prmt(q, 0u, 0x9180u);   // [b0, sx(b0), b1, sx(b1)]
  const uint32_t t23 = prmt(q, 0u, 0xB3A2u);   // [b2, sx(b2), b3, sx(b3)]
  lo = bf16x2_mul((t01 & 0x087F087Fu) << 4, mul);
  hi = bf16x2_mul((t23 & 0x087F087Fu) << 4, mul);
}

}  // namespace fp8blk
