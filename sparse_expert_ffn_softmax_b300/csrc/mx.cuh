// OCP microscaling "MXFP8" quantisation on the device: 32 consecutive values share
// one power-of-two scale 2^s (stored as the E8M0 byte s + 127) and each value is the
// FP8 E4M3 code of v / 2^s (sign, 4 exponent bits with bias 7, 3 mantissa bits,
// largest finite magnitude 448). The shared exponent is s = floor(log2(max |v|)) - 8
// (8 is the exponent of E4M3's largest power of two), clamped below at -127; the
// block maximum then scales into [256, 512) and the conversion saturates at 448.
// Lower-precision experts: "Mixture of Experts (MoE)" (learn.starphix.com),
// "Quantization".
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {
namespace mx {

// E8M0 byte of a block whose largest magnitude is amax (fp32, finite): the biased
// exponent field of amax less 8, at least 0 (s = byte - 127). For a normal amax the
// field is floor(log2 amax) + 127; a zero or subnormal amax gives byte 0 (s = -127).
__device__ __forceinline__ uint32_t scale_byte(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 8;
  return e > 0 ? (uint32_t)e : 0u;
}

// 2^-s for the scale byte b (s = b - 127): the fp32 with exponent field 254 - b,
// a normal number for every byte 0 .. 253.
__device__ __forceinline__ float inv_scale(uint32_t b) { return __uint_as_float((254u - b) << 23); }

// Four fp32 values -> four E4M3 codes (round to nearest even, saturating at +-448),
// byte i of the result from v_i. The conversion instruction packs its first source
// into the upper byte of each pair.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v1), "f"(v0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v3), "f"(v2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Byte offset of the scale array inside a region holding `rows` rows of K codes:
// the codes [rows, K] first, the scales [rows, K / 32] from the next 256-byte boundary.
__host__ __device__ __forceinline__ int64_t scale_offset(int64_t rows, int64_t K) {
  return (rows * K + 255) / 256 * 256;
}

}  // namespace mx
}  // namespace moe
