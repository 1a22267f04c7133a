// MX element/scale encoding shared by the quantize kernels and the GEMM epilogues
// that emit MX operands directly.
//
// Rule (OCP Microscaling v1.0): amax = max |v| over a 32-element block; E =
// clamp(floor(log2 amax) - emax, -127, 127), emax 8 (e4m3) / 2 (e2m1); scale
// code E + 127; code = RNE(v * 2^-E) saturated to the largest finite value,
// sign of zero kept; a block holding NaN or Inf gets scale 0xFF and zero codes.
// For bf16 inputs floor(log2 amax) is the exponent field minus 127 (zero and
// subnormal amax clamp to E = -127), and v * 2^-E is exact in fp32 for every
// value that can round to a non-zero code, so the conversion instruction's
// single rounding is the rule's rounding.
#pragma once
#include "ptx.cuh"

namespace pgg {

constexpr int kE4M3 = 1;
constexpr int kE2M1 = 2;

template <int FMT>
__device__ __forceinline__ int emax() { return FMT == kE4M3 ? 8 : 2; }

// amax bits (bf16 magnitude bits, ordered as integers) -> (scale code, fp32 multiplier 2^-E);
// returns false for a non-finite block.
template <int FMT>
__device__ __forceinline__ bool block_scale(uint32_t amax_bits, uint32_t& code, float& mult) {
  if (amax_bits >= 0x7F80u) {
    code = 0xFFu;
    mult = 0.0f;
    return false;
  }
  int e = (int)(amax_bits >> 7) - 127 - emax<FMT>();
  e = max(e, -127);  // upper clamp is never reached from bf16 (max exponent 127)
  code = (uint32_t)(e + 127);
  mult = __uint_as_float((uint32_t)(127 - e) << 23);
  return true;
}

// two fp32 -> two e4m3 bytes (lo in the low byte)
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// two fp32 -> one byte of two e2m1 nibbles (lo in the low nibble)
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}


// One 32-element block held by one thread as bf16 bit patterns (v16[j] = bits of
// element j): writes the block's codes (32 bytes e4m3 / 16 bytes e2m1, 16-byte
// aligned) and returns its scale code.
template <int FMT>
__device__ __forceinline__ uint32_t quantize_block32(const uint32_t (&v16)[32], uint8_t* codes) {
  uint32_t am = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) am = max(am, v16[j] & 0x7FFFu);
  uint32_t sc;
  float mult;
  const bool fin = block_scale<FMT>(am, sc, mult);
  float f[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) f[j] = fin ? __uint_as_float(v16[j] << 16) * mult : 0.0f;
  if (FMT == kE4M3) {
    uint4 o[2];
    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ow[k] = cvt_e4m3x2(f[4 * k], f[4 * k + 1]) | (cvt_e4m3x2(f[4 * k + 2], f[4 * k + 3]) << 16);
    reinterpret_cast<uint4*>(codes)[0] = o[0];
    reinterpret_cast<uint4*>(codes)[1] = o[1];
  } else {
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      ow[k] = cvt_e2m1x2(f[8 * k], f[8 * k + 1]) | (cvt_e2m1x2(f[8 * k + 2], f[8 * k + 3]) << 8) |
              (cvt_e2m1x2(f[8 * k + 4], f[8 * k + 5]) << 16) | (cvt_e2m1x2(f[8 * k + 6], f[8 * k + 7]) << 24);
    *reinterpret_cast<uint4*>(codes) = o;
  }
  return sc;
}

// The same block held as 16 words of bf16 pairs (element 2k in the low half of w[k]), as
// the GEMM epilogues store it; the amax is a tree over the pairs (the max is associative,
// so the result is the same as a running max, with a 5-deep dependency chain instead of 32).
template <int FMT>
__device__ __forceinline__ uint32_t quantize_block32_packed(const uint32_t (&w)[16], uint8_t* codes) {
  uint32_t m[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) m[k] = max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu);
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1)
#pragma unroll
    for (int k = 0; k < d; ++k) m[k] = max(m[k], m[k + d]);
  uint32_t sc;
  float mult;
  const bool fin = block_scale<FMT>(m[0], sc, mult);
  float f[32];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    f[2 * k] = fin ? __uint_as_float(w[k] << 16) * mult : 0.0f;
    f[2 * k + 1] = fin ? __uint_as_float(w[k] & 0xFFFF0000u) * mult : 0.0f;
  }
  if (FMT == kE4M3) {
    uint4 o[2];
    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ow[k] = cvt_e4m3x2(f[4 * k], f[4 * k + 1]) | (cvt_e4m3x2(f[4 * k + 2], f[4 * k + 3]) << 16);
    reinterpret_cast<uint4*>(codes)[0] = o[0];
    reinterpret_cast<uint4*>(codes)[1] = o[1];
  } else {
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      ow[k] = cvt_e2m1x2(f[8 * k], f[8 * k + 1]) | (cvt_e2m1x2(f[8 * k + 2], f[8 * k + 3]) << 8) |
              (cvt_e2m1x2(f[8 * k + 4], f[8 * k + 5]) << 16) | (cvt_e2m1x2(f[8 * k + 6], f[8 * k + 7]) << 24);
    *reinterpret_cast<uint4*>(codes) = o;
  }
  return sc;
}

}  // namespace pgg
