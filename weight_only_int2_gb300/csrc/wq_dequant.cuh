// bf16 dequantization of packed code slices, shared by the tensor-core GEMM
// (whose A operand it produces) and the embedding gather (whose output it is).
//
// "vLLM Can Run INT5-7", section 1: the weights are dequantized back to bf16,
// w = s * (q - 2^(b-1)); "Qwen3.8-27B-INT6-Mixed-AutoRound" model card,
// section "Findings": the dense LSB-first rows being read.
#pragma once

#include <stdint.h>

namespace wq {
namespace dq {

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 32 bits of the slice starting at bit p (compile-time p after unrolling).
template <int B>
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[B], int p) {
  const int i = p >> 5, sh = p & 31;
  if (sh == 0) return w[i];
  const uint32_t nx = (i + 1 < B) ? w[i + 1] : 0u;
  return __funnelshift_r(w[i], nx, sh);
}

// One 32-code slice (B packed words, LSB-first) -> 16 words holding the bf16
// pairs RN(s * (q - z)) for codes (2c, 2c+1). Codes are placed in the
// mantissa of bf16 128.0 (0x4300: 7 mantissa bits, unit spacing), so
// (128 + q) - (128 + z) is exact and the scale multiply rounds once.
template <int B>
__device__ __forceinline__ void dequant_slice(const uint32_t (&w)[B], uint32_t s2, uint32_t (&o)[16]) {
  constexpr uint32_t kMagic = 0x43004300u;
  if constexpr (B == 8) {
    // 8-bit codes do not fit 7 mantissa bits: take q & 127 into the mantissa
    // and subtract 256 (bit 7 clear) or 128 (bit 7 set), i.e. q - 128.
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t t = __byte_perm(w[c >> 1], 0u, (c & 1) ? 0x4342u : 0x4140u);
      const uint32_t v = (t & 0x007F007Fu) | kMagic;
      const uint32_t zz = (~t & 0x00800080u) | kMagic;
      o[c] = bf16x2_mul(bf16x2_sub(v, zz), s2);
    }
  } else {
    constexpr uint32_t kM = (1u << B) - 1u;
    constexpr uint32_t kZ = 0x4300u | (1u << (B - 1));  // bf16 of 128 + 2^(B-1)
    constexpr uint32_t kZ2 = kZ | (kZ << 16);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t win = window<B>(w, 2 * c * B);
      const uint32_t v = (win & kM) | ((win << (16 - B)) & (kM << 16)) | kMagic;
      o[c] = bf16x2_mul(bf16x2_sub(v, kZ2), s2);
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// The per-(row, group) constant that dequant_slice_zp subtracts or adds, for
// a zero point zp in [0, 2^B - 1]: B <= 7: bf16 (128 + zp) twice (exact,
// zp < 128); B = 8: bf16 (128 - zp) twice (exact, |128 - zp| <= 128).
template <int B>
__device__ __forceinline__ uint32_t zero_pair(uint32_t zp) {
  uint32_t h;
  if constexpr (B == 8) {
    h = __float_as_uint(128.0f - static_cast<float>(zp)) >> 16;  // an integer: the low half is zero
  } else {
    h = 0x4300u | (zp & ((1u << B) - 1u));
  }
  return h | (h << 16);
}

// As dequant_slice, with a zero point per (row, group) [model card "Findings",
// second bullet: asymmetric groups]: RN(s * (q - zp)), q - zp exact.
// B <= 7: (128 + q) - (128 + zp). B = 8: (q - 128) + (128 - zp), both terms
// and the sum (|q - zp| <= 255) exact in bf16. zc2 = zero_pair<B>(zp).
template <int B>
__device__ __forceinline__ void dequant_slice_zp(const uint32_t (&w)[B], uint32_t s2, uint32_t zc2, uint32_t (&o)[16]) {
  constexpr uint32_t kMagic = 0x43004300u;
  if constexpr (B == 8) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t t = __byte_perm(w[c >> 1], 0u, (c & 1) ? 0x4342u : 0x4140u);
      const uint32_t v = (t & 0x007F007Fu) | kMagic;
      const uint32_t zz = (~t & 0x00800080u) | kMagic;
      o[c] = bf16x2_mul(bf16x2_add(bf16x2_sub(v, zz), zc2), s2);
    }
  } else {
    constexpr uint32_t kM = (1u << B) - 1u;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t win = window<B>(w, 2 * c * B);
      const uint32_t v = (win & kM) | ((win << (16 - B)) & (kM << 16)) | kMagic;
      o[c] = bf16x2_mul(bf16x2_sub(v, zc2), s2);
    }
  }
}

}  // namespace dq
}  // namespace wq
