// Bit-unpacking helpers shared by the weight-streaming GEMM kernels: the
// per-width pairing of the 32 codes of a b-word slice into 16 registers of two
// 16-bit floats, the slice loads from shared memory and the warp-level MMA.
//
// Layout being read: "Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section
// "Findings" (dense LSB-first rows of ceil(K*bits/32) words).
#pragma once

#include "wq_device.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace wq {
namespace unpack {

// ---------------------------------------------------------------------------
// Pairing of the 32 codes of a slice into 16 registers.
// {lo, hi, s, o_lo, o_hi}: the window W = slice >> s (bits below the slice
// read as zero) holds code `lo` at bit o_lo and code `hi` at bit 16 + o_hi,
// with o <= (mantissa bits - b). Found by exhaustive search for the fewest
// shifts; every width's table covers each of the 32 codes exactly once.
// ---------------------------------------------------------------------------
struct PairSpec {
  int lo, hi, s, olo, ohi;
};

template <int B>
__host__ __device__ constexpr bool uses_fp16() {
  return !(B == 2 || B == 4);
}

template <int B>
__host__ __device__ constexpr PairSpec pair_spec(int p) {
  if constexpr (B == 2) {
    return PairSpec{16 * (p >> 3) + (p & 7), 16 * (p >> 3) + (p & 7) + 8, 32 * (p >> 3) + 2 * (p & 7), 0, 0};
  } else if constexpr (B == 4) {
    return PairSpec{8 * (p >> 2) + (p & 3), 8 * (p >> 2) + (p & 3) + 4, 32 * (p >> 2) + 4 * (p & 3), 0, 0};
  } else if constexpr (B == 3) {
    constexpr PairSpec t[16] = {{0, 3, -7, 7, 0},    {1, 6, 0, 3, 2},     {2, 7, 0, 6, 5},
                                {4, 8, 5, 7, 3},     {5, 9, 8, 7, 3},     {10, 14, 23, 7, 3},
                                {11, 16, 32, 1, 0},  {12, 17, 32, 4, 3},  {13, 18, 32, 7, 6},
                                {15, 19, 38, 7, 3},  {20, 24, 53, 7, 3},  {21, 25, 56, 7, 3},
                                {22, 27, 64, 2, 1},  {23, 29, 64, 5, 7},  {26, 30, 71, 7, 3},
                                {28, 31, 77, 7, 0}};
    return t[p];
  } else if constexpr (B == 5) {
    constexpr PairSpec t[16] = {{0, 3, -5, 5, 4},    {1, 4, 0, 5, 4},     {2, 5, 5, 5, 4},
                                {6, 9, 25, 5, 4},    {7, 10, 32, 3, 2},   {8, 11, 35, 5, 4},
                                {12, 15, 55, 5, 4},  {13, 17, 64, 1, 5},  {14, 18, 69, 1, 5},
                                {16, 19, 75, 5, 4},  {20, 23, 96, 4, 3},  {21, 24, 100, 5, 4},
                                {22, 25, 105, 5, 4}, {26, 29, 128, 2, 1}, {27, 30, 130, 5, 4},
                                {28, 31, 135, 5, 4}};
    return t[p];
  } else if constexpr (B == 6) {
    constexpr PairSpec t[16] = {{0, 3, 0, 0, 2},     {1, 4, 4, 2, 4},     {2, 5, 10, 2, 4},
                                {6, 8, 32, 4, 0},    {7, 9, 38, 4, 0},    {10, 12, 56, 4, 0},
                                {11, 14, 64, 2, 4},  {13, 15, 74, 4, 0},  {16, 19, 96, 0, 2},
                                {17, 20, 100, 2, 4}, {18, 21, 106, 2, 4}, {22, 24, 128, 4, 0},
                                {23, 25, 134, 4, 0}, {26, 28, 152, 4, 0}, {27, 30, 160, 2, 4},
                                {29, 31, 170, 4, 0}};
    return t[p];
  } else if constexpr (B == 7) {
    constexpr PairSpec t[16] = {{0, 2, -3, 3, 1},     {1, 3, 4, 3, 1},     {4, 6, 25, 3, 1},
                                {5, 7, 32, 3, 1},     {8, 10, 53, 3, 1},   {9, 11, 60, 3, 1},
                                {12, 14, 81, 3, 1},   {13, 15, 88, 3, 1},  {16, 18, 109, 3, 1},
                                {17, 19, 116, 3, 1},  {20, 22, 137, 3, 1}, {21, 23, 144, 3, 1},
                                {24, 26, 165, 3, 1},  {25, 27, 172, 3, 1}, {28, 30, 193, 3, 1},
                                {29, 31, 200, 3, 1}};
    return t[p];
  } else {
    constexpr PairSpec t[16] = {{0, 2, 0, 0, 0},      {1, 3, 6, 2, 2},      {4, 6, 32, 0, 0},
                                {5, 7, 38, 2, 2},     {8, 10, 64, 0, 0},    {9, 11, 70, 2, 2},
                                {12, 14, 96, 0, 0},   {13, 15, 102, 2, 2},  {16, 18, 128, 0, 0},
                                {17, 19, 134, 2, 2},  {20, 22, 160, 0, 0},  {21, 23, 166, 2, 2},
                                {24, 26, 192, 0, 0},  {25, 27, 198, 2, 2},  {28, 30, 224, 0, 0},
                                {29, 31, 230, 2, 2}};
    return t[p];
  }
}

template <int B>
__device__ __forceinline__ uint32_t slice_window(const uint32_t (&w)[B], int s) {
  if (s < 0) return w[0] << (-s);
  const int i = s >> 5, sh = s & 31;
  const uint32_t a = w[i];
  const uint32_t b = (i + 1 < B) ? w[i + 1] : 0u;
  return sh == 0 ? a : __funnelshift_r(a, b, sh);
}

// 32 codes held in B words -> 16 registers of two 16-bit floats MAGIC + q*2^o.
template <int B>
__device__ __forceinline__ void unpack_slice(const uint32_t (&w)[B], uint32_t (&r)[16]) {
  constexpr uint32_t kMagic = uses_fp16<B>() ? 0x64006400u : 0x43004300u;
  constexpr uint32_t kM = (1u << B) - 1u;
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const PairSpec sp = pair_spec<B>(p);
    const uint32_t mask = (kM << sp.olo) | (kM << (16 + sp.ohi));
    r[p] = lop3_and_or(slice_window<B>(w, sp.s), mask, kMagic);
  }
}

// Loads this thread's B words of row `row` of a stage (row pitch 4*B words).
template <int B>
__device__ __forceinline__ void load_slice(const uint32_t* stage, int row, int t, uint32_t (&w)[B]) {
  const uint32_t* src = stage + row * 4 * B + t * B;
  if constexpr (B % 4 == 0) {
#pragma unroll
    for (int i = 0; i < B; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + i);
      w[i] = v.x;
      w[i + 1] = v.y;
      w[i + 2] = v.z;
      w[i + 3] = v.w;
    }
  } else if constexpr (B % 2 == 0) {
#pragma unroll
    for (int i = 0; i < B; i += 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(src + i);
      w[i] = v.x;
      w[i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < B; ++i) w[i] = src[i];
  }
}

template <bool kFp16>
__device__ __forceinline__ void mma16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kFp16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    mma_bf16_16816(c, a0, a1, a2, a3, b0, b1);
  }
}


// ---------------------------------------------------------------------------
// Activation staging. A thread owns slice t (32 consecutive activations) of
// one (token, group); the four lanes of a quad hold the four slices of the
// group. The 16 fragment words follow the code pairing of width B, each value
// pre-scaled by 2^-o of its code (and, for fp16, by a power of two that keeps
// the group below 2^15). `corr` receives MAGIC*sum x 2^-o + z*sum x over the
// whole group and `scale_back` the power of two to undo (quad reductions: all
// 32 lanes of the warp must call this together).
// ---------------------------------------------------------------------------
template <bool kInt8>
__device__ __forceinline__ void load_slice_x(const void* src, bool valid, float (&v)[32]) {
  if (!valid) {
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] = 0.0f;
    return;
  }
  if constexpr (!kInt8) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 q = p[c];
      const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * c + 2 * e] = __uint_as_float(wv[e] << 16);
        v[8 * c + 2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
      }
    }
  } else {
    const int4* p = reinterpret_cast<const int4*>(src);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int4 q = p[c];
      const int wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 16; ++e)
        v[16 * c + e] = static_cast<float>(static_cast<int8_t>((wv[e >> 2] >> (8 * (e & 3))) & 0xFF));
    }
  }
}

template <int B>
__device__ __forceinline__ void make_fragments(const float (&v)[32], uint32_t (&frag)[16], float& corr,
                                               float& scale_back, float& xsum) {
  constexpr bool kF16 = uses_fp16<B>();
  constexpr float kMagic = kF16 ? 1024.0f : 128.0f;
  constexpr float kZero = static_cast<float>(1 << (B - 1));
  float inv = 1.0f;
  scale_back = 1.0f;
  if constexpr (kF16) {
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < 32; ++c) amax = fmaxf(amax, fabsf(v[c]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    // amax < 2^(ebits - 126); scale so that the group stays below 2^15
    const int ebits = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
    const int e = max(0, ebits - 126 - 15);
    inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    scale_back = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  }
  float sum = 0.0f, sum_o = 0.0f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const PairSpec sp = pair_spec<B>(q);
    const float flo = 1.0f / static_cast<float>(1 << sp.olo);
    const float fhi = 1.0f / static_cast<float>(1 << sp.ohi);
    const float xlo = v[sp.lo], xhi = v[sp.hi];
    sum += xlo + xhi;
    sum_o = fmaf(xlo, flo, fmaf(xhi, fhi, sum_o));
    // one paired round-to-nearest conversion per register (lo in the low half)
    if constexpr (kF16) {
      const __half2 h = __floats2half2_rn(xlo * flo * inv, xhi * fhi * inv);
      frag[q] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __nv_bfloat162 h = __floats2bfloat162_rn(xlo, xhi);
      frag[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
  sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
  sum_o += __shfl_xor_sync(0xFFFFFFFFu, sum_o, 1);
  sum_o += __shfl_xor_sync(0xFFFFFFFFu, sum_o, 2);
  corr = fmaf(kMagic, sum_o, kZero * sum);
  xsum = sum;
}

// The same without the plain group sum (symmetric groups only).
template <int B>
__device__ __forceinline__ void make_fragments(const float (&v)[32], uint32_t (&frag)[16], float& corr,
                                               float& scale_back) {
  float xsum;
  make_fragments<B>(v, frag, corr, scale_back, xsum);
}

}  // namespace unpack
}  // namespace wq
