// Repack (int8 codes -> dense LSB-first bitstream) and its inverse.
//
// Layout: "Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section "Findings",
// first bullet: a row of K b-bit codes takes ceil(K*bits/32) 32-bit words and
// codes may straddle words. Code k sits at stream bits [k*b, k*b+b), stream
// bit j being bit j%32 of word j/32. The repack step itself is the "Repack"
// job of "vLLM Quantization", section "How it works".
//
// Work unit: 32 consecutive codes of a row occupy exactly `bits` whole words,
// so one thread turns one 32-byte slice of codes into `bits` output words and
// no two threads touch the same word.
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

template <int B>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ codes,
                                                     int64_t n_units, int64_t units_per_row,
                                                     int64_t K, uint32_t* __restrict__ packed,
                                                     int32_t* __restrict__ bad_count) {
  const int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int bad = 0;
  if (u < n_units) {
    const int64_t row = u / units_per_row;
    const int64_t unit = u - row * units_per_row;
    const uint4* src = reinterpret_cast<const uint4*>(codes + row * K + unit * 32);
    const uint4 v0 = src[0];
    const uint4 v1 = src[1];
    const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    constexpr uint32_t kMask = (1u << B) - 1u;
    uint32_t out[B];
#pragma unroll
    for (int w = 0; w < B; ++w) out[w] = 0u;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const uint32_t q = (in[c >> 2] >> (8 * (c & 3))) & 0xFFu;
      bad += (q > kMask) ? 1 : 0;
      const uint32_t v = q & kMask;
      const int p = c * B;  // stream bit offset inside this unit
      out[p >> 5] |= v << (p & 31);
      if ((p & 31) + B > 32) out[(p >> 5) + 1] |= v >> (32 - (p & 31));
    }
    uint32_t* dst = packed + row * (units_per_row * B) + unit * B;
#pragma unroll
    for (int w = 0; w < B; ++w) dst[w] = out[w];
  }
  if (bad_count != nullptr) {
    const int warp_bad = __reduce_add_sync(0xFFFFFFFFu, bad);
    if ((threadIdx.x & 31) == 0 && warp_bad != 0) atomicAdd(bad_count, warp_bad);
  }
}

template <int B>
__global__ void __launch_bounds__(256) unpack_kernel(const uint32_t* __restrict__ packed,
                                                     int64_t n_units, int64_t units_per_row,
                                                     int64_t K, uint8_t* __restrict__ codes) {
  const int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= n_units) return;
  const int64_t row = u / units_per_row;
  const int64_t unit = u - row * units_per_row;
  const uint32_t* src = packed + row * (units_per_row * B) + unit * B;
  uint32_t w[B + 1];
#pragma unroll
  for (int i = 0; i < B; ++i) w[i] = src[i];
  w[B] = 0u;
  constexpr uint32_t kMask = (1u << B) - 1u;
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = 0u;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int p = c * B;
    const uint32_t win = ((p & 31) == 0) ? w[p >> 5] : __funnelshift_r(w[p >> 5], w[(p >> 5) + 1], p & 31);
    out[c >> 2] |= (win & kMask) << (8 * (c & 3));
  }
  uint4* dst = reinterpret_cast<uint4*>(codes + row * K + unit * 32);
  dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
  dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

}  // namespace

cudaError_t launch_repack(const Ctx& c, const uint8_t* codes, int64_t N, int64_t K, int bits,
                          uint32_t* packed, int32_t* bad_count) {
  const int64_t upr = K / 32;
  const int64_t n_units = N * upr;
  if (n_units == 0) return cudaSuccess;
  const dim3 block(256);
  const dim3 grid(static_cast<unsigned>((n_units + 255) / 256));
  switch (bits) {
#define WQ_CASE(b)                                                                        \
  case b:                                                                                 \
    repack_kernel<b><<<grid, block, 0, c.stream>>>(codes, n_units, upr, K, packed, bad_count); \
    break;
    WQ_CASE(2) WQ_CASE(3) WQ_CASE(4) WQ_CASE(5) WQ_CASE(6) WQ_CASE(7) WQ_CASE(8)
#undef WQ_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_unpack(const Ctx& c, const uint32_t* packed, int64_t N, int64_t K, int bits,
                          uint8_t* codes) {
  const int64_t upr = K / 32;
  const int64_t n_units = N * upr;
  if (n_units == 0) return cudaSuccess;
  const dim3 block(256);
  const dim3 grid(static_cast<unsigned>((n_units + 255) / 256));
  switch (bits) {
#define WQ_CASE(b)                                                                     \
  case b:                                                                              \
    unpack_kernel<b><<<grid, block, 0, c.stream>>>(packed, n_units, upr, K, codes);    \
    break;
    WQ_CASE(2) WQ_CASE(3) WQ_CASE(4) WQ_CASE(5) WQ_CASE(6) WQ_CASE(7) WQ_CASE(8)
#undef WQ_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace wq
