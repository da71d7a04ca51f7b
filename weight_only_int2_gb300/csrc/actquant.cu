// Per-token dynamic int8 activation quantization.
//
// "int8 activations (W4A8) are now a one-flag serve-time knob ...", section
// "Under the hood": activations are quantized per token to int8 at run time.
// The page leaves the arithmetic open; this kernel implements the reading the
// library documents: IEEE float32, sx = amax / 127 by correctly rounded
// division, xq = clamp(round_half_even(x / sx), -127, 127) with x / sx also a
// correctly rounded division, and sx = 0, xq = 0 for an all-zero row.
//
// One CTA per token row; the row is read twice (the second pass hits L2).
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 256;

// kBf16Codes: write each code as a bf16 value (exact, |q| <= 127) instead of
// int8, for the W4A8 tensor-core GEMM whose operands are bf16, and in the K
// order of its weight operand: within each block of 8 columns the codes of
// columns 0, 4, 1, 5, 2, 6, 3, 7 (the kernel pairs 4-bit weight codes k and
// k + 4 of a word; any order shared by both operands gives the same sums).
template <bool kBf16Codes>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint16_t* __restrict__ x,
                                                            int64_t K, void* __restrict__ xq_out,
                                                            float* __restrict__ sx) {
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * K);
  const int64_t chunks = K / 8;  // 8 bf16 per 16-byte chunk

  float amax = 0.0f;
  for (int64_t i = threadIdx.x; i < chunks; i += kThreads) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  __shared__ float red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);

  const float s = __fdiv_rn(m, 127.0f);
  if (threadIdx.x == 0) sx[row] = s;

  for (int64_t i = threadIdx.x; i < chunks; i += kThreads) {
    int q[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (s > 0.0f) {
      const uint4 v = xr[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t word = w[j >> 1];
        const float f = __uint_as_float((j & 1) ? (word & 0xFFFF0000u) : (word << 16));
        q[j] = max(-127, min(127, __float2int_rn(__fdiv_rn(f, s))));
      }
    }
    if constexpr (kBf16Codes) {
      // small integers convert exactly; bf16 bits are the top half of fp32
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = (__float_as_uint(static_cast<float>(q[j])) >> 16) |
               (__float_as_uint(static_cast<float>(q[j + 4])) & 0xFFFF0000u);
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(xq_out) + row * K)[i] = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) packed[j >> 2] |= (static_cast<uint32_t>(q[j]) & 0xFFu) << (8 * (j & 3));
      reinterpret_cast<uint2*>(static_cast<int8_t*>(xq_out) + row * K)[i] = make_uint2(packed[0], packed[1]);
    }
  }
}

}  // namespace

cudaError_t launch_act_quant(const Ctx& c, const uint16_t* x, int64_t M, int64_t K, int8_t* xq,
                             float* sx) {
  if (M == 0) return cudaSuccess;
  act_quant_kernel<false><<<static_cast<unsigned>(M), kThreads, 0, c.stream>>>(x, K, xq, sx);
  return cudaGetLastError();
}

cudaError_t launch_act_quant_bf16(const Ctx& c, const uint16_t* x, int64_t M, int64_t K, uint16_t* xqb,
                                  float* sx) {
  if (M == 0) return cudaSuccess;
  act_quant_kernel<true><<<static_cast<unsigned>(M), kThreads, 0, c.stream>>>(x, K, xqb, sx);
  return cudaGetLastError();
}

}  // namespace wq
