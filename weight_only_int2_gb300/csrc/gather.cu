// Quantized embedding gather on the dense layout, any bit width 2..8.
//
// "vLLM Can Run INT5-7", section 3, and the "Qwen3.8-27B-INT6-Mixed-AutoRound"
// model card, section "Findings", first bullet: the embedding path is a
// dequantize-and-gather of table rows, and the word-aligned kernel the card
// describes cannot read widths that do not divide 32. This kernel reads the
// dense ceil(D*bits/32)-word rows directly, so every width works.
//
// out[t, d] = bf16_RNE(float(s[id, d/128]) * float(q[id, d] - 2^(bits-1))).
// The float32 product is exact, so one bf16 rounding of it is the definition.
// It is computed as in the tensor-core GEMM's dequant: the codes in the
// mantissa of bf16 128.0, an exact sub.bf16x2 of 128 + z, and a mul.bf16x2 by
// the scale, which rounds the exact product once (no int-to-float
// conversions); q == zero point with a negative scale yields -0.0.
//
// One CTA per token. Thread u reads the b words of its 32-code slices u,
// u + 128, ... straight from global memory (the warp's loads cover one
// contiguous span of the row, in the widest loads the alignment of u * b
// words allows), all of a pass before expanding any, and writes 64 output
// bytes per slice. No shared-memory staging of the input: any row length
// works.
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_dequant.cuh"

namespace wq {
namespace {

constexpr int kThreads = 128;
// Slices a thread loads before expanding any. A token's row is one round trip
// to memory after its id's (D = 5120: 160 slices, at most two per thread);
// measured at T = 4096: 13.1 us against 13.8 with one slice in flight, and
// 64- or 32-thread CTAs with three or five slices per thread (more tokens in
// flight per SM) are slower (14.4, 15.0 us).
constexpr int kPerPass = 2;
constexpr size_t kStageMaxBytes = 48 * 1024;  // rows staged whole (no opt-in needed)

// Words u * B .. u * B + B - 1 of a row (the row starts 16-byte aligned).
template <int B>
__device__ __forceinline__ void load_slice_words(const uint32_t* __restrict__ row, int64_t u, uint32_t (&w)[B + 1]) {
  const uint32_t* src = row + u * B;
  if constexpr (B % 4 == 0) {
#pragma unroll
    for (int i = 0; i < B; i += 4) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + i));
      w[i] = v.x, w[i + 1] = v.y, w[i + 2] = v.z, w[i + 3] = v.w;
    }
  } else if constexpr (B % 2 == 0) {
#pragma unroll
    for (int i = 0; i < B; i += 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(src + i));
      w[i] = v.x, w[i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < B; ++i) w[i] = __ldg(src + i);
  }
  w[B] = 0u;
}

// Shared -> global bulk copy of `bytes` (a multiple of 16, both addresses
// 16-byte aligned), and the wait until it has read its shared-memory source.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_store_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// kStage: the output row is assembled in shared memory and written by one
// bulk copy (rows up to kStageMaxBytes), instead of four 16-byte stores per
// slice per thread, which fill the SM's global-memory instruction queue.
template <int B, bool kStage>
__global__ void __launch_bounds__(kThreads) gather_kernel(
    const int32_t* __restrict__ ids, const uint32_t* __restrict__ packed,
    const uint16_t* __restrict__ scales, int64_t V, int64_t D, uint16_t* __restrict__ out,
    int32_t* __restrict__ bad_count) {
  extern __shared__ __align__(128) uint4 sout[];
  const int64_t t = blockIdx.x;
  const int64_t id = ids[t];
  const int64_t units = D / 32;
  uint4* orow = reinterpret_cast<uint4*>(out + t * D);

  if (id < 0 || id >= V) {  // the whole CTA
    for (int64_t u = threadIdx.x; u < units; u += kThreads) {
#pragma unroll
      for (int j = 0; j < 4; ++j) orow[u * 4 + j] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (threadIdx.x == 0 && bad_count != nullptr) atomicAdd(bad_count, 1);
    return;
  }

  const uint32_t* prow = packed + id * units * B;
  const uint16_t* srow = scales + id * (D / 128);
  uint4* dst = kStage ? sout : orow;
  // kPerPass slices per thread and pass, all loaded before any is expanded,
  // so that a row of up to kPerPass * kThreads slices costs one round trip
  // to memory after the id's
  for (int64_t u0 = threadIdx.x; u0 < units; u0 += kPerPass * kThreads) {
    uint32_t win[kPerPass][B + 1];
    uint32_t sb[kPerPass];
#pragma unroll
    for (int h = 0; h < kPerPass; ++h) {
      const int64_t u = u0 + h * kThreads;
      if (u < units) {
        load_slice_words<B>(prow, u, win[h]);
        sb[h] = __ldg(srow + (u >> 2));
      }
    }
#pragma unroll
    for (int h = 0; h < kPerPass; ++h) {
      const int64_t u = u0 + h * kThreads;
      if (u < units) {
        uint32_t w[B];
#pragma unroll
        for (int i = 0; i < B; ++i) w[i] = win[h][i];
        uint32_t o[16];
        dq::dequant_slice<B>(w, sb[h] | (sb[h] << 16), o);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[u * 4 + j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      }
    }
  }
  if constexpr (kStage) {
    fence_proxy_async_smem();  // this thread's row bytes, before the copy reads them
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(orow, sout, static_cast<uint32_t>(D * 2));
      bulk_store_wait_read();  // the shared memory stays valid until read
    }
  }
}

template <int B>
cudaError_t launch_b(const Ctx& c, const int32_t* ids, int64_t T, const uint32_t* packed,
                     const uint16_t* scales, int64_t V, int64_t D, uint16_t* out,
                     int32_t* bad_count) {
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  if (row_bytes <= kStageMaxBytes)
    gather_kernel<B, true><<<static_cast<unsigned>(T), kThreads, row_bytes, c.stream>>>(ids, packed, scales, V, D,
                                                                                       out, bad_count);
  else
    gather_kernel<B, false><<<static_cast<unsigned>(T), kThreads, 0, c.stream>>>(ids, packed, scales, V, D, out,
                                                                                bad_count);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const Ctx& c, const int32_t* ids, int64_t T, const uint32_t* packed,
                          const uint16_t* scales, int64_t V, int64_t D, int bits, uint16_t* out,
                          int32_t* bad_count) {
  if (T == 0) return cudaSuccess;
  switch (bits) {
    case 2: return launch_b<2>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 3: return launch_b<3>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 4: return launch_b<4>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 5: return launch_b<5>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 6: return launch_b<6>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 7: return launch_b<7>(c, ids, T, packed, scales, V, D, out, bad_count);
    case 8: return launch_b<8>(c, ids, T, packed, scales, V, D, out, bad_count);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wq
