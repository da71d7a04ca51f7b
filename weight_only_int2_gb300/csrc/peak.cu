// Throughput probe of the warp-level tensor-core instruction (mma.sync) in the
// two forms the W4A8 discussion weighs against each other ("int8 activations
// (W4A8) ...", section "Under the hood": int8 x int8 products accumulated in
// int32, against the bf16 path): m16n8k32 s8 x s8 -> s32 and m16n8k16
// bf16 x bf16 -> f32. Every warp runs kChains independent accumulator chains
// of `iters` instructions on all-ones operands, so each instruction adds K
// (32 or 16) to every accumulator element and each thread's checksum is
// exactly kChains * 4 * K * iters: the probe proves it did the work it is
// timed for. The caller times the launch (CUDA events) and divides the
// operations, blocks * 8 warps * kChains * iters * 2*16*8*K, by the time.
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kChains = 8;
constexpr int kPeakThreads = 256;

template <int kKind>  // 0: s8 m16n8k32 (s32 accumulators), 1: bf16 m16n8k16 (f32 accumulators)
__global__ void __launch_bounds__(kPeakThreads) mma_peak_kernel(int64_t iters, int32_t* out) {
  // all-ones operands: four int8 ones, or two bf16 ones, per register; kept
  // opaque so that the instructions take them from registers each time
  uint32_t one = kKind == 0 ? 0x01010101u : 0x3F803F80u;
  asm volatile("" : "+r"(one));
  int64_t sum = 0;
  if constexpr (kKind == 0) {
    int32_t acc[kChains][4] = {};
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < kChains; ++c)
        asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
            : "r"(one), "r"(one), "r"(one), "r"(one), "r"(one), "r"(one));
    }
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += acc[c][e];
  } else {
    float acc[kChains][4] = {};
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < kChains; ++c)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(acc[c][0]), "+f"(acc[c][1]), "+f"(acc[c][2]), "+f"(acc[c][3])
            : "r"(one), "r"(one), "r"(one), "r"(one), "r"(one), "r"(one));
    }
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += static_cast<int64_t>(acc[c][e]);  // exact: below 2^24
  }
  out[static_cast<int64_t>(blockIdx.x) * kPeakThreads + threadIdx.x] = static_cast<int32_t>(sum);
}

}  // namespace
}  // namespace wq

extern "C" wq_status wq_debug_mma_peak(int kind, int64_t iters, int blocks, int32_t* out, void* stream) {
  using namespace wq;
  set_error("");
  if ((kind != 0 && kind != 1) || iters < 1 || iters > 1000000 || blocks < 1 || blocks > 65535 ||
      out == nullptr) {
    set_error("wq_debug_mma_peak: kind 0 or 1, iters in 1..1000000, blocks in 1..65535, out non-NULL");
    return WQ_EINVAL;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == 0)
    mma_peak_kernel<0><<<blocks, kPeakThreads, 0, s>>>(iters, out);
  else
    mma_peak_kernel<1><<<blocks, kPeakThreads, 0, s>>>(iters, out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("wq_debug_mma_peak launch: %s", cudaGetErrorString(e));
    return WQ_ECUDA;
  }
  return WQ_OK;
}
