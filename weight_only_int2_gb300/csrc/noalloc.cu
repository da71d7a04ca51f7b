// wna16_gemm_noalloc: the WNA16 linear layer for callers that cannot
// allocate device memory.
//
// Who needs it: a serving engine that reserves (nearly) all device memory up
// front for its KV-cache pool cannot hand this library a workspace buffer on
// the request path -- a cudaMalloc there may fail, stall the device, or take
// memory the engine already promised elsewhere -- and a plain C caller may
// have no allocator or workspace lifetime to manage at all. This entry point
// takes only inputs and outputs; the split-K scratch the GEMM needs lives in a
// fixed array that belongs to the library.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes. Every
// GPU that loads the library holds it until the process exits, and every call
// on a device shares it, so calls whose executions overlap on the GPU race.
// Its first use on a device resolves the array's device address with
// cudaGetSymbolAddress (the array's name is only a host-side stand-in); that
// first call should therefore come before any stream capture.
#include "wq.h"
#include "wq_device.cuh"
#include "wq_internal.h"

#include <mutex>

namespace wq {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

}  // namespace
}  // namespace wq

using namespace wq;

extern "C" wq_status wna16_gemm_noalloc(const wq_bf16* x, int64_t M, const uint32_t* Wpacked,
                                        const wq_bf16* scales, int64_t N, int64_t K, int bits, int group,
                                        wq_bf16* y, void* stream) {
  // The same argument checks as wna16_gemm, plus the scratch limit. A
  // 32..64-token shape that the tensor-core kernel takes needs no scratch;
  // that is known once the device's SM count is.
  size_t need = wna16_workspace_bytes(M, N, K, bits);
  const bool maybe_tc = M >= 32 && M < kPrefillMinTokens && bits >= 2 && bits <= 8 && group == 128 &&
                        prefill_supported(M, N, K, bits);
  if (need > kNoAllocScratchBytes && !maybe_tc) {
    set_error("wna16_gemm_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu-byte array "
              "(use wna16_gemm with a caller-provided workspace)",
              need, kNoAllocScratchBytes);
    return WQ_EINVAL;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("wna16_gemm_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    return WQ_ECUDA;
  }
  if (maybe_tc) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      set_error("wna16_gemm_noalloc: SM count: %s", cudaGetErrorString(e));
      return WQ_ECUDA;
    }
    if (route_wna16(M, N, K, bits, sms) == Route::kTensorCore) need = 0;
    if (need > kNoAllocScratchBytes) {
      set_error("wna16_gemm_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu-byte array "
                "(use wna16_gemm with a caller-provided workspace)",
                need, kNoAllocScratchBytes);
      return WQ_EINVAL;
    }
  }
  if (dev < 0 || dev >= kMaxDev) {
    set_error("wna16_gemm_noalloc: device index %d too large", dev);
    return WQ_EUNSUPPORTED;
  }
  void* ptr = nullptr;
  {
    // Set-up, once per device with that device current: the device address of
    // the scratch array (a kernel given the host-side symbol would fault).
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        set_error("wna16_gemm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return WQ_ECUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    ptr = g_scratch_ptr[dev];
  }
  if (need > 0) {
    // The split-K region must start at zero; clear it rather than rely on the
    // contents left by the previous call.
    e = cudaMemsetAsync(ptr, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      set_error("wna16_gemm_noalloc: clearing the scratch: %s", cudaGetErrorString(e));
      return WQ_ECUDA;
    }
  }
  return wna16_gemm(x, M, Wpacked, scales, N, K, bits, group, y, need > 0 ? ptr : nullptr, need, stream);
}
