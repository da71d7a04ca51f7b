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
//
// Order of a call: every argument check of wna16_gemm first (nothing is
// enqueued for a call that fails them), then the route and its scratch need,
// then the clearing of that region and the GEMM, both on the caller's stream.
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

wq_status too_big(size_t need) {
  set_error("wna16_gemm_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu-byte array "
            "(use wna16_gemm with a caller-provided workspace)",
            need, kNoAllocScratchBytes);
  return WQ_EINVAL;
}

// The device address of the scratch array on device `dev` (current), looked
// up once per device with that device current.
wq_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDev) {
    set_error("wna16_gemm_noalloc: device index %d too large", dev);
    return WQ_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_error("wna16_gemm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      return WQ_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return WQ_OK;
}

}  // namespace
}  // namespace wq

using namespace wq;

extern "C" wq_status wna16_gemm_noalloc(const wq_bf16* x, int64_t M, const uint32_t* Wpacked,
                                        const wq_bf16* scales, int64_t N, int64_t K, int bits, int group,
                                        wq_bf16* y, void* stream) {
  set_error("");
  // 1. The argument checks of wna16_gemm, before anything touches the device.
  wq_status st = wna16_check_args(x, M, Wpacked, scales, N, K, bits, group, y);
  if (st != WQ_OK) return st;
  // 2. The scratch limit: the documented need when it is known without the
  //    device, else (32..64 tokens, where the tensor-core kernel may take the
  //    shape) the need of the route the device picks.
  const size_t need_q = wna16_workspace_bytes(M, N, K, bits);
  if (need_q > kNoAllocScratchBytes && !maybe_tensor_core(M, N, K, bits)) return too_big(need_q);
  Ctx c{};
  Route r = Route::kNone;
  st = wna16_route(M, N, K, bits, stream, &c, &r);
  if (st != WQ_OK) return st;
  const size_t need = route_workspace_bytes(r, M, N, K);
  if (need > kNoAllocScratchBytes) return too_big(need);
  // 3. Clear the region the route uses (the split-K partials and counters
  //    must start at zero), then run the GEMM on it, both on `stream`.
  void* ptr = nullptr;
  if (need > 0) {
    st = scratch_address(c.device, &ptr);
    if (st != WQ_OK) return st;
    const cudaError_t e = cudaMemsetAsync(ptr, 0, need, c.stream);
    if (e != cudaSuccess) {
      set_error("wna16_gemm_noalloc: clearing the scratch: %s", cudaGetErrorString(e));
      return WQ_ECUDA;
    }
  }
  return wna16_launch(c, r, x, M, Wpacked, scales, N, K, bits, y, ptr);
}

extern "C" wq_status wq_debug_noalloc_scratch(void* buf, size_t bytes, int to_scratch, void* stream) {
  set_error("");
  if (buf == nullptr || (to_scratch != 0 && to_scratch != 1) || bytes > kNoAllocScratchBytes) {
    set_error("wq_debug_noalloc_scratch: buf must be non-NULL, to_scratch 0 or 1, bytes <= %zu",
              kNoAllocScratchBytes);
    return WQ_EINVAL;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("wq_debug_noalloc_scratch: cudaGetDevice: %s", cudaGetErrorString(e));
    return WQ_ECUDA;
  }
  void* ptr = nullptr;
  const wq_status st = scratch_address(dev, &ptr);
  if (st != WQ_OK) return st;
  if (bytes == 0) return WQ_OK;
  e = to_scratch ? cudaMemcpyAsync(ptr, buf, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream))
                 : cudaMemcpyAsync(buf, ptr, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error("wq_debug_noalloc_scratch: copy: %s", cudaGetErrorString(e));
    return WQ_ECUDA;
  }
  return WQ_OK;
}
