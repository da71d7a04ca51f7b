// C ABI of libwq: argument checks, per-device state, TMA descriptors and
// dispatch to the kernels. See include/wq.h for the contract of each call.
#include "wq.h"
#include "wq_device.cuh"
#include "wq_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace wq {

// Per-device status word: kernels record a bounded-wait timeout here.
__device__ unsigned g_status_word;

namespace {

thread_local char t_err[512] = "";

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  unsigned* status = nullptr;
  int sm_count = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

wq_status fail(wq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return s;
}

wq_status cuda_fail(cudaError_t e, const char* where) {
  return fail(WQ_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Fills `c` for the current device; sets up the device's state on first use.
wq_status get_ctx(void* stream, Ctx* c) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WQ_EUNSUPPORTED, "device index %d too large", dev);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_status_word);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
      d.status = static_cast<unsigned*>(p);
      d.sm_count = sms;
      d.ready = true;
    }
    c->status = d.status;
    c->sm_count = d.sm_count;
  }
  c->device = dev;
  c->stream = static_cast<cudaStream_t>(stream);
  return WQ_OK;
}

wq_status check_bits(int bits) {
  if (bits < 2 || bits > 8) return fail(WQ_EINVAL, "bits must be in 2..8 (got %d)", bits);
  return WQ_OK;
}

// Sizes become grid dimensions and 32-bit TMA coordinates: all below 2^31.
constexpr int64_t kMaxDim = 0x7FFFFFFF;
// Experts of one grouped call (each tile looks its expert up in the offsets).
constexpr int kMaxExperts = 1024;

wq_status check_group_k(int group, int64_t K, const char* kname) {
  if (group != 128) return fail(WQ_EUNSUPPORTED, "group must be 128 (got %d)", group);
  if (K <= 0 || K % 128 != 0 || K > kMaxDim)
    return fail(WQ_EINVAL, "%s must be a positive multiple of 128 below 2^31 (got %lld)", kname, (long long)K);
  return WQ_OK;
}

wq_status check_size(int64_t v, const char* name) {
  if (v < 1 || v > kMaxDim) return fail(WQ_EINVAL, "%s must be in 1..2^31-1 (got %lld)", name, (long long)v);
  return WQ_OK;
}

// A split-K workspace: non-NULL, 16-byte aligned, at least `need` bytes.
wq_status check_workspace(const void* workspace, size_t ws_bytes, size_t need) {
  if (workspace == nullptr) return fail(WQ_EINVAL, "workspace is NULL");
  if (!aligned16(workspace)) return fail(WQ_EINVAL, "workspace is not 16-byte aligned");
  if (ws_bytes < need) return fail(WQ_EINVAL, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  return WQ_OK;
}

// The message of a shape no kernel takes.
wq_status no_route(int64_t M, int64_t N, int64_t K) {
  return fail(WQ_EUNSUPPORTED,
              "no kernel takes M = %lld, N = %lld, K = %lld: below the tensor-core kernel's token counts "
              "the streaming kernels take K <= 1048576",
              (long long)M, (long long)N, (long long)K);
}

#define WQ_TRY(expr)            \
  do {                          \
    wq_status _s = (expr);      \
    if (_s != WQ_OK) return _s; \
  } while (0)

#define WQ_PTR(p)                                                         \
  do {                                                                    \
    if ((p) == nullptr) return fail(WQ_EINVAL, "%s is NULL", #p);          \
    if (!aligned16(p)) return fail(WQ_EINVAL, "%s is not 16-byte aligned", #p); \
  } while (0)

}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
}

wq_status wna16_check_args(const uint16_t* x, int64_t M, const uint32_t* Wpacked, const uint16_t* scales,
                           int64_t N, int64_t K, int bits, int group, const uint16_t* y) {
  WQ_TRY(check_bits(bits));
  WQ_TRY(check_group_k(group, K, "K"));
  WQ_TRY(check_size(M, "M"));
  WQ_TRY(check_size(N, "N"));
  WQ_PTR(x);
  WQ_PTR(Wpacked);
  WQ_PTR(scales);
  WQ_PTR(y);
  return WQ_OK;
}

bool maybe_tensor_core(int64_t M, int64_t N, int64_t K, int bits) {
  return M >= 32 && M < kPrefillMinTokens && prefill_supported(M, N, K, bits);
}

wq_status wna16_route(int64_t M, int64_t N, int64_t K, int bits, void* stream, Ctx* c, Route* r, bool zp) {
  WQ_TRY(get_ctx(stream, c));
  *r = zp ? route_wna16_zp(M, N, K, bits, c->sm_count) : route_wna16(M, N, K, bits, c->sm_count);
  if (*r == Route::kNone) return no_route(M, N, K);
  return WQ_OK;
}

wq_status wna16_launch(const Ctx& c, Route r, const uint16_t* x, int64_t M, const uint32_t* Wpacked,
                       const uint16_t* scales, int64_t N, int64_t K, int bits, uint16_t* y, void* workspace,
                       const uint8_t* zeros) {
  GemvArgs a{};
  a.mode = GemvMode::kWna16;
  a.x = x;
  a.packed = Wpacked;
  a.scales = scales;
  a.zeros = zeros;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.y = y;
  a.ws = static_cast<float*>(workspace);
  cudaError_t e = r == Route::kTensorCore ? launch_prefill(c, x, Wpacked, scales, M, N, K, bits, y, zeros)
                                          : launch_routed(c, r, a);
  if (e != cudaSuccess) return t_err[0] ? WQ_ECUDA : cuda_fail(e, "wna16_gemm launch");
  return WQ_OK;
}

static bool ensure_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr) set_error("cuTensorMapEncodeTiled is not available from the driver");
  return g_encode != nullptr;
}

// A descriptor is a pure function of its encoding arguments (the address
// included), so an encoded one can be reused whenever the same arguments
// recur, whatever happened to the memory in between. A call's descriptors are
// looked up in a small table before the driver encodes them: the per-call
// host work of a decode step is then a table lookup instead of two driver
// calls per GEMM.
struct TmapKey {
  const void* base;
  uint64_t cols, rows;
  uint32_t box_cols, box_rows;
  int dtype, swizzle, promo;
  bool operator==(const TmapKey& o) const {
    return base == o.base && cols == o.cols && rows == o.rows && box_cols == o.box_cols &&
           box_rows == o.box_rows && dtype == o.dtype && swizzle == o.swizzle && promo == o.promo;
  }
};
constexpr int kTmapSlots = 256;
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool used;
};
static std::mutex g_tmap_mu;
static TmapEntry g_tmap[kTmapSlots];

static bool encode_2d_cached(CUtensorMap* map, CUtensorMapDataType dt, uint32_t esize, const void* base,
                             uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                             CUtensorMapSwizzle sw, CUtensorMapL2promotion promo, CUresult* res) {
  const TmapKey key{base, cols, rows, box_cols, box_rows, static_cast<int>(dt), static_cast<int>(sw),
                    static_cast<int>(promo)};
  uint64_t h = reinterpret_cast<uintptr_t>(base) * 0x9E3779B97F4A7C15ull;
  h ^= (cols * 31 + rows) * 0xC2B2AE3D27D4EB4Full;
  h ^= (static_cast<uint64_t>(box_cols) << 32 | box_rows) + static_cast<uint64_t>(key.dtype * 7 + key.swizzle);
  const int slot = static_cast<int>((h >> 32) % kTmapSlots);
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    if (g_tmap[slot].used && g_tmap[slot].key == key) {
      *map = g_tmap[slot].map;
      *res = CUDA_SUCCESS;
      return true;
    }
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  *res = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (*res != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  g_tmap[slot] = TmapEntry{key, *map, true};
  return true;
}

bool make_tmap_u32_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint32_t box_cols, uint32_t box_rows, int swizzle_bytes) {
  if (!ensure_encode()) return false;
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (swizzle_bytes != 0) {
    set_error("make_tmap_u32_2d: unsupported swizzle span %d", swizzle_bytes);
    return false;
  }
  CUresult r;
  if (!encode_2d_cached(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, cols, rows, box_cols, box_rows, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, &r)) {
    set_error("cuTensorMapEncodeTiled(u32 %llux%llu box %ux%u) failed: %d", (unsigned long long)cols,
              (unsigned long long)rows, box_cols, box_rows, static_cast<int>(r));
    return false;
  }
  return true;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                       uint32_t box_cols, uint32_t box_rows) {
  if (!ensure_encode()) return false;
  CUresult r;
  if (!encode_2d_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, box_cols, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, &r)) {
    set_error("cuTensorMapEncodeTiled(bf16 %llux%llu box %ux%u) failed: %d", (unsigned long long)cols,
              (unsigned long long)rows, box_cols, box_rows, static_cast<int>(r));
    return false;
  }
  return true;
}

bool make_tmap_bf16_2d_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                             uint32_t box_cols, uint32_t box_rows) {
  if (!ensure_encode()) return false;
  CUresult r;
  if (!encode_2d_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, box_cols, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, &r)) {
    set_error("cuTensorMapEncodeTiled(bf16 %llux%llu box %ux%u) failed: %d", (unsigned long long)cols,
              (unsigned long long)rows, box_cols, box_rows, static_cast<int>(r));
    return false;
  }
  return true;
}

}  // namespace wq

using namespace wq;

extern "C" {

size_t wq_packed_words_per_row(int64_t K, int bits) {
  if (K < 0 || bits < 1 || bits > 32) return 0;
  return static_cast<size_t>((K * bits + 31) / 32);
}

const char* wq_last_error(void) { return t_err; }

const char* wq_version(void) { return "wq 0.1 (sm_103a)"; }

wq_status wna16_repack(const uint8_t* codes, const wq_bf16* scales, int64_t N, int64_t K, int bits,
                       int group, uint32_t* packed, wq_bf16* scales_out, int32_t* bad_count,
                       void* stream) {
  t_err[0] = 0;
  WQ_TRY(check_bits(bits));
  WQ_TRY(check_group_k(group, K, "K"));
  WQ_TRY(check_size(N, "N"));
  WQ_PTR(codes);
  WQ_PTR(scales);
  WQ_PTR(packed);
  WQ_PTR(scales_out);
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  cudaError_t e = launch_repack(c, codes, N, K, bits, packed, bad_count);
  if (e != cudaSuccess) return cuda_fail(e, "repack launch");
  if (scales_out != scales) {
    e = cudaMemcpyAsync(scales_out, scales, static_cast<size_t>(N) * (K / 128) * 2,
                        cudaMemcpyDeviceToDevice, c.stream);
    if (e != cudaSuccess) return cuda_fail(e, "scale copy");
  }
  return WQ_OK;
}

size_t wna16_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits) {
  if (M < 1 || N < 1 || K < 128) return 0;
  return stream_workspace_bytes(M, N, K, bits);
}

wq_status wna16_gemm(const wq_bf16* x, int64_t M, const uint32_t* Wpacked, const wq_bf16* scales,
                     int64_t N, int64_t K, int bits, int group, wq_bf16* y, void* workspace,
                     size_t ws_bytes, void* stream) {
  t_err[0] = 0;
  WQ_TRY(wna16_check_args(x, M, Wpacked, scales, N, K, bits, group, y));
  // The documented size is checked before any device call, except for a
  // 32..64-token shape the tensor-core GEMM may take (known from the SM
  // count); then the route's own need, whatever the query said.
  const size_t need = stream_workspace_bytes(M, N, K, bits);
  if (need > 0 && !maybe_tensor_core(M, N, K, bits)) WQ_TRY(check_workspace(workspace, ws_bytes, need));
  Ctx c{};
  Route r = Route::kNone;
  WQ_TRY(wna16_route(M, N, K, bits, stream, &c, &r));
  const size_t need_r = route_workspace_bytes(r, M, N, K);
  if (need_r > 0) WQ_TRY(check_workspace(workspace, ws_bytes, need_r));
  return wna16_launch(c, r, x, M, Wpacked, scales, N, K, bits, y, workspace);
}

size_t wna16_zp_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits) {
  if (M < 1 || N < 1 || K < 128) return 0;
  return stream_workspace_bytes_zp(M, N, K, bits);
}

wq_status wna16_gemm_zp(const wq_bf16* x, int64_t M, const uint32_t* Wpacked, const wq_bf16* scales,
                        const uint8_t* zeros, int64_t N, int64_t K, int bits, int group, wq_bf16* y,
                        void* workspace, size_t ws_bytes, void* stream) {
  t_err[0] = 0;
  WQ_TRY(wna16_check_args(x, M, Wpacked, scales, N, K, bits, group, y));
  WQ_PTR(zeros);
  const size_t need = stream_workspace_bytes_zp(M, N, K, bits);
  if (need > 0 && !maybe_tensor_core(M, N, K, bits)) WQ_TRY(check_workspace(workspace, ws_bytes, need));
  Ctx c{};
  Route r = Route::kNone;
  WQ_TRY(wna16_route(M, N, K, bits, stream, &c, &r, true));
  const size_t need_r = route_workspace_bytes(r, M, N, K);
  if (need_r > 0) WQ_TRY(check_workspace(workspace, ws_bytes, need_r));
  return wna16_launch(c, r, x, M, Wpacked, scales, N, K, bits, y, workspace, zeros);
}

wq_status wna16_moe_gemm(const wq_bf16* x, int64_t M, const int32_t* expert_offsets, int64_t E,
                         const uint32_t* Wpacked, const wq_bf16* scales, int64_t N, int64_t K, int bits, int group,
                         wq_bf16* y, void* stream) {
  t_err[0] = 0;
  WQ_TRY(check_bits(bits));
  WQ_TRY(check_group_k(group, K, "K"));
  WQ_TRY(check_size(M, "M"));
  WQ_TRY(check_size(N, "N"));
  if (E < 1 || E > kMaxExperts) return fail(WQ_EINVAL, "E must be in 1..%d (got %lld)", kMaxExperts, (long long)E);
  if (E * N > kMaxDim) return fail(WQ_EINVAL, "E * N must be below 2^31 (got %lld)", (long long)(E * N));
  WQ_PTR(x);
  WQ_PTR(Wpacked);
  WQ_PTR(scales);
  WQ_PTR(y);
  if (expert_offsets == nullptr || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
    return fail(WQ_EINVAL, "expert_offsets must be a non-NULL, 4-byte aligned device pointer");
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  cudaError_t e = launch_moe(c, x, expert_offsets, E, Wpacked, scales, M, N, K, bits, y);
  if (e != cudaSuccess) return t_err[0] ? WQ_ECUDA : cuda_fail(e, "wna16_moe_gemm launch");
  return WQ_OK;
}

wq_status act_quant_int8(const wq_bf16* x, int64_t M, int64_t K, int8_t* xq, float* sx,
                         void* stream) {
  t_err[0] = 0;
  WQ_TRY(check_size(M, "M"));
  WQ_TRY(check_group_k(128, K, "K"));
  WQ_PTR(x);
  WQ_PTR(xq);
  WQ_PTR(sx);
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  cudaError_t e = launch_act_quant(c, x, M, K, xq, sx);
  if (e != cudaSuccess) return cuda_fail(e, "act_quant launch");
  return WQ_OK;
}

static size_t al256(size_t v) { return (v + 255) / 256 * 256; }

size_t w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 128) return 0;
  return stream_workspace_bytes(M, N, K, 4);
}

size_t w4a8_scratch_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 128) return 0;
  // codes (int8, or bf16 for the tensor-core path) then the per-token scales
  return al256(static_cast<size_t>(M) * K * 2) + al256(static_cast<size_t>(M) * 4);
}

// W4A8 in full (w4a8_gemm), or its per-group accumulators through the same
// route and kernel (acc != nullptr: wq_debug_w4a8_group_acc).
static wq_status w4a8_body(const wq_bf16* x, int64_t M, const uint32_t* Wpacked4, const wq_bf16* scales,
                           int64_t N, int64_t K, int group, wq_bf16* y, int32_t* acc, void* workspace,
                           size_t ws_bytes, void* scratch, size_t scratch_bytes, void* stream) {
  WQ_TRY(check_group_k(group, K, "K"));
  WQ_TRY(check_size(M, "M"));
  WQ_TRY(check_size(N, "N"));
  WQ_PTR(x);
  WQ_PTR(Wpacked4);
  WQ_PTR(scales);
  if (acc != nullptr) {
    WQ_PTR(acc);
  } else {
    WQ_PTR(y);
  }
  WQ_PTR(scratch);
  const size_t need_s = w4a8_scratch_bytes(M, K);
  if (scratch_bytes < need_s)
    return fail(WQ_EINVAL, "scratch too small: %zu < %zu bytes", scratch_bytes, need_s);
  const size_t need = w4a8_workspace_bytes(M, N, K);
  const bool uses_ws = acc == nullptr;  // the group-accumulator mode needs no split-K partials
  if (uses_ws && need > 0 && !maybe_tensor_core(M, N, K, 4)) WQ_TRY(check_workspace(workspace, ws_bytes, need));
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  const Route r = route_w4a8(M, N, K, c.sm_count);
  if (r == Route::kNone) return no_route(M, N, K);
  const size_t need_r = uses_ws ? route_workspace_bytes(r, M, N, K) : 0;
  if (need_r > 0) {
    WQ_TRY(check_workspace(workspace, ws_bytes, need_r));
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), s0 = reinterpret_cast<uintptr_t>(scratch);
    if (w0 < s0 + need_s && s0 < w0 + need_r) return fail(WQ_EINVAL, "scratch overlaps the workspace");
  }
  uint8_t* sb = static_cast<uint8_t*>(scratch);
  int8_t* xq = reinterpret_cast<int8_t*>(sb);
  float* sx = reinterpret_cast<float*>(sb + al256(static_cast<size_t>(M) * K * 2));
  GemvArgs a{};
  a.mode = acc != nullptr ? GemvMode::kW4a8GroupAcc : GemvMode::kW4a8;
  a.packed = Wpacked4;
  a.scales = scales;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = 4;
  a.y = y;
  a.acc = acc;
  if (r == Route::kDecodePair) {
    // few tokens: the decode kernel quantizes the activations per token in
    // its staging (same arithmetic as act_quant_int8), no separate pass
    a.x = x;
    cudaError_t e = launch_decode2(c, a);
    if (e != cudaSuccess) return t_err[0] ? WQ_ECUDA : cuda_fail(e, "w4a8_gemm launch");
    return WQ_OK;
  }
  if (r == Route::kTensorCore) {
    // many tokens: the codes as exact bf16 values into the tensor-core
    // kernel, which accumulates each group exactly and applies s and sx
    uint16_t* xqb = reinterpret_cast<uint16_t*>(sb);
    cudaError_t e = launch_act_quant_bf16(c, x, M, K, xqb, sx);
    if (e != cudaSuccess) return cuda_fail(e, "act_quant launch");
    e = launch_w4a8_tc(c, xqb, sx, Wpacked4, scales, M, N, K, y, acc);
    if (e != cudaSuccess) return t_err[0] ? WQ_ECUDA : cuda_fail(e, "w4a8_gemm launch");
    return WQ_OK;
  }
  cudaError_t e = launch_act_quant(c, x, M, K, xq, sx);
  if (e != cudaSuccess) return cuda_fail(e, "act_quant launch");
  a.xq = xq;
  a.sx = sx;
  a.ws = static_cast<float*>(workspace);
  e = launch_routed(c, r, a);
  if (e != cudaSuccess) return t_err[0] ? WQ_ECUDA : cuda_fail(e, "w4a8_gemm launch");
  return WQ_OK;
}

wq_status w4a8_gemm(const wq_bf16* x, int64_t M, const uint32_t* Wpacked4, const wq_bf16* scales,
                    int64_t N, int64_t K, int group, wq_bf16* y, void* workspace, size_t ws_bytes,
                    void* scratch, size_t scratch_bytes, void* stream) {
  t_err[0] = 0;
  return w4a8_body(x, M, Wpacked4, scales, N, K, group, y, nullptr, workspace, ws_bytes, scratch, scratch_bytes,
                   stream);
}

wq_status qembed_gather(const int32_t* ids, int64_t T, const uint32_t* Wpacked, const wq_bf16* scales,
                        int64_t V, int64_t D, int bits, int group, wq_bf16* out, int32_t* bad_count,
                        void* stream) {
  t_err[0] = 0;
  WQ_TRY(check_bits(bits));
  WQ_TRY(check_group_k(group, D, "D"));
  if (T < 0 || T > kMaxDim) return fail(WQ_EINVAL, "T must be in 0..2^31-1 (got %lld)", (long long)T);
  WQ_TRY(check_size(V, "V"));
  if (T == 0) return WQ_OK;
  WQ_PTR(ids);
  WQ_PTR(Wpacked);
  WQ_PTR(scales);
  WQ_PTR(out);
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  cudaError_t e = launch_gather(c, ids, T, Wpacked, scales, V, D, bits, out, bad_count);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return WQ_OK;
}

wq_status wq_debug_decode_plan(int64_t M, int64_t N, int64_t K, int bits, int sm_count, int64_t* out14) {
  t_err[0] = 0;
  WQ_PTR(out14);
  if (bits < 2 || bits > 8 || sm_count < 1) return fail(WQ_EINVAL, "bits must be in 2..8 and sm_count >= 1");
  decode2_plan_info(M, N, K, bits, sm_count, out14);
  return WQ_OK;
}

wq_status wq_debug_route(int64_t M, int64_t N, int64_t K, int bits, int w4a8, int sm_count, int* route) {
  t_err[0] = 0;
  if (route == nullptr) return fail(WQ_EINVAL, "route is NULL");
  if (sm_count < 1) return fail(WQ_EINVAL, "sm_count must be >= 1");
  if (w4a8 < 0 || w4a8 > 2) return fail(WQ_EINVAL, "kind must be 0, 1 or 2");
  if (w4a8 == 1) {
    if (bits != 4) return fail(WQ_EINVAL, "W4A8 weights are 4-bit (got bits = %d)", bits);
  } else {
    WQ_TRY(check_bits(bits));
  }
  WQ_TRY(check_group_k(128, K, "K"));
  WQ_TRY(check_size(M, "M"));
  WQ_TRY(check_size(N, "N"));
  const Route r = w4a8 == 1   ? route_w4a8(M, N, K, sm_count)
                  : w4a8 == 2 ? route_wna16_zp(M, N, K, bits, sm_count)
                              : route_wna16(M, N, K, bits, sm_count);
  *route = static_cast<int>(r);
  return WQ_OK;
}

wq_status wq_debug_unpack(const uint32_t* packed, int64_t N, int64_t K, int bits, uint8_t* codes,
                          void* stream) {
  t_err[0] = 0;
  WQ_TRY(check_bits(bits));
  WQ_TRY(check_group_k(128, K, "K"));
  WQ_TRY(check_size(N, "N"));
  WQ_PTR(packed);
  WQ_PTR(codes);
  Ctx c{};
  WQ_TRY(get_ctx(stream, &c));
  cudaError_t e = launch_unpack(c, packed, N, K, bits, codes);
  if (e != cudaSuccess) return cuda_fail(e, "unpack launch");
  return WQ_OK;
}

wq_status wq_debug_w4a8_group_acc(const wq_bf16* x, int64_t M, const uint32_t* Wpacked4, const wq_bf16* scales,
                                  int64_t N, int64_t K, int32_t* acc, void* scratch, size_t scratch_bytes,
                                  void* stream) {
  t_err[0] = 0;
  if (acc == nullptr) return fail(WQ_EINVAL, "acc is NULL");
  return w4a8_body(x, M, Wpacked4, scales, N, K, 128, nullptr, acc, nullptr, 0, scratch, scratch_bytes, stream);
}

wq_status wq_check_status(void) {
  t_err[0] = 0;
  Ctx c{};
  WQ_TRY(get_ctx(nullptr, &c));
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  unsigned v = 0;
  e = cudaMemcpy(&v, c.status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpy(c.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    if (v == kStatusTimeout) return fail(WQ_ETIMEOUT, "a kernel gave up on a pipeline wait");
    return fail(WQ_ECUDA, "device status word %u", v);
  }
  return WQ_OK;
}

}  // extern "C"
