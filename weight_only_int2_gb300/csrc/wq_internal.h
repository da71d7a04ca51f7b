// Host-side declarations shared by the translation units of libwq.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "wq.h"

namespace wq {

// Per-call launch context filled by the C-ABI layer.
struct Ctx {
  cudaStream_t stream;
  unsigned* status;  // device address of this device's status word
  int device;
  int sm_count;
};

// Records a one-line error for wq_last_error() (thread-local).
void set_error(const char* fmt, ...);

// A kernel's dynamic shared-memory limit per device, raised on demand and
// never lowered, under a lock: host threads that launch concurrently never
// see a limit below the one they raised (a lowered limit would fail their
// launch). One instance per kernel instantiation (a static in its launcher).
struct SmemLimit {
  std::mutex mu;
  size_t bytes[64] = {};
};
template <typename Kernel>
cudaError_t raise_smem_limit(SmemLimit& lim, Kernel kern, int device, size_t bytes) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(lim.mu);
  if (lim.bytes[device] >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) lim.bytes[device] = bytes;
  return e;
}

// Builds a 2-D tiled TMA descriptor over a row-major matrix of 32-bit words.
// swizzle_bytes 0 (none), 32, 64 or 128: the shared-memory tile is written
// with that TMA swizzle (16-byte chunk index XOR address bits 7 and up; the
// destination must be aligned to the pattern). Returns false (and records the
// reason) if the driver rejects it.
bool make_tmap_u32_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint32_t box_cols, uint32_t box_rows, int swizzle_bytes = 0);

// Builds a 2-D tiled TMA descriptor over a row-major bf16 matrix (no swizzle).
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                       uint32_t box_cols, uint32_t box_rows);

// Builds a 2-D tiled TMA descriptor over a row-major bf16 matrix with 128-byte
// swizzling (box inner extent of 64 elements).
bool make_tmap_bf16_2d_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                             uint32_t box_cols, uint32_t box_rows);

// ---- launchers (return cudaSuccess or the launch error) ----------------------

cudaError_t launch_repack(const Ctx& c, const uint8_t* codes, int64_t N, int64_t K, int bits,
                          uint32_t* packed, int32_t* bad_count);

cudaError_t launch_unpack(const Ctx& c, const uint32_t* packed, int64_t N, int64_t K, int bits,
                          uint8_t* codes);

cudaError_t launch_act_quant(const Ctx& c, const uint16_t* x, int64_t M, int64_t K, int8_t* xq,
                             float* sx);

// Same quantization, codes written as bf16 values (exact) for the W4A8
// tensor-core GEMM, in its K order: within each block of 8 columns the codes
// of columns 0, 4, 1, 5, 2, 6, 3, 7.
cudaError_t launch_act_quant_bf16(const Ctx& c, const uint16_t* x, int64_t M, int64_t K, uint16_t* xqb,
                                  float* sx);

cudaError_t launch_gather(const Ctx& c, const int32_t* ids, int64_t T, const uint32_t* packed,
                          const uint16_t* scales, int64_t V, int64_t D, int bits, uint16_t* out,
                          int32_t* bad_count);

// Weight-streaming GEMM (warp MMA, split-K). Modes of the same main loop.
enum class GemvMode { kWna16 = 0, kW4a8 = 1, kW4a8GroupAcc = 2 };

struct GemvArgs {
  GemvMode mode;
  const uint16_t* x;   // kWna16: bf16 activations [M, K]
  const int8_t* xq;    // W4A8 modes: int8 activations [M, K]
  const float* sx;     // kW4a8: per-token scale [M]
  const uint32_t* packed;
  const uint16_t* scales;
  const uint8_t* zeros;  // kWna16, asymmetric groups: zero points [N, K/128], or null
  int64_t M, N, K;
  int bits;
  uint16_t* y;         // bf16 [M, N] (kWna16, kW4a8)
  int32_t* acc;        // int32 [M, N, K/128] (kW4a8GroupAcc)
  float* ws;           // fp32 [M, N] split-K partials (zero at rest)
  uint32_t* counters;  // split-K arrival counters (zero at rest)
};

// Workspace bytes the weight-streaming GEMM needs for this shape.
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Whether the chunked kernel takes K: a CTA keeps the scales of its groups in
// shared memory, at most 128 groups, and a longer K splits over up to 64
// CTAs (K <= 1048576).
bool gemv_supported(int64_t K);

cudaError_t launch_gemv(const Ctx& c, const GemvArgs& a);

// Persistent decode kernel (M <= 16, K a multiple of 1024).
bool decode_supported(int64_t M, int64_t N, int64_t K, int bits, int sm_count);
size_t decode_workspace_bytes(int64_t M, int64_t N);
cudaError_t launch_decode(const Ctx& c, const GemvArgs& a);

// Tensor-core GEMM for many tokens (tcgen05, dequantize-then-multiply).
constexpr int64_t kPrefillMinTokens = 65;
bool prefill_supported(int64_t M, int64_t N, int64_t K, int bits);
// zeros: asymmetric groups, uint8 [N, K/128] zero points (low `bits` bits
// used), or nullptr for the symmetric zero point 2^(bits-1).
cudaError_t launch_prefill(const Ctx& c, const uint16_t* x, const uint32_t* packed, const uint16_t* scales,
                           int64_t M, int64_t N, int64_t K, int bits, uint16_t* y, const uint8_t* zeros);

// Mixture of experts on the same kernel: tokens sorted by expert, expert e
// owning rows [offsets[e], offsets[e+1]) of x [M, K] and y [M, N] (offsets: a
// device array of E + 1 values, clamped into [0, M] by the kernel); its
// weights are rows e N .. e N + N - 1 of the stacked packed [E N, words] and
// scales [E N, K/128].
cudaError_t launch_moe(const Ctx& c, const uint16_t* x, const int32_t* offsets, int64_t E, const uint32_t* packed,
                       const uint16_t* scales, int64_t M, int64_t N, int64_t K, int bits, uint16_t* y);

// W4A8 on the tensor cores with exact per-group integer accumulation
// (w4a8tc.cu): xqb holds the per-token int8 codes as bf16 values [M, K] and sx
// the token scales [M]; writes y [M, N], or with acc != nullptr the group
// accumulators acc [M, N, K/128] (int32) instead.
cudaError_t launch_w4a8_tc(const Ctx& c, const uint16_t* xqb, const float* sx, const uint32_t* packed4,
                           const uint16_t* scales, int64_t M, int64_t N, int64_t K, uint16_t* y, int32_t* acc);

// From kPrefillMinTokens tokens on, always; from 32 tokens when the layer has
// at least one 128-row tile per two SMs. Measured at K = 5120 (b = 5..7): the
// tensor-core kernel takes ~41-43 us for any M in 17..64 (one CTA dequantizes
// a whole row tile), the streaming kernel 41-46 us at M = 17..32 and 80 us at
// M = 64 for 17408 rows, but 21-37 us for 5120 rows (40 tiles: 112 SMs idle
// in the tensor-core kernel). The workspace queries keep sizing the
// streaming kernel below kPrefillMinTokens, an upper bound either way.
inline bool use_prefill(int64_t M, int64_t N, int64_t K, int bits, int sm_count) {
  if (!prefill_supported(M, N, K, bits)) return false;
  if (M >= kPrefillMinTokens) return true;
  return M >= 32 && 2 * ((N + 127) / 128) >= sm_count;
}

// Decode by CTA pairs (M <= 16, K % 1024 == 0): no workspace, no grid-wide
// synchronisation. Mode kWna16 (bf16 x), or kW4a8 with a.x the bf16
// activations, which the kernel quantizes per token itself.
bool decode2_shape(int64_t M, int64_t K);
// Whether the pair kernel takes this shape whatever the device's SM count (>= 2).
// zp: asymmetric groups (the plan also keeps the plain group sums of x).
bool decode2_fits_any(int64_t M, int64_t N, int64_t K, int bits, bool zp = false);
// The CTA-pair decode plan for a shape, for host-side checks: out[14] =
// {ok, C, H, nchunk, T, ksplit, NS, G, Gh, sbox, sx0, NT, smem bytes, max ring slots}.
int decode2_plan_info(int64_t M, int64_t N, int64_t K, int bits, int sm_count, int64_t* out);
bool decode2_supported(int64_t M, int64_t N, int64_t K, int bits, int sm_count, bool zp = false);
cudaError_t launch_decode2(const Ctx& c, const GemvArgs& a);

// The kernel a GEMM call launches, by shape (host only). The entry points
// dispatch on it and wq_debug_route reports it; the values are the header's
// WQ_ROUTE_* numbers.
// kNone: no kernel takes the shape (the entry points return WQ_EUNSUPPORTED).
enum class Route : int { kNone = 0, kDecodePair = 1, kDecodeSplitK = 2, kChunked = 3, kTensorCore = 4 };

inline Route route_stream(int64_t M, int64_t N, int64_t K, int bits, int sm_count, bool pair_ok) {
  if (pair_ok && decode2_supported(M, N, K, bits, sm_count)) return Route::kDecodePair;
  if (decode_supported(M, N, K, bits, sm_count)) return Route::kDecodeSplitK;
  return gemv_supported(K) ? Route::kChunked : Route::kNone;
}

inline Route route_wna16(int64_t M, int64_t N, int64_t K, int bits, int sm_count) {
  if (use_prefill(M, N, K, bits, sm_count)) return Route::kTensorCore;
  return route_stream(M, N, K, bits, sm_count, true);
}

// Asymmetric groups (a zero point per row and group): the kernels of
// route_wna16 but the persistent split-K decode kernel, which has no
// zero-point mode; the chunked kernel takes those shapes.
inline Route route_wna16_zp(int64_t M, int64_t N, int64_t K, int bits, int sm_count) {
  if (use_prefill(M, N, K, bits, sm_count)) return Route::kTensorCore;
  if (decode2_supported(M, N, K, bits, sm_count, true)) return Route::kDecodePair;
  return gemv_supported(K) ? Route::kChunked : Route::kNone;
}

// W4A8: the pair kernel quantizes few tokens itself; for many tokens the codes
// go as exact bf16 values into the W4A8 tensor-core kernel (w4a8tc.cu, exact
// per-group accumulation); otherwise int8 codes feed the split-K streaming
// kernels.
inline Route route_w4a8(int64_t M, int64_t N, int64_t K, int sm_count) {
  if (decode2_supported(M, N, K, 4, sm_count)) return Route::kDecodePair;
  if (use_prefill(M, N, K, 4, sm_count)) return Route::kTensorCore;
  return route_stream(M, N, K, 4, sm_count, false);
}

// Launches a streaming route (every route but the tensor-core one, whose
// kernel takes other arguments).
inline cudaError_t launch_routed(const Ctx& c, Route r, const GemvArgs& a) {
  switch (r) {
    case Route::kDecodePair: return launch_decode2(c, a);
    case Route::kDecodeSplitK: return launch_decode(c, a);
    case Route::kChunked: return launch_gemv(c, a);
    default: return cudaErrorInvalidValue;
  }
}

// Workspace a route uses: the split-K partials and counters of the streaming
// kernels; none for the pair kernel and the tensor-core GEMM.
inline size_t route_workspace_bytes(Route r, int64_t M, int64_t N, int64_t K) {
  if (r == Route::kChunked) return gemv_workspace_bytes(M, N, K);
  if (r == Route::kDecodeSplitK) return decode_workspace_bytes(M, N);
  return 0;
}

// The workspace query, without the SM count: zero when no SM count sends the
// shape to a streaming kernel (65 or more tokens, or a shape the pair kernel
// takes on every device); otherwise enough for either streaming kernel, an
// upper bound for 32..64 tokens, which the tensor-core GEMM takes on layers
// with a 128-row tile for every two SMs.
inline size_t stream_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits) {
  if (M >= kPrefillMinTokens && prefill_supported(M, N, K, bits)) return 0;
  if (decode2_fits_any(M, N, K, bits)) return 0;
  const size_t a = gemv_workspace_bytes(M, N, K), b = decode_workspace_bytes(M, N);
  return a > b ? a : b;
}

// The same query for asymmetric groups (route_wna16_zp): no split-K decode
// kernel, and the pair kernel's plan keeps the group sums of x as well.
inline size_t stream_workspace_bytes_zp(int64_t M, int64_t N, int64_t K, int bits) {
  if (M >= kPrefillMinTokens && prefill_supported(M, N, K, bits)) return 0;
  if (decode2_fits_any(M, N, K, bits, true)) return 0;
  return gemv_workspace_bytes(M, N, K);
}

// ---- the WNA16 entry point in steps (api.cu), shared by wna16_gemm and the
// allocation-free variant so that both validate and route identically ----

// Every argument check that needs no device call (bits, group, sizes,
// pointers); records the message and returns WQ_EINVAL/WQ_EUNSUPPORTED.
wq_status wna16_check_args(const uint16_t* x, int64_t M, const uint32_t* Wpacked, const uint16_t* scales, int64_t N,
                     int64_t K, int bits, int group, const uint16_t* y);
// A 32..64-token shape that the tensor-core kernel may take (decided with the
// SM count): its workspace is checked only if the route turns out to use it.
bool maybe_tensor_core(int64_t M, int64_t N, int64_t K, int bits);
// The device context and the kernel the shape takes (device queries, no
// launch); WQ_EUNSUPPORTED when no kernel takes it.
// zp: the call has zero points (route_wna16_zp).
wq_status wna16_route(int64_t M, int64_t N, int64_t K, int bits, void* stream, Ctx* c, Route* r, bool zp = false);
// Launches route r (arguments already checked; workspace as the route needs;
// zeros null for symmetric groups).
wq_status wna16_launch(const Ctx& c, Route r, const uint16_t* x, int64_t M, const uint32_t* Wpacked,
                       const uint16_t* scales, int64_t N, int64_t K, int bits, uint16_t* y, void* workspace,
                       const uint8_t* zeros = nullptr);

}  // namespace wq
