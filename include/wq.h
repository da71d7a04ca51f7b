/*
 * wq.h -- C ABI of the weight-only quantized linear layer library (libwq.so).
 *
 * The layer computes y = x . dequant(W)^T, where x holds bf16 activations
 * [M, K] and W holds b-bit integer codes (b in 2..8) with one bf16 scale per
 * (output row, 128-wide group along K) and the symmetric zero point 2^(b-1).
 * It also provides the W4A8 variant (per-token int8 activations, int4 codes
 * widened to int8, integer accumulation per group) and the dequantize-and-
 * gather of a quantized embedding table.
 *
 * Sources, cited by page title and section:
 *  [CARD]  "Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section "Findings"
 *          (dense pack-quantized layout of ceil(in_features*bits/32) words per
 *          row; symmetric groups above four bits; the embedding gather).
 *  [INT57] "vLLM Can Run INT5-7", sections 1 and 3 (bit widths 2..8; quantized
 *          embed_tokens / lm_head).
 *  [VQ]    "vLLM Quantization", section "How it works" (create, repack, run).
 *  [W4A8]  "int8 activations (W4A8) are now a one-flag serve-time knob ...",
 *          section "Under the hood" (per-token dynamic int8 activations, int4
 *          weights widened losslessly to int8, negative group scales).
 *
 * Conventions for every call
 *  - bf16 data is passed as raw 16-bit patterns (wq_bf16).
 *  - Every buffer pointer is a DEVICE pointer, owned and allocated by the
 *    caller, 16-byte aligned, row-major and contiguous. The library never
 *    allocates or frees memory and never synchronizes, except in
 *    wq_check_status().
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream);
 *    all work is enqueued asynchronously on it.
 *  - group must be 128 and K (or D) a positive multiple of 128.
 *  - Sizes (M, N, K, T, V, D) are below 2^31; they become grid dimensions and
 *    32-bit TMA coordinates. Larger values return WQ_EINVAL.
 *  - Return codes: WQ_OK, or WQ_EINVAL for bad arguments (returned
 *    synchronously, nothing enqueued), WQ_EUNSUPPORTED for a valid but
 *    unimplemented configuration, WQ_ECUDA when a CUDA call or a launch fails.
 *    wq_last_error() gives a one-line reason for the last failure on the
 *    calling thread.
 *  - Kernels never trap. A pipeline wait that exceeds its bound records
 *    WQ_ETIMEOUT in a per-device status word and the kernel returns early;
 *    wq_check_status() reads and clears that word.
 *
 * Packed layout ("v1", identical to the compressed-tensors dense layout [CARD]):
 *  row n of W is ceil(K*bits/32) little-endian uint32 words; code k occupies
 *  stream bits [k*bits, k*bits + bits), where stream bit j is bit (j % 32) of
 *  word j / 32 (least significant bit first, the bit order of the word-aligned
 *  formula quoted in [CARD]). Because K is a multiple of 128, every
 *  (row, group) block is exactly 16*bits bytes at a 16-byte-aligned offset.
 *  Scales are bf16 [N, K/128].
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WQ_OK = 0,
  WQ_EINVAL = 1,
  WQ_EUNSUPPORTED = 2,
  WQ_ECUDA = 3,
  WQ_ETIMEOUT = 4
} wq_status;

typedef uint16_t wq_bf16; /* raw bf16 bit pattern */

/* Words per packed row: ceil(K * bits / 32) [CARD]. Host-only, never fails
 * (returns 0 for bits outside 1..32 or K < 0). */
size_t wq_packed_words_per_row(int64_t K, int bits);

/* Repack ("Repack: reorder weights into the layout the kernel wants" [VQ]).
 *  codes      [N, K] uint8, one code per byte, expected in [0, 2^bits - 1].
 *  scales     [N, K/128] bf16, any sign [W4A8].
 *  packed     [N, ceil(K*bits/32)] uint32 output in the v1 layout.
 *  scales_out [N, K/128] bf16 output (a copy; may equal `scales`).
 *  bad_count  optional (NULL allowed) device int32; the number of codes above
 *             2^bits - 1 is ADDED to it. Such codes are packed as their low
 *             `bits` bits.
 *  bits in 2..8. */
wq_status wna16_repack(const uint8_t* codes, const wq_bf16* scales, int64_t N, int64_t K,
                       int bits, int group, uint32_t* packed, wq_bf16* scales_out,
                       int32_t* bad_count, void* stream);

/* Bytes of workspace wna16_gemm needs for this shape, without asking the
 * device: 0 when no GPU sends the shape to a split-K streaming kernel (65 or
 * more tokens, or a few-token shape the CTA-pair decode kernel takes whatever
 * the SM count); otherwise enough for either streaming kernel (an upper bound
 * for 32..64 tokens; see wna16_gemm). wq_debug_route names the kernel. */
size_t wna16_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits);

/* WNA16 linear layer [INT57 s.1, CARD]:
 *   y[m, n] = sum_k x[m, k] * s[n, k/128] * (q[n, k] - 2^(bits-1)),
 * float32 accumulation, y rounded to bf16 (round-to-nearest-even).
 *  x        [M, K] bf16.        Wpacked [N, ceil(K*bits/32)] uint32 (v1 layout).
 *  scales   [N, K/128] bf16.    y       [M, N] bf16 output.
 *  workspace, ws_bytes: device scratch of at least wna16_workspace_bytes(),
 *             an upper bound (a 32..64-token shape that runs on the
 *             tensor-core kernel needs none: 32 <= M <= 64 on a layer with a
 *             128-row tile for every two SMs);
 *             it must be zero-filled before its first use and every call that
 *             returns WQ_OK leaves it zero-filled again (a call that fails with
 *             WQ_ECUDA, or whose kernel timed out as wq_check_status reports,
 *             may leave partial sums: zero it before reuse). Calls that may run
 *             concurrently must not share one workspace. May be NULL when the
 *             required size is 0, or when the kernel the call takes uses none;
 *             a call whose kernel uses one returns WQ_EINVAL without it.
 *  Reproducibility: the CTA-pair decode and tensor-core kernels reduce in a
 *  fixed order, so repeated calls give the same bits; the split-K streaming
 *  kernels (WQ_ROUTE_DECODE_SPLITK, WQ_ROUTE_CHUNKED) add their partial sums
 *  with fp32 atomics in arrival order, so their results may differ between
 *  calls in the last bits (each within the documented accuracy).
 *  M >= 1, N >= 1, bits in 2..8, K <= 1048576 below the tensor-core kernel's
 *  token counts (fewer than 65 tokens, see wq_debug_route); larger K there
 *  returns WQ_EUNSUPPORTED. */
wq_status wna16_gemm(const wq_bf16* x, int64_t M, const uint32_t* Wpacked, const wq_bf16* scales,
                     int64_t N, int64_t K, int bits, int group, wq_bf16* y,
                     void* workspace, size_t ws_bytes, void* stream);

/* WNA16 linear layer with asymmetric groups [CARD "Findings", second bullet:
 * a zero point per group instead of the symmetric 2^(bits-1), the option the
 * pages' four-bit tier used and their serving path lacked above four bits]:
 *   y[m, n] = sum_k x[m, k] * s[n, k/128] * (q[n, k] - zp[n, k/128]),
 * float32 accumulation, y rounded to bf16.
 *  zeros    [N, K/128] uint8, one zero point per (row, group); its low `bits`
 *           bits are used (the method's zero points lie in [0, 2^bits - 1]).
 *  Every other argument as wna16_gemm; workspace at least
 *  wna16_zp_workspace_bytes(). Same kernels as wna16_gemm, except that
 *  few-token shapes whose K half does not fit the CTA-pair decode kernel go
 *  to the chunked kernel. */
wq_status wna16_gemm_zp(const wq_bf16* x, int64_t M, const uint32_t* Wpacked, const wq_bf16* scales,
                        const uint8_t* zeros, int64_t N, int64_t K, int bits, int group, wq_bf16* y,
                        void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes wna16_gemm_zp needs (same contract as
 * wna16_workspace_bytes). */
size_t wna16_zp_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits);

/* Mixture-of-experts WNA16 layer, all experts in one launch [CARD "Findings",
 * third bullet: the pages' serving path has no fused MoE WNA16 GEMM at 5/6/7
 * bits]. The tokens come sorted by expert: expert e owns token rows
 * [expert_offsets[e], expert_offsets[e+1]) of x and y and applies its own
 * layer to them,
 *   y[m, n] = sum_k x[m, k] * s_e[n, k/128] * (q_e[n, k] - 2^(bits-1)).
 *  x              [M, K] bf16, tokens sorted by expert.
 *  expert_offsets [E + 1] int32 DEVICE array (4-byte aligned): 0, ..., M,
 *                 nondecreasing; the kernel clamps each value into [0, M] and
 *                 to at least the previous one, so no offsets can make it
 *                 read or write outside x and y (tokens outside every range
 *                 are then left unwritten).
 *  Wpacked        [E * N, ceil(K*bits/32)] uint32: the E layers' packed rows
 *                 stacked (v1 layout); scales [E * N, K/128] bf16 likewise.
 *  y              [M, N] bf16 output.
 *  1 <= E <= 1024, E * N < 2^31, bits in 2..8. Runs on the tensor-core
 *  kernel whatever the token counts (tiles of 128 or 256 tokens of one
 *  expert); needs no workspace. */
wq_status wna16_moe_gemm(const wq_bf16* x, int64_t M, const int32_t* expert_offsets, int64_t E,
                         const uint32_t* Wpacked, const wq_bf16* scales, int64_t N, int64_t K, int bits, int group,
                         wq_bf16* y, void* stream);

/* WNA16 linear layer without a workspace argument, for callers that cannot
 * allocate device memory (no counterpart on the source pages; it is a
 * packaging of wna16_gemm). A serving engine that has reserved nearly all
 * device memory up front for its KV-cache pool cannot supply a workspace on
 * the request path, where a cudaMalloc may fail, stall the device or take
 * memory promised elsewhere; a plain C caller may have no allocator at all.
 * Same arguments and results as wna16_gemm, minus the workspace: the split-K
 * scratch is a fixed 4 MiB __device__ array owned by the library, held by
 * every GPU that loads it until the process exits.
 *  - Shapes whose wna16_workspace_bytes() exceeds 4 MiB (about M*N > 1M)
 *    return WQ_EINVAL with a message, unless they run on the tensor-core
 *    kernel, which needs no scratch (32 <= M <= 64 on a layer with a
 *    128-row tile for every two SMs); use wna16_gemm for the others.
 *  - Every argument check of wna16_gemm runs first: a call with bad
 *    arguments returns WQ_EINVAL (or WQ_EUNSUPPORTED) with nothing enqueued
 *    and the array untouched.
 *  - The scratch region used is cleared on `stream` before the GEMM, so no
 *    state carries over between calls; calls whose executions overlap on the
 *    GPU (other streams, other host threads) share the array and race.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
wq_status wna16_gemm_noalloc(const wq_bf16* x, int64_t M, const uint32_t* Wpacked,
                             const wq_bf16* scales, int64_t N, int64_t K, int bits, int group,
                             wq_bf16* y, void* stream);

/* Per-token dynamic int8 activation quantization [W4A8], IEEE float32:
 *   sx[m] = max_k |x[m, k]| / 127 (IEEE division),
 *   xq[m, k] = clamp(round_half_even(x[m, k] / sx[m]), -127, 127)
 * (IEEE division, not a reciprocal multiply); an all-zero row gives sx = 0 and
 * xq = 0. x [M, K] bf16 -> xq [M, K] int8, sx [M] float32. Non-finite inputs
 * give unspecified results. */
wq_status act_quant_int8(const wq_bf16* x, int64_t M, int64_t K, int8_t* xq, float* sx,
                         void* stream);

/* Bytes of zero-at-rest workspace w4a8_gemm needs (split-K partials; 0 when
 * none). Same contract as the workspace of wna16_gemm. */
size_t w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Bytes of scratch w4a8_gemm needs for the quantized activations (xq [M, K]
 * int8 and sx [M] float32). Its contents need not be zero and are left
 * undefined. */
size_t w4a8_scratch_bytes(int64_t M, int64_t K);

/* W4A8 linear layer [W4A8]: act_quant_int8(x) (into `scratch`; for M <= 16
 * and K % 1024 == 0 inside the decode kernel, same arithmetic), then with
 * int4 codes q and zero point 8,
 *   acc[m, n, g] = sum_{k in group g} xq[m, k] * (q[n, k] - 8)   (exact, int32)
 *   y[m, n] = bf16( sx[m] * sum_g s[n, g] * acc[m, n, g] ),
 * the group sum in float32 over g in order. Every route computes each
 * acc[m, n, g] exactly (integer-valued products and sums below 2^24 on the
 * tensor cores, one accumulator per group) before applying s[n, g];
 * wq_debug_w4a8_group_acc returns them.
 *  Wpacked4 [N, K/8] uint32 (v1 layout, bits = 4); scales [N, K/128] bf16.
 *  workspace, ws_bytes: at least w4a8_workspace_bytes(); zero-fill and NULL
 *             contract as for wna16_gemm.
 *  scratch, scratch_bytes: at least w4a8_scratch_bytes(); must not overlap the
 *             workspace.
 *  The shape limits of wna16_gemm apply (WQ_EUNSUPPORTED). */
wq_status w4a8_gemm(const wq_bf16* x, int64_t M, const uint32_t* Wpacked4, const wq_bf16* scales,
                    int64_t N, int64_t K, int group, wq_bf16* y, void* workspace,
                    size_t ws_bytes, void* scratch, size_t scratch_bytes, void* stream);

/* Quantized embedding gather [INT57 s.3, CARD "Findings" first bullet], any
 * bits in 2..8 on the dense layout:
 *   out[t, d] = bf16_RNE( float(s[ids[t], d/128]) * float(q[ids[t], d] - 2^(bits-1)) )
 * (the float32 product is exact, so this is one rounding; a zero code offset
 * times a negative scale gives -0.0).
 *  ids [T] int32; Wpacked [V, ceil(D*bits/32)] uint32; scales [V, D/128] bf16;
 *  out [T, D] bf16. Ids outside [0, V) produce a +0.0 row and, when bad_count
 *  is not NULL, are added to *bad_count. T >= 0 (T = 0 enqueues nothing). */
wq_status qembed_gather(const int32_t* ids, int64_t T, const uint32_t* Wpacked,
                        const wq_bf16* scales, int64_t V, int64_t D, int bits, int group,
                        wq_bf16* out, int32_t* bad_count, void* stream);

/* ---- test and debug entry points ---------------------------------------- */

/* The launch plan of the CTA-pair decode kernel for a shape (host only, no
 * device call), for checks of its invariants. out14 receives, in order:
 * usable (1/0), clusters C, chunk rows H, chunks, 32-row tiles T, warps per
 * tile ksplit, ring slots NS, groups G, groups per K half, scale-box width,
 * scale-box start of the second half, token groups of 8, dynamic shared
 * memory bytes, and the most ring slots the kernel supports. The entries
 * after the first are meaningful only when it is 1. WQ_EINVAL for bits
 * outside 2..8, sm_count < 1 or a NULL out14. */
wq_status wq_debug_decode_plan(int64_t M, int64_t N, int64_t K, int bits, int sm_count, int64_t* out14);

/* Which kernel wna16_gemm (kind = 0), w4a8_gemm (kind = 1, bits = 4) or
 * wna16_gemm_zp (kind = 2) launches for a shape on a device with sm_count SMs
 * (host only, no device call). The entry points dispatch on the same
 * function. *route receives one of: */
#define WQ_ROUTE_NONE 0          /* no kernel takes the shape: the call returns WQ_EUNSUPPORTED */
#define WQ_ROUTE_DECODE_PAIR 1   /* CTA-pair decode kernel: M <= 16, K % 1024 == 0 */
#define WQ_ROUTE_DECODE_SPLITK 2 /* persistent split-K decode kernel (uses the workspace) */
#define WQ_ROUTE_CHUNKED 3       /* chunked split-K streaming kernel (uses the workspace) */
#define WQ_ROUTE_TENSOR_CORE 4   /* tcgen05 tensor-core GEMM: M >= 65, or 32..64 tokens on a
                                    layer with a 128-row tile for every two SMs */
/* WQ_EINVAL for a NULL route, sm_count < 1, kind not 0..2, bits outside 2..8
 * (not 4 with kind 1), K not a positive multiple of 128, or M, N < 1. */
wq_status wq_debug_route(int64_t M, int64_t N, int64_t K, int bits, int kind, int sm_count, int* route);

/* Inverse of the repack for the codes: packed [N, ceil(K*bits/32)] ->
 * codes [N, K] uint8. */
wq_status wq_debug_unpack(const uint32_t* packed, int64_t N, int64_t K, int bits,
                          uint8_t* codes, void* stream);

/* Throughput probe of the warp-level tensor-core instruction (mma.sync) in
 * the two forms the W4A8 discussion weighs [W4A8 "Under the hood": int8
 * products accumulated in int32, against bf16]: kind 0 runs m16n8k32
 * s8 x s8 -> s32, kind 1 m16n8k16 bf16 x bf16 -> f32. `blocks` CTAs of 8
 * warps each run 8 independent chains of `iters` instructions on all-ones
 * operands and write one int32 checksum per thread to out [blocks * 256]
 * (device memory, caller-owned), which must equal 8 * 4 * K * iters with
 * K = 32 (kind 0) or 16 (kind 1). The caller times the launch on `stream`:
 * operations = blocks * 8 * 8 * iters * 2*16*8*K. WQ_EINVAL for kind not 0/1,
 * iters outside 1..1000000, blocks outside 1..65535 or a NULL out. */
wq_status wq_debug_mma_peak(int kind, int64_t iters, int blocks, int32_t* out, void* stream);

/* The exact per-group integer accumulators of the W4A8 main loop [W4A8]:
 *   acc[m, n, g] = sum_{k in group g} xq[m, k] * (q[n, k] - 8),
 * with xq = act_quant_int8(x), computed by the kernel that w4a8_gemm launches
 * for the same shape (same route, same quantization of x, same main loop),
 * which writes these int32 sums instead of y. Arguments as w4a8_gemm, with
 * acc [M, N, K/128] int32 in place of y and no workspace (the accumulators
 * need no split-K partials). */
wq_status wq_debug_w4a8_group_acc(const wq_bf16* x, int64_t M, const uint32_t* Wpacked4,
                                  const wq_bf16* scales, int64_t N, int64_t K, int32_t* acc,
                                  void* scratch, size_t scratch_bytes, void* stream);

/* Test hook of the CTA-pair decode kernel, for checking the bounded-wait error
 * path without any fault: from the next launch on the current device, every
 * pipeline wait of that kernel gives up after wait_limit_ns (0: the default
 * bound of 2 s), and its producers stop issuing weight stages at stage
 * stop_stage of their sequence (-1: never). The copies already issued all
 * land; the consumers waiting for the first stage never issued give up,
 * record WQ_ETIMEOUT (read by wq_check_status) and finish the kernel, whose
 * outputs are then incomplete. Call again with (-1, 0) to restore normal
 * operation. Synchronous. */
wq_status wq_debug_decode_wait_fault(int64_t stop_stage, uint64_t wait_limit_ns);

/* Copies `bytes` (at most 4 MiB) between the caller's device buffer `buf` and
 * the start of wna16_gemm_noalloc's scratch array on the current device
 * (to_scratch = 1: buf -> scratch; 0: scratch -> buf), asynchronously on
 * `stream`. For tests that plant a sentinel in the array or read it back.
 * Like wna16_gemm_noalloc, it has no counterpart on the source pages. */
wq_status wq_debug_noalloc_scratch(void* buf, size_t bytes, int to_scratch, void* stream);

/* Reads and clears the status word of the current device (synchronizes the
 * device). Returns WQ_OK, WQ_ETIMEOUT if a kernel gave up on a pipeline wait,
 * or WQ_ECUDA if the device reports an error. */
wq_status wq_check_status(void);

/* One-line description of the last error on the calling thread ("" if none). */
const char* wq_last_error(void);

/* Library version string. */
const char* wq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
