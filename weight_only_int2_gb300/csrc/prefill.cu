// Prefill GEMM (many tokens): y = x . dequant(W)^T on the 5th-generation
// tensor cores (tcgen05.mma kind::f16, bf16 operands, fp32 accumulator in
// tensor memory).
//
// Method: "vLLM Can Run INT5-7", section 1 (WNA16 for widths 2..8, dequantize
// then multiply); model card "Qwen3.8-27B-INT6-Mixed-AutoRound", section
// "Findings" (dense LSB-first packing, symmetric zero point 2^(b-1), bf16
// group-128 scales of either sign); "vLLM Quantization", section "Key points"
// (at large batch the layer is compute bound: the weights are dequantized on
// chip and the product runs on the tensor cores).
//
// One CTA computes a tile of 128 weight rows x TN tokens, D[row, token] in
// tensor memory (MMA M = 128 rows, N = TN tokens; the weights are the A
// operand so that a dequantized tile serves TN tokens). K advances in stages
// of 64 (half a quantization group). Warp roles:
//   warp 0      TMA producer for the activation tile [TN x 64] (128-byte
//               swizzle, zero fill past M) of each stage.
//   warp 1      allocates tensor memory; one thread issues 4 MMAs of K = 16
//               per stage and commits them to the stage's "empty" barrier.
//   warp 2      TMA producer for the packed weights, one group [128 rows x
//               16*b bytes] per load, into a ring of 2 slots.
//   warps 3-10  dequantize: each thread turns one 32-code slice of one row
//               into bf16 RN(s * (q - z)) (q - z exact, one rounding) and
//               stores it in the K-major 128-byte-swizzled layout the MMA
//               reads; afterwards the same 8 warps drain the accumulator
//               (tcgen05.ld) and store bf16 outputs.
// All mbarrier waits are bounded; a timeout records WQ_ETIMEOUT and the roles
// stop early, the outputs of that CTA are then not written.
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kBK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kNS = 4;    // activation / dequantized-weight stages
constexpr int kNP = 2;    // packed-weight slots (one group each)
constexpr int kDeqWarps = 8;
constexpr int kThreads = (3 + kDeqWarps) * 32;  // 352
constexpr int kWStageBytes = kBM * kBK * 2;     // 16 KB

template <int B, int TN>
struct Layout {
  static constexpr int kXStage = TN * kBK * 2;
  static constexpr int kPSlot = kBM * 16 * B;  // one group of 128 rows
  static constexpr int kXOff = 0;
  static constexpr int kWOff = kNS * kXStage;
  static constexpr int kPOff = kWOff + kNS * kWStageBytes;
  static constexpr int kBytes = kPOff + kNP * kPSlot;
  static constexpr size_t kSmem = static_cast<size_t>(kBytes) + 1024;  // + alignment slack
};

struct PParams {
  const uint16_t* scales;  // bf16 [N, G]
  int64_t M, N, K;
  int G;
  uint16_t* y;       // bf16 [M, N]
  const float* sx;   // per-token output factor [M] or null
  unsigned* status;
};

// ---- tcgen05 helpers (inline PTX) -----------------------------------------

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (bits
// 16-29, unused for this layout; 1), stride byte offset >> 4 (bits 32-45),
// fixed 0b001 (bits 46-48), swizzle mode 2 = 128 B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at
// bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 consecutive fp32 columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- dequantization --------------------------------------------------------

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 32 bits of the slice starting at bit p (compile-time p after unrolling).
template <int B>
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[B], int p) {
  const int i = p >> 5, sh = p & 31;
  if (sh == 0) return w[i];
  const uint32_t nx = (i + 1 < B) ? w[i + 1] : 0u;
  return __funnelshift_r(w[i], nx, sh);
}

// One 32-code slice (B packed words, LSB-first) -> 16 words holding the bf16
// pairs RN(s * (q - z)) for codes (2c, 2c+1). Codes are placed in the
// mantissa of bf16 128.0 (0x4300: 7 mantissa bits, unit spacing), so
// (128 + q) - (128 + z) is exact and the scale multiply rounds once.
template <int B>
__device__ __forceinline__ void dequant_slice(const uint32_t (&w)[B], uint32_t s2, uint32_t (&o)[16]) {
  constexpr uint32_t kMagic = 0x43004300u;
  if constexpr (B == 8) {
    // 8-bit codes do not fit 7 mantissa bits: take q & 127 into the mantissa
    // and subtract 256 (bit 7 clear) or 128 (bit 7 set), i.e. q - 128.
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t t = __byte_perm(w[c >> 1], 0u, (c & 1) ? 0x4342u : 0x4140u);
      const uint32_t v = (t & 0x007F007Fu) | kMagic;
      const uint32_t zz = (~t & 0x00800080u) | kMagic;
      o[c] = bf16x2_mul(bf16x2_sub(v, zz), s2);
    }
  } else {
    constexpr uint32_t kM = (1u << B) - 1u;
    constexpr uint32_t kZ = 0x4300u | (1u << (B - 1));  // bf16 of 128 + 2^(B-1)
    constexpr uint32_t kZ2 = kZ | (kZ << 16);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t win = window<B>(w, 2 * c * B);
      const uint32_t v = (win & kM) | ((win << (16 - B)) & (kM << 16)) | kMagic;
      o[c] = bf16x2_mul(bf16x2_sub(v, kZ2), s2);
    }
  }
}

template <int B>
__device__ __forceinline__ void load_words(const uint8_t* src, uint32_t (&w)[B]) {
  if constexpr (B % 4 == 0) {
#pragma unroll
    for (int j = 0; j < B / 4; ++j) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[j];
      w[4 * j] = v.x, w[4 * j + 1] = v.y, w[4 * j + 2] = v.z, w[4 * j + 3] = v.w;
    }
  } else if constexpr (B % 2 == 0) {
#pragma unroll
    for (int j = 0; j < B / 2; ++j) {
      const uint2 v = reinterpret_cast<const uint2*>(src)[j];
      w[2 * j] = v.x, w[2 * j + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < B; ++j) w[j] = reinterpret_cast<const uint32_t*>(src)[j];
  }
}

template <int B, int TN, bool kTok>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                   const PParams p) {
  using L = Layout<B, TN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t xfull[kNS], wfull[kNS], empty[kNS], pfull[kNP], pempty[kNP], accb;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* xs = base + L::kXOff;
  uint8_t* ws = base + L::kWOff;
  uint8_t* ps = base + L::kPOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBM;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TN;
  const int G = p.G;
  const int S = 2 * G;  // stages

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&wfull[s], kDeqWarps);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kNP; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], kDeqWarps);
    }
    mbar_init(&accb, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(TN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ---- activations: stage i covers k = 64 i .. 64 i + 63
    if (lane == 0) {
      for (int i = 0; i < S && !s_abort; ++i) {
        const int s = i % kNS;
        if (i >= kNS && !mbar_wait_bounded(&empty[s], ((i / kNS) - 1) & 1)) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&xfull[s], L::kXStage);
        tma_load_2d(xs + s * L::kXStage, &xmap, i * kBK, static_cast<int>(m0), &xfull[s]);
      }
    }
  } else if (warp == 2) {
    // ---- packed weights: group g (128 codes of 128 rows) into slot g % 2
    if (lane == 0) {
      for (int g = 0; g < G && !s_abort; ++g) {
        const int sl = g % kNP;
        if (g >= kNP && !mbar_wait_bounded(&pempty[sl], ((g / kNP) - 1) & 1)) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&pfull[sl], L::kPSlot);
        tma_load_2d(ps + sl * L::kPSlot, &wmap, g * 4 * B, static_cast<int>(n0), &pfull[sl]);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kBM, TN);
      for (int i = 0; i < S; ++i) {
        const int s = i % kNS;
        const uint32_t par = (i / kNS) & 1;
        if (s_abort || !mbar_wait_bounded(&wfull[s], par) || !mbar_wait_bounded(&xfull[s], par)) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t aa = smem_u32(ws + s * kWStageBytes);
        const uint32_t bb = smem_u32(xs + s * L::kXStage);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // K = 16 bf16 = 32 bytes further along the 128-byte swizzled rows
          umma_bf16(tmem, sw128_desc(aa + 32 * kk), sw128_desc(bb + 32 * kk), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(&accb);  // fires once every MMA issued above has completed
    }
  } else {
    // ---- dequantize: thread -> (row r, 32-code half sl of the stage)
    const int dt = threadIdx.x - 3 * 32;  // 0..255
    const int r = dt >> 1, sl = dt & 1;
    const int64_t row = n0 + r;
    const bool row_ok = row < p.N;
    const uint16_t* srow = p.scales + (row_ok ? row : 0) * static_cast<int64_t>(G);
    uint8_t* wdst = ws + (r >> 3) * 1024 + (r & 7) * 128;
    uint16_t sb = row_ok ? srow[0] : static_cast<uint16_t>(0);
    for (int i = 0; i < S; ++i) {
      const int s = i % kNS, g = i >> 1, h = i & 1, pslot = g % kNP;
      // every decision below is warp-uniform (the warp later meets at
      // __syncwarp and tcgen05.ld)
      bool go = !s_abort;
      if (go && h == 0) go = mbar_wait_bounded(&pfull[pslot], (g / kNP) & 1);
      if (go && i >= kNS) go = mbar_wait_bounded(&empty[s], ((i / kNS) - 1) & 1);
      if (!__all_sync(0xFFFFFFFFu, go)) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        break;
      }
      const uint32_t s2 = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(sb) << 16);
      uint32_t w[B];
      load_words<B>(ps + pslot * L::kPSlot + r * 16 * B + (2 * h + sl) * 4 * B, w);
      if (h == 1 && g + 1 < G && row_ok) sb = srow[g + 1];  // next group's scale
      uint32_t o[16];
      dequant_slice<B>(w, s2, o);
      uint8_t* dst = wdst + s * kWStageBytes;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = 4 * sl + q;  // 16-byte chunk of the 128-byte row
        *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) =
            make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
      fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wfull[s]);
        if (h == 1) mbar_arrive(&pempty[pslot]);
      }
    }

    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows);
    // the two warps of a lane quarter split the TN token columns.
    const int quarter = warp & 3, half = (warp - 3) >> 2;
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&accb, 0));
    if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
    tc_fence_after();
    const int64_t n = n0 + quarter * 32 + lane;
#pragma unroll 1
    for (int cb = half * (TN / 2); cb < (half + 1) * (TN / 2); cb += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cb, v);
      if (ok && !s_abort && n < p.N) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t m = m0 + cb + j;
          if (m < p.M) {
            const float f = __uint_as_float(v[j]) * (kTok ? p.sx[m] : 1.0f);
            p.y[m * p.N + n] = float_to_bf16_bits_rn(f);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TN) : "memory");
  }
}

template <int B, int TN, bool kTok>
cudaError_t plaunch(const Ctx& c, const CUtensorMap& xmap, const CUtensorMap& wmap, const PParams& prm) {
  constexpr size_t smem = Layout<B, TN>::kSmem;
  static_assert(smem <= 227 * 1024, "prefill stage layout exceeds shared memory");
  static bool configured[64] = {};
  if (c.device < 0 || c.device >= 64) return cudaErrorInvalidDevice;
  if (!configured[c.device]) {
    const cudaError_t e = cudaFuncSetAttribute(prefill_kernel<B, TN, kTok>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured[c.device] = true;
  }
  const dim3 grid(static_cast<unsigned>((prm.N + kBM - 1) / kBM), static_cast<unsigned>((prm.M + TN - 1) / TN));
  prefill_kernel<B, TN, kTok><<<grid, kThreads, smem, c.stream>>>(xmap, wmap, prm);
  return cudaGetLastError();
}

template <int TN>
cudaError_t plaunch_b(const Ctx& c, int bits, const CUtensorMap& xmap, const CUtensorMap& wmap,
                      const PParams& prm) {
  if (prm.sx != nullptr) {
    // per-token output factor: the W4A8 path (4-bit weights)
    return bits == 4 ? plaunch<4, TN, true>(c, xmap, wmap, prm) : cudaErrorInvalidValue;
  }
  switch (bits) {
    case 2: return plaunch<2, TN, false>(c, xmap, wmap, prm);
    case 3: return plaunch<3, TN, false>(c, xmap, wmap, prm);
    case 4: return plaunch<4, TN, false>(c, xmap, wmap, prm);
    case 5: return plaunch<5, TN, false>(c, xmap, wmap, prm);
    case 6: return plaunch<6, TN, false>(c, xmap, wmap, prm);
    case 7: return plaunch<7, TN, false>(c, xmap, wmap, prm);
    case 8: return plaunch<8, TN, false>(c, xmap, wmap, prm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int prefill_tile_tokens(int64_t M) { return M <= 128 ? 128 : 256; }

bool prefill_supported(int64_t M, int64_t N, int64_t K, int bits) {
  // K a whole number of groups (then every TMA coordinate and row stride is
  // a multiple of 16 bytes); N, M within the 32-bit TMA coordinate range.
  return M > 16 && M < (int64_t(1) << 31) && N >= 1 && N < (int64_t(1) << 31) && K >= 128 && K % 128 == 0 &&
         bits >= 2 && bits <= 8;
}

cudaError_t launch_prefill(const Ctx& c, const uint16_t* x, const uint32_t* packed, const uint16_t* scales,
                           int64_t M, int64_t N, int64_t K, int bits, uint16_t* y, const float* sx) {
  const int tn = prefill_tile_tokens(M);
  CUtensorMap xmap, wmap;
  if (!make_tmap_bf16_2d_sw128(&xmap, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBK,
                               static_cast<uint32_t>(tn)))
    return cudaErrorInvalidValue;
  const uint64_t words = static_cast<uint64_t>(K) * bits / 32;
  if (!make_tmap_u32_2d(&wmap, packed, words, static_cast<uint64_t>(N), 4u * bits, kBM))
    return cudaErrorInvalidValue;
  PParams prm{};
  prm.scales = scales;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.G = static_cast<int>(K / 128);
  prm.y = y;
  prm.sx = sx;
  prm.status = c.status;
  return tn == 128 ? plaunch_b<128>(c, bits, xmap, wmap, prm) : plaunch_b<256>(c, bits, xmap, wmap, prm);
}

}  // namespace wq
