// Weight-streaming quantized GEMM: y = x . dequant(W)^T for small M (decode),
// the W4A8 variant, and the exact W4A8 group accumulators.
//
// The layer: "vLLM Can Run INT5-7", section 1 (WNA16 for every width 2..8);
// the "Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section "Findings"
// (dense layout, symmetric groups: zero point 2^(b-1), one bf16 scale per
// (row, 128-group), any sign); "vLLM Quantization", section "Key points"
// (decode waits on memory); "int8 activations (W4A8) ...", section "Under the
// hood" (per-token int8 activations, int4 weights widened losslessly,
// integer accumulation, negative scales).
//
// Design (GB300):
//  * Swap-AB warp MMA: W rows are the MMA's M dimension (16 rows per warp),
//    tokens its N dimension (8 per n-tile), so M = 1..64 wastes no weight
//    bandwidth. mma.sync m16n8k16 with fp32 accumulators.
//  * Each warp streams its 16 rows through its own 4-stage TMA pipeline
//    (2-D tensor map; one box = 16 rows x one 128-code group = 16*b bytes per
//    row). No cross-warp synchronisation inside the main loop.
//  * Each thread owns the 32 codes of one b-word slice of a group (32 codes
//    fill exactly b words, so no code straddles two threads). The order of
//    the contraction inside an MMA is free as long as the activations follow
//    it, so codes are paired per register in whatever order is cheapest: for
//    every pair one 32-bit window of the slice (one funnel shift, often none)
//    holds both codes, and one LOP3 masks them into the mantissas of two
//    16-bit floats of value MAGIC + q * 2^o (o = the code's offset inside its
//    half). fp16 (MAGIC = 1024, 10 mantissa bits) is used for b in {3,5,6,7,8},
//    bf16 (MAGIC = 128, 7 bits, o = 0) for b in {2,4}.
//  * The factor 2^-o of each contraction index is folded into the staged
//    activations (exact power-of-two scaling). Per (token, group) the MMA then
//    yields sum_k x_k (q_k + MAGIC 2^-o_k); subtracting
//    corr = MAGIC sum_k x_k 2^-o_k + z sum_k x_k (computed once per CTA) leaves
//    sum_k x_k (q_k - z), which is scaled by s[n, g]. For fp16 the activations
//    of a (token, group) are additionally scaled by a power of two that keeps
//    them below 2^15, and the group result is scaled back.
//  * W4A8: int8 activations and int4 codes (bf16 path, o = 0) are exact and
//    every partial sum of one 128-group is an integer below 2^24, so the fp32
//    accumulator equals the int32 accumulator bit for bit.
//  * Split-K over groups for occupancy: partial sums go to a zero-at-rest fp32
//    workspace with atomics; the last CTA of a row block (arrival counter)
//    converts to bf16 and zeroes the workspace again.
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_unpack.cuh"

#include <algorithm>

namespace wq {
namespace {

using namespace unpack;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 16;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 128
constexpr int kStages = 4;
constexpr int kXGroupsTimesNT = 16;     // x chunk: NT * XC == 16 groups of 8 tokens
constexpr int kMaxGroupsPerCta = 128;   // groups per CTA (its scales live in smem); K splits above
constexpr int kMaxSplits = 64;          // K <= 64 * 128 * 128 = 1048576

struct Params {
  const uint16_t* x;
  const int8_t* xq;
  const float* sx;
  const uint16_t* scales;
  const uint8_t* zeros;  // asymmetric groups (kWna16): [N, G], or null
  int64_t M, N, K;
  int G;     // groups along K
  int gper;  // groups per split
  uint16_t* y;
  int32_t* acc;
  float* ws;
  uint32_t* counters;
  unsigned* status;
};

// ---------------------------------------------------------------------------
// Activation staging for one chunk of groups.
// Thread job (j, gi, g, t): token m0 + 8j + g, group gabs0 + gi, slice t
// (32 consecutive activations, read with 16-byte loads). It writes the four
// 16-byte MMA B fragments of that slice; the quad t = 0..3 then reduces the
// group's correction term.
// ---------------------------------------------------------------------------
template <int B, int NT, int MODE>
__device__ __forceinline__ void stage_x(const Params& p, int64_t m0, int gabs0, int nc, uint4* xs4,
                                        float* corr, float* scl, float* xsm) {
  constexpr int XC = kXGroupsTimesNT / NT;
  constexpr int kJobs = NT * XC * 32;
  static_assert(kJobs % kThreads == 0, "staging jobs must divide evenly");
  constexpr bool kInt8 = MODE != static_cast<int>(GemvMode::kWna16);
#pragma unroll
  for (int rep = 0; rep < kJobs / kThreads; ++rep) {
    const int job = rep * kThreads + threadIdx.x;
    const int ln = job & 31, gi = (job >> 5) % XC, j = (job >> 5) / XC;
    const int t = ln & 3;
    const int64_t tok = m0 + j * 8 + (ln >> 2);
    const bool valid = gi < nc && tok < p.M;
    const int64_t k0 = static_cast<int64_t>(gabs0 + gi) * 128 + 32 * t;
    const void* src = kInt8 ? static_cast<const void*>(p.xq + (valid ? tok * p.K + k0 : 0))
                            : static_cast<const void*>(p.x + (valid ? tok * p.K + k0 : 0));
    float v[32];
    load_slice_x<kInt8>(src, valid, v);
    uint32_t frag[16];
    float cr, sb, xsum;
    make_fragments<B>(v, frag, cr, sb, xsum);
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2)
      xs4[((j * XC + gi) * 4 + i2) * 32 + ln] =
          make_uint4(frag[4 * i2], frag[4 * i2 + 1], frag[4 * i2 + 2], frag[4 * i2 + 3]);
    if (t == 0) {
      const int tokl = j * 8 + (ln >> 2);
      corr[tokl * XC + gi] = cr;
      scl[tokl * XC + gi] = sb;
      xsm[tokl * XC + gi] = xsum;
    }
  }
}

template <int B, int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ CUtensorMap tmap,
                                                          const Params p) {
  constexpr int XC = kXGroupsTimesNT / NT;            // groups per x chunk
  constexpr int kStageBytes = kRowsPerWarp * 16 * B;  // 16 rows x (16*B bytes)
  constexpr int kStageWords = kStageBytes / 4;
  constexpr bool kF16 = uses_fp16<B>();

  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* wbuf_all = reinterpret_cast<uint32_t*>(smem);
  uint4* xs4 = reinterpret_cast<uint4*>(smem + kWarps * kStages * kStageBytes);
  float* corr = reinterpret_cast<float*>(xs4 + NT * XC * 4 * 32);
  float* scl = corr + NT * 8 * XC;
  float* xsm = scl + NT * 8 * XC;  // plain group sums of x (asymmetric groups)
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(xsm + NT * 8 * XC);
  uint16_t* ssm = reinterpret_cast<uint16_t*>(bars_all + kWarps * kStages);  // [128][gper]
  uint8_t* zsm = reinterpret_cast<uint8_t*>(ssm + kRowsPerCta * p.gper);      // [128][gper] zero points
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t rb0 = static_cast<int64_t>(blockIdx.x) * kRowsPerCta;
  const int64_t row0 = rb0 + warp * kRowsPerWarp;
  const bool warp_active = row0 < p.N;
  const int gbeg = blockIdx.y * p.gper;
  const int ngroups = min(p.G - gbeg, p.gper);
  const int64_t m0 = static_cast<int64_t>(blockIdx.z) * (NT * 8);
  uint32_t* wbuf = wbuf_all + warp * kStages * kStageWords;
  uint64_t* bars = bars_all + warp * kStages;

  // Pipeline prologue: first kStages groups of this warp's 16 rows.
  if (warp_active && lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    for (int s = 0; s < kStages && s < ngroups; ++s) {
      mbar_arrive_expect_tx(&bars[s], kStageBytes);
      tma_load_2d(wbuf + s * kStageWords, &tmap, (gbeg + s) * 4 * B, static_cast<int>(row0), &bars[s]);
    }
  }
  __syncwarp();

  // Scales of this CTA's rows and groups (the group-accumulator mode has none).
  if constexpr (MODE != static_cast<int>(GemvMode::kW4a8GroupAcc)) {
    for (int idx = threadIdx.x; idx < kRowsPerCta * ngroups; idx += kThreads) {
      const int r = idx / ngroups, gi = idx - r * ngroups;
      const int64_t row = rb0 + r;
      ssm[r * p.gper + gi] = (row < p.N) ? p.scales[row * p.G + gbeg + gi] : static_cast<uint16_t>(0);
      if (p.zeros != nullptr)
        zsm[r * p.gper + gi] = (row < p.N) ? p.zeros[row * p.G + gbeg + gi] : static_cast<uint8_t>(0);
    }
  }
  constexpr float kZero = static_cast<float>(1 << (B - 1));
  constexpr uint32_t kZMask = (1u << B) - 1u;

  const int rl_g = warp * kRowsPerWarp + g;  // local index of this thread's first row
  const int64_t r_g = row0 + g, r_g8 = row0 + g + 8;
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;

  bool aborted = false;
  int it = 0;  // group index within this split
  for (int cb = 0; cb < ngroups; cb += XC) {
    const int nc = min(XC, ngroups - cb);
    const int gabs0 = gbeg + cb;
    __syncthreads();  // previous chunk fully consumed (and scales written)
    stage_x<B, NT, MODE>(p, m0, gabs0, nc, xs4, corr, scl, xsm);
    __syncthreads();

    if (!warp_active) {
      it += nc;
      continue;
    }
    if (aborted) continue;
    for (int gi = 0; gi < nc; ++gi, ++it) {
      const int slot = it % kStages;
      if (!mbar_wait_bounded(&bars[slot], (it / kStages) & 1)) {
        record_status(p.status, kStatusTimeout);
        aborted = true;
        break;
      }
      const uint32_t* st = wbuf + slot * kStageWords;
      uint32_t wa[B], wb[B];
      load_slice<B>(st, g, t, wa);
      load_slice<B>(st, g + 8, t, wb);
      uint32_t ra[16], rb[16];
      unpack_slice<B>(wa, ra);
      unpack_slice<B>(wb, rb);
      __syncwarp();
      if (lane == 0 && it + kStages < ngroups) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[slot], kStageBytes);
        tma_load_2d(wbuf + slot * kStageWords, &tmap, (gbeg + it + kStages) * 4 * B,
                    static_cast<int>(row0), &bars[slot]);
      }
      float s_g = 0.0f, s_g8 = 0.0f;
      if constexpr (MODE != static_cast<int>(GemvMode::kW4a8GroupAcc)) {
        s_g = bf16_bits_to_float(ssm[rl_g * p.gper + it]);
        s_g8 = bf16_bits_to_float(ssm[(rl_g + 8) * p.gper + it]);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float c0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint4* xb = xs4 + ((j * XC + gi) * 4) * 32 + lane;
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const uint4 bv = xb[i2 * 32];
          mma16<kF16>(c0, ra[4 * i2], rb[4 * i2], ra[4 * i2 + 1], rb[4 * i2 + 1], bv.x, bv.y);
          mma16<kF16>(c1, ra[4 * i2 + 2], rb[4 * i2 + 2], ra[4 * i2 + 3], rb[4 * i2 + 3], bv.z, bv.w);
        }
        const int tl0 = j * 8 + 2 * t;
        float cr0 = corr[tl0 * XC + gi], cr1 = corr[(tl0 + 1) * XC + gi];
        float cr2 = cr0, cr3 = cr1;
        const float sc0 = scl[tl0 * XC + gi], sc1 = scl[(tl0 + 1) * XC + gi];
        if (MODE == static_cast<int>(GemvMode::kWna16) && p.zeros != nullptr) {
          // asymmetric groups: the correction carries (zp - 2^(b-1)) sum x
          const float zd_g = static_cast<float>(zsm[rl_g * p.gper + it] & kZMask) - kZero;
          const float zd_g8 = static_cast<float>(zsm[(rl_g + 8) * p.gper + it] & kZMask) - kZero;
          const float x0 = xsm[tl0 * XC + gi], x1 = xsm[(tl0 + 1) * XC + gi];
          cr2 = fmaf(zd_g8, x0, cr0);
          cr3 = fmaf(zd_g8, x1, cr1);
          cr0 = fmaf(zd_g, x0, cr0);
          cr1 = fmaf(zd_g, x1, cr1);
        }
        const float d0 = fmaf(sc0, c0[0] + c1[0], -cr0);
        const float d1 = fmaf(sc1, c0[1] + c1[1], -cr1);
        const float d2 = fmaf(sc0, c0[2] + c1[2], -cr2);
        const float d3 = fmaf(sc1, c0[3] + c1[3], -cr3);
        if constexpr (MODE == static_cast<int>(GemvMode::kW4a8GroupAcc)) {
          const int64_t tk0 = m0 + tl0, tk1 = tk0 + 1;
          const int64_t G = p.G;
          const int gabs = gabs0 + gi;
          if (r_g < p.N) {
            if (tk0 < p.M) p.acc[(tk0 * p.N + r_g) * G + gabs] = __float2int_rn(d0);
            if (tk1 < p.M) p.acc[(tk1 * p.N + r_g) * G + gabs] = __float2int_rn(d1);
          }
          if (r_g8 < p.N) {
            if (tk0 < p.M) p.acc[(tk0 * p.N + r_g8) * G + gabs] = __float2int_rn(d2);
            if (tk1 < p.M) p.acc[(tk1 * p.N + r_g8) * G + gabs] = __float2int_rn(d3);
          }
        } else {
          acc[j][0] = fmaf(s_g, d0, acc[j][0]);
          acc[j][1] = fmaf(s_g, d1, acc[j][1]);
          acc[j][2] = fmaf(s_g8, d2, acc[j][2]);
          acc[j][3] = fmaf(s_g8, d3, acc[j][3]);
        }
      }
    }
  }

  // Drain: if a wait gave up, give the copies still in flight a bounded chance
  // to land before the CTA's shared memory is released.
  if (aborted && lane == 0) {
    for (int k = it; k < ngroups && k < it + kStages; ++k)
      mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1);
  }

  if constexpr (MODE == static_cast<int>(GemvMode::kW4a8GroupAcc)) {
    return;
  } else {
    const bool split = gridDim.y > 1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t row = (e < 2) ? r_g : r_g8;
        const int64_t tok = m0 + j * 8 + 2 * t + (e & 1);
        if (!warp_active || row >= p.N || tok >= p.M) continue;
        float v = acc[j][e];
        if constexpr (MODE == static_cast<int>(GemvMode::kW4a8)) v *= p.sx[tok];
        if (!split) {
          p.y[tok * p.N + row] = float_to_bf16_bits_rn(v);
        } else {
          atomicAdd(p.ws + tok * p.N + row, v);
        }
      }
    }
    if (split) {
      __threadfence();
      __syncthreads();
      const unsigned cidx = blockIdx.z * gridDim.x + blockIdx.x;
      if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&p.counters[cidx], 1u);
        s_last = (prev == gridDim.y - 1) ? 1 : 0;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int idx = threadIdx.x; idx < NT * 8 * kRowsPerCta; idx += kThreads) {
          const int64_t tok = m0 + idx / kRowsPerCta;
          const int64_t row = rb0 + idx % kRowsPerCta;
          if (tok >= p.M || row >= p.N) continue;
          float* cell = p.ws + tok * p.N + row;
          p.y[tok * p.N + row] = float_to_bf16_bits_rn(__ldcg(cell));
          *cell = 0.0f;
        }
        if (threadIdx.x == 0) p.counters[cidx] = 0u;
      }
    }
  }
}

template <int B, int NT>
size_t smem_bytes(int gper) {
  constexpr int XC = kXGroupsTimesNT / NT;
  return static_cast<size_t>(kWarps) * kStages * kRowsPerWarp * 16 * B      // weight stages
         + static_cast<size_t>(NT) * XC * 4 * 32 * 16                       // B fragments
         + static_cast<size_t>(NT) * 8 * XC * 4 * 3                         // corrections, scales, sums
         + static_cast<size_t>(kWarps) * kStages * 8                        // mbarriers
         + ((static_cast<size_t>(kRowsPerCta) * gper * 3 + 15) / 16) * 16;  // group scales, zero points
}

struct Plan {
  int nt;
  int mchunks;
  int row_blocks;
  int splits;
  int gper;
};

// Split-K choice: minimise (waves of resident CTAs) x (groups per CTA plus a
// fixed per-CTA cost of about three groups), with at most kMaxGroupsPerCta
// groups per CTA (a longer K always splits).
Plan make_plan(int64_t M, int64_t N, int64_t K, int sm_count) {
  Plan pl{};
  pl.nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8));
  pl.mchunks = static_cast<int>((M + pl.nt * 8 - 1) / (pl.nt * 8));
  pl.row_blocks = static_cast<int>((N + kRowsPerCta - 1) / kRowsPerCta);
  const int G = static_cast<int>(K / 128);
  const int min_splits = (G + kMaxGroupsPerCta - 1) / kMaxGroupsPerCta;
  int best_gper = (G + min_splits - 1) / min_splits;
  if (M <= 64) {
    const int64_t base = static_cast<int64_t>(pl.row_blocks) * pl.mchunks;
    const int64_t resident = 2LL * sm_count;
    int64_t best_cost = -1;
    for (int s = 1; s <= std::min(G, kMaxSplits); ++s) {
      const int gper = (G + s - 1) / s;
      if (gper > kMaxGroupsPerCta) continue;
      const int splits = (G + gper - 1) / gper;
      const int64_t ctas = base * splits;
      const int64_t cost = ((ctas + resident - 1) / resident) * (gper + 3);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_gper = gper;
      }
    }
  }
  pl.gper = best_gper;
  pl.splits = (G + pl.gper - 1) / pl.gper;
  return pl;
}

template <int B, int NT, int MODE>
cudaError_t launch_t(const Ctx& c, const CUtensorMap& tmap, const Params& prm, const Plan& pl) {
  // The shared-memory opt-in is a per-device function attribute: raise it to
  // the largest size this instantiation can ask for, once per device.
  static SmemLimit limit;
  const cudaError_t e = raise_smem_limit(limit, gemv_kernel<B, NT, MODE>, c.device,
                                         static_cast<size_t>(smem_bytes<B, NT>(kMaxGroupsPerCta)));
  if (e != cudaSuccess) return e;
  const size_t smem = smem_bytes<B, NT>(pl.gper);
  const dim3 grid(pl.row_blocks, pl.splits, pl.mchunks);
  gemv_kernel<B, NT, MODE><<<grid, kThreads, smem, c.stream>>>(tmap, prm);
  return cudaGetLastError();
}

template <int B, int MODE>
cudaError_t launch_nt(const Ctx& c, const CUtensorMap& tmap, const Params& prm, const Plan& pl) {
  switch (pl.nt) {
    case 1: return launch_t<B, 1, MODE>(c, tmap, prm, pl);
    case 2: return launch_t<B, 2, MODE>(c, tmap, prm, pl);
    case 4: return launch_t<B, 4, MODE>(c, tmap, prm, pl);
    default: return launch_t<B, 8, MODE>(c, tmap, prm, pl);
  }
}

}  // namespace

bool gemv_supported(int64_t K) { return K / 128 <= static_cast<int64_t>(kMaxSplits) * kMaxGroupsPerCta; }

size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)K;
  if (M > 64) return 0;
  const int64_t row_blocks = (N + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8));
  const int64_t mchunks = (M + nt * 8 - 1) / (nt * 8);
  const size_t part = static_cast<size_t>(M) * N * 4;
  const size_t cnt = static_cast<size_t>(row_blocks * mchunks) * 4;
  return ((part + 255) / 256) * 256 + ((cnt + 255) / 256) * 256;
}

cudaError_t launch_gemv(const Ctx& c, const GemvArgs& a) {
  if (!gemv_supported(a.K)) {
    set_error("K = %lld exceeds the supported maximum of %d", static_cast<long long>(a.K),
              kMaxSplits * kMaxGroupsPerCta * 128);
    return cudaErrorInvalidValue;
  }
  const Plan pl = make_plan(a.M, a.N, a.K, c.sm_count);
  if (pl.gper > kMaxGroupsPerCta) {
    set_error("chunked plan: %d groups per CTA exceed %d", pl.gper, kMaxGroupsPerCta);
    return cudaErrorInvalidValue;
  }
  CUtensorMap tmap;
  const uint64_t words = static_cast<uint64_t>(a.K) * a.bits / 32;
  if (!make_tmap_u32_2d(&tmap, a.packed, words, static_cast<uint64_t>(a.N), 4u * a.bits, kRowsPerWarp))
    return cudaErrorInvalidValue;
  Params prm{};
  prm.x = a.x;
  prm.xq = a.xq;
  prm.sx = a.sx;
  prm.scales = a.scales;
  prm.zeros = a.mode == GemvMode::kWna16 ? a.zeros : nullptr;
  prm.M = a.M;
  prm.N = a.N;
  prm.K = a.K;
  prm.G = static_cast<int>(a.K / 128);
  prm.gper = pl.gper;
  prm.y = a.y;
  prm.acc = a.acc;
  prm.status = c.status;
  if (pl.splits > 1 && a.mode != GemvMode::kW4a8GroupAcc) {
    if (a.ws == nullptr) return cudaErrorInvalidValue;
    const size_t part = static_cast<size_t>(a.M) * a.N * 4;
    prm.ws = a.ws;
    prm.counters = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(a.ws) + ((part + 255) / 256) * 256);
  }
  switch (a.mode) {
    case GemvMode::kWna16:
      switch (a.bits) {
        case 2: return launch_nt<2, 0>(c, tmap, prm, pl);
        case 3: return launch_nt<3, 0>(c, tmap, prm, pl);
        case 4: return launch_nt<4, 0>(c, tmap, prm, pl);
        case 5: return launch_nt<5, 0>(c, tmap, prm, pl);
        case 6: return launch_nt<6, 0>(c, tmap, prm, pl);
        case 7: return launch_nt<7, 0>(c, tmap, prm, pl);
        case 8: return launch_nt<8, 0>(c, tmap, prm, pl);
        default: return cudaErrorInvalidValue;
      }
    case GemvMode::kW4a8:
      return launch_nt<4, 1>(c, tmap, prm, pl);
    case GemvMode::kW4a8GroupAcc:
      return launch_nt<4, 2>(c, tmap, prm, pl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
