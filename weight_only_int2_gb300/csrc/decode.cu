// Persistent decode GEMM for M <= 16 tokens: y = x . dequant(W)^T streamed
// from HBM at close to full bandwidth.
//
// Method: "vLLM Can Run INT5-7", section 1 (WNA16 for widths 2..8); model card
// "Qwen3.8-27B-INT6-Mixed-AutoRound", section "Findings" (dense layout,
// symmetric 2^(b-1) zero point, bf16 group-128 scales of any sign); "vLLM
// Quantization", section "Key points" (decode waits on memory); W4A8 per
// "int8 activations (W4A8) ...", section "Under the hood".
//
// Design (GB300):
//  * One CTA of 16 warps per SM, launched cooperatively. The work is cut into
//    units of (32 output rows, one K-split of gs groups). Each CTA owns an
//    equal, contiguous range of units (split-major order, so a CTA touches at
//    most two K-splits); inside the CTA, warps take units dynamically from a
//    shared counter, so no warp idles while another still holds two units.
//  * Each warp runs its own TMA ring over the stages of the units it takes,
//    prefetching across unit boundaries; one stage is 32 rows x one 128-code
//    group, and the first stage of a unit also brings the unit's 32 x gs
//    group scales (second tensor map) into one of two per-warp buffers.
//  * A warp unit is two m16 MMA tiles that share every activation fragment.
//    Unpack (pairing tables of wq_unpack.cuh) happens just in time, four pair
//    registers per row per MMA step; swap-AB m16n8k16, fp32 accumulators.
//  * The activations of the CTA's K-splits are staged once into shared memory
//    in MMA fragment order before the weight prologue is issued, so their
//    small loads are not queued behind the weight traffic.
//  * Split-K partials go to a zero-at-rest fp32 workspace with fire-and-forget
//    atomics. After one bounded grid-wide barrier every CTA converts its slice
//    of the sums to bf16 and zeroes it again. (A per-unit arrival counter with
//    acquire-release semantics serialised every unit's epilogue.)
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_unpack.cuh"

#include <algorithm>

namespace wq {
namespace {

using namespace unpack;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 32;        // output rows per unit
constexpr int kMaxXJobs = 2;     // activation staging jobs per warp (2 splits x NT x gs <= 32)
constexpr size_t kSmemLimit = 227 * 1024;

template <int B>
__host__ __device__ constexpr int stages_for() {
  return B <= 6 ? 3 : 2;
}

struct DParams {
  const uint16_t* x;
  const int8_t* xq;
  const float* sx;
  int64_t M, N, K;
  int G;
  int S;       // K splits
  int gs;      // groups per split (the last split may hold fewer, but >= stages)
  int R;       // 32-row tiles
  int64_t U;   // units = S * R, split-major
  int sbox;    // columns of a scale box (multiple of 8, >= gs + misalignment)
  uint16_t* y;
  int32_t* acc;
  float* ws;
  uint32_t* counters;
  unsigned* status;
};

__device__ __forceinline__ int split_groups(const DParams& p, int s) { return min(p.gs, p.G - s * p.gs); }

template <int B>
__device__ __forceinline__ void unpack_quad(const uint32_t (&w)[B], int i2, uint32_t (&r)[4]) {
  constexpr uint32_t kMagic = uses_fp16<B>() ? 0x64006400u : 0x43004300u;
  constexpr uint32_t kM = (1u << B) - 1u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const PairSpec sp = pair_spec<B>(4 * i2 + q);
    const uint32_t mask = (kM << sp.olo) | (kM << (16 + sp.ohi));
    r[q] = lop3_and_or(slice_window<B>(w, sp.s), mask, kMagic);
  }
}

template <int B, int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ CUtensorMap wmap,
                                                            const __grid_constant__ CUtensorMap smap,
                                                            const DParams p) {
  constexpr int NS = stages_for<B>();
  constexpr int kStageBytes = kRows * 16 * B;  // 32 rows x one group
  constexpr int kStageWords = kStageBytes / 4;
  constexpr bool kF16 = uses_fp16<B>();
  constexpr bool kInt8 = MODE != static_cast<int>(GemvMode::kWna16);
  constexpr bool kAcc = MODE == static_cast<int>(GemvMode::kW4a8GroupAcc);

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_next;             // next CTA-local unit to hand out
  __shared__ int s_uq[kWarps][4];    // per-warp queue of taken units (-1 = none left)
  const int gs = p.gs;
  const int sbox_elems = kRows * p.sbox;
  uint32_t* wring_all = reinterpret_cast<uint32_t*>(smem);
  uint16_t* sbuf_all = reinterpret_cast<uint16_t*>(smem + kWarps * NS * kStageBytes);
  uint4* xs4 = reinterpret_cast<uint4*>(sbuf_all + kWarps * 2 * sbox_elems);
  float* corr = reinterpret_cast<float*>(xs4 + 2 * NT * gs * 128);
  float* scl = corr + 2 * NT * 8 * gs;
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(scl + 2 * NT * 8 * gs);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t cb = static_cast<int64_t>(blockIdx.x) * p.U / gridDim.x;
  const int64_t ce = (static_cast<int64_t>(blockIdx.x) + 1) * p.U / gridDim.x;
  const int nunits = static_cast<int>(ce - cb);
  const int s_first = static_cast<int>(cb / p.R);
  const int r_first = static_cast<int>(cb - static_cast<int64_t>(s_first) * p.R);
  const int s_last = (nunits > 0) ? static_cast<int>((ce - 1) / p.R) : s_first - 1;

  uint32_t* wring = wring_all + warp * NS * kStageWords;
  uint16_t* sbuf = sbuf_all + warp * 2 * sbox_elems;
  uint64_t* bars = bars_all + warp * NS;

  if (threadIdx.x == 0) s_next = 0;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- activation staging, part 1: issue this warp's global loads first
  const int nsplit = s_last - s_first + 1;
  const int xjobs = nsplit * NT * gs;  // warp-jobs (ls, j, gi); each covers one group of 8 tokens
  float xv[kMaxXJobs][32];
  bool xvalid[kMaxXJobs];
#pragma unroll
  for (int q = 0; q < kMaxXJobs; ++q) {
    const int job = warp + q * kWarps;
    const int gi = job % gs, j = (job / gs) % NT, ls = job / (gs * NT);
    const int s = s_first + ls;
    const bool live = job < xjobs && gi < split_groups(p, s) && j * 8 < p.M;
    const int64_t tok = j * 8 + (lane >> 2);
    const bool valid = live && tok < p.M;
    const int64_t k0 = static_cast<int64_t>(s * gs + gi) * 128 + 32 * t;
    const void* src = kInt8 ? static_cast<const void*>(p.xq + (valid ? tok * p.K + k0 : 0))
                            : static_cast<const void*>(p.x + (valid ? tok * p.K + k0 : 0));
    load_slice_x<kInt8>(src, valid, xv[q]);
    xvalid[q] = live;
  }

  // ---- TMA issue side (lane 0): units taken from the CTA counter
  int qw = 0, qr = 0;     // queue write / read positions
  int is_ = 0, ir = 0;    // split and tile of the unit being issued
  int ig = 0, igc = 0;    // group within it, and its group count
  bool more = true;       // units may remain to be issued
  int64_t issued = 0;
  auto take_unit = [&]() {
    const int lu = atomicAdd(&s_next, 1);
    if (lu >= nunits) {
      s_uq[warp][qw++ & 3] = -1;
      more = false;
      return;
    }
    s_uq[warp][qw++ & 3] = lu;
    ir = r_first + lu;
    is_ = s_first;
    if (ir >= p.R) {
      ir -= p.R;
      ++is_;
    }
    ig = 0;
    igc = split_groups(p, is_);
  };
  auto issue_next = [&](int slot) {
    const bool with_scales = ig == 0 && !kAcc;
    mbar_arrive_expect_tx(&bars[slot], kStageBytes + (with_scales ? 2u * sbox_elems : 0u));
    tma_load_2d(wring + slot * kStageWords, &wmap, (is_ * gs + ig) * 4 * B, ir * kRows, &bars[slot]);
    if (with_scales)
      tma_load_2d(sbuf + ((qw - 1) & 1) * sbox_elems, &smap, (is_ * gs) & ~7, ir * kRows, &bars[slot]);
    ++issued;
    if (++ig == igc) take_unit();
  };
  // The weight prologue goes out once this warp's activation loads are in
  // flight (so they are not queued behind it) and fills the ring while the
  // fragments below are built.
  if (lane == 0) {
    take_unit();
    for (int s = 0; s < NS && more; ++s) issue_next(s);
  }
  // ---- activation staging, part 2: fragments, corrections
#pragma unroll
  for (int q = 0; q < kMaxXJobs; ++q) {
    const int job = warp + q * kWarps;
    if (job >= xjobs) break;  // warp-uniform
    const int gi = job % gs, j = (job / gs) % NT, ls = job / (gs * NT);
    uint32_t frag[16];
    float cr, sb;
    make_fragments<B>(xv[q], frag, cr, sb);
    if (xvalid[q]) {
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2)
        xs4[(((ls * NT + j) * gs + gi) * 4 + i2) * 32 + lane] =
            make_uint4(frag[4 * i2], frag[4 * i2 + 1], frag[4 * i2 + 2], frag[4 * i2 + 3]);
      if (t == 0) {
        const int idx = (ls * NT * 8 + j * 8 + (lane >> 2)) * gs + gi;
        corr[idx] = cr;
        scl[idx] = sb;
      }
    }
  }
  __syncthreads();

  // ---- main loop over the units this warp takes
  bool aborted = false;
  int slot = 0;          // ring slot of the next stage to consume
  uint32_t phase = 0;    // its mbarrier phase parity
  int64_t consumed = 0;  // stages consumed
  while (!aborted) {
    __syncwarp();  // lane 0's queue writes before every lane's read
    const int lu = s_uq[warp][qr & 3];
    const int par = qr & 1;
    ++qr;
    if (lu < 0) break;
    int r = r_first + lu, s = s_first;
    if (r >= p.R) {
      r -= p.R;
      ++s;
    }
    const int gc = split_groups(p, s);
    const int ls = s - s_first;
    const uint16_t* sunit = sbuf + par * sbox_elems + ((s * gs) & 7);
    const int64_t row0 = static_cast<int64_t>(r) * kRows + g;  // rows row0 + {0, 8, 16, 24}
    float acc[NT][2][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][h][e] = 0.0f;

    for (int gi = 0; gi < gc; ++gi) {
      if (!mbar_wait_bounded(&bars[slot], phase)) {
        record_status(p.status, kStatusTimeout);
        aborted = true;
        break;
      }
      const uint32_t* st = wring + slot * kStageWords;
      uint32_t w0[B], w1[B], w2[B], w3[B];
      load_slice<B>(st, g, t, w0);
      load_slice<B>(st, g + 8, t, w1);
      load_slice<B>(st, g + 16, t, w2);
      load_slice<B>(st, g + 24, t, w3);
      float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (!kAcc) {
#pragma unroll
        for (int q = 0; q < 4; ++q) sc[q] = bf16_bits_to_float(sunit[(g + 8 * q) * p.sbox + gi]);
      }
      float c[NT][2][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[j][h][e] = 0.0f;
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        uint32_t a0[4], a1[4], a2[4], a3[4];
        unpack_quad<B>(w0, i2, a0);
        unpack_quad<B>(w1, i2, a1);
        unpack_quad<B>(w2, i2, a2);
        unpack_quad<B>(w3, i2, a3);
        if (i2 == 3) {
          // every lane has read its slices: the slot may be refilled
          __syncwarp();
          if (lane == 0 && more) issue_next(slot);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint4 bv = xs4[(((ls * NT + j) * gs + gi) * 4 + i2) * 32 + lane];
          mma16<kF16>(c[j][0], a0[0], a1[0], a0[1], a1[1], bv.x, bv.y);
          mma16<kF16>(c[j][1], a2[0], a3[0], a2[1], a3[1], bv.x, bv.y);
          mma16<kF16>(c[j][0], a0[2], a1[2], a0[3], a1[3], bv.z, bv.w);
          mma16<kF16>(c[j][1], a2[2], a3[2], a2[3], a3[3], bv.z, bv.w);
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int ti0 = (ls * NT * 8 + j * 8 + 2 * t) * gs + gi, ti1 = ti0 + gs;
        const float cr0 = corr[ti0], cr1 = corr[ti1], sl0 = scl[ti0], sl1 = scl[ti1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float d0 = fmaf(sl0, c[j][h][0], -cr0);
          const float d1 = fmaf(sl1, c[j][h][1], -cr1);
          const float d2 = fmaf(sl0, c[j][h][2], -cr0);
          const float d3 = fmaf(sl1, c[j][h][3], -cr1);
          if constexpr (kAcc) {
            const int64_t tk0 = j * 8 + 2 * t, tk1 = tk0 + 1;
            const int64_t G = p.G, gabs = static_cast<int64_t>(s) * gs + gi;
            const int64_t ra = row0 + 16 * h, rb = ra + 8;
            if (ra < p.N) {
              if (tk0 < p.M) p.acc[(tk0 * p.N + ra) * G + gabs] = __float2int_rn(d0);
              if (tk1 < p.M) p.acc[(tk1 * p.N + ra) * G + gabs] = __float2int_rn(d1);
            }
            if (rb < p.N) {
              if (tk0 < p.M) p.acc[(tk0 * p.N + rb) * G + gabs] = __float2int_rn(d2);
              if (tk1 < p.M) p.acc[(tk1 * p.N + rb) * G + gabs] = __float2int_rn(d3);
            }
          } else {
            acc[j][h][0] = fmaf(sc[2 * h], d0, acc[j][h][0]);
            acc[j][h][1] = fmaf(sc[2 * h], d1, acc[j][h][1]);
            acc[j][h][2] = fmaf(sc[2 * h + 1], d2, acc[j][h][2]);
            acc[j][h][3] = fmaf(sc[2 * h + 1], d3, acc[j][h][3]);
          }
        }
      }
      ++consumed;
      if (++slot == NS) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (aborted) break;

    // ---- unit epilogue: partial sums (or the final value when S == 1)
    if constexpr (!kAcc) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t row = row0 + 16 * h + ((e >> 1) << 3);
            const int64_t tok = j * 8 + 2 * t + (e & 1);
            if (row >= p.N || tok >= p.M) continue;
            float v = acc[j][h][e];
            if constexpr (MODE == static_cast<int>(GemvMode::kW4a8)) v *= p.sx[tok];
            if (p.S == 1) {
              p.y[tok * p.N + row] = float_to_bf16_bits_rn(v);
            } else {
              atomicAdd(p.ws + tok * p.N + row, v);
            }
          }
        }
      }
    }
  }

  // Drain: if a wait gave up, give the copies still in flight a bounded chance
  // to land before the CTA's shared memory is released.
  if (aborted && lane == 0) {
    for (int64_t q = consumed; q < issued; ++q) {
      mbar_wait_bounded(&bars[slot], phase);
      if (++slot == NS) {
        slot = 0;
        phase ^= 1u;
      }
    }
  }

  // ---- split-K finish: one grid-wide barrier (the launch is cooperative, so
  // every CTA is resident), then each CTA converts its slice of the fp32
  // partial sums to bf16 and zeroes those workspace cells again.
  if constexpr (!kAcc) {
    if (p.S > 1) {
      __shared__ int s_ok;
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned* arrive = p.counters;
        unsigned* flag = p.counters + 1;
        __threadfence();  // this CTA's partial sums before its arrival
        const unsigned old = atomicAdd(arrive, 1u);
        int ok = 1;
        if (old == gridDim.x - 1) {
          *arrive = 0u;
          __threadfence();
          atomicExch(flag, 1u);
        } else {
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(flag) == 0u) {
            __nanosleep(256);
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              record_status(p.status, kStatusTimeout);
              ok = 0;
              break;
            }
          }
        }
        __threadfence();
        s_ok = ok;
      }
      __syncthreads();
      const int64_t total = p.M * p.N;
      const int64_t per = (total + gridDim.x - 1) / gridDim.x;
      const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
      const int64_t b1 = min(total, b0 + per);
      for (int64_t i = b0 + threadIdx.x; i < b1; i += kThreads) {
        p.y[i] = float_to_bf16_bits_rn(__ldcg(p.ws + i));
        p.ws[i] = 0.0f;
      }
      // leave: the last CTA out re-arms the barrier for the next launch
      __syncthreads();
      if (threadIdx.x == 0 && s_ok) {
        unsigned* leave = p.counters + 2;
        __threadfence();
        if (atomicAdd(leave, 1u) == gridDim.x - 1) {
          *leave = 0u;
          p.counters[1] = 0u;
        }
      }
    }
  }
}

size_t dsmem_bytes(int B, int NT, int gs, int sbox) {
  const int NS = B <= 6 ? 3 : 2;
  return static_cast<size_t>(kWarps) * NS * kRows * 16 * B   // weight rings
         + static_cast<size_t>(kWarps) * 2 * kRows * sbox * 2  // scale boxes
         + static_cast<size_t>(2) * NT * gs * 128 * 16       // B fragments
         + static_cast<size_t>(2) * NT * 8 * gs * 4 * 2      // corrections, range factors
         + static_cast<size_t>(kWarps) * NS * 8;             // mbarriers
}

struct DPlan {
  int nt, S, gs, R, sbox;
  int64_t U;
  bool ok;
};

DPlan make_dplan(int64_t M, int64_t N, int64_t K, int bits, int sm_count) {
  DPlan pl{};
  pl.ok = false;
  // K % 1024 == 0 keeps the rows of the scale matrix 16-byte multiples (TMA)
  if (M > 16 || K % 1024 != 0) return pl;
  const int NS = bits <= 6 ? 3 : 2;
  pl.nt = M <= 8 ? 1 : 2;
  const int G = static_cast<int>(K / 128);
  pl.R = static_cast<int>((N + kRows - 1) / kRows);
  double best = -1.0;
  for (int s = 1; s <= G; ++s) {
    const int gs = (G + s - 1) / s;
    const int S = (G + gs - 1) / gs;
    // activations of two splits must fit the per-warp staging jobs
    if (2 * pl.nt * gs > kMaxXJobs * kWarps) continue;
    // every unit holds >= NS groups: the TMA lookahead spans at most the next
    // unit, so two scale buffers per warp suffice
    if (gs < NS || G - (S - 1) * gs < NS) continue;
    const int64_t U = static_cast<int64_t>(S) * pl.R;
    const int64_t per_cta = (U + sm_count - 1) / sm_count;
    if (per_cta + 1 > pl.R) continue;  // a CTA must touch at most two splits
    const int sbox = ((gs + 7 + 7) / 8) * 8;
    if (dsmem_bytes(bits, pl.nt, gs, sbox) > kSmemLimit) continue;
    // Busiest warp: units are handed out dynamically inside a CTA, so it
    // holds ceil(per_cta / 16) units; CTAs also drift apart by about half a
    // unit. Partial sums cost atomics per split.
    const int64_t per_warp = (per_cta + kWarps - 1) / kWarps;
    const double cost = static_cast<double>(per_warp) * gs + 0.5 * gs +
                        (S > 1 ? 0.25 * static_cast<double>(M) * S * N / (sm_count * 1024.0) : 0.0);
    if (best < 0 || cost < best - 1e-9) {
      best = cost;
      pl.S = S;
      pl.gs = gs;
      pl.U = U;
      pl.sbox = sbox;
    }
  }
  pl.ok = best >= 0;
  return pl;
}

template <int B, int NT, int MODE>
cudaError_t dlaunch(const Ctx& c, const CUtensorMap& wmap, const CUtensorMap& smap, const DParams& prm) {
  // Raise the per-device dynamic shared-memory opt-in when a launch needs more
  // than any earlier one did.
  static SmemLimit limit;
  const size_t smem = dsmem_bytes(B, NT, prm.gs, prm.sbox);
  const cudaError_t e = raise_smem_limit(limit, decode_kernel<B, NT, MODE>, c.device, smem);
  if (e != cudaSuccess) return e;
  // Cooperative launch: the split-K finish waits on every CTA of the grid,
  // which is only safe when all of them are guaranteed to be resident.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(c.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<B, NT, MODE>, wmap, smap, prm);
}

template <int B, int MODE>
cudaError_t dlaunch_nt(const Ctx& c, int nt, const CUtensorMap& wmap, const CUtensorMap& smap,
                       const DParams& prm) {
  return nt == 1 ? dlaunch<B, 1, MODE>(c, wmap, smap, prm) : dlaunch<B, 2, MODE>(c, wmap, smap, prm);
}

}  // namespace

size_t decode_workspace_bytes(int64_t M, int64_t N) {
  if (M > 16) return 0;
  const size_t part = static_cast<size_t>(M) * N * 4;
  return ((part + 255) / 256) * 256 + 256;  // partial sums, then the grid-barrier words
}

bool decode_supported(int64_t M, int64_t N, int64_t K, int bits, int sm_count) {
  return make_dplan(M, N, K, bits, sm_count).ok;
}

cudaError_t launch_decode(const Ctx& c, const GemvArgs& a) {
  const DPlan pl = make_dplan(a.M, a.N, a.K, a.bits, c.sm_count);
  if (!pl.ok) return cudaErrorInvalidValue;
  CUtensorMap wmap, smap;
  const uint64_t words = static_cast<uint64_t>(a.K) * a.bits / 32;
  if (!make_tmap_u32_2d(&wmap, a.packed, words, static_cast<uint64_t>(a.N), 4u * a.bits, kRows))
    return cudaErrorInvalidValue;
  if (a.mode != GemvMode::kW4a8GroupAcc) {
    if (!make_tmap_bf16_2d(&smap, a.scales, static_cast<uint64_t>(a.K / 128), static_cast<uint64_t>(a.N),
                           static_cast<uint32_t>(pl.sbox), kRows))
      return cudaErrorInvalidValue;
  } else {
    smap = wmap;  // unused
  }
  DParams prm{};
  prm.x = a.x;
  prm.xq = a.xq;
  prm.sx = a.sx;
  prm.M = a.M;
  prm.N = a.N;
  prm.K = a.K;
  prm.G = static_cast<int>(a.K / 128);
  prm.S = pl.S;
  prm.gs = pl.gs;
  prm.R = pl.R;
  prm.U = pl.U;
  prm.sbox = pl.sbox;
  prm.y = a.y;
  prm.acc = a.acc;
  prm.status = c.status;
  if (pl.S > 1 && a.mode != GemvMode::kW4a8GroupAcc) {
    if (a.ws == nullptr) return cudaErrorInvalidValue;
    const size_t part = static_cast<size_t>(a.M) * a.N * 4;
    prm.ws = a.ws;
    prm.counters = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(a.ws) + ((part + 255) / 256) * 256);
  }
  switch (a.mode) {
    case GemvMode::kWna16:
      switch (a.bits) {
        case 2: return dlaunch_nt<2, 0>(c, pl.nt, wmap, smap, prm);
        case 3: return dlaunch_nt<3, 0>(c, pl.nt, wmap, smap, prm);
        case 4: return dlaunch_nt<4, 0>(c, pl.nt, wmap, smap, prm);
        case 5: return dlaunch_nt<5, 0>(c, pl.nt, wmap, smap, prm);
        case 6: return dlaunch_nt<6, 0>(c, pl.nt, wmap, smap, prm);
        case 7: return dlaunch_nt<7, 0>(c, pl.nt, wmap, smap, prm);
        case 8: return dlaunch_nt<8, 0>(c, pl.nt, wmap, smap, prm);
        default: return cudaErrorInvalidValue;
      }
    case GemvMode::kW4a8:
      return dlaunch_nt<4, 1>(c, pl.nt, wmap, smap, prm);
    case GemvMode::kW4a8GroupAcc:
      return dlaunch_nt<4, 2>(c, pl.nt, wmap, smap, prm);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
