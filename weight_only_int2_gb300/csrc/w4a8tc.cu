// W4A8 GEMM for many tokens on the 5th-generation tensor cores, with the
// integer accumulation per quantization group that the method prescribes.
//
// Method: "int8 activations (W4A8) are now a one-flag serve-time knob ...",
// section "Under the hood": activations quantized per token to int8, int4
// weight codes widened losslessly to int8, integer accumulation, then the
// group scale (either sign) and the token scale:
//   acc[m, n, g] = sum_{k in group g} xq[m, k] * (q[n, k] - 8)
//   y[m, n]      = sx[m] * sum_g s[n, g] * acc[m, n, g].
//
// Exactness: the A operand is q - 8 (in [-8, 7]) and the B operand the int8
// code xq (in [-127, 127]), both exact in bf16; every product is an integer
// of magnitude <= 1016 and every partial sum of a group of 128 stays below
// 2^17, so the fp32 accumulation of one group in tensor memory is the exact
// integer acc[m, n, g] whatever the order. Each group therefore gets its own
// accumulator; the scale is applied in fp32 when the group is read out.
//
// Persistent kernel, one CTA per SM; a tile is 128 weight rows (MMA M) x TN
// tokens (MMA N): 160, or 128 where 160 would pad the tokens more. Tensor
// memory (512 columns): two group accumulators of TN columns (group g in
// buffer g % 2, so the MMAs of one group overlap the read-out of the other)
// and a ring of kNA = (512 - 2 TN) / 32 stages of the A operand, 64 codes
// each (8 stages at TN = 128, 6 at TN = 160).
// Warp roles (24 warps in six warpgroups). Reading a group out and writing
// the A operand are done by different warps, so that neither waits for the
// other: an accumulator is freed as soon as its MMAs end, and the A operand
// of the next groups is written while they run. The read-out warpgroups take
// 96 registers a thread (setmaxnreg) from the two others, which keep 48, so
// that every read-out load of a group is in flight at once.
//   warp 0      TMA producer for the activation codes [TN x 64] (bf16,
//               128-byte swizzle, zero fill past M) of each stage.
//   warp 1      allocates tensor memory; one thread issues, per group, the
//               waits for its accumulator and its two stages, one fence, 8
//               MMAs of K = 16 and one commit (the group's barrier: its
//               accumulator is complete and its slots are free).
//   warp 2      TMA producer for the packed 4-bit weights, one group
//               [128 rows x 64 bytes] per load.
//   warp 3      idle (completes the first warpgroup).
//   warps 4-7   the A operand: a thread turns the 128 codes of one weight row
//               of a group into q - 8 and stores them to its TMEM lane (the
//               group's two stages), once the MMAs that read those slots
//               before have ended.
//   warps 8-23  read-out: warp (set c, quarter) takes token columns
//               c TN / 4 .. + TN / 4 - 1 of its 32 rows of every group (all
//               its loads in flight at once, one wait), frees the
//               accumulator and adds s[n, g] * acc into fp32 running sums;
//               after the last group of a tile it stores bf16(sx[m] * sum).
// kAcc: write the exact accumulators acc[m, n, g] as int32 instead of y (the
// test and debug mode of the same kernel).
// All mbarrier waits are bounded; a timeout records WQ_ETIMEOUT and every
// role stops early (outputs are then incomplete).
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kNB = 8;          // stage barriers (full), indexed by stage mod 8
constexpr int kNG = 8;          // group barriers (gdone), indexed by group mod 8
constexpr int kTmemCols = 512;
constexpr int kMaxNX = 8;       // activation stages in shared memory (<= kNB)
constexpr int kMaxNP = 8;       // packed-weight slots, one group each (even)
constexpr int kAWarps = 4;      // the A operand: one warp per TMEM lane quarter
constexpr int kRWarps = 16;     // read-out: 4 column sets x 4 lane quarters
constexpr int kAWarp0 = 4;
constexpr int kRWarp0 = kAWarp0 + kAWarps;
constexpr int kThreads = (kRWarp0 + kRWarps) * 32;  // 768: 80 registers a thread at launch
// setmaxnreg split of the 768 x 80 registers the block is launched with:
// warpgroups 0 and 1 (producers, MMA, A operand) give 32 each of theirs to
// the four read-out warpgroups: 256 x 48 + 512 x 96 = 768 x 80.
constexpr int kRegsLow = 48, kRegsHigh = 96;
static_assert(256 * kRegsLow + 512 * kRegsHigh <= kThreads * 80, "register split above the launch's registers");
constexpr int kPSlot = kBM * 64;                    // one group of 128 rows of 4-bit codes

template <int TN>
struct WLayout {
  static constexpr int kNA = (kTmemCols - 2 * TN) / 32;  // A stages in tensor memory
  static constexpr int kACol = 2 * TN;                    // A ring: columns [2 TN, 512)
  static_assert(kNA >= 4 && kNA % 2 == 0 && kNA <= kNB, "A ring must hold whole groups");
  static constexpr int kCols = TN / 4;  // token columns of one read-out warp
  static_assert(kCols % 8 == 0, "read-out in loads of eight columns");
  static constexpr int kXStage = TN * kBK * 2;
  static constexpr int kBudget = 227 * 1024 - 1024 - 512;  // minus alignment slack and static smem
  static constexpr bool fits(int nx, int np) { return nx * kXStage + np * kPSlot <= kBudget; }
  static constexpr int pick_nx() {
    for (int nx = kMaxNX; nx >= 3; --nx)
      if (fits(nx, 4)) return nx;
    return 0;
  }
  static constexpr int kNX = pick_nx();
  static constexpr int pick_np() {
    for (int np = kMaxNP; np >= 2; np -= 2)
      if (fits(kNX, np)) return np;
    return 0;
  }
  static constexpr int kNP = pick_np();
  static_assert(kNX >= 3 && kNP >= 4 && kNP % 2 == 0, "W4A8 rings do not fit shared memory");
  static constexpr int kPOff = kNX * kXStage;
  static constexpr size_t kSmem = static_cast<size_t>(kPOff + kNP * kPSlot) + 1024;  // + alignment slack
};

struct WParams {
  const uint16_t* scales;  // bf16 [N, G]
  int64_t M, N, K;
  int G;
  int row_tiles, tok_tiles;  // ceil(N / 128), ceil(M / TN)
  uint16_t* y;               // bf16 [M, N]
  const float* sx;           // per-token scale [M]
  int32_t* acc;              // kAcc: int32 [M, N, G]
  unsigned* status;
};

// 32 codes of 4 bits (4 words, LSB-first) -> 16 words of bf16 pairs
// (q - 8), exactly: word i holds codes 8i .. 8i + 7, and output column
// 4i + j holds the pair (8i + j, 8i + j + 4), which one shift and one AND-OR
// put into the mantissas of bf16 128.0 (unit spacing); 136 = 128 + 8 is
// then subtracted. The activation codes are staged in the same K order
// (within each block of 8: 0, 4, 1, 5, 2, 6, 3, 7), so the products pair up.
__device__ __forceinline__ void exact_slice4(const uint32_t (&w)[4], uint32_t (&o)[16]) {
  constexpr uint32_t kMagic = 0x43004300u;  // bf16 (128, 128)
  constexpr uint32_t kZ2 = 0x43084308u;     // bf16 (136, 136)
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t v = lop3_and_or(w[c >> 2] >> (4 * (c & 3)), 0x000F000Fu, kMagic);
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(kZ2));
    o[c] = r;
  }
}

template <int TN, bool kAcc>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                   const WParams p) {
  using L = WLayout<TN>;
  constexpr int NX = L::kNX, NA = L::kNA, NP = L::kNP, kCols = L::kCols;
  extern __shared__ uint8_t smem_raw[];
  // full[j]: stage (j mod kNB) has its activation bytes and its A operand
  //          (arrivals: the activation producer's expect-tx + the A warps);
  // gdone[g]: the MMAs of group (g mod kNG) completed (one commit per group,
  //          after both its stages): the group's accumulator is complete, its
  //          two A slots are free and, NX stages later in the sequence, its
  //          activation slots;
  // pfull/pempty: packed-weight slots;
  // acce[b]: group accumulator b read out.
  __shared__ __align__(8) uint64_t full[kNB], gdone[kNG], pfull[kMaxNP], pempty[kMaxNP], acce[2];
  // the group barrier that releases stage j of the sequence, and its phase
  auto gbar = [&](uint32_t j) -> uint64_t* { return &gdone[(j >> 1) % kNG]; };
  auto gphase = [](uint32_t j) -> uint32_t { return ((j >> 1) / kNG) & 1u; };
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* xs = base;
  uint8_t* ps = base + L::kPOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int S = 2 * G;  // stages per tile
  // static schedule: tiles blockIdx.x, blockIdx.x + gridDim.x, ...; row
  // tiles vary fastest so that CTAs running together share activation tiles
  const int first = blockIdx.x, step = gridDim.x;
  const int ntiles = p.row_tiles * p.tok_tiles;
  const int my_tiles = first < ntiles ? (ntiles - 1 - first) / step + 1 : 0;
  const uint32_t total_groups = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNB; ++s) mbar_init(&full[s], kAWarps + 1);
    for (int s = 0; s < kNG; ++s) mbar_init(&gdone[s], 1);
    for (int s = 0; s < NP; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], kAWarps);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&acce[b], kRWarps);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp < kAWarp0) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
  if (warp == 0) {
    // ---- activation codes: stage i of a tile covers k = 64 i .. 64 i + 63;
    // slot it % NX is free once stage it - NX is done (NX <= kNB: the done
    // barrier of that stage cannot be a whole lap ahead)
    if (lane == 0) {
      uint32_t it = 0;
      for (int t = first; t < ntiles && !s_abort; t += step) {
        const int m0 = (t / p.row_tiles) * TN;
        for (int i = 0; i < S; ++i, ++it) {
          if (it >= static_cast<uint32_t>(NX)) {
            const uint32_t j = it - NX;
            if (!mbar_wait_backoff<256>(gbar(j), gphase(j))) {
              record_status(p.status, kStatusTimeout);
              s_abort = 1;
              break;
            }
          }
          uint64_t* fb = &full[it % kNB];
          mbar_arrive_expect_tx(fb, L::kXStage);
          tma_load_2d(xs + (it % NX) * L::kXStage, &xmap, i * kBK, m0, fb);
        }
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- packed weights: group gi into slot gi % NP
    if (lane == 0) {
      uint32_t gi = 0;
      for (int t = first; t < ntiles && !s_abort; t += step) {
        const int n0 = (t % p.row_tiles) * kBM;
        for (int g = 0; g < G; ++g, ++gi) {
          const uint32_t sl = gi % NP;
          if (gi >= static_cast<uint32_t>(NP) && !mbar_wait_backoff<256>(&pempty[sl], ((gi / NP) - 1) & 1)) {
            record_status(p.status, kStatusTimeout);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&pfull[sl], kPSlot);
          tma_load_2d(ps + sl * kPSlot, &wmap, g * 16, n0, &pfull[sl]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue (one thread): group gi accumulates into buffer gi % 2,
    // once the group that used that buffer before has been read out
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kBM, TN);
      uint32_t it = 0;
      bool ok = true;
      for (uint32_t gi = 0; gi < total_groups && ok; ++gi) {
        const uint32_t b = gi & 1u;
        if (gi >= 2 && (s_abort || !mbar_wait_bounded(&acce[b], ((gi >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        // both stages of the group, then one fence, 8 MMAs and one commit
        if (s_abort || !mbar_wait_bounded(&full[it % kNB], (it / kNB) & 1) ||
            !mbar_wait_bounded(&full[(it + 1) % kNB], ((it + 1) / kNB) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t bb = smem_u32(xs + ((it + h) % NX) * L::kXStage);
          const uint32_t aa = tmem + L::kACol + ((it + h) % NA) * (kBK / 2);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_ta(tmem + b * TN, aa + 8 * kk, sw128_desc(bb + 32 * kk), idesc, (h > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(gbar(it));  // fires when the group's MMAs complete
        it += 2;
      }
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // idle
  } else if (warp < kRWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    // ---- A operand (warps 4..7). Warp w owns TMEM lane quarter q = w % 4
    // (rows 32 q .. 32 q + 31 of the tile) and writes stages 2 gi, 2 gi + 1
    // of every group gi into slots (2 gi) % NA, (2 gi + 1) % NA, once the
    // MMAs of the group NA / 2 before (the slots' previous group) have
    // completed.
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    for (uint32_t gi = 0; gi < total_groups; ++gi) {
      const uint32_t it = 2 * gi, pslot = gi % NP;
      bool go = !s_abort;
      if (go) go = mbar_wait_bounded(&pfull[pslot], (gi / NP) & 1);
      if (go && it >= static_cast<uint32_t>(NA)) go = mbar_wait_bounded(gbar(it - NA), gphase(it - NA));
      if (!__all_sync(0xFFFFFFFFu, go)) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        break;
      }
      // row r: the four 16-byte chunks of the 64-byte row, loaded with the
      // TMA 64-byte swizzle (chunk c sits at c ^ ((r >> 1) & 3))
      const uint8_t* prow = ps + pslot * kPSlot + r * 64;
      uint4 v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint4*>(prow + ((c ^ packed_xor<4>(r)) << 4));
      // the slot may be refilled once every lane's reads are done: the refill
      // is a TMA (async-proxy) write, which these generic-proxy reads are
      // ordered before only by a proxy fence in each reading thread
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pempty[pslot]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // chunk c: codes 32 c .. 32 c + 31 = half c % 2 of stage it + c / 2
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        uint32_t o[16];
        exact_slice4(w, o);
        tmem_st16(tmem + lane_base + L::kACol + ((it + c / 2) % NA) * (kBK / 2) + 16 * (c & 1), o);
      }
      tmem_wait_st();
      tc_fence_before();  // the A tiles before the arrivals the MMA waits on
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full[it % kNB]);
        mbar_arrive(&full[(it + 1) % kNB]);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ---- read-out (warps 8..23). Warp w owns TMEM lane quarter q = w % 4
    // (rows 32 q .. 32 q + 31) and token columns c kCols .. + kCols - 1,
    // c = (w - 8) / 4, of every group's accumulator.
    const int cset = (warp - kRWarp0) / 4;
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float run[kCols];
#pragma unroll
    for (int j = 0; j < kCols; ++j) run[j] = 0.0f;
    // group gi of the sequence is group g of tile t; the row, the token
    // columns and the scale row change once per tile (no division per group)
    int t = first, g = 0;
    int64_t n = static_cast<int64_t>(t % p.row_tiles) * kBM + r;
    int64_t m0 = static_cast<int64_t>(t / p.row_tiles) * TN + cset * kCols;
    // the scale s[n, g] of the group read out next, loaded one group ahead
    float s_next = (!kAcc && my_tiles > 0 && n < p.N) ? bf16_bits_to_float(p.scales[n * G]) : 0.0f;
    for (uint32_t gi = 0; gi < total_groups; ++gi) {
      const uint32_t b = gi & 1u;
      if (!__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_bounded(&gdone[gi % kNG], (gi / kNG) & 1))) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        break;
      }
      tc_fence_after();
      const float sc = s_next;
      if constexpr (!kAcc) {
        if (g + 1 < G) {
          s_next = n < p.N ? bf16_bits_to_float(p.scales[n * G + g + 1]) : 0.0f;
        } else if (t + step < ntiles) {
          const int64_t n2 = static_cast<int64_t>((t + step) % p.row_tiles) * kBM + r;
          s_next = n2 < p.N ? bf16_bits_to_float(p.scales[n2 * G]) : 0.0f;
        }
      }
      const uint32_t col0 = tmem + lane_base + b * TN + cset * kCols;
      // every load of the warp's columns in flight, one wait, then free the
      // buffer and use the values
      uint32_t v[kCols];
      tmem_ld_cols<kCols>(col0, v);
      tmem_wait_ld_all<kCols>(v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
      if constexpr (kAcc) {
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < kCols; ++j) {
            const int64_t m = m0 + j;
            if (m < p.M) p.acc[(m * p.N + n) * G + g] = __float2int_rn(__uint_as_float(v[j]));
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < kCols; ++j) run[j] = fmaf(sc, __uint_as_float(v[j]), run[j]);
      }
      if constexpr (!kAcc) {
        if (g == G - 1) {
          // the tile's last group: y = bf16(sx[m] * sum), then start over
          if (n < p.N) {
            uint16_t* dst = p.y + m0 * p.N + n;
            // eight token columns at a time (the compiler barrier keeps the
            // token-scale loads of later columns from being hoisted, which
            // would need registers beside the running sums)
#pragma unroll
            for (int j0 = 0; j0 < kCols; j0 += 8) {
#pragma unroll
              for (int j = j0; j < j0 + 8; ++j) {
                const int64_t m = m0 + j;
                if (m < p.M) dst[static_cast<int64_t>(j) * p.N] = float_to_bf16_bits_rn(run[j] * p.sx[m]);
              }
              asm volatile("" ::: "memory");
            }
          }
#pragma unroll
          for (int j = 0; j < kCols; ++j) run[j] = 0.0f;
        }
      }
      if (++g == G) {  // next tile
        g = 0;
        t += step;
        n = static_cast<int64_t>(t % p.row_tiles) * kBM + r;
        m0 = static_cast<int64_t>(t / p.row_tiles) * TN + cset * kCols;
      }
    }
  }

  // every warp arrives here converged (role branches end with __syncwarp or
  // are warp-uniform), so the barrier waits for all of them
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int TN, bool kAcc>
cudaError_t wlaunch(const Ctx& c, const CUtensorMap& xmap, const CUtensorMap& wmap, const WParams& prm) {
  constexpr size_t smem = WLayout<TN>::kSmem;
  static_assert(smem <= 227 * 1024, "W4A8 stage layout exceeds shared memory");
  static SmemLimit limit;
  const cudaError_t e = raise_smem_limit(limit, w4a8_tc_kernel<TN, kAcc>, c.device, smem);
  if (e != cudaSuccess) return e;
  WParams q = prm;
  q.row_tiles = static_cast<int>((prm.N + kBM - 1) / kBM);
  q.tok_tiles = static_cast<int>((prm.M + TN - 1) / TN);
  const int tiles = q.row_tiles * q.tok_tiles;
  const int grid = tiles < c.sm_count ? tiles : c.sm_count;  // persistent: one CTA per SM
  w4a8_tc_kernel<TN, kAcc><<<grid, kThreads, smem, c.stream>>>(xmap, wmap, q);
  return cudaGetLastError();
}

template <int TN>
cudaError_t launch_tn(const Ctx& c, const uint16_t* xqb, const uint32_t* packed4, const WParams& prm) {
  CUtensorMap xmap, wmap;
  if (!make_tmap_bf16_2d_sw128(&xmap, xqb, static_cast<uint64_t>(prm.K), static_cast<uint64_t>(prm.M), kBK, TN))
    return cudaErrorInvalidValue;
  // 4-bit rows of a group are 64 bytes: loaded with the 64-byte swizzle so
  // that the rows of a tile spread over the shared-memory banks
  if (!make_tmap_u32_2d(&wmap, packed4, static_cast<uint64_t>(prm.K) / 8, static_cast<uint64_t>(prm.N), 16u, kBM,
                        64))
    return cudaErrorInvalidValue;
  return prm.acc != nullptr ? wlaunch<TN, true>(c, xmap, wmap, prm) : wlaunch<TN, false>(c, xmap, wmap, prm);
}

// Tokens per tile: 160 (less A-operand work per token) unless its last tile
// would pad the tokens by more than a few per cent beyond 128-token tiles.
int w4a8_tile_tokens(int64_t M) {
  const int64_t p128 = (M + 127) / 128 * 128, p160 = (M + 159) / 160 * 160;
  return p160 * 100 <= p128 * 104 ? 160 : 128;
}

}  // namespace

cudaError_t launch_w4a8_tc(const Ctx& c, const uint16_t* xqb, const float* sx, const uint32_t* packed4,
                           const uint16_t* scales, int64_t M, int64_t N, int64_t K, uint16_t* y, int32_t* acc) {
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return cudaErrorInvalidValue;
  WParams prm{};
  prm.scales = scales;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.G = static_cast<int>(K / 128);
  prm.y = y;
  prm.sx = sx;
  prm.acc = acc;
  prm.status = c.status;
  return w4a8_tile_tokens(M) == 160 ? launch_tn<160>(c, xqb, packed4, prm) : launch_tn<128>(c, xqb, packed4, prm);
}

}  // namespace wq
