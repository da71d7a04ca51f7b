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
// = 128 tokens (MMA N). Tensor memory (512 columns): two group accumulators
// of TN columns (group g in buffer g % 2, so the MMAs of one group overlap
// the read-out of the other) and a ring of kNA = (512 - 2 TN) / 32 = 8
// stages of the A operand (64 codes each).
// Warp roles:
//   warp 0      TMA producer for the activation codes [TN x 64] (bf16,
//               128-byte swizzle, zero fill past M) of each stage.
//   warp 1      allocates tensor memory; one thread issues, per group, the
//               waits for its accumulator and its two stages, one fence, 8
//               MMAs of K = 16 and one commit (the group's barrier: its
//               accumulator is complete and its slots are free).
//   warp 2      TMA producer for the packed 4-bit weights, one group
//               [128 rows x 64 bytes] per load.
//   warps 3-18  four teams of 4 warps. Team j writes the A operand of the
//               stages j (mod 4): a thread turns the 64 codes of one weight
//               row into q - 8 and stores them to its TMEM lane. Every one of
//               the 16 warps reads out every group: warp (j, quarter) takes
//               TN / 4 token columns of its 32 rows, frees the accumulator,
//               and adds s[n, g] * acc into fp32 running sums; after the last
//               group of a tile it stores bf16(sx[m] * sum). A warp reads a
//               group out as soon as its MMAs end, then writes the A operand
//               of the group kNA / 2 ahead into the slots they freed, so the
//               tensor core always has the next groups queued.
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
constexpr int kNP = 4;          // packed-weight slots, one group each (even)
constexpr int kTeamWarps = 4;   // one team: 128 rows x 64 codes
constexpr int kTeams = 4;       // team j takes stages j (mod 4)
constexpr int kDeqWarps = kTeams * kTeamWarps;
constexpr int kThreads = (3 + kDeqWarps) * 32;  // 608
constexpr int kPSlot = kBM * 64;                // one group of 128 rows of 4-bit codes
// Tokens per tile (MMA N). 128 leaves room for an 8-stage A ring beside the
// two accumulators and keeps the running sums (32 per thread) in registers;
// 192 (a 4-stage ring, 48 sums) measured slower at every token count from
// 512 to 8192, its running sums spilling at the register limit of 19 warps.
constexpr int kTN = 128;

template <int TN>
struct WLayout {
  static constexpr int kNA = (kTmemCols - 2 * TN) / 32;  // A stages in tensor memory
  static constexpr int kACol = 2 * TN;                    // A ring: columns [2 TN, 512)
  static constexpr int kLead = kNA / 2;                   // groups of A a warp writes ahead
  static_assert(kNA >= 4 && kNA % kTeams == 0 && kNA <= kNB, "A ring must give each team whole slots");
  static constexpr int kXStage = TN * kBK * 2;
  static constexpr int kBudget = 227 * 1024 - 1024 - 512;  // minus alignment slack and static smem
  static constexpr int pick_nx() {
    for (int nx = kMaxNX; nx >= 3; --nx)
      if (nx * kXStage + kNP * kPSlot <= kBudget) return nx;
    return 0;
  }
  static constexpr int kNX = pick_nx();
  static_assert(kNX >= 3, "W4A8 rings do not fit shared memory");
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
  constexpr int NX = L::kNX, NA = L::kNA;
  constexpr int kCols = TN / kTeams;  // token columns a warp reads out
  extern __shared__ uint8_t smem_raw[];
  // full[j]: stage (j mod kNB) has its activation bytes and its A operand
  //          (arrivals: the activation producer's expect-tx + one team);
  // gdone[g]: the MMAs of group (g mod kNG) completed (one commit per group,
  //          after both its stages): the group's accumulator is complete, its
  //          two A slots are free and, NX stages later in the sequence, its
  //          activation slots;
  // pfull/pempty: packed-weight slots;
  // acce[b]: group accumulator b read out.
  __shared__ __align__(8) uint64_t full[kNB], gdone[kNG], pfull[kNP], pempty[kNP], acce[2];
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
    for (int s = 0; s < kNB; ++s) mbar_init(&full[s], kTeamWarps + 1);
    for (int s = 0; s < kNG; ++s) mbar_init(&gdone[s], 1);
    for (int s = 0; s < kNP; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], 2 * kTeamWarps);  // the two teams that share a group
    }
    for (int b = 0; b < 2; ++b) mbar_init(&acce[b], kDeqWarps);
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
    // ---- packed weights: group gi into slot gi % kNP
    if (lane == 0) {
      uint32_t gi = 0;
      for (int t = first; t < ntiles && !s_abort; t += step) {
        const int n0 = (t % p.row_tiles) * kBM;
        for (int g = 0; g < G; ++g, ++gi) {
          const uint32_t sl = gi % kNP;
          if (gi >= static_cast<uint32_t>(kNP) && !mbar_wait_backoff<256>(&pempty[sl], ((gi / kNP) - 1) & 1)) {
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
  } else {
    // ---- A operand + read-out (warps 3..18). Warp w owns TMEM lane quarter
    // q = w % 4 (rows 32 q .. 32 q + 31 of the tile); team j = (w - 3) / 4
    // writes the A operand of stages it = j (mod 4) (groups of parity j / 2,
    // half j % 2) and reads token columns j * kCols .. + kCols - 1 out of
    // every group's accumulator.
    const int dw = warp - 3;
    const int team = dw / kTeamWarps;
    const int q = warp & 3;
    const int h = team & 1, gpar = team >> 1;
    const int r = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;

    // writes the A operand of group gi (this team's half); warp-uniform,
    // false on timeout
    auto write_a = [&](uint32_t gi) -> bool {
      const uint32_t it = 2 * gi + h, a = it % NA, pslot = gi % kNP;
      bool go = !s_abort;
      if (go) go = mbar_wait_backoff<32>(&pfull[pslot], (gi / kNP) & 1);
      if (go && it >= static_cast<uint32_t>(NA)) go = mbar_wait_backoff<32>(gbar(it - NA), gphase(it - NA));
      if (!__all_sync(0xFFFFFFFFu, go)) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        return false;
      }
      // half h of row r: 16-byte chunks 2h, 2h + 1 of the 64-byte row,
      // loaded with the TMA 64-byte swizzle (chunk c sits at c ^ ((r >> 1) & 3))
      const uint8_t* prow = ps + pslot * kPSlot + r * 64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c = 2 * h + half;
        const uint4 v = *reinterpret_cast<const uint4*>(prow + ((c ^ packed_xor<4>(r)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[16];
        exact_slice4(w, o);
        tmem_st16(tmem + lane_base + L::kACol + a * (kBK / 2) + 16 * half, o);
      }
      tmem_wait_st();
      tc_fence_before();  // the A tile before the arrival the MMA waits on
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full[it % kNB]);
        mbar_arrive(&pempty[pslot]);
      }
      return true;
    };

    float run[kCols];
#pragma unroll
    for (int j = 0; j < kCols; ++j) run[j] = 0.0f;

    bool failed = false;  // a wait of this warp gave up (warp-uniform)
    // the A operand of the first kLead groups
    for (uint32_t gi = 0; gi < static_cast<uint32_t>(L::kLead) && gi < total_groups; ++gi)
      if (static_cast<int>(gi & 1) == gpar && !failed && !write_a(gi)) failed = true;
    // group gi of the sequence is group g of tile t; the row, the token
    // columns and the scale row change once per tile (no division per group)
    int t = first, g = 0;
    int64_t n = static_cast<int64_t>(t % p.row_tiles) * kBM + r;
    int64_t m0 = static_cast<int64_t>(t / p.row_tiles) * TN + team * kCols;
    // the scale s[n, g] of the group read out next, loaded one group ahead
    float s_next = (!kAcc && n < p.N) ? bf16_bits_to_float(p.scales[n * G]) : 0.0f;
    for (uint32_t gi = 0; gi < total_groups; ++gi) {
      // 1. read out group gi: the MMAs of group gi + 2 wait for this buffer,
      //    so it comes first; the A operand is needed one group later
      const uint32_t b = gi & 1u;
      if (failed || !__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_backoff<32>(&gdone[gi % kNG], (gi / kNG) & 1))) {
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
      const uint32_t col0 = tmem + lane_base + b * TN + team * kCols;
      // consumes 16 columns of the group: running sums, or (kAcc) the
      // integer accumulators themselves
      auto use16 = [&](int c, const uint32_t (&v)[16]) {
        if constexpr (kAcc) {
          if (n < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int64_t m = m0 + 16 * c + j;
              if (m < p.M) p.acc[(m * p.N + n) * G + g] = __float2int_rn(__uint_as_float(v[j]));
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) run[16 * c + j] = fmaf(sc, __uint_as_float(v[j]), run[16 * c + j]);
        }
      };
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
      };
      if constexpr (kCols <= 32) {
        // every load in flight at once, one wait, then free the buffer
        uint32_t v[kCols / 16][16];
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) tmem_ld16_nowait(col0 + 16 * c, v[c]);
        tmem_wait_ld();
        release();
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) use16(c, v[c]);
      } else {
        // 16 columns at a time (registers: the running sums stay resident)
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) {
          uint32_t v[16];
          tmem_ld16_nowait(col0 + 16 * c, v);
          tmem_wait_ld();
          if (c == kCols / 16 - 1) release();
          use16(c, v);
        }
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
        m0 = static_cast<int64_t>(t / p.row_tiles) * TN + team * kCols;
      }
      // 2. the A operand kLead groups ahead (its slot was freed by the MMAs
      //    of group gi, which have completed)
      const uint32_t ga = gi + L::kLead;
      if (ga < total_groups && static_cast<int>(ga & 1) == gpar && !failed && !write_a(ga)) failed = true;
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

}  // namespace

cudaError_t launch_w4a8_tc(const Ctx& c, const uint16_t* xqb, const float* sx, const uint32_t* packed4,
                           const uint16_t* scales, int64_t M, int64_t N, int64_t K, uint16_t* y, int32_t* acc) {
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return cudaErrorInvalidValue;
  CUtensorMap xmap, wmap;
  if (!make_tmap_bf16_2d_sw128(&xmap, xqb, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBK, kTN))
    return cudaErrorInvalidValue;
  // 4-bit rows of a group are 64 bytes: loaded with the 64-byte swizzle so
  // that the rows of a tile spread over the shared-memory banks
  if (!make_tmap_u32_2d(&wmap, packed4, static_cast<uint64_t>(K) / 8, static_cast<uint64_t>(N), 16u, kBM, 64))
    return cudaErrorInvalidValue;
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
  return acc != nullptr ? wlaunch<kTN, true>(c, xmap, wmap, prm) : wlaunch<kTN, false>(c, xmap, wmap, prm);
}

}  // namespace wq
