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
// Persistent kernel, one CTA per SM. A tile is 128 weight rows x TN tokens,
// D[row, token] in tensor memory (MMA M = 128 rows, N = TN tokens: the
// weights are the A operand, so a dequantized tile serves TN tokens). Tiles
// are taken in a static round-robin over the grid, weight-row tiles varying
// fastest. K advances in stages of 64 (half a quantization group).
// Tensor memory (512 columns): the fp32 accumulator in columns 0..TN-1 and a
// ring of 8 dequantized A stages (32 columns each) in columns 256..511, so
// the weights never pass through shared memory once dequantized; shared
// memory holds up to 8 activation stages and 2-12 packed-weight groups.
// Warp roles:
//   warp 0      TMA producer for the activation tile [TN x 64] (128-byte
//               swizzle, zero fill past M) of each stage.
//   warp 1      allocates tensor memory; one thread issues, per group (two
//               stages), the stages' barrier waits, one fence, 8 MMAs of
//               K = 16 (A from tensor memory, B from shared memory) and one
//               commit, which releases both stages' slots; each finished
//               tile is committed to the accumulator's "full" barrier.
//   warp 2      TMA producer for the packed weights, one group [128 rows x
//               16*b bytes] per load.
//   warps 3-18  four teams of 4 warps; team j takes every fourth stage. A
//               thread turns the 64 codes of one weight row into bf16
//               RN(s * (q - z)) (q - z exact, one rounding; z = 2^(b-1), or
//               the group's zero point for asymmetric groups) and writes them
//               to its TMEM lane (tcgen05.st). The same warps read the
//               accumulator out after each tile (tcgen05.ld), release it,
//               and store bf16 outputs.
// All mbarrier waits are bounded; a timeout records WQ_ETIMEOUT and every
// role stops early (outputs are then incomplete).
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_dequant.cuh"
#include "wq_tc.cuh"

namespace wq {
namespace {

constexpr int kBM = 128;     // weight rows per tile (MMA M)
constexpr int kBK = 64;      // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kNA = 8;       // A stages in tensor memory
constexpr int kACol = 256;   // A ring: TMEM columns [256, 512), 32 per stage
constexpr int kTmemCols = 512;
// Stages per wait, fence and commit of the MMA thread: that thread's
// synchronisation per stage (~0.1 us) rivals the tensor time of a stage of
// four 128 x 256 x 16 MMAs (~0.26 us), so it takes the two stages of a group
// together (measured: 0.79 of the bf16 peak at M = 8192 against 0.71 per
// stage; four stages per commit starve the A ring at 0.54).
constexpr int kSPC = 2;
constexpr int kMaxNX = 8;    // activation stages in shared memory (upper bound, at most kNA)
constexpr int kMaxNP = 12;   // packed-weight slots, one group each (upper bound)
constexpr int kTeamWarps = 4;                  // one team: 128 rows x 64 codes
constexpr int kTeams = 4;                      // team j takes stages j (mod 4)
constexpr int kDeqWarps = kTeams * kTeamWarps;
constexpr int kThreads = (3 + kDeqWarps) * 32;  // 608
static_assert(kNA % kTeams == 0, "each team must own whole A slots");

// Shared memory: activation stages (3..8) and packed-weight slots (2..12).
// Preference: at least 5 activation stages beside 4 packed slots, else the
// deepest activation ring with 2 slots; then as many packed slots as the rest
// of shared memory holds. Few tokens per tile (TN = 128) leave room for 8 to
// 12 groups of weights in flight, which is what a tile that is bound by the
// weight stream needs. The slot count is even: a slot's previous group then
// has the same parity, so the teams that wait on it have consumed that
// previous phase (a parity wait is only sound when the phase before the
// awaited one has completed).
template <int B, int TN>
struct Layout {
  static constexpr int kXStage = TN * kBK * 2;
  static constexpr int kPSlot = kBM * 16 * B;  // one group of 128 rows
  static constexpr int kBudget = 227 * 1024 - 1024 - 512;  // minus alignment slack and static smem
  static constexpr bool fits(int nx, int np) { return nx * kXStage + np * kPSlot <= kBudget; }
  static constexpr int pick_nx() {
    for (int nx = kMaxNX; nx >= 5; --nx)
      if (fits(nx, 4)) return nx;
    for (int nx = kMaxNX; nx >= 3; --nx)
      if (fits(nx, 2)) return nx;
    return 0;
  }
  static constexpr int kNX = pick_nx();
  static constexpr int pick_np() {
    for (int np = kMaxNP; np >= 2; np -= 2)
      if (fits(kNX, np)) return np;
    return 0;
  }
  static constexpr int kNP = pick_np();
  // the activation producer refills a slot once the MMAs of the stage kNX
  // back have completed; that also proves the "full" phase kNA stages back
  // complete only while kNX <= kNA
  static_assert(kNX <= kNA, "activation ring deeper than the A ring");
  static_assert(kNX >= 3 && kNP >= 2 && kNP % 2 == 0 && fits(kNX, kNP), "prefill rings do not fit shared memory");
  static constexpr int kXOff = 0;
  static constexpr int kPOff = kNX * kXStage;
  static constexpr int kBytes = kPOff + kNP * kPSlot;
  static constexpr size_t kSmem = static_cast<size_t>(kBytes) + 1024;  // + alignment slack
};

struct PParams {
  const uint16_t* scales;  // bf16 [N, G]
  const uint8_t* zeros;    // asymmetric groups: zero points [N, G], or null (2^(b-1))
  int64_t M, N, K;
  int G;
  int row_tiles, tok_tiles;  // ceil(N / 128), ceil(M / TN) (without offsets)
  // Mixture of experts: the tokens come sorted by expert, expert e owning
  // rows [offsets[e], offsets[e+1]) of x and y; its weights are rows
  // e N .. e N + N - 1 of the stacked packed tensor and scales. Null for a
  // single dense layer (E = 1).
  const int32_t* offsets;
  int E;
  uint16_t* y;       // bf16 [M, N]
  unsigned* status;
};

using namespace tc;

// A token tile of the concatenated per-expert sequence: its expert, its
// first token and the end of that expert's tokens. The offsets are clamped
// into [0, M] and made nondecreasing, so no tile can reach outside x or y.
struct TokTile {
  int e;
  int64_t m0, mend;
};
__device__ __forceinline__ int64_t clamped_offset(const PParams& p, int e, int64_t prev) {
  int64_t v = p.offsets[e];
  v = v < prev ? prev : v;
  return v > p.M ? p.M : v;
}
template <int TN>
__device__ __forceinline__ TokTile tok_tile(const PParams& p, int tt) {
  if (p.offsets == nullptr) return TokTile{0, static_cast<int64_t>(tt) * TN, p.M};
  int acc = 0;
  int64_t prev = clamped_offset(p, 0, 0);
  for (int e = 0; e < p.E; ++e) {
    const int64_t nxt = clamped_offset(p, e + 1, prev);
    const int nt = static_cast<int>((nxt - prev + TN - 1) / TN);
    if (tt < acc + nt) return TokTile{e, prev + static_cast<int64_t>(tt - acc) * TN, nxt};
    acc += nt;
    prev = nxt;
  }
  return TokTile{p.E - 1, p.M, p.M};  // past the last tile: no tokens
}
// Token tiles of the whole sequence (sum over experts of ceil(tokens / TN)).
template <int TN>
__device__ __forceinline__ int tok_tiles_total(const PParams& p) {
  if (p.offsets == nullptr) return p.tok_tiles;
  int acc = 0;
  int64_t prev = clamped_offset(p, 0, 0);
  for (int e = 0; e < p.E; ++e) {
    const int64_t nxt = clamped_offset(p, e + 1, prev);
    acc += static_cast<int>((nxt - prev + TN - 1) / TN);
    prev = nxt;
  }
  return acc;
}

// ---- dequantization: wq_dequant.cuh -----------------------------------------

using dq::dequant_slice;
using dq::dequant_slice_zp;

template <int B, int TN>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                   const PParams p) {
  using L = Layout<B, TN>;
  constexpr int NX = L::kNX, NP = L::kNP;
  extern __shared__ uint8_t smem_raw[];
  // full[j]: stage (j mod kNA) has its activation bytes and its A tile
  //          (arrivals: the activation producer's expect-tx + one team);
  // done[p]: the MMAs of stage pair (p mod kNA/2) completed (one commit per
  //          pair: the MMA thread takes two stages per wait, fence and
  //          commit), which frees the pair's two A slots and, kNX stages
  //          later in the sequence, their activation slots;
  // pfull/pempty: packed-weight slots; tfull/tempty: the accumulator.
  constexpr int kND = kNA / kSPC;  // commit barriers
  __shared__ __align__(8) uint64_t full[kNA], done[kND], pfull[kMaxNP], pempty[kMaxNP], tfull, tempty;
  // the commit barrier that releases stage j of the sequence, and its phase
  auto pair_bar = [&](uint32_t j) -> uint64_t* { return &done[(j / kSPC) % kND]; };
  auto pair_phase = [](uint32_t j) -> uint32_t { return ((j / kSPC) / kND) & 1u; };
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_tok_tiles;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* xs = base + L::kXOff;
  uint8_t* ps = base + L::kPOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int S = 2 * G;  // stages per tile
  // static schedule: tiles blockIdx.x, blockIdx.x + gridDim.x, ...; row
  // tiles vary fastest so that CTAs running together share activation tiles
  const int first = blockIdx.x, step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNA; ++s) mbar_init(&full[s], kTeamWarps + 1);
    for (int s = 0; s < kND; ++s) mbar_init(&done[s], 1);
    for (int s = 0; s < NP; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], 2 * kTeamWarps);  // the two teams that share a group
    }
    mbar_init(&tfull, 1);
    mbar_init(&tempty, kDeqWarps);
    s_abort = 0;
    s_tok_tiles = tok_tiles_total<TN>(p);
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
  const int ntiles = p.row_tiles * s_tok_tiles;

  if (warp == 0) {
    // ---- activations: stage i of a tile covers k = 64 i .. 64 i + 63; slot
    // it % NX is free once stage it - NX is done
    if (lane == 0) {
      uint32_t it = 0;  // stages of this CTA's sequence
      for (int t = first; t < ntiles && !s_abort; t += step) {
        const int m0 = static_cast<int>(tok_tile<TN>(p, t / p.row_tiles).m0);
        for (int i = 0; i < S; ++i, ++it) {
          if (it >= static_cast<uint32_t>(NX)) {
            const uint32_t j = it - NX;
            if (!mbar_wait_bounded(pair_bar(j), pair_phase(j))) {
              record_status(p.status, kStatusTimeout);
              s_abort = 1;
              break;
            }
          }
          uint64_t* fb = &full[it % kNA];
          mbar_arrive_expect_tx(fb, L::kXStage);
          tma_load_2d(xs + (it % NX) * L::kXStage, &xmap, i * kBK, m0, fb);
        }
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- packed weights: group g (128 codes of 128 rows) into slot g % NP
    if (lane == 0) {
      uint32_t gi = 0;  // groups of this CTA's sequence
      for (int t = first; t < ntiles && !s_abort; t += step) {
        // rows of the stacked weights: expert e's layer starts at row e N
        const int n0 = tok_tile<TN>(p, t / p.row_tiles).e * static_cast<int>(p.N) + (t % p.row_tiles) * kBM;
        for (int g = 0; g < G; ++g, ++gi) {
          const uint32_t sl = gi % NP;
          if (gi >= static_cast<uint32_t>(NP) && !mbar_wait_bounded(&pempty[sl], ((gi / NP) - 1) & 1)) {
            record_status(p.status, kStatusTimeout);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&pfull[sl], L::kPSlot);
          tma_load_2d(ps + sl * L::kPSlot, &wmap, g * 4 * B, n0, &pfull[sl]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue (one thread): per stage one wait, 4 MMAs, one commit
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kBM, TN);
      uint32_t it = 0, tc = 0;
      for (int t = first; t < ntiles && !s_abort; t += step, ++tc) {
        // the first MMA of a tile overwrites the accumulator: the previous
        // tile must have been drained
        if (tc >= 1 && !mbar_wait_bounded(&tempty, (tc - 1) & 1)) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        bool ok = true;
        // kSPC = 2 stages (one group) per wait, fence and commit; a tile
        // has an even number of stages, so pairs never straddle tiles
        for (int i = 0; i < S; i += kSPC, it += kSPC) {
          bool got = !s_abort;
#pragma unroll
          for (int hh = 0; hh < kSPC; ++hh)
            if (got) got = mbar_wait_bounded(&full[(it + hh) % kNA], ((it + hh) / kNA) & 1);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < kSPC; ++hh) {
            const uint32_t bb = smem_u32(xs + ((it + hh) % NX) * L::kXStage);
            const uint32_t aa = tmem + kACol + ((it + hh) % kNA) * (kBK / 2);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              // K = 16: 8 more A columns, 32 more bytes along the swizzled B rows
              umma_bf16_ta(tmem, aa + 8 * kk, sw128_desc(bb + 32 * kk), idesc, (i + hh > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(pair_bar(it));  // fires when the pair's MMAs complete
        }
        umma_commit(&tfull);  // fires once the tile's MMAs have completed
        if (!ok) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ---- dequantize + drain (warps 3..18). Warp w owns TMEM lane quarter
    // q = w % 4: A rows / accumulator rows 32 q .. 32 q + 31 of the tile.
    // Team j = (w - 3) / 4 takes the stages it = j (mod 4) of the CTA's
    // sequence: groups gi = j / 2 (mod 2), half j % 2 of each group; its
    // thread dequantizes the 64 codes of row r = 32 q + lane into A slot
    // it % kNA. The same warps read the accumulator out: warp (j, q) takes
    // token columns j * TN / 4 .. + TN / 4 - 1 of rows 32 q ...
    const int dw = warp - 3;
    const int team = dw / kTeamWarps;
    const int q = warp & 3;
    const int h = team & 1, gpar = team >> 1;
    const int r = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // the scale of the next group this thread dequantizes, loaded one use ahead
    int nt = first, ng = gpar;
    while (ng >= G && nt < ntiles) ng -= G, nt += step;
    // the scale bits and (asymmetric groups) the zero point of that group,
    // as scale | zero << 16
    int s_nt = -1;
    int64_t s_wrow = 0;  // stacked row of this thread's weight row in tile s_nt (or -1)
    auto load_scale = [&]() -> uint32_t {
      uint32_t v = 0;
      if (nt < ntiles) {
        if (nt != s_nt) {
          s_nt = nt;
          const int64_t row = static_cast<int64_t>(nt % p.row_tiles) * kBM + r;
          s_wrow = row < p.N ? static_cast<int64_t>(tok_tile<TN>(p, nt / p.row_tiles).e) * p.N + row : -1;
        }
        if (s_wrow >= 0) {
          v = p.scales[s_wrow * G + ng];
          if (p.zeros != nullptr) v |= static_cast<uint32_t>(p.zeros[s_wrow * G + ng]) << 16;
        }
      }
      ng += 2;
      while (ng >= G && nt < ntiles) ng -= G, nt += step;
      return v;
    };
    // read this warp's share of tile t's accumulator (k-th tile of the CTA),
    // release the accumulator, then store; warp-uniform, false on timeout
    auto drain = [&](int k, int t) -> bool {
      constexpr int kCols = TN / kTeams;
      if (!__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_bounded(&tfull, k & 1))) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        return false;
      }
      tc_fence_after();
      uint32_t v[kCols / 32][32];
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) tmem_ld32(tmem + lane_base + team * kCols + 32 * c, v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty);
      const TokTile tk = tok_tile<TN>(p, t / p.row_tiles);
      const int64_t n = static_cast<int64_t>(t % p.row_tiles) * kBM + r;
      const int64_t m0 = tk.m0 + team * kCols;
      if (n < p.N) {
        uint16_t* dst = p.y + m0 * p.N + n;
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t m = m0 + 32 * c + j;
            if (m < tk.mend) {
              const float f = __uint_as_float(v[c][j]);
              dst[static_cast<int64_t>(32 * c + j) * p.N] = float_to_bf16_bits_rn(f);
            }
          }
        }
      }
      return true;
    };

    uint32_t sb = load_scale();
    uint32_t gi = 0;    // groups of the CTA's sequence
    int pend_k = -1, pend_t = 0;  // tile whose accumulator this warp has not read yet
    bool stop = false;  // warp-uniform
    int k = 0;
    for (int t = first; t < ntiles && !stop; t += step, ++k) {
      const uint32_t it0 = static_cast<uint32_t>(k) * static_cast<uint32_t>(S);  // the tile's first stage
      for (int g = 0; g < G; ++g, ++gi) {
        if (static_cast<int>(gi & 1) != gpar) continue;
        const uint32_t it = 2 * gi + h, a = it % kNA, pslot = gi % NP;
        // stage it - kNA in this tile needs this tile's MMAs, which need the
        // previous tile's accumulator drained: drain it first
        if (pend_k >= 0 && it >= static_cast<uint32_t>(kNA) && it - kNA >= it0) {
          if (!drain(pend_k, pend_t)) {
            stop = true;
            break;
          }
          pend_k = -1;
        }
        // every decision below is warp-uniform (the warp meets at __syncwarp
        // and the .sync.aligned tcgen05 instructions)
        bool go = !s_abort;
        if (go) go = mbar_wait_bounded(&pfull[pslot], (gi / NP) & 1);
        if (go && it >= static_cast<uint32_t>(kNA)) go = mbar_wait_bounded(pair_bar(it - kNA), pair_phase(it - kNA));
        if (!__all_sync(0xFFFFFFFFu, go)) {
          if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
          s_abort = 1;
          stop = true;
          break;
        }
        const uint32_t s2 = (sb & 0xFFFFu) | (sb << 16);
        const uint32_t zc2 = dq::zero_pair<B>(sb >> 16);
        sb = load_scale();
        uint32_t w[2 * B];
        const uint8_t* prow = ps + pslot * L::kPSlot + r * 16 * B;
        if constexpr (packed_swizzle_bytes(B) != 0) {
          // half h = 16-byte chunks B/2 * h .. + B/2 - 1 of the row, swizzled
#pragma unroll
          for (int j = 0; j < B / 2; ++j) {
            const int c = (B / 2) * h + j;
            const uint4 v = *reinterpret_cast<const uint4*>(prow + ((c ^ packed_xor<B>(r)) << 4));
            w[4 * j] = v.x, w[4 * j + 1] = v.y, w[4 * j + 2] = v.z, w[4 * j + 3] = v.w;
          }
        } else {
          load_words<2 * B>(prow + h * 8 * B, w);
        }
        uint32_t o[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t wsl[B], os[16];
#pragma unroll
          for (int j = 0; j < B; ++j) wsl[j] = w[half * B + j];
          if (p.zeros != nullptr) {
            dequant_slice_zp<B>(wsl, s2, zc2, os);
          } else {
            dequant_slice<B>(wsl, s2, os);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) o[16 * half + j] = os[j];
        }
        tmem_st32(tmem + lane_base + kACol + a * (kBK / 2), o);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();  // the A tile before the arrival the MMA waits on
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[a]);
          mbar_arrive(&pempty[pslot]);
        }
      }
      if (stop) break;
      // at most one tile pending: drain the previous one before moving on
      if (pend_k >= 0 && !drain(pend_k, pend_t)) break;
      pend_k = k;
      pend_t = t;
    }
    if (!stop && pend_k >= 0) drain(pend_k, pend_t);
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

template <int B, int TN>
cudaError_t plaunch(const Ctx& c, const CUtensorMap& xmap, const CUtensorMap& wmap, const PParams& prm) {
  constexpr size_t smem = Layout<B, TN>::kSmem;
  static_assert(smem <= 227 * 1024, "prefill stage layout exceeds shared memory");
  static SmemLimit limit;
  const cudaError_t e = raise_smem_limit(limit, prefill_kernel<B, TN>, c.device, smem);
  if (e != cudaSuccess) return e;
  PParams q = prm;
  q.row_tiles = static_cast<int>((prm.N + kBM - 1) / kBM);
  q.tok_tiles = static_cast<int>((prm.M + TN - 1) / TN);
  // with experts the tiles are known on the device only: at most one
  // partial token tile per expert beyond ceil(M / TN)
  const int64_t tiles64 = static_cast<int64_t>(q.row_tiles) * (q.tok_tiles + (prm.offsets ? prm.E : 0));
  const int tiles = tiles64 < c.sm_count ? static_cast<int>(tiles64) : c.sm_count;
  const int grid = tiles;  // persistent: one CTA per SM
  prefill_kernel<B, TN><<<grid, kThreads, smem, c.stream>>>(xmap, wmap, q);
  return cudaGetLastError();
}

template <int TN>
cudaError_t plaunch_b(const Ctx& c, int bits, const CUtensorMap& xmap, const CUtensorMap& wmap,
                      const PParams& prm) {
  switch (bits) {
    case 2: return plaunch<2, TN>(c, xmap, wmap, prm);
    case 3: return plaunch<3, TN>(c, xmap, wmap, prm);
    case 4: return plaunch<4, TN>(c, xmap, wmap, prm);
    case 5: return plaunch<5, TN>(c, xmap, wmap, prm);
    case 6: return plaunch<6, TN>(c, xmap, wmap, prm);
    case 7: return plaunch<7, TN>(c, xmap, wmap, prm);
    case 8: return plaunch<8, TN>(c, xmap, wmap, prm);
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

static cudaError_t launch_tc(const Ctx& c, const uint16_t* x, const uint32_t* packed, const uint16_t* scales,
                             const uint8_t* zeros, const int32_t* offsets, int64_t E, int64_t M, int64_t N, int64_t K,
                             int bits, uint16_t* y) {
  // tokens per tile from the tokens per expert (all of them for one layer)
  const int tn = prefill_tile_tokens((M + E - 1) / E);
  CUtensorMap xmap, wmap;
  if (!make_tmap_bf16_2d_sw128(&xmap, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBK,
                               static_cast<uint32_t>(tn)))
    return cudaErrorInvalidValue;
  const uint64_t words = static_cast<uint64_t>(K) * bits / 32;
  // rows of a power-of-two pitch (2, 4, 8 bits: 32, 64, 128 bytes) would put
  // every row on the same banks; the TMA swizzle of that span spreads them
  if (!make_tmap_u32_2d(&wmap, packed, words, static_cast<uint64_t>(E * N), 4u * bits, kBM,
                        packed_swizzle_bytes(bits)))
    return cudaErrorInvalidValue;
  PParams prm{};
  prm.scales = scales;
  prm.zeros = zeros;
  prm.offsets = offsets;
  prm.E = static_cast<int>(E);
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.G = static_cast<int>(K / 128);
  prm.y = y;
  prm.status = c.status;
  return tn == 128 ? plaunch_b<128>(c, bits, xmap, wmap, prm) : plaunch_b<256>(c, bits, xmap, wmap, prm);
}

cudaError_t launch_prefill(const Ctx& c, const uint16_t* x, const uint32_t* packed, const uint16_t* scales,
                           int64_t M, int64_t N, int64_t K, int bits, uint16_t* y, const uint8_t* zeros) {
  return launch_tc(c, x, packed, scales, zeros, nullptr, 1, M, N, K, bits, y);
}

cudaError_t launch_moe(const Ctx& c, const uint16_t* x, const int32_t* offsets, int64_t E, const uint32_t* packed,
                       const uint16_t* scales, int64_t M, int64_t N, int64_t K, int bits, uint16_t* y) {
  return launch_tc(c, x, packed, scales, nullptr, offsets, E, M, N, K, bits, y);
}

}  // namespace wq
