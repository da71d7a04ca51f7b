// Decode GEMM for M <= 16 tokens, streamed by CTA pairs: y = x . dequant(W)^T
// at close to HBM bandwidth with no split-K workspace and no grid barrier.
//
// Method: "vLLM Can Run INT5-7", section 1 (WNA16 for widths 2..8); model card
// "Qwen3.8-27B-INT6-Mixed-AutoRound", section "Findings" (dense LSB-first
// layout, symmetric 2^(b-1) zero point, bf16 group-128 scales of any sign);
// "vLLM Quantization", section "Key points" (decode waits on memory); W4A8
// per "int8 activations (W4A8) ...", section "Under the hood" (the per-token
// int8 quantization of the activations is done here, in the staging).
//
// Design (GB300):
//  * Clusters of two CTAs, one CTA per SM. The output rows are cut into
//    equal contiguous ranges, one per cluster; CTA q of the pair takes K half
//    q of every row in the range, so each CTA stages only half of the
//    activations (as MMA fragments) and the two halves meet once per chunk
//    through distributed shared memory. Nothing goes through global memory
//    but the weights, the scales, x and y.
//  * A range is streamed in chunks of H <= 256 rows (one TMA box high). A
//    producer warp keeps a deep ring of [H rows x one 128-code group] stages
//    in flight (about 100-150 KB per SM) plus the chunk's scale box (its own
//    barrier: all consumer warps read it, whatever stages they own).
//  * 16 consumer warps: a warp owns a 32-row tile of the chunk (two m16 MMA
//    tiles sharing the activation fragments) and every ksplit-th group of the
//    CTA's half; unpack by code pairing (wq_unpack.cuh), swap-AB m16n8k16,
//    fp32 accumulators with the group scale applied per group.
//  * Per chunk: the warps of a tile reduce in shared memory in a fixed order;
//    each CTA pushes its sums of the rows its peer finalises into the peer's
//    inbox with remote asynchronous 16-byte stores that count their bytes on
//    the peer's "ready" barrier; each CTA then writes half the rows. A
//    "consumed" arrival frees the inbox for the next chunk; after the last
//    chunk each CTA leaves on its own.
//  * Programmatic dependent launch: the kernel lets the next one in the
//    stream launch at once; the producer streams weights and scales (never
//    written by these kernels) right away, the consumers wait for the
//    previous kernel before reading activations or writing outputs.
// All waits are bounded (WQ_ETIMEOUT on expiry).
#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_unpack.cuh"
#include "wq_cluster.cuh"

namespace wq {
namespace {

using namespace unpack;

constexpr int kCWarps = 16;                      // consumer warps
constexpr int kThreads2 = (kCWarps + 1) * 32;    // + one producer warp
constexpr int kTileRows = 32;                    // rows per warp tile
constexpr int kMaxH = 256;                       // rows per chunk (TMA box limit)
constexpr int kMaxStages = 24;                   // ring slots at most (a small layer streams whole)
constexpr int kXBatch = 3;                       // activation jobs a warp loads at once
constexpr size_t kSmemCap = 227 * 1024 - 1024;   // dynamic smem budget (alignment slack)

struct D2Params {
  const uint16_t* x;   // bf16 [M, K]
  int64_t M, N, K;
  int G, Gh;           // groups, groups per K half
  int C;               // clusters
  int H, nchunk, T;    // chunk rows, chunks per range, 32-row tiles per chunk
  int ksplit;          // consumer warps per tile (each takes every ksplit-th group)
  int NS;              // ring stages
  int sbox, sx0;       // scale box width, and the box start of each half (x0 of half q = q * sx0)
  uint16_t* y;
  int32_t* acc;        // kMode 2: int32 [M, N, G] group accumulators
  const uint8_t* zeros;  // kMode 3: zero points [N, G]
  unsigned* status;
};

// The bound of every wait of this kernel, and a test hook: a producer stops
// issuing at this stage of its sequence (-1: never). Set through
// wq_debug_decode_wait_fault, so that a test can make a wait run out: the
// copies already issued all land, and the consumers that wait for the first
// stage never issued give up after the bound, record WQ_ETIMEOUT and finish
// the kernel normally.
__constant__ uint64_t c_wait_limit_ns = kWaitLimitNs;
__constant__ int64_t c_stop_stage = -1;

using namespace cl;

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory");
}
// m16n8k16 MMA with f32 accumulators, D = A B + C (kZero: C = 0). Not
// volatile: the compiler may schedule it like any other arithmetic.
template <bool kF16, bool kZero>
__device__ __forceinline__ void mma16c(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  if constexpr (kZero) {
    if constexpr (kF16)
      asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
          : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
    else
      asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
          : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
  } else {
    if constexpr (kF16)
      asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
      asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <int B>
__device__ __forceinline__ void unpack_quad2(const uint32_t (&w)[B], int i2, uint32_t (&r)[4]) {
  constexpr uint32_t kMagic = uses_fp16<B>() ? 0x64006400u : 0x43004300u;
  constexpr uint32_t kM = (1u << B) - 1u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const PairSpec sp = pair_spec<B>(4 * i2 + q);
    const uint32_t mask = (kM << sp.olo) | (kM << (16 + sp.ohi));
    r[q] = lop3_and_or(slice_window<B>(w, sp.s), mask, kMagic);
  }
}

// Shared-memory carve-up, identical on host (planning) and device. A ring
// slot and a scale buffer hold the H rows their TMA box brings; the warps of
// the last tile also read the rows up to T * 32 - 1 past them (bytes of the
// next region, whose results are never written), which stay inside the
// allocation since the scale buffers and the fragments follow the ring.
struct D2Smem {
  size_t ring, slot, sbuf, shalf, xs, corr, scl, xsum, part, inbox, bars, total;
};
// zp: asymmetric groups, which also keep the plain group sums of x.
__host__ __device__ inline D2Smem d2_smem(int B, int NT, int T, int H, int Gh, int sbox, int NS, bool zp = false) {
  D2Smem s{};
  auto al = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  s.slot = al(static_cast<size_t>(H) * 16 * B, 128);
  s.ring = 0;
  s.sbuf = s.ring + NS * s.slot;
  s.shalf = al(static_cast<size_t>(H) * sbox * 2, 128);  // one of the two scale buffers
  s.xs = al(s.sbuf + 2 * s.shalf, 128);
  s.corr = s.xs + static_cast<size_t>(NT) * Gh * 4 * 32 * 16;
  s.scl = s.corr + static_cast<size_t>(NT) * 8 * Gh * 4;
  s.xsum = s.scl + static_cast<size_t>(NT) * 8 * Gh * 4;
  s.part = al(s.xsum + (zp ? static_cast<size_t>(NT) * 8 * Gh * 4 : 0), 16);
  s.inbox = s.part + static_cast<size_t>(T) * kTileRows * NT * 8 * 4;
  s.bars = al(s.inbox + static_cast<size_t>(T) * (kTileRows / 2) * NT * 8 * 4, 8);
  s.total = s.bars + (2 * kMaxStages + 6) * 8;
  return s;
}

// kMode 0: WNA16. kMode 3: WNA16 with asymmetric groups (a zero point per
// (row, group): the correction of a group grows by (zp - 2^(b-1)) sum x).
// kMode 1: W4A8 (x quantized per token in the staging).
// kMode 2: W4A8, and instead of y the exact per-group integer accumulators
// acc[m, n, g] = sum_{k in g} xq[m, k] (q[n, k] - 8) are written (the test
// and debug mode of the same main loop; the reduction and exchange still run).
template <int B, int NT, int kMode>
__global__ void __launch_bounds__(kThreads2, 1) decode2_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap smap,
                                                              const D2Params p) {
  constexpr bool kQuant = kMode == 1 || kMode == 2;
  constexpr bool kZp = kMode == 3;
  constexpr bool kF16 = uses_fp16<B>();
  constexpr int kTok = NT * 8;  // token columns of the partial-sum buffer
  extern __shared__ uint8_t smem_raw[];
  __shared__ volatile int s_abort;
  __shared__ float s_sx[16];       // W4A8: per-token activation scales
  __shared__ float s_f[16];        // W4A8: 2^k, k = clamp(1 - exponent(sx), -126, 127)
  __shared__ float s_sxn[16];      // W4A8: sx 2^k
  __shared__ float s_rcp[16];      // W4A8: RN(1 / (sx 2^k))
  __shared__ float s_wmax[kCWarps];  // W4A8: per-warp partial maxima
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int Gh = p.Gh, T = p.T, NS = p.NS, ksplit = p.ksplit, H = p.H;
  const D2Smem L = d2_smem(B, NT, T, H, Gh, p.sbox, NS, kZp);
  uint8_t* ring = base + L.ring;
  uint16_t* sbuf = reinterpret_cast<uint16_t*>(base + L.sbuf);
  uint4* xs4 = reinterpret_cast<uint4*>(base + L.xs);
  float* corr = reinterpret_cast<float*>(base + L.corr);
  float* scl = reinterpret_cast<float*>(base + L.scl);
  float* xsm = reinterpret_cast<float*>(base + L.xsum);  // kZp: plain group sums of x
  float* part = reinterpret_cast<float*>(base + L.part);    // this CTA's sums, [T*32 rows][kTok]
  float* inbox = reinterpret_cast<float*>(base + L.inbox);  // the peer's sums of our half, [T*16][kTok]
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.bars);  // [kMaxStages]
  uint64_t* empty = full + kMaxStages;                           // [kMaxStages]
  uint64_t* cdone = empty + kMaxStages;  // [2]: consumers done with scale buffer k % 2
  uint64_t* rbar = cdone + 2;            // the peer's sums of the chunk are ready
  uint64_t* dbar = rbar + 1;             // the peer has read our sums of the chunk
  uint64_t* sfull = dbar + 1;            // [2]: scale box of chunk k landed in buffer k % 2

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t q = cluster_rank();  // K half of this CTA
  const uint32_t peer = q ^ 1u;
  const int64_t cid = cluster_id_x();
  const int64_t r0 = cid * p.N / p.C, r1 = (cid + 1) * p.N / p.C;  // the pair's rows
  const int nck = static_cast<int>((r1 - r0 + H - 1) / H);      // chunks (the same in both CTAs)
  const int gbase = static_cast<int>(q) * Gh;                    // first group of this half
  const int scol0 = static_cast<int>(q) * p.sx0;                 // scale box start column
  const int sbox_elems = static_cast<int>(L.shalf / 2);  // elements between the two scale buffers
  const uint32_t stage_bytes = static_cast<uint32_t>(H) * 16u * B;
  const uint32_t scale_bytes = static_cast<uint32_t>(H) * p.sbox * 2u;

  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint64_t lim = c_wait_limit_ns;

  if (warp == kCWarps) {
    // ---- producer: initialise the barriers, then stream at once. Shared
    // memory still holds the barrier words of the previous kernel on this SM:
    // the consumers learn of the initialisation through named barrier 2,
    // which the producer only arrives on, after a CTA-scope release fence
    // (they wait on it, then fence, before their first barrier operation);
    // the peer CTA learns of it through the cluster barrier.
    if (lane == 0) {
      // the two descriptors are fetched while the barriers are set up
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&smap)) : "memory");
      for (int s = 0; s < NS; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], T);  // the T warps (one per tile) that read a stage
      }
      mbar_init(&cdone[0], kCWarps);
      mbar_init(&cdone[1], kCWarps);
      mbar_init(rbar, 1);
      mbar_init(dbar, 1);
      mbar_init(&sfull[0], 1);
      mbar_init(&sfull[1], 1);
      s_abort = 0;
      fence_mbar_init();
      asm volatile("fence.acq_rel.cta;" ::: "memory");
    }
    __syncwarp();
    cluster_arrive();
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads2) : "memory");
    // chunk k = rows r0 + k H .. + H - 1; stage = one group of this CTA's K
    // half; the chunk's first stage also brings its scale box
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int k = 0; k < nck && !stop; ++k) {
        const int rc = static_cast<int>(r0 + static_cast<int64_t>(k) * H);
        if (k >= 2 && !mbar_wait_bounded(&cdone[k & 1], ((k >> 1) - 1) & 1, lim)) {
          record_status(p.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        // the chunk's scale box, on its own barrier: every consumer warp of
        // the chunk reads it, whichever stages it owns
        mbar_arrive_expect_tx(&sfull[k & 1], scale_bytes);
        tma_load_2d(sbuf + (k & 1) * sbox_elems, &smap, scol0, rc, &sfull[k & 1]);
        for (int gl = 0; gl < Gh; ++gl, ++it) {
          const uint32_t s = it % NS;
          if (static_cast<int64_t>(it) == c_stop_stage) {  // test hook: stop issuing here
            stop = true;
            break;
          }
          if (s_abort || (it >= static_cast<uint32_t>(NS) && !mbar_wait_bounded(&empty[s], ((it / NS) - 1) & 1, lim))) {
            record_status(p.status, kStatusTimeout);
            s_abort = 1;
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(ring + s * L.slot, &wmap, (gbase + gl) * 4 * B, rc, &full[s]);
        }
      }
    }
    __syncwarp();
    cluster_wait();
  } else {
    // ---- consumers
    cluster_arrive();
    const bool active = warp < T * ksplit;
    const int tile = warp % T, kr = warp / T;
    const int g = lane >> 2, t = lane & 3;

    // activation fragments of this K half, built once while the producer
    // streams weights. A task is one (token, group) of the half: the four
    // lanes t = 0..3 of a lane quad take its 128 activations, eight tasks per
    // warp pass, so that a few tokens still fill whole warps. The fragments
    // and corrections of the token columns past M are zero (scale 1); they
    // are written first, since they do not wait for the previous kernel,
    // whose output the activations are.
    const int ntask = static_cast<int>(p.M) * Gh;
    const int nwt = (ntask + 7) / 8;  // warp tasks: eight tasks each
    {
      const int zt0 = static_cast<int>(p.M), nz = NT * 8 - zt0;
      for (int e = threadIdx.x; e < nz * Gh * 16; e += kCWarps * 32) {
        const int tk = zt0 + e / (Gh * 16), rem = e % (Gh * 16);
        const int gz = rem >> 4, i2 = (rem >> 2) & 3, tt = rem & 3;
        xs4[(((tk >> 3) * Gh + gz) * 4 + i2) * 32 + (tk & 7) * 4 + tt] = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int e = threadIdx.x; e < nz * Gh; e += kCWarps * 32) {
        corr[zt0 * Gh + e] = 0.0f;
        scl[zt0 * Gh + e] = 1.0f;
        if constexpr (kZp) xsm[zt0 * Gh + e] = 0.0f;
      }
    }
    griddep_wait();
    // Each warp issues the loads of up to kXBatch of its passes (warp task
    // q * kCWarps + warp for its q-th pass) before building any fragments.
    uint4 rawv[kXBatch][4];
    auto load_x_batch = [&](int q0, uint4 (&dst)[kXBatch][4]) {
#pragma unroll
      for (int b = 0; b < kXBatch; ++b) {
        const int task = ((q0 + b) * kCWarps + warp) * 8 + g;
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[b][c] = make_uint4(0u, 0u, 0u, 0u);
        if (task < ntask) {
          const int tok = task / Gh, gl = task % Gh;
          const int64_t k0 = static_cast<int64_t>(gbase + gl) * 128 + 32 * t;
          const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(tok) * p.K + k0);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[b][c] = src[c];
        }
      }
    };
    // W4A8: the first batch is in flight during the amax pass below
    if constexpr (kQuant) load_x_batch(0, rawv);
    if constexpr (kQuant) {
      // W4A8: per-token int8 quantization of the activations, here instead of
      // a separate pass. Every CTA needs the scales of all tokens, whichever
      // K half it owns: amax over the whole row, split over 16 / Mp warps per
      // token (Mp = M rounded up to a power of two), then sx = amax / 127 by
      // IEEE division, as the activation-quant kernel does.
      const int mp = p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : p.M <= 8 ? 8 : 16;
      const int wpt = kCWarps / mp, tok = warp / wpt, part = warp % wpt;
      const int nch = static_cast<int>(p.K / 8);  // 16-byte chunks of a row
      float amax = 0.0f;
      if (tok < p.M) {
        const uint4* row = reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(tok) * p.K);
        const int stride = wpt * 32;
        for (int i0 = part * 32 + lane; i0 < nch; i0 += 4 * stride) {
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int idx = i0 + u * stride;
            v[u] = idx < nch ? row[idx] : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              amax = fmaxf(amax, fabsf(__uint_as_float(wv[e] << 16)));
              amax = fmaxf(amax, fabsf(__uint_as_float(wv[e] & 0xFFFF0000u)));
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      if (lane == 0) s_wmax[warp] = amax;
      consumer_sync();
      if (threadIdx.x < p.M) {
        float a = 0.0f;
        for (int w = 0; w < wpt; ++w) a = fmaxf(a, s_wmax[threadIdx.x * wpt + w]);
        const float sxv = __fdiv_rn(a, 127.0f);
        // a power of two that brings sx into [1, 2): x / sx = (x 2^k) / (sx 2^k)
        // and both scalings are exact (bar an x 2^k that underflows, whose
        // quotient is below 2^-126 and quantizes to 0 either way)
        int e = 0;
        (void)frexpf(sxv, &e);
        const int k = max(-126, min(127, 1 - e));
        const float f = sxv > 0.0f ? __uint_as_float(static_cast<uint32_t>(127 + k) << 23) : 0.0f;
        s_sx[threadIdx.x] = sxv;
        s_f[threadIdx.x] = f;
        s_sxn[threadIdx.x] = sxv * f;
        s_rcp[threadIdx.x] = sxv > 0.0f ? __frcp_rn(sxv * f) : 0.0f;
      }
      consumer_sync();
    }
    for (int q0 = 0; q0 * kCWarps + warp < nwt; q0 += kXBatch) {  // warp-uniform
      if (!kQuant || q0 != 0) load_x_batch(q0, rawv);
#pragma unroll
      for (int b = 0; b < kXBatch; ++b) {
        const int wt = (q0 + b) * kCWarps + warp;
        if (wt >= nwt) break;  // warp-uniform
        const int task = wt * 8 + g;
        const bool valid = task < ntask;  // lane quads past the last task build zeros
        const int tok = valid ? task / Gh : 0, gl = valid ? task % Gh : 0;
        float xv[32];
        raw_to_float(rawv[b], xv);
        if constexpr (kQuant) {
          // xq = clamp(round_half_even(x / sx), -127, 127); an all-zero row
          // (sx = 0) quantizes to zeros. The codes are exact in bf16.
          const float f = valid ? s_f[tok] : 0.0f;
          const float sxn = valid ? s_sxn[tok] : 0.0f;
          const float rcp = valid ? s_rcp[tok] : 0.0f;
          // RN(x / sx) = RN(x' / sx') with x' = x 2^k, sx' = sx 2^k in [1, 2),
          // by Markstein's correction of the product with y = RN(1 / sx'):
          // q0 = RN(x' y), r = x' - q0 sx' exactly (fma), RN(q0 + r y) is the
          // correctly rounded quotient (IBM J. Res. Dev. 34(1), 1990). With
          // sx' in [2^-22, 2) (below 1 only for a subnormal sx, where k stops
          // at 127) and |x'| <= 256 nothing overflows, and an underflowing
          // quotient rounds to 0 as the exact one does. sx = 0 gives f = 0
          // and zeros throughout.
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float xs = xv[c] * f;
            const float q0 = xs * rcp;
            const float r = fmaf(-q0, sxn, xs);
            xv[c] = static_cast<float>(max(-127, min(127, __float2int_rn(fmaf(r, rcp, q0)))));
          }
        }
        uint32_t frag[16];
        float cr, sb, xsum;
        make_fragments<B>(xv, frag, cr, sb, xsum);  // every lane: it shuffles within its quad
        if (valid) {
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2)
            xs4[(((tok >> 3) * Gh + gl) * 4 + i2) * 32 + (tok & 7) * 4 + t] =
                make_uint4(frag[4 * i2], frag[4 * i2 + 1], frag[4 * i2 + 2], frag[4 * i2 + 3]);
          if (t == 0) {
            corr[tok * Gh + gl] = cr;
            scl[tok * Gh + gl] = sb;
            if constexpr (kZp) xsm[tok * Gh + gl] = xsum;
          }
        }
      }
    }
    consumer_sync();
    // the producer has initialised the barriers (named barrier 2)
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads2) : "memory");
    asm volatile("fence.acq_rel.cta;" ::: "memory");

    bool stop = false;  // warp-uniform
    uint32_t slot_cur = static_cast<uint32_t>(kr), phase_cur = 0;  // this warp's next stage: slot, phase
    for (int k = 0; k < nck; ++k) {
      const int64_t rc = r0 + static_cast<int64_t>(k) * H;
      const uint16_t* sbk = sbuf + (k & 1) * sbox_elems;
      float acc[NT][2][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][h][e] = 0.0f;

      // the chunk's scales (every active warp waits on every chunk's phase)
      if (active && !stop && !__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_bounded(&sfull[k & 1], (k >> 1) & 1, lim))) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        stop = true;
      }
      if (active && !stop) {
        const int rowt = tile * kTileRows + g;  // rows rowt + {0, 8, 16, 24} of the chunk
        for (int gl = kr; gl < Gh; gl += ksplit) {
          // stage it = k Gh + gl sits in slot it % NS, phase it / NS; a warp's
          // stages advance by ksplit, which divides NS and Gh, so both are
          // carried along instead of divided out
          const uint32_t s = slot_cur, phase = phase_cur;
          // kZp: the zero points of this thread's four rows in this group,
          // loaded before the stage wait (global memory, so their latency
          // overlaps it), as zp - 2^(b-1)
          float zd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if constexpr (kZp) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int64_t row = rc + rowt + 8 * qq;
              if (row < r1)
                zd[qq] = static_cast<float>(p.zeros[row * p.G + gbase + gl] & ((1u << B) - 1u)) -
                         static_cast<float>(1 << (B - 1));
            }
          }
          slot_cur += static_cast<uint32_t>(ksplit);
          if (slot_cur >= static_cast<uint32_t>(NS)) {
            slot_cur -= static_cast<uint32_t>(NS);
            phase_cur ^= 1u;
          }
          if (!__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_bounded(&full[s], phase, lim))) {
            if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
            s_abort = 1;
            stop = true;
            break;
          }
          const uint32_t* st = reinterpret_cast<const uint32_t*>(ring + s * L.slot);
          uint32_t w0[B], w1[B], w2[B], w3[B];
          load_slice<B>(st, rowt, t, w0);
          load_slice<B>(st, rowt + 8, t, w1);
          load_slice<B>(st, rowt + 16, t, w2);
          load_slice<B>(st, rowt + 24, t, w3);
          // the slot may be refilled once every lane's reads are done: the
          // refill is a TMA (async-proxy) write, which the generic-proxy reads
          // above are ordered before only by a proxy fence in each reading
          // thread (without it, a read still in flight could see the next
          // stage's bytes)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          const int scol = gbase + gl - scol0;
          float sc[4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) sc[qq] = bf16_bits_to_float(sbk[(rowt + 8 * qq) * p.sbox + scol]);
          float c[NT][2][4];
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            uint32_t a0[4], a1[4], a2[4], a3[4];
            unpack_quad2<B>(w0, i2, a0);
            unpack_quad2<B>(w1, i2, a1);
            unpack_quad2<B>(w2, i2, a2);
            unpack_quad2<B>(w3, i2, a3);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const uint4 bv = xs4[((j * Gh + gl) * 4 + i2) * 32 + lane];
              if (i2 == 0) {  // the group's chains start from zero
                mma16c<kF16, true>(c[j][0], a0[0], a1[0], a0[1], a1[1], bv.x, bv.y);
                mma16c<kF16, true>(c[j][1], a2[0], a3[0], a2[1], a3[1], bv.x, bv.y);
              } else {
                mma16c<kF16, false>(c[j][0], a0[0], a1[0], a0[1], a1[1], bv.x, bv.y);
                mma16c<kF16, false>(c[j][1], a2[0], a3[0], a2[1], a3[1], bv.x, bv.y);
              }
              mma16c<kF16, false>(c[j][0], a0[2], a1[2], a0[3], a1[3], bv.z, bv.w);
              mma16c<kF16, false>(c[j][1], a2[2], a3[2], a2[3], a3[3], bv.z, bv.w);
            }
          }
          if constexpr (kMode == 2) {
            // the group's exact integer sums: xq (128 + q) - 136 xq
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const int ti0 = (j * 8 + 2 * t) * Gh + gl, ti1 = ti0 + Gh;
              const float cr0 = corr[ti0], cr1 = corr[ti1], sl0 = scl[ti0], sl1 = scl[ti1];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int tok = j * 8 + 2 * t + (e & 1);
                  const int rl = tile * kTileRows + g + 16 * hh + 8 * (e >> 1);
                  const int64_t row = rc + rl;
                  if (tok < p.M && rl < H && row < r1) {
                    const float v = (e & 1) ? fmaf(sl1, c[j][hh][e], -cr1) : fmaf(sl0, c[j][hh][e], -cr0);
                    p.acc[(static_cast<int64_t>(tok) * p.N + row) * p.G + gbase + gl] = __float2int_rn(v);
                  }
                }
            }
          }
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const int ti0 = (j * 8 + 2 * t) * Gh + gl, ti1 = ti0 + Gh;
            const float cr0 = corr[ti0], cr1 = corr[ti1], sl0 = scl[ti0], sl1 = scl[ti1];
            if constexpr (kZp) {
              // rows rowt + 16 h (e = 0, 1) and rowt + 16 h + 8 (e = 2, 3)
              const float x0 = xsm[ti0], x1 = xsm[ti1];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                acc[j][h][0] = fmaf(sc[2 * h], fmaf(sl0, c[j][h][0], -fmaf(zd[2 * h], x0, cr0)), acc[j][h][0]);
                acc[j][h][1] = fmaf(sc[2 * h], fmaf(sl1, c[j][h][1], -fmaf(zd[2 * h], x1, cr1)), acc[j][h][1]);
                acc[j][h][2] =
                    fmaf(sc[2 * h + 1], fmaf(sl0, c[j][h][2], -fmaf(zd[2 * h + 1], x0, cr0)), acc[j][h][2]);
                acc[j][h][3] =
                    fmaf(sc[2 * h + 1], fmaf(sl1, c[j][h][3], -fmaf(zd[2 * h + 1], x1, cr1)), acc[j][h][3]);
              }
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                acc[j][h][0] = fmaf(sc[2 * h], fmaf(sl0, c[j][h][0], -cr0), acc[j][h][0]);
                acc[j][h][1] = fmaf(sc[2 * h], fmaf(sl1, c[j][h][1], -cr1), acc[j][h][1]);
                acc[j][h][2] = fmaf(sc[2 * h + 1], fmaf(sl0, c[j][h][2], -cr0), acc[j][h][2]);
                acc[j][h][3] = fmaf(sc[2 * h + 1], fmaf(sl1, c[j][h][3], -cr1), acc[j][h][3]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cdone[k & 1]);  // done with scale buffer k % 2

      // the peer has consumed its inbox of the previous chunk: it may be
      // written again
      if (k >= 1 && !__all_sync(0xFFFFFFFFu, mbar_wait_cluster_bounded(dbar, (k - 1) & 1, lim))) {
        if (lane == 0 && !s_abort) record_status(p.status, kStatusTimeout);
        s_abort = 1;
        stop = true;
      }
      // reduce the ksplit warps of each tile, in a fixed order
      for (int r = 0; r < ksplit; ++r) {
        if (active && kr == r) {
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int rl = tile * kTileRows + g + 16 * h + 8 * (e >> 1);
                float* d = part + rl * kTok + j * 8 + 2 * t + (e & 1);
                *d = (r == 0) ? acc[j][h][e] : *d + acc[j][h][e];
              }
        }
        consumer_sync();
      }
      // the peer's barriers exist (it arrived on the cluster barrier after
      // initialising them) before anything of ours reaches its memory
      if (k == 0) cluster_wait();
      // push our sums of the rows the peer finalises into its inbox: remote
      // 16-byte asynchronous stores, each counting its bytes on the peer's
      // "ready" barrier, which completes once all have landed (and its own
      // CTA has announced the byte count of the chunk)
      const int half_rows = T * (kTileRows / 2);
      {
        const int nvec = half_rows * (kTok / 4);
        if (threadIdx.x == 0) mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(nvec) * 16u);
        const uint32_t pin = map_peer(smem_u32(inbox), peer);
        const uint32_t prbar = map_peer(smem_u32(rbar), peer);
        for (int e = threadIdx.x; e < nvec; e += kCWarps * 32) {
          const int rr = e / (kTok / 4), c4 = e % (kTok / 4);
          const float4 v = *reinterpret_cast<const float4*>(part + (static_cast<int>(peer) * half_rows + rr) * kTok + 4 * c4);
          st_async_peer_v4(pin + 16u * static_cast<uint32_t>(rr * (kTok / 4) + c4), v, prbar);
        }
      }
      // the peer's sums of our rows are in our inbox: combine, write y
      const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait_cluster_bounded(rbar, k & 1, lim));
      if (!ready && threadIdx.x == 0) {
        record_status(p.status, kStatusTimeout);
        s_abort = 1;
      }
      // (a thread takes four token columns of one row: 16-byte reads of
      // consecutive words, no bank conflicts; the quads past M are skipped)
      if (kMode != 2 && ready) {
        const int mq = (static_cast<int>(p.M) + 3) / 4;  // token quads holding real tokens
        for (int e = threadIdx.x; e < half_rows * mq; e += kCWarps * 32) {
          const int rr = e / mq, c4 = e % mq;
          const int rl = static_cast<int>(q) * half_rows + rr;
          const int64_t row = rc + rl;
          if (rl < H && row < r1) {  // tile rows past H are not the chunk's
            const float4 a = *reinterpret_cast<const float4*>(part + rl * kTok + 4 * c4);
            const float4 b = *reinterpret_cast<const float4*>(inbox + rr * kTok + 4 * c4);
            const float v[4] = {a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tok = 4 * c4 + i;
              if (tok < p.M) {
                float vi = v[i];
                if constexpr (kQuant) vi *= s_sx[tok];
                p.y[tok * p.N + row] = float_to_bf16_bits_rn(vi);
              }
            }
          }
        }
      }
      // our inbox has been read: the peer may fill it again (after the last
      // chunk nothing more is sent, and each CTA leaves on its own: every
      // access of one CTA to the other's shared memory, the peer's sums and
      // its arrival on "ready", has completed once that CTA's wait on
      // "ready" returned)
      if (k + 1 < nck) {
        consumer_sync();
        if (threadIdx.x == 0) mbar_arrive_remote(map_peer(smem_u32(dbar), peer));
      }
    }
  }
  __syncthreads();
}

struct D2Plan {
  D2Params prm;
  int NT;
  size_t smem;
  bool ok;
};

D2Plan make_d2plan(int64_t M, int64_t N, int64_t K, int bits, int sm_count, bool zp = false) {
  D2Plan pl{};
  pl.ok = false;
  // K % 1024 == 0: the scale rows are 16-byte multiples (TMA) and each K half
  // is a whole number of groups
  if (M < 1 || M > 16 || N < 1 || K < 1024 || K % 1024 != 0 || sm_count < 2) return pl;
  if (N >= (int64_t(1) << 31)) return pl;
  D2Params& p = pl.prm;
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = static_cast<int>(K / 128);
  p.Gh = p.G / 2;
  const int64_t max_c = sm_count / 2;
  const int64_t by_rows = (N + kTileRows - 1) / kTileRows;  // at least a 32-row tile per pair
  p.C = static_cast<int>(by_rows < max_c ? by_rows : max_c);
  const int64_t rows_max = (N + p.C - 1) / p.C;
  p.nchunk = static_cast<int>((rows_max + kMaxH - 1) / kMaxH);
  p.H = static_cast<int>((rows_max + p.nchunk - 1) / p.nchunk);
  p.T = (p.H + kTileRows - 1) / kTileRows;
  p.sx0 = (p.Gh / 8) * 8;
  p.sbox = ((p.G - p.sx0 + 7) / 8) * 8;  // covers [0, Gh) and [Gh, G) from their box starts
  if (p.sbox < p.Gh || p.sbox > 256) return pl;
  pl.NT = M <= 8 ? 1 : 2;
  // Stage gl of a chunk belongs to the warps with kr = gl % ksplit. With
  // ksplit dividing both Gh and the ring depth NS, slot s always belongs to
  // the warps kr = s % ksplit, so whoever waits on a slot's "full" barrier
  // has consumed that slot's previous phase (a parity wait is only sound then).
  p.ksplit = 0;
  p.NS = 0;
  for (int ks = kCWarps / p.T; ks >= 1 && p.NS == 0; --ks) {
    if (ks > p.Gh || p.Gh % ks != 0) continue;
    for (int ns = (kMaxStages / ks) * ks; ns >= ks && ns >= 2; ns -= ks) {
      if (d2_smem(bits, pl.NT, p.T, p.H, p.Gh, p.sbox, ns, zp).total <= kSmemCap) {
        p.ksplit = ks;
        p.NS = ns;
        break;
      }
    }
  }
  if (p.NS < 2 || p.ksplit < 1) return pl;
  pl.smem = d2_smem(bits, pl.NT, p.T, p.H, p.Gh, p.sbox, p.NS, zp).total + 1024;  // + base alignment
  pl.ok = true;
  return pl;
}

template <int B, int NT, int kMode>
cudaError_t d2launch(const Ctx& c, const CUtensorMap& wmap, const CUtensorMap& smap, const D2Plan& pl) {
  static SmemLimit limit;  // dynamic smem opted in so far, per device
  auto kern = decode2_kernel<B, NT, kMode>;
  const cudaError_t e = raise_smem_limit(limit, kern, c.device, pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pl.prm.C), 1, 1);
  cfg.blockDim = dim3(kThreads2, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel of the stream finishes: the kernel
  // reads only weights and scales before griddepcontrol.wait
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, wmap, smap, pl.prm);
}

template <int kMode>
cudaError_t d2launch_b(const Ctx& c, int bits, const CUtensorMap& wmap, const CUtensorMap& smap, const D2Plan& pl) {
  if constexpr (kMode == 1 || kMode == 2) {
    if (bits != 4) return cudaErrorInvalidValue;
    return pl.NT == 1 ? d2launch<4, 1, kMode>(c, wmap, smap, pl) : d2launch<4, 2, kMode>(c, wmap, smap, pl);
  } else {
#define WQ_D2(BB)                                                                 \
  case BB:                                                                        \
    return pl.NT == 1 ? d2launch<BB, 1, kMode>(c, wmap, smap, pl) : d2launch<BB, 2, kMode>(c, wmap, smap, pl);
    switch (bits) {
      WQ_D2(2)
      WQ_D2(3)
      WQ_D2(4)
      WQ_D2(5)
      WQ_D2(6)
      WQ_D2(7)
      WQ_D2(8)
      default: return cudaErrorInvalidValue;
    }
#undef WQ_D2
  }
}

}  // namespace

bool decode2_supported(int64_t M, int64_t N, int64_t K, int bits, int sm_count, bool zp) {
  return bits >= 2 && bits <= 8 && make_d2plan(M, N, K, bits, sm_count, zp).ok;
}

bool decode2_shape(int64_t M, int64_t K) { return M >= 1 && M <= 16 && K >= 1024 && K % 1024 == 0; }

// The plan exists on every device with at least two SMs when its smallest
// configuration (ksplit 1, two ring slots) fits at the largest chunk any SM
// count gives: a chunk has at most min(N, kMaxH) rows, and the shared-memory
// footprint grows with the rows, the tiles and the ring depth.
bool decode2_fits_any(int64_t M, int64_t N, int64_t K, int bits, bool zp) {
  if (bits < 2 || bits > 8 || !decode2_shape(M, K) || N < 1 || N >= (int64_t(1) << 31)) return false;
  const int G = static_cast<int>(K / 128), Gh = G / 2;
  const int sx0 = (Gh / 8) * 8, sbox = ((G - sx0 + 7) / 8) * 8;
  if (sbox < Gh || sbox > 256) return false;
  const int H = static_cast<int>(N < kMaxH ? N : kMaxH);
  const int T = (H + kTileRows - 1) / kTileRows;
  return d2_smem(bits, M <= 8 ? 1 : 2, T, H, Gh, sbox, 2, zp).total <= kSmemCap;
}

int decode2_plan_info(int64_t M, int64_t N, int64_t K, int bits, int sm_count, int64_t* out) {
  const D2Plan pl = make_d2plan(M, N, K, bits, sm_count);
  const D2Params& p = pl.prm;
  const int64_t v[14] = {pl.ok ? 1 : 0, p.C, p.H, p.nchunk, p.T, p.ksplit, p.NS, p.G, p.Gh,
                         p.sbox, p.sx0, pl.NT, static_cast<int64_t>(pl.smem), kMaxStages};
  for (int i = 0; i < 14; ++i) out[i] = v[i];
  return pl.ok ? 1 : 0;
}

cudaError_t launch_decode2(const Ctx& c, const GemvArgs& a) {
  // the W4A8 modes here take a.x, the bf16 activations, and quantize them per
  // token in the kernel; kW4a8GroupAcc writes a.acc instead of a.y
  const bool zp = a.mode == GemvMode::kWna16 && a.zeros != nullptr;
  const int mode = a.mode == GemvMode::kWna16 ? (zp ? 3 : 0) : a.mode == GemvMode::kW4a8 ? 1 : 2;
  if (a.x == nullptr || (mode == 2 && a.acc == nullptr)) return cudaErrorInvalidValue;
  const D2Plan pl = make_d2plan(a.M, a.N, a.K, a.bits, c.sm_count, zp);
  if (!pl.ok) return cudaErrorInvalidValue;
  D2Plan q = pl;
  q.prm.x = a.x;
  q.prm.y = a.y;
  q.prm.acc = a.acc;
  q.prm.zeros = a.zeros;
  q.prm.status = c.status;
  CUtensorMap wmap, smap;
  const uint64_t words = static_cast<uint64_t>(a.K) * a.bits / 32;
  if (!make_tmap_u32_2d(&wmap, a.packed, words, static_cast<uint64_t>(a.N), 4u * a.bits,
                        static_cast<uint32_t>(pl.prm.H)))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&smap, a.scales, static_cast<uint64_t>(pl.prm.G), static_cast<uint64_t>(a.N),
                         static_cast<uint32_t>(pl.prm.sbox), static_cast<uint32_t>(pl.prm.H)))
    return cudaErrorInvalidValue;
  if (mode == 1) return d2launch_b<1>(c, a.bits, wmap, smap, q);
  if (mode == 2) return d2launch_b<2>(c, a.bits, wmap, smap, q);
  if (mode == 3) return d2launch_b<3>(c, a.bits, wmap, smap, q);
  return d2launch_b<0>(c, a.bits, wmap, smap, q);
}

}  // namespace wq

extern "C" wq_status wq_debug_decode_wait_fault(int64_t stop_stage, uint64_t wait_limit_ns) {
  using namespace wq;
  const uint64_t lim = wait_limit_ns == 0 ? kWaitLimitNs : wait_limit_ns;
  const int64_t stage = stop_stage < 0 ? -1 : stop_stage;
  cudaError_t e = cudaMemcpyToSymbol(c_wait_limit_ns, &lim, sizeof(lim));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(c_stop_stage, &stage, sizeof(stage));
  if (e != cudaSuccess) {
    set_error("wq_debug_decode_wait_fault: %s", cudaGetErrorString(e));
    return WQ_ECUDA;
  }
  return WQ_OK;
}
