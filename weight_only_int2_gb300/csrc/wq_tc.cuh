// tcgen05 (5th-generation tensor core) helpers shared by the tensor-core
// GEMM kernels: shared-memory matrix and instruction descriptors, MMA issue
// with the A operand in tensor memory, commits, tensor-memory loads and
// stores, and the swizzled packed-weight tile addressing. Inline PTX for
// sm_103a.
#pragma once

#include "wq_device.cuh"

namespace wq {
namespace tc {

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

// MMA with the A operand in tensor memory: A row m is TMEM lane m, and 32-bit
// column j of the operand holds the bf16 pair (k = 2j, 2j + 1); one K = 16
// step reads 8 columns starting at a_tmem.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Thread t of the warp writes 32 consecutive 32-bit columns of TMEM lane
// (base lane + t); completes with tcgen05.wait::st.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (base + t).
// Completes with tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// N (a multiple of 8) consecutive 32-bit columns of 32 lanes, as loads of
// 8 columns, all in flight; completes with tmem_wait_ld_all.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N % 8 == 0, "columns in loads of 8");
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[8 * c]), "=r"(r[8 * c + 1]), "=r"(r[8 * c + 2]), "=r"(r[8 * c + 3]), "=r"(r[8 * c + 4]),
                   "=r"(r[8 * c + 5]), "=r"(r[8 * c + 6]), "=r"(r[8 * c + 7])
                 : "r"(taddr + 8 * c));
  }
}
// tcgen05.wait::ld for the registers of tmem_ld_cols: each group of eight is
// named by an empty statement after the wait, so that no use of them can be
// moved above it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_all(uint32_t (&r)[N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int c = 0; c < N / 8; ++c)
    asm volatile(""
                 : "+r"(r[8 * c]), "+r"(r[8 * c + 1]), "+r"(r[8 * c + 2]), "+r"(r[8 * c + 3]), "+r"(r[8 * c + 4]),
                   "+r"(r[8 * c + 5]), "+r"(r[8 * c + 6]), "+r"(r[8 * c + 7]));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Thread t of the warp writes 16 consecutive 32-bit columns of TMEM lane
// (base lane + t); completes with tcgen05.wait::st.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The packed tile's shared-memory rows are 16*B bytes apart. For B = 2, 4, 8
// that is a TMA swizzle span (32, 64, 128 B) and the tile is loaded swizzled:
// the 16-byte chunk c of row r sits at chunk c ^ packed_xor<B>(r).
__host__ __device__ constexpr int packed_swizzle_bytes(int b) {
  return b == 8 ? 128 : (b == 4 ? 64 : (b == 2 ? 32 : 0));
}
template <int B>
__device__ __forceinline__ int packed_xor(int r) {
  if constexpr (B == 8) return r & 7;         // address bits 4-6 ^= 7-9
  else if constexpr (B == 4) return (r >> 1) & 3;  // bits 4-5 ^= 7-8
  else if constexpr (B == 2) return (r >> 2) & 1;  // bit 4 ^= bit 7
  else return 0;
}

// N consecutive 32-bit words from shared memory, in the widest loads the
// alignment allows (16 bytes when N % 4 == 0, else 8 when N is even).
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* src, uint32_t (&w)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[j];
      w[4 * j] = v.x, w[4 * j + 1] = v.y, w[4 * j + 2] = v.z, w[4 * j + 3] = v.w;
    }
  } else if constexpr (N % 2 == 0) {
#pragma unroll
    for (int j = 0; j < N / 2; ++j) {
      const uint2 v = reinterpret_cast<const uint2*>(src)[j];
      w[2 * j] = v.x, w[2 * j + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) w[j] = reinterpret_cast<const uint32_t*>(src)[j];
  }
}

}  // namespace tc
}  // namespace wq
