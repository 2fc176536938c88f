// tcgen05 (fifth-generation tensor core) and TMA building blocks shared by
// the tensor-core GEMMs: TMEM allocation, the MMA with its commit, TMEM loads,
// the shared-memory and instruction descriptors, and the split of a matrix's
// (tile, k-block) iterations into equal contiguous ranges, one per CTA.
#pragma once

#include "ptx.cuh"

namespace lps {
namespace tc {

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A . B^T, both operands K-major bf16 in shared memory.
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes, 8-row groups 1024 bytes apart (the
// stride byte offset); the leading byte offset is unused for this layout.
// Bits: start address >> 4 at 0..13, LBO >> 4 at 16..29, SBO >> 4 at 32..45,
// descriptor version 1 at 46..47, layout type 2 (128-byte swizzle) at 61..63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// Instruction descriptor of kind::f16: D fp32 (bits 4..5 = 1), A and B bf16
// (bits 7..9 and 10..12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at
// bits 17..22, M >> 4 at bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---- work split ----------------------------------------------------------------

// CTA c of G takes iterations [range_start(c), range_start(c + 1)) of T. The
// launchers keep T * G below 2^32, so 32-bit unsigned arithmetic is exact
// (and far cheaper than 64-bit division on the GPU).
__device__ __forceinline__ long long range_start(int c, long long T, int G) {
  return static_cast<long long>(static_cast<uint32_t>(c) * static_cast<uint32_t>(T) / static_cast<uint32_t>(G));
}
// The CTA whose range holds iteration i: the largest c with range_start(c) <= i.
__device__ __forceinline__ int owner_of(long long i, long long T, int G) {
  return static_cast<int>((static_cast<uint32_t>(i + 1) * static_cast<uint32_t>(G) - 1u) / static_cast<uint32_t>(T));
}

struct Run {
  int tile, k0, k1;  // k-blocks [k0, k1) of tile `tile`
};
// Run number `n` of a CTA whose range is [beg, end); false past the last run.
__device__ __forceinline__ bool run_at(long long beg, long long end, int nkb, int n, Run* r) {
  if (beg >= end) return false;
  const long long t0 = beg / nkb;
  const long long t = t0 + n;
  const long long lo = t * nkb > beg ? t * nkb : beg;
  if (lo >= end) return false;
  const long long hi = (t + 1) * nkb < end ? (t + 1) * nkb : end;
  r->tile = static_cast<int>(t);
  r->k0 = static_cast<int>(lo - t * nkb);
  r->k1 = static_cast<int>(hi - t * nkb);
  return true;
}

}  // namespace tc
}  // namespace lps
