// Inline-PTX building blocks for sm_103a: mbarriers, 1D bulk (TMA) copies into
// shared memory, L2 eviction hints, programmatic dependent launch, and bounded
// waits that report a timeout instead of spinning forever.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lps {

// Device-side error reports. A status is two ints: word 0 collects the kind
// bits below (OR-ed), word 1 keeps the first report whole (kind bits, the
// kernel id at bits 8..11 and a detail above), so the host can name the
// kernel that failed first.
enum : int {
  kErrWaitFull = 1,    // a consumer gave up waiting for a bulk copy
  kErrWaitEmpty = 2,   // a producer gave up waiting for a buffer to be released
  kErrDrain = 4,       // draining in-flight copies after an error also timed out
  kErrBadArg = 8,      // a kernel saw an argument outside its supported range
  kErrBarrier = 16,    // a grid-wide barrier wait gave up
};
// Kernel ids of the reports (bits 8..11); bit 12 marks the batch > 1 GEMM.
enum : int {
  kKidQkv = 1,         // RMSNorm + QKV + RoPE + KV append
  kKidResidual = 2,    // o-proj or down projection + residual
  kKidSwiglu = 3,      // RMSNorm + gate/up + SwiGLU
  kKidHead = 4,        // final RMSNorm + LM head
  kKidAttn = 5,        // split-K attention
  kKidAttnCombine = 6, // split-K attention, the last CTA's merge
  kKidEmbed = 7,       // embedding row
  kKidStage = 8,       // the persistent stage kernel
  kKidTcGemm = 9,      // prefill-chunk GEMM on tcgen05
  kKidChunkAttn = 10,  // prefill-chunk attention (and its merge)
  kKidPrep = 11,       // prefill-chunk RMSNorm / split of the activations
  kKidSkinnyBit = 1 << 12,
};

// Every mbarrier wait gives up after this many SM cycles (about two seconds at
// the maximum clock) unless a kernel's parameters set a shorter limit (a test
// hook). The per-SM cycle counter is used because it is monotonic on the SM
// that spins; a global timer read can step backwards between SMs' updates, and
// an unsigned difference of two such reads would wrap.
constexpr long long kWaitLimitCycles = 4000000000ll;
// Waiting for the copies a thread issued itself to land before its CTA ends
// (after an error) keeps this bound, whatever the parameters say: a copy must
// never land in the shared memory of a CTA that has ended.
constexpr long long kDrainLimitCycles = 200000000ll;  // about 0.1 s

// The wait limit a kernel uses: the parameter when positive, else the default.
__host__ __device__ __forceinline__ long long wait_cycles(long long param) {
  return param > 0 ? param : kWaitLimitCycles;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ long long cycles() { return clock64(); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false after `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = cycles();
  while (!mbar_try_wait(bar, parity)) {
    if (cycles() - t0 > limit) return false;
  }
  return true;
}

// Launch tracing: a record is two 64-bit words, both zero before the launch:
// word 0 collects ~(earliest start) by atomicMax, word 1 the latest end, in
// %globaltimer nanoseconds. t == nullptr when tracing is off.
// One non-blocking look at phase `parity` of `bar`: true once it has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_start(unsigned long long* t) {
  if (t && threadIdx.x == 0) atomicMax(t, ~global_ns());
}
__device__ __forceinline__ void trace_end(unsigned long long* t) {
  if (t && (threadIdx.x & 31) == 0) atomicMax(t + 1, global_ns());
}

// L2 policy that lets streamed-once data (weights, KV rows) be evicted first.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// 16-byte global -> shared copy through L2 (bytes < 16 zero-fill the rest)
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Record an error: `code` = kind bits | kernel id << 8 | detail << 13.
__device__ __forceinline__ void report_error(int* status, int code) {
  if (status) {
    atomicOr(status, code & 0xff);
    atomicCAS(status + 1, 0, code);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// bf16 pair in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four signed int8 in a 32-bit word -> four exact floats, by the magic-number
// construction: flipping the sign bit biases each byte to u = q + 128, the
// bit pattern 0x4B0000uu is the float 2^23 + u, and subtracting 2^23 + 128
// leaves q exactly.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float& a, float& b, float& c, float& d) {
  const uint32_t u = w ^ 0x80808080u;
  const float bias = 8388736.0f;  // 2^23 + 128
  a = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - bias;
  b = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - bias;
  c = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - bias;
  d = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - bias;
}

}  // namespace lps
