// Weight-streaming GEMV for one sequence (batch 1), bf16 or int8-row-scale
// weights, fp32 accumulation, with fused input RMSNorm and fused epilogues
// (RoPE + KV-cache append, residual add, SwiGLU, plain store).
//
// Decode is weight-bandwidth bound (ninfer pipeline-stages.md, "What it is and
// is not"), so the kernel is built to keep HBM busy:
//   - one persistent CTA per SM; CTA c owns units [c*U/G, (c+1)*U/G), a single
//     contiguous byte range of the packed weights;
//   - a producer warp streams that range through a ring of shared-memory
//     buffers with 1D bulk copies (cp.async.bulk + mbarrier complete_tx) and
//     an L2 evict-first hint; it issues the first ring's worth before the
//     programmatic-dependent-launch wait, because weights never depend on the
//     previous kernel, so the prefetch overlaps the previous kernel's tail;
//   - eight consumer warps split each row's K into 16-byte chunks (thread t
//     owns chunks t, t+256, ...) and keep the matching slice of the input
//     vector (RMSNorm already applied) in registers, so shared memory is read
//     once per weight byte;
//   - every reduction has one fixed order (chunks ascending, a warp xor tree,
//     warps ascending), independent of grid size and stream: identical inputs
//     give identical bits in every stage plan.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kWarps = 8;                   // consumer warps
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;   // plus one producer warp
constexpr int kMaxChunks = 8;               // 16-byte chunks of a row per consumer thread
constexpr int kMaxRowsPerBuf = 32;
constexpr int kMaxBuf = 16;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kBufTarget = 16 * 1024;
constexpr int kFixedSmem = 2 * kMaxBuf * 8 + (2 * kWarps * kMaxRowsPerBuf + kWarps) * 4 + 16;
constexpr uint64_t kDrainLimitNs = 100000000ull;

template <bool INT8>
struct Elem {
  static constexpr int kPerChunk = INT8 ? 16 : 8;  // elements per 16-byte chunk
  static constexpr int kBytes = INT8 ? 1 : 2;
};

__device__ __forceinline__ float chunk_dot(uint4 w, const float* x, float acc, bool /*bf16*/) {
  acc = fmaf(bf16lo(w.x), x[0], acc);
  acc = fmaf(bf16hi(w.x), x[1], acc);
  acc = fmaf(bf16lo(w.y), x[2], acc);
  acc = fmaf(bf16hi(w.y), x[3], acc);
  acc = fmaf(bf16lo(w.z), x[4], acc);
  acc = fmaf(bf16hi(w.z), x[5], acc);
  acc = fmaf(bf16lo(w.w), x[6], acc);
  acc = fmaf(bf16hi(w.w), x[7], acc);
  return acc;
}

__device__ __forceinline__ float chunk_dot_i8(uint4 w, const float* x, float acc) {
  float a, b, c, d;
  i8x4_to_f32(w.x, a, b, c, d);
  acc = fmaf(a, x[0], acc); acc = fmaf(b, x[1], acc); acc = fmaf(c, x[2], acc); acc = fmaf(d, x[3], acc);
  i8x4_to_f32(w.y, a, b, c, d);
  acc = fmaf(a, x[4], acc); acc = fmaf(b, x[5], acc); acc = fmaf(c, x[6], acc); acc = fmaf(d, x[7], acc);
  i8x4_to_f32(w.z, a, b, c, d);
  acc = fmaf(a, x[8], acc); acc = fmaf(b, x[9], acc); acc = fmaf(c, x[10], acc); acc = fmaf(d, x[11], acc);
  i8x4_to_f32(w.w, a, b, c, d);
  acc = fmaf(a, x[12], acc); acc = fmaf(b, x[13], acc); acc = fmaf(c, x[14], acc); acc = fmaf(d, x[15], acc);
  return acc;
}

// All 256 consumers meet at named barrier 1; returns true if any passed `bad`.
__device__ __forceinline__ bool consumers_sync_or(bool bad) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(bad)), "n"(kConsumers)
      : "memory");
  return r != 0;
}

template <bool INT8, bool NORM, int EPI, int MC>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int EPC = Elem<INT8>::kPerChunk;
  constexpr int EB = Elem<INT8>::kBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>(static_cast<long long>(p.units) * cta / G);
  const int u1 = static_cast<int>(static_cast<long long>(p.units) * (cta + 1) / G);
  const int nunits = u1 - u0;
  const int ups = p.units_per_buf;
  const int nbufs = (nunits + ups - 1) / ups;
  const uint32_t row_bytes = static_cast<uint32_t>(p.K) * EB;
  const uint32_t unit_bytes = row_bytes * p.unit_rows;
  const uint32_t buf_bytes = unit_bytes * ups;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.nbuf) * buf_bytes);
  uint64_t* empty = full + p.nbuf;
  float* red = reinterpret_cast<float*>(empty + p.nbuf);  // [2][kWarps][kMaxRowsPerBuf]
  float* nred = red + 2 * kWarps * kMaxRowsPerBuf;        // [kWarps]

  if (tid == 0) {
    for (int i = 0; i < p.nbuf; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kWarps) {
    // Producer: stream this CTA's weight range through the ring.
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      const uint8_t* src = static_cast<const uint8_t*>(p.w) + static_cast<size_t>(u0) * unit_bytes;
      for (int i = 0; i < nbufs; ++i) {
        const int slot = i % p.nbuf;
        if (i >= p.nbuf && !mbar_wait(&empty[slot], ((i / p.nbuf) - 1) & 1)) {
          report_error(p.status, kErrWaitEmpty);
          break;
        }
        const int nu = min(ups, nunits - i * ups);
        const uint32_t bytes = static_cast<uint32_t>(nu) * unit_bytes;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(smem + static_cast<size_t>(slot) * buf_bytes, src + static_cast<size_t>(i) * buf_bytes, bytes,
                 &full[slot], pol);
      }
    }
    return;
  }

  // Consumers. Inputs written by the previous kernel are read only after the wait.
  pdl_wait();
  const int nch = static_cast<int>(row_bytes / 16);
  float x[MC * EPC];
#pragma unroll
  for (int j = 0; j < MC; ++j) {
    const int c = tid + kConsumers * j;
    const float* src = NORM ? p.h : p.x;
#pragma unroll
    for (int e = 0; e < EPC; e += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nch) v = *reinterpret_cast<const float4*>(src + c * EPC + e);
      x[j * EPC + e + 0] = v.x;
      x[j * EPC + e + 1] = v.y;
      x[j * EPC + e + 2] = v.z;
      x[j * EPC + e + 3] = v.w;
    }
  }
  if (NORM) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < MC * EPC; ++i) ss = fmaf(x[i], x[i], ss);
    ss = warp_sum(ss);
    if (lane == 0) nred[warp] = ss;
    consumers_sync_or(false);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += nred[w];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
#pragma unroll
    for (int j = 0; j < MC; ++j) {
      const int c = tid + kConsumers * j;
#pragma unroll
      for (int e = 0; e < EPC; e += 4) {
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < nch) g = *reinterpret_cast<const float4*>(p.gain + c * EPC + e);
        x[j * EPC + e + 0] = x[j * EPC + e + 0] * inv * g.x;
        x[j * EPC + e + 1] = x[j * EPC + e + 1] * inv * g.y;
        x[j * EPC + e + 2] = x[j * EPC + e + 2] * inv * g.z;
        x[j * EPC + e + 3] = x[j * EPC + e + 3] * inv * g.w;
      }
    }
  }

  for (int i = 0; i < nbufs; ++i) {
    const int slot = i % p.nbuf;
    const bool got = mbar_wait(&full[slot], (i / p.nbuf) & 1);
    const int nu = min(ups, nunits - i * ups);
    const int nrows = nu * p.unit_rows;
    const uint8_t* buf = smem + static_cast<size_t>(slot) * buf_bytes;
    float* rb = red + (i & 1) * kWarps * kMaxRowsPerBuf;
    for (int r = 0; r < nrows; ++r) {
      const uint8_t* row = buf + static_cast<size_t>(r) * row_bytes;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < MC; ++j) {
        const int c = tid + kConsumers * j;
        if (c < nch) {
          const uint4 wv = *reinterpret_cast<const uint4*>(row + c * 16);
          if (INT8)
            acc = chunk_dot_i8(wv, x + j * EPC, acc);
          else
            acc = chunk_dot(wv, x + j * EPC, acc, true);
        }
      }
      acc = warp_sum(acc);
      if (lane == 0) rb[warp * kMaxRowsPerBuf + r] = acc;
    }
    if (consumers_sync_or(!got)) {
      // A copy never arrived: record it, drain what may still be in flight, stop.
      if (tid == 0) {
        report_error(p.status, kErrWaitFull);
        for (int j = i; j < min(nbufs, i + p.nbuf); ++j) {
          const uint64_t t0 = globaltimer_ns();
          bool ok = false;
          while (!(ok = mbar_try_wait(&full[j % p.nbuf], (j / p.nbuf) & 1)))
            if (globaltimer_ns() - t0 > kDrainLimitNs) break;
          if (!ok) {
            report_error(p.status, kErrDrain);
            break;
          }
        }
      }
      return;
    }
    if (tid == 0) mbar_arrive(&empty[slot]);
    if (tid < nu) {
      const int u = u0 + i * ups + tid;
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) y0 += rb[w * kMaxRowsPerBuf + tid * p.unit_rows];
      if (EPI == kEpiQkv || EPI == kEpiSwiglu) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) y1 += rb[w * kMaxRowsPerBuf + tid * p.unit_rows + 1];
      }
      if (INT8) {
        y0 *= p.wscale[u * p.unit_rows];
        if (EPI == kEpiQkv || EPI == kEpiSwiglu) y1 *= p.wscale[u * p.unit_rows + 1];
      }
      if (EPI == kEpiQkv) {
        const int half = p.hd >> 1;
        const int hh = u / half, ii = u - hh * half;
        if (hh < p.nq) {
          const float2 cs = p.rope[ii];
          p.out[hh * p.hd + ii] = y0 * cs.x - y1 * cs.y;
          p.out[hh * p.hd + ii + half] = y0 * cs.y + y1 * cs.x;
        } else if (hh < p.nq + p.nkv) {
          const float2 cs = p.rope[ii];
          const size_t base = (static_cast<size_t>(hh - p.nq) * p.max_ctx + p.pos) * p.hd;
          p.kc[base + ii] = __float2bfloat16_rn(y0 * cs.x - y1 * cs.y);
          p.kc[base + ii + half] = __float2bfloat16_rn(y0 * cs.y + y1 * cs.x);
        } else {
          const size_t base = (static_cast<size_t>(hh - p.nq - p.nkv) * p.max_ctx + p.pos) * p.hd;
          p.vc[base + ii] = __float2bfloat16_rn(y0);
          p.vc[base + ii + half] = __float2bfloat16_rn(y1);
        }
      } else if (EPI == kEpiResidual) {
        p.h_out[u] = p.h_in[u] + y0;
      } else if (EPI == kEpiSwiglu) {
        p.out[u] = y0 / (1.0f + expf(-y0)) * y1;
      } else {
        p.out[u] = y0;
      }
    }
  }
}

template <bool INT8, bool NORM, int EPI, int MC>
cudaError_t launch_mc(const GemvParams& p, const GemvPlan& plan, cudaStream_t s, bool pdl) {
  auto kern = gemv_kernel<INT8, NORM, EPI, MC>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget + kFixedSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Chunks per consumer thread, rounded up to an instantiated count.
template <bool INT8, bool NORM, int EPI>
cudaError_t launch_one(const GemvParams& p, const GemvPlan& plan, cudaStream_t s, bool pdl) {
  const int nch = p.K * Elem<INT8>::kBytes / 16;
  const int mc = (nch + kConsumers - 1) / kConsumers;
  if (mc <= 1) return launch_mc<INT8, NORM, EPI, 1>(p, plan, s, pdl);
  if (mc <= 2) return launch_mc<INT8, NORM, EPI, 2>(p, plan, s, pdl);
  if (mc <= 4) return launch_mc<INT8, NORM, EPI, 4>(p, plan, s, pdl);
  if (mc <= 8) return launch_mc<INT8, NORM, EPI, 8>(p, plan, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace

GemvPlan gemv_plan(int rows, int K, int unit_rows, bool int8, int num_sms) {
  GemvPlan g{};
  const int row_bytes = K * (int8 ? 1 : 2);
  const int unit_bytes = row_bytes * unit_rows;
  const int units = rows / unit_rows;
  int ups = kBufTarget / unit_bytes;
  ups = ups < 1 ? 1 : ups;
  if (ups * unit_rows > kMaxRowsPerBuf) ups = kMaxRowsPerBuf / unit_rows;
  const int buf_bytes = ups * unit_bytes;
  int nbuf = kSmemBudget / buf_bytes;
  nbuf = nbuf > kMaxBuf ? kMaxBuf : nbuf;
  g.units_per_buf = ups;
  g.nbuf = nbuf;
  g.grid = units < num_sms ? units : num_sms;
  g.smem = nbuf * buf_bytes + kFixedSmem;
  return g;
}

// Shapes the kernel supports: rows of whole 16-byte chunks, at most kMaxChunks
// chunks per consumer thread, and a ring of at least two units.
bool gemv_supported(int K, int unit_rows, bool int8) {
  const int row_bytes = K * (int8 ? 1 : 2);
  if (K <= 0 || row_bytes % 16) return false;
  if (row_bytes / 16 > kMaxChunks * kConsumers) return false;
  if (2 * unit_rows * row_bytes > kSmemBudget) return false;
  return true;
}

cudaError_t launch_gemv(const GemvParams& p, int epi, bool norm, bool int8, const GemvPlan& plan, cudaStream_t s,
                        bool pdl) {
  if (int8) {
    if (epi == kEpiQkv && norm) return launch_one<true, true, kEpiQkv>(p, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_one<true, false, kEpiResidual>(p, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_one<true, true, kEpiSwiglu>(p, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_one<true, true, kEpiStore>(p, plan, s, pdl);
  } else {
    if (epi == kEpiQkv && norm) return launch_one<false, true, kEpiQkv>(p, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_one<false, false, kEpiResidual>(p, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_one<false, true, kEpiSwiglu>(p, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_one<false, true, kEpiStore>(p, plan, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lps
