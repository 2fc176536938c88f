// Weight-streaming GEMV for one sequence (batch 1), bf16 or int8-row-scale
// weights, fp32 accumulation, with fused input RMSNorm and fused epilogues
// (RoPE + KV-cache append, residual add, SwiGLU, plain store).
//
// Decode is weight-bandwidth bound (ninfer pipeline-stages.md, "What it is and
// is not"), so the kernel is built to keep HBM busy and never stall on itself:
//   - one persistent CTA per SM; CTA c owns units [c*U/G, (c+1)*U/G), a single
//     contiguous byte range of the packed weights;
//   - a producer warp streams that range through a ring of shared-memory
//     buffers with 1D bulk copies (cp.async.bulk + mbarrier complete_tx) and
//     an L2 evict-first hint; it fills the ring without the programmatic-
//     dependent-launch wait, because weights never depend on the previous
//     kernel, so the prefetch overlaps that kernel's tail and this kernel's
//     own prologue;
//   - the consumers fetch the input vector (and the RMSNorm gain, before the
//     dependency wait) in one round of loads per thread, and each lane loads
//     its next unit's epilogue inputs before waiting for the buffer;
//   - buffer i belongs to consumer warp i mod NW and sits in slot i mod nbuf,
//     with nbuf a multiple of NW: every slot is owned by one warp, which waits
//     on its phases strictly in order (a warp sharing slots with others could
//     run ahead and mistake an older completed phase of the same parity for
//     its buffer). Each warp works through whole rows on its own (no CTA-wide
//     barrier in the main loop), up to four rows at once with independent
//     accumulators, and applies the epilogue itself;
//   - the input vector (RMSNorm already applied) sits in shared memory as
//     float4 planes, so the lanes' reads of weights and inputs are free of
//     bank conflicts;
//   - every reduction has one fixed order (lane l sums chunks l, l+32, ... in
//     ascending order, then a warp xor tree), independent of grid size, warp
//     and stream: identical inputs give identical bits in every stage plan.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kMaxWarps = 8;        // consumer warps
// Producer lanes issuing copies. More lanes fill the ring faster at kernel
// start but measured slower on whole decode steps: the burst queues ahead of
// the previous kernel's completion and of this kernel's input-vector loads.
constexpr int kIssueLanes = 1;
constexpr int kMaxBuf = 16;
constexpr int kMaxRows = 4;         // rows per buffer
constexpr int kBufTarget = 16 * 1024;
constexpr int kReserve = 2 * kMaxBuf * 8 + kMaxWarps * 4 + 64;  // barriers + norm partials

template <bool INT8>
struct Elem {
  static constexpr int kPerChunk = INT8 ? 16 : 8;  // elements per 16-byte chunk
  static constexpr int kBytes = INT8 ? 1 : 2;
  static constexpr int kPlanes = kPerChunk / 4;    // float4 planes of the input vector
};

__device__ __forceinline__ float dot_bf16(uint4 w, const float4 a, const float4 b, float acc) {
  acc = fmaf(bf16lo(w.x), a.x, acc);
  acc = fmaf(bf16hi(w.x), a.y, acc);
  acc = fmaf(bf16lo(w.y), a.z, acc);
  acc = fmaf(bf16hi(w.y), a.w, acc);
  acc = fmaf(bf16lo(w.z), b.x, acc);
  acc = fmaf(bf16hi(w.z), b.y, acc);
  acc = fmaf(bf16lo(w.w), b.z, acc);
  acc = fmaf(bf16hi(w.w), b.w, acc);
  return acc;
}

__device__ __forceinline__ float dot_i8x4(uint32_t w, const float4 a, float acc) {
  float q0, q1, q2, q3;
  i8x4_to_f32(w, q0, q1, q2, q3);
  acc = fmaf(q0, a.x, acc);
  acc = fmaf(q1, a.y, acc);
  acc = fmaf(q2, a.z, acc);
  acc = fmaf(q3, a.w, acc);
  return acc;
}

__device__ __forceinline__ void consumers_sync(int nthreads) { named_bar_sync(1, nthreads); }

template <bool INT8, bool NORM, int EPI, int RB>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1) gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int EB = Elem<INT8>::kBytes;
  constexpr int NP = Elem<INT8>::kPlanes;
  // error-report ids follow the epilogues' order
  static_assert(kEpiQkv + 1 == kKidQkv && kEpiResidual + 1 == kKidResidual && kEpiSwiglu + 1 == kKidSwiglu &&
                    kEpiStore + 1 == kKidHead,
                "kernel ids");
  constexpr int kid = EPI + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NW = p.nwarps;
  const int G = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>(static_cast<long long>(p.units) * cta / G);
  const int u1 = static_cast<int>(static_cast<long long>(p.units) * (cta + 1) / G);
  const int nunits = u1 - u0;
  const int ups = p.units_per_buf;
  const int nbufs = (nunits + ups - 1) / ups;
  const uint32_t row_bytes = static_cast<uint32_t>(p.K) * EB;
  const uint32_t unit_bytes = row_bytes * p.unit_rows;
  const uint32_t buf_bytes = unit_bytes * ups;
  const int nch = static_cast<int>(row_bytes / 16);  // 16-byte chunks per row
  float4* xs = reinterpret_cast<float4*>(smem + static_cast<size_t>(p.nbuf) * buf_bytes);  // [NP][nch]
  uint64_t* full = reinterpret_cast<uint64_t*>(xs + static_cast<size_t>(NP) * nch);
  uint64_t* empty = full + p.nbuf;
  float* nred = reinterpret_cast<float*>(empty + p.nbuf);

  trace_start(p.trace);
  if (tid == 0) {
    for (int i = 0; i < p.nbuf; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == NW) {
    // Producer: lane l of the first IL lanes streams buffers l, l + IL, ...
    // of this CTA's weight range (buffer i into slot i mod nbuf, every slot
    // owned by one lane). The lanes poll their slots together, so no lane's
    // wait blocks another's copy.
    const int IL = p.nbuf % kIssueLanes == 0 ? kIssueLanes : 1;
    const uint64_t pol = l2_evict_first();
    const uint8_t* src = static_cast<const uint8_t*>(p.w) + static_cast<size_t>(u0) * unit_bytes;
    const long long limit = wait_cycles(p.wait_limit);
    int i = lane;
    bool done = lane >= IL || i >= nbufs, failed = false;
    long long t0 = cycles();
    while (true) {
      bool ready = false;
      const int slot = i % p.nbuf;
      if (!done) ready = i < p.nbuf || mbar_test(&empty[slot], ((i / p.nbuf) - 1) & 1);
      if (ready) {
        const int nu = min(ups, nunits - i * ups);
        const uint32_t bytes = static_cast<uint32_t>(nu) * unit_bytes;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(smem + static_cast<size_t>(slot) * buf_bytes, src + static_cast<size_t>(i) * buf_bytes, bytes,
                 &full[slot], pol);
        i += IL;
        done = i >= nbufs;
        t0 = cycles();
      } else if (!done && cycles() - t0 > limit) {
        report_error(p.status, kErrWaitEmpty | (kid << 8));
        done = failed = true;
      }
      if (__all_sync(0xffffffffu, done)) break;
      if (!__any_sync(0xffffffffu, ready)) __nanosleep(64);  // nothing to issue yet
    }
    {
      // Consumers may have left early after an error: the last buffer this
      // lane issued into each slot lands before the CTA may end (that slot's
      // phase cannot move past it, since nothing later was issued there). On
      // the normal path these copies have landed or are about to.
      (void)failed;
      for (int j = max(lane, i - IL * (p.nbuf / IL)); j < i; j += IL)
        if (!mbar_wait(&full[j % p.nbuf], (j / p.nbuf) & 1, kDrainLimitCycles)) {
          report_error(p.status, kErrDrain | (kid << 8));
          break;
        }
    }
    return;
  }

  // Consumers: the input vector into shared memory. The RMSNorm gain does not
  // depend on the previous kernel, so it is fetched before the dependency wait;
  // the vector itself is fetched after it, every load of a thread issued at once.
  const int nthreads = NW * 32;
  const int K4 = p.K / 4;
  const float4* src4 = reinterpret_cast<const float4*>(NORM ? p.h : p.x);
  const float4* g4 = reinterpret_cast<const float4*>(p.gain);
  constexpr int XR = NORM ? 8 : 20;  // float4 per thread held in registers
  const bool in_regs = K4 <= XR * nthreads;
  float4 gr[NORM ? XR : 1];
  if (NORM && in_regs) {
#pragma unroll
    for (int r = 0; r < XR; ++r) {
      const int k4 = tid + r * nthreads;
      if (k4 < K4) gr[r] = g4[k4];
    }
  }
  pdl_wait();
  if (in_regs) {
    float4 xr[XR];
#pragma unroll
    for (int r = 0; r < XR; ++r) {
      const int k4 = tid + r * nthreads;
      if (k4 < K4) xr[r] = src4[k4];
    }
    if (NORM) {
      float ss = 0.f;
#pragma unroll
      for (int r = 0; r < XR; ++r) {
        if (tid + r * nthreads < K4) {
          ss = fmaf(xr[r].x, xr[r].x, ss);
          ss = fmaf(xr[r].y, xr[r].y, ss);
          ss = fmaf(xr[r].z, xr[r].z, ss);
          ss = fmaf(xr[r].w, xr[r].w, ss);
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) nred[warp] = ss;
      consumers_sync(nthreads);
      float tot = 0.f;
      for (int w = 0; w < NW; ++w) tot += nred[w];
      const float inv = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
#pragma unroll
      for (int r = 0; r < XR; ++r) {
        const float4 g = gr[NORM ? r : 0];
        xr[r] = make_float4(xr[r].x * inv * g.x, xr[r].y * inv * g.y, xr[r].z * inv * g.z, xr[r].w * inv * g.w);
      }
    }
#pragma unroll
    for (int r = 0; r < XR; ++r) {
      const int k4 = tid + r * nthreads;
      if (k4 < K4) xs[(k4 % NP) * nch + k4 / NP] = xr[r];
    }
  } else {
    // vectors too long for registers: passes over global memory
    float inv = 1.f;
    if (NORM) {
      float ss = 0.f;
      for (int k4 = tid; k4 < K4; k4 += nthreads) {
        const float4 v = src4[k4];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) nred[warp] = ss;
      consumers_sync(nthreads);
      float tot = 0.f;
      for (int w = 0; w < NW; ++w) tot += nred[w];
      inv = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
    }
    for (int k4 = tid; k4 < K4; k4 += nthreads) {
      float4 v = src4[k4];
      if (NORM) {
        const float4 g = g4[k4];
        v = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
      }
      xs[(k4 % NP) * nch + k4 / NP] = v;
    }
  }
  consumers_sync(nthreads);

  for (int i = warp; i < nbufs; i += NW) {
    const int slot = i % p.nbuf;
    const int nu = min(ups, nunits - i * ups);
    // Lane j's epilogue inputs for unit j of this buffer, loaded before the
    // wait so that their latency hides behind it and the dot products.
    float s0 = 1.f, s1 = 1.f, e0 = 0.f, e1 = 0.f;
    if (lane < nu) {
      const int u = u0 + i * ups + lane;
      if (INT8) {
        s0 = p.wscale[u * p.unit_rows];
        if (EPI == kEpiQkv || EPI == kEpiSwiglu) s1 = p.wscale[u * p.unit_rows + 1];
      }
      if (EPI == kEpiQkv) {
        const int half = p.hd >> 1;
        const int hh = u / half;
        if (hh < p.nq + p.nkv) {
          const float2 cs = p.rope[u - hh * half];
          e0 = cs.x;
          e1 = cs.y;
        }
      }
      if (EPI == kEpiResidual) e0 = p.h_in[u];
    }
    if (!mbar_wait(&full[slot], (i / p.nbuf) & 1, wait_cycles(p.wait_limit))) {
      // A copy did not arrive in time: record it and stop; the producer waits
      // for the copies it issued before the CTA ends.
      if (lane == 0) {
        report_error(p.status, kErrWaitFull | (kid << 8) | (min(i, 0x3ffff) << 13));
      }
      return;
    }
    const int rows = nu * p.unit_rows;
    const uint8_t* buf = smem + static_cast<size_t>(slot) * buf_bytes;
    float acc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] = 0.f;
#pragma unroll 2
    for (int c = lane; c < nch; c += 32) {
      float4 xv[NP];
#pragma unroll
      for (int pl = 0; pl < NP; ++pl) xv[pl] = xs[pl * nch + c];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r < rows) {
          const uint4 wv = *reinterpret_cast<const uint4*>(buf + r * row_bytes + c * 16);
          if (INT8) {
            acc[r] = dot_i8x4(wv.x, xv[0], acc[r]);
            acc[r] = dot_i8x4(wv.y, xv[1], acc[r]);
            acc[r] = dot_i8x4(wv.z, xv[2], acc[r]);
            acc[r] = dot_i8x4(wv.w, xv[3], acc[r]);
          } else {
            acc[r] = dot_bf16(wv, xv[0], xv[NP - 1], acc[r]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // the buffer is no longer read
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] = warp_sum(acc[r]);

    // epilogue: lane j finishes unit j of this buffer
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      if (j < nu && lane == j) {
        const int u = u0 + i * ups + j;
        float y0 = 0.f, y1 = 0.f;
        if (EPI == kEpiQkv || EPI == kEpiSwiglu) {
          if (2 * j + 1 < RB) {
            y0 = acc[2 * j];
            y1 = acc[2 * j + 1];
          }
        } else {
          y0 = acc[j];
        }
        if (INT8) {
          y0 *= s0;
          if (EPI == kEpiQkv || EPI == kEpiSwiglu) y1 *= s1;
        }
        if (EPI == kEpiQkv) {
          const int half = p.hd >> 1;
          const int hh = u / half, ii = u - hh * half;
          if (hh < p.nq) {
            p.out[hh * p.hd + ii] = y0 * e0 - y1 * e1;
            p.out[hh * p.hd + ii + half] = y0 * e1 + y1 * e0;
          } else if (hh < p.nq + p.nkv) {
            const size_t base = (static_cast<size_t>(hh - p.nq) * p.max_ctx + p.pos) * p.hd;
            p.kc[base + ii] = __float2bfloat16_rn(y0 * e0 - y1 * e1);
            p.kc[base + ii + half] = __float2bfloat16_rn(y0 * e1 + y1 * e0);
          } else {
            const size_t base = (static_cast<size_t>(hh - p.nq - p.nkv) * p.max_ctx + p.pos) * p.hd;
            p.vc[base + ii] = __float2bfloat16_rn(y0);
            p.vc[base + ii + half] = __float2bfloat16_rn(y1);
          }
        } else if (EPI == kEpiResidual) {
          p.h_out[u] = e0 + y0;
        } else if (EPI == kEpiSwiglu) {
          p.out[u] = y0 / (1.0f + expf(-y0)) * y1;
        } else {
          p.out[u] = y0;
        }
      }
    }
  }
  trace_end(p.trace);
}


template <bool INT8, bool NORM, int EPI, int RB>
cudaError_t launch_rb(const GemvParams& p, const GemvPlan& plan, cudaStream_t s, bool pdl) {
  auto kern = gemv_kernel<INT8, NORM, EPI, RB>;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(kern, plan.smem, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3((plan.nwarps + 1) * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool INT8, bool NORM, int EPI>
cudaError_t launch_one(const GemvParams& p, const GemvPlan& plan, cudaStream_t s, bool pdl) {
  const int rb = p.units_per_buf * p.unit_rows;
  if (rb <= 1) return launch_rb<INT8, NORM, EPI, 1>(p, plan, s, pdl);
  if (rb <= 2) return launch_rb<INT8, NORM, EPI, 2>(p, plan, s, pdl);
  if (rb <= 4) return launch_rb<INT8, NORM, EPI, 4>(p, plan, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace

// Ring sizing: buffers of whole units (about 16 KB, at most four rows), as many
// as fit beside the input vector in the opt-in shared memory, one consumer warp
// per buffer up to eight.
GemvPlan gemv_plan(int rows, int K, int unit_rows, bool int8, int num_sms, int max_smem) {
  GemvPlan g{};
  const int row_bytes = K * (int8 ? 1 : 2);
  const int unit_bytes = row_bytes * unit_rows;
  const int units = rows / unit_rows;
  int ups = kBufTarget / unit_bytes;
  ups = ups < 1 ? 1 : ups;
  if (ups * unit_rows > kMaxRows) ups = kMaxRows / unit_rows;
  const int buf_bytes = ups * unit_bytes;
  const int avail = max_smem - K * 4 - kReserve;
  int room = avail / buf_bytes;
  room = room > kMaxBuf ? kMaxBuf : room;
  // nbuf = nwarps * depth: among 8 to 4 warps the most slots that fit
  // (then the most warps); with room for fewer than four buffers, one each
  int best_w = room, best_n = room;
  if (room >= 4) {
    best_n = 0;
    for (int w : {8, 7, 6, 5, 4}) {
      const int n = (room / w) * w;
      if (n > best_n) {
        best_w = w;
        best_n = n;
      }
    }
  }
  g.units_per_buf = ups;
  g.nbuf = best_n;
  g.nwarps = best_w;
  g.grid = units < num_sms ? units : num_sms;
  g.smem = best_n * buf_bytes + K * 4 + kReserve;
  return g;
}

// Shapes the kernel supports: rows of whole 16-byte chunks and a ring of at
// least two buffers beside the input vector.
bool gemv_supported(int K, int unit_rows, bool int8, int max_smem) {
  const int row_bytes = K * (int8 ? 1 : 2);
  if (K <= 0 || row_bytes % 16) return false;
  return 2 * unit_rows * row_bytes + K * 4 + kReserve <= max_smem;
}


cudaError_t launch_gemv(const GemvParams& p, int epi, bool norm, bool int8, const GemvPlan& plan, cudaStream_t s,
                        bool pdl) {
  GemvParams q = p;
  q.nwarps = plan.nwarps;
  if (int8) {
    if (epi == kEpiQkv && norm) return launch_one<true, true, kEpiQkv>(q, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_one<true, false, kEpiResidual>(q, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_one<true, true, kEpiSwiglu>(q, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_one<true, true, kEpiStore>(q, plan, s, pdl);
  } else {
    if (epi == kEpiQkv && norm) return launch_one<false, true, kEpiQkv>(q, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_one<false, false, kEpiResidual>(q, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_one<false, true, kEpiSwiglu>(q, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_one<false, true, kEpiStore>(q, plan, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lps
