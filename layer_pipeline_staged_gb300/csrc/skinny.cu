// Skinny GEMM for batch 2..8 on tensor cores: Y[b][r] = sum_k W[r][k] X[b][k],
// bf16 or int8-row-scale weights, with the same fused RMSNorm input and
// epilogues as the batch-1 GEMV. At batch > 1 every weight byte serves B
// sequences, so the weights are read once per step for the whole batch
// (memra_engine::pp, batch_pp_on: the batched step takes the same stage split).
//
// Weights are re-laid at bind time into tiles of 16*MT packed rows x KC columns,
// ordered [unit][k-chunk]; inside a tile each row's 16-byte chunks are
// XOR-swizzled by (row mod 8), so a tile is one contiguous bulk copy and the
// fragment loads from shared memory are free of bank conflicts.
//
// CTA c owns a contiguous range of units (16*MT rows each) and streams its
// tiles through a ring (producer warp, 1D bulk copies, mbarriers). The
// k-chunks of a unit are split over NW consumer warps (tile i -> warp i mod NW,
// slots owned by one warp each); each warp runs mma.sync m16n8k16 (bf16 in,
// fp32 accumulate) with the weights as the A operand (int8 weights widened to
// bf16, exact for |q| <= 127) and the activations as B. Every fp32 activation
// is written exactly as three bf16 parts, hi = bf16(x), mid = bf16(x - hi),
// lo = x - hi - mid, one B column each (column c of the 3B is sequence c / 3,
// part c mod 3), so the products are exact and only the fp32 accumulation
// rounds. A fixed permutation of k inside each 16-wide k-step (the same for A
// and B) lets every lane fetch 4 consecutive weights. The warps' partial sums
// of a unit are added in warp order, then the epilogue runs.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kMaxWarps = 4;
constexpr int kMaxBuf = 16;
constexpr uint64_t kTileTarget = 16 * 1024;
constexpr int kCols = 3 * kMaxBatch;                  // B columns: three exact bf16 parts per sequence
constexpr int kRedFloats = 2 * kMaxWarps * 32 * kCols;  // [parity][warp][rows of a unit (<=32)][column]
constexpr int kReserve = 2 * kMaxBuf * 8 + kRedFloats * 4 + 2 * kMaxBatch * 4 * 8 + 128;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Part `part` (0: hi, 1: mid, 2: lo) of the exact three-way bf16 split of x:
// hi = bf16(x), mid = bf16(x - hi), lo = x - hi - mid (each difference is exact
// in fp32, and lo fits in bf16 because x has 24 significant bits).
__device__ __forceinline__ float split3(float x, int part) {
  const float hi = bf16_round(x);
  if (part == 0) return hi;
  const float r = x - hi;
  const float mid = bf16_round(r);
  return part == 1 ? mid : r - mid;
}

// c += A.B for one 16-wide k-step. The tensor core sums the 16 exact products
// from a zero accumulator and the result is added to c with an ordinary
// (round-to-nearest) fp32 add, so long sums do not pile up the accumulator's
// truncation.
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  float d0, d1, d2, d3;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
  c[0] += d0;
  c[1] += d1;
  c[2] += d2;
  c[3] += d3;
}

// Four int8 (one word) -> two bf16x2 words, exactly (|q| <= 127 needs 7 bits).
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  float a, b, c, d;
  i8x4_to_f32(w, a, b, c, d);
  lo = pack_bf16(a, b);
  hi = pack_bf16(c, d);
}

// The consumer warps meet at named barrier 1; returns true if any passed `bad`.
__device__ __forceinline__ bool consumers_or(bool bad, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(bad)), "r"(nthreads)
      : "memory");
  return r != 0;
}

template <bool INT8, bool NORM, int EPI, int NT, int MT>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1) skinny_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int EB = INT8 ? 1 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int NW = p.nwarps, B = p.batch;
  const int G = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>(static_cast<long long>(p.units) * cta / G);
  const int u1 = static_cast<int>(static_cast<long long>(p.units) * (cta + 1) / G);
  const int nk = p.KP / p.KC;
  const int ntiles = (u1 - u0) * nk;
  const uint32_t row_bytes = static_cast<uint32_t>(p.KC) * EB;
  const uint32_t tile_bytes = row_bytes * 16 * MT;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.nbuf) * tile_bytes);
  uint64_t* empty = full + p.nbuf;
  float* red = reinterpret_cast<float*>(empty + p.nbuf);  // [2][NW][16*MT][8]
  float* nred = red + kRedFloats;                          // [kMaxBatch][NW] norm partials
  float* inv_s = nred + kMaxBatch * kMaxWarps;             // [kMaxBatch]

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
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      const uint8_t* src = static_cast<const uint8_t*>(p.w) + static_cast<size_t>(u0) * nk * tile_bytes;
      for (int i = 0; i < ntiles; ++i) {
        const int slot = i % p.nbuf;
        if (i >= p.nbuf && !mbar_wait(&empty[slot], ((i / p.nbuf) - 1) & 1)) {
          report_error(p.status, kErrWaitEmpty | ((EPI + 1) << 8) | (1 << 11));
          break;
        }
        mbar_arrive_expect_tx(&full[slot], tile_bytes);
        bulk_g2s(smem + static_cast<size_t>(slot) * tile_bytes, src + static_cast<size_t>(i) * tile_bytes, tile_bytes,
                 &full[slot], pol);
      }
    }
    return;
  }

  pdl_wait();
  const int nthreads = NW * 32;
  // RMSNorm factor of every sequence (fixed order: thread-strided sums, warp tree, warps in order)
  if (NORM) {
    for (int b = 0; b < B; ++b) {
      const float4* h4 = reinterpret_cast<const float4*>(p.x + static_cast<size_t>(b) * p.K);
      float ss = 0.f;
      for (int k4 = tid; k4 < p.K / 4; k4 += nthreads) {
        const float4 v = h4[k4];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) nred[b * kMaxWarps + warp] = ss;
    }
    named_bar_sync(1, nthreads);
    if (tid < B) {
      float tot = 0.f;
      for (int w = 0; w < NW; ++w) tot += nred[tid * kMaxWarps + w];
      inv_s[tid] = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
    }
    named_bar_sync(1, nthreads);
  }

  // this lane's B-operand column of n-tile j: column 8j + g8 = sequence (8j + g8) / 3, part (8j + g8) mod 3
  int part[NT];
  float inv[NT];
  const float* xrow[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int col = 8 * j + g8, b = col / 3;
    part[j] = col - 3 * b;
    xrow[j] = b < B ? p.x + static_cast<size_t>(b) * p.K : nullptr;
    inv[j] = (NORM && b < B) ? inv_s[b] : 1.f;
  }

  float acc[MT][NT][4];
  bool bad = false;  // a bounded wait gave up: keep the barrier count, skip work, leave together
  for (int i = warp; i < ntiles; i += NW) {
    const int unit_local = i / nk, c = i - unit_local * nk;
    if (c == warp) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[mt][j][0] = acc[mt][j][1] = acc[mt][j][2] = acc[mt][j][3] = 0.f;
    }
    const int slot = i % p.nbuf;
    if (!bad && !mbar_wait(&full[slot], (i / p.nbuf) & 1)) {
      bad = true;
      if (lane == 0) report_error(p.status, kErrWaitFull | ((EPI + 1) << 8) | (1 << 11));
    }
    const uint8_t* tile = smem + static_cast<size_t>(slot) * tile_bytes;
    const int k_base = c * p.KC;
#pragma unroll 2
    for (int ks = 0; ks < (bad ? 0 : p.KC / 16); ++ks) {
      const int k0 = k_base + 16 * ks + 4 * t4;  // this lane's 4 consecutive k (permuted k order)
      uint32_t bf[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (xrow[j] && k0 < p.K) {  // columns past K are padding (zero weights, zero input)
          v = *reinterpret_cast<const float4*>(xrow[j] + k0);
          if (NORM) {
            const float4 gg = *reinterpret_cast<const float4*>(p.gain + k0);
            v = make_float4(v.x * inv[j] * gg.x, v.y * inv[j] * gg.y, v.z * inv[j] * gg.z, v.w * inv[j] * gg.w);
          }
        }
        bf[j][0] = pack_bf16(split3(v.x, part[j]), split3(v.y, part[j]));
        bf[j][1] = pack_bf16(split3(v.z, part[j]), split3(v.w, part[j]));
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a[4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // rows g8 and g8 + 8 of this m-tile
          const int r = 16 * mt + g8 + 8 * hf;
          if (INT8) {
            const uint32_t off = r * row_bytes + ((ks ^ (r & 7)) << 4) + 4 * t4;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + off);
            i8x4_to_bf16x4(w, a[hf], a[2 + hf]);
          } else {
            const int ch = 2 * ks + (t4 >> 1);
            const uint32_t off = r * row_bytes + ((ch ^ (r & 7)) << 4) + 8 * (t4 & 1);
            const uint2 w = *reinterpret_cast<const uint2*>(tile + off);
            a[hf] = w.x;
            a[2 + hf] = w.y;
          }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_bf16(acc[mt][j], a, bf[j][0], bf[j][1]);
      }
    }
    __syncwarp();
    if (lane == 0 && !bad) mbar_arrive(&empty[slot]);

    // the unit's last k-chunk of this warp: hand the partial sums over, then merge and finish
    if (c + NW >= nk) {
      float* rb = red + (unit_local & 1) * (kMaxWarps * 32 * kCols);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int col = 8 * j + 2 * t4;  // columns col, col + 1 of rows g8 and g8 + 8
          if (col < kCols) {
            rb[(warp * 32 + 16 * mt + g8) * kCols + col] = acc[mt][j][0];
            rb[(warp * 32 + 16 * mt + g8) * kCols + col + 1] = acc[mt][j][1];
            rb[(warp * 32 + 16 * mt + g8 + 8) * kCols + col] = acc[mt][j][2];
            rb[(warp * 32 + 16 * mt + g8 + 8) * kCols + col + 1] = acc[mt][j][3];
          }
        }
      if (consumers_or(bad, nthreads)) {
        // drain this warp's own copies that may still be in flight (bounded), then stop
        if (lane == 0)
          for (int j = i + NW; j < min(ntiles, i + p.nbuf); j += NW)
            if (!mbar_wait(&full[j % p.nbuf], (j / p.nbuf) & 1, 200000000ll)) break;
        return;
      }
      // one thread per (row, or row pair, of the unit) x sequence
      const int per = (EPI == kEpiQkv || EPI == kEpiSwiglu) ? 2 : 1;
      const int items = (16 * MT / per) * B;
      for (int it = tid; it < items; it += nthreads) {
        const int b = it % B, rl = (it / B) * per;  // first row (local) of the item
        const int r = (u0 + unit_local) * 16 * MT + rl;  // packed row
        if (r >= p.rows) continue;                       // padding rows of the last unit
        float y[2] = {0.f, 0.f};
        for (int k = 0; k < per; ++k) {
          float s = 0.f;
          for (int w = 0; w < NW; ++w) {
            const float* c3 = rb + (w * 32 + rl + k) * kCols + 3 * b;
            s += (c3[0] + c3[1]) + c3[2];
          }
          y[k] = s;
        }
        if (INT8) {
          y[0] *= p.wscale[r];
          if (per == 2) y[1] *= p.wscale[r + 1];
        }
        if (EPI == kEpiQkv) {
          const int u = r >> 1, half = p.hd >> 1;
          const int hh = u / half, ii = u - hh * half;
          const float2 cs = p.rope[static_cast<size_t>(p.pos[b]) * half + ii];
          if (hh < p.nq) {
            float* q = p.out + static_cast<size_t>(b) * p.out_stride;
            q[hh * p.hd + ii] = y[0] * cs.x - y[1] * cs.y;
            q[hh * p.hd + ii + half] = y[0] * cs.y + y[1] * cs.x;
          } else if (hh < p.nq + p.nkv) {
            const size_t base = static_cast<size_t>(b) * p.kv_stride +
                                (static_cast<size_t>(hh - p.nq) * p.max_ctx + p.pos[b]) * p.hd;
            p.kc[base + ii] = __float2bfloat16_rn(y[0] * cs.x - y[1] * cs.y);
            p.kc[base + ii + half] = __float2bfloat16_rn(y[0] * cs.y + y[1] * cs.x);
          } else {
            const size_t base = static_cast<size_t>(b) * p.kv_stride +
                                (static_cast<size_t>(hh - p.nq - p.nkv) * p.max_ctx + p.pos[b]) * p.hd;
            p.vc[base + ii] = __float2bfloat16_rn(y[0]);
            p.vc[base + ii + half] = __float2bfloat16_rn(y[1]);
          }
        } else if (EPI == kEpiResidual) {
          const size_t o = static_cast<size_t>(b) * p.out_stride + r;
          p.h_out[o] = p.h_in[o] + y[0];
        } else if (EPI == kEpiSwiglu) {
          p.out[static_cast<size_t>(b) * p.out_stride + (r >> 1)] = y[0] / (1.0f + expf(-y[0])) * y[1];
        } else {
          p.out[static_cast<size_t>(b) * p.out_stride + r] = y[0];
        }
      }
    }
  }
}

int g_max_smem = 0;

template <bool INT8, bool NORM, int EPI, int NT, int MT>
cudaError_t launch_t(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t s, bool pdl) {
  auto kern = skinny_kernel<INT8, NORM, EPI, NT, MT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g_max_smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
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
cudaError_t launch_e(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t s, bool pdl) {
  const int nt = (3 * p.batch + 7) / 8;  // 8-column n-tiles for 3B columns
  if (plan.mt == 2) {
    if (nt == 1) return launch_t<INT8, NORM, EPI, 1, 2>(p, plan, s, pdl);
    if (nt == 2) return launch_t<INT8, NORM, EPI, 2, 2>(p, plan, s, pdl);
    return launch_t<INT8, NORM, EPI, 3, 2>(p, plan, s, pdl);
  }
  if (nt == 1) return launch_t<INT8, NORM, EPI, 1, 1>(p, plan, s, pdl);
  if (nt == 2) return launch_t<INT8, NORM, EPI, 2, 1>(p, plan, s, pdl);
  return launch_t<INT8, NORM, EPI, 3, 1>(p, plan, s, pdl);
}

}  // namespace

void skinny_set_max_smem(int bytes) { g_max_smem = bytes; }

// KC: the widest of 512..64 columns dividing K with a tile of at most 16 KB and at
// least eight 16-byte chunks per row; MT = 2 when every CTA gets eight or more
// 32-row units; NW: 4, 2 or 1 warps, dividing the k-chunk count; the ring: as many
// tiles as fit, a multiple of NW.
SkinnyPlan skinny_plan(int rows, int K, bool int8, int num_sms, int max_smem) {
  SkinnyPlan g{};
  const int eb = int8 ? 1 : 2;
  g.mt = (rows % 32 == 0 && rows / 32 >= 8 * num_sms) ? 2 : 1;
  int kc = 0;
  for (int want : {4, 2, 1}) {  // the widest tile, little K padding, k-chunks splitting over `want` warps
    for (int c : {1024, 512, 256, 128, 64}) {
      const int nk = (K + c - 1) / c;
      if (c * eb * 16 * g.mt <= static_cast<int>(kTileTarget) && c * eb >= 128 && (nk * c - K) * 8 <= K &&
          nk % want == 0) {
        kc = c;
        break;
      }
    }
    if (kc) break;
  }
  g.kc = kc;
  if (!kc) return g;
  const int nk = (K + kc - 1) / kc;
  g.kp = nk * kc;
  g.nwarps = nk % 4 == 0 ? 4 : (nk % 2 == 0 ? 2 : 1);
  const int tile = kc * eb * 16 * g.mt;
  int room = (max_smem - kReserve) / tile;
  room = room > kMaxBuf ? kMaxBuf : room;
  g.nbuf = room / g.nwarps * g.nwarps;
  const int units = (rows + 16 * g.mt - 1) / (16 * g.mt);
  g.units = units;
  g.rows_p = units * 16 * g.mt;
  g.grid = units < num_sms ? units : num_sms;
  g.smem = g.nbuf * tile + kReserve;
  return g;
}

bool skinny_supported(int rows, int K, bool int8, int num_sms, int max_smem) {
  if (rows % 2 || K % 16) return false;
  const SkinnyPlan g = skinny_plan(rows, K, int8, num_sms, max_smem);
  return g.kc > 0 && g.nbuf >= g.nwarps && g.nbuf >= 2;
}

cudaError_t launch_skinny(const SkinnyParams& p, int epi, bool norm, bool int8, const SkinnyPlan& plan, cudaStream_t s,
                          bool pdl) {
  SkinnyParams q = p;
  q.nwarps = plan.nwarps;
  q.nbuf = plan.nbuf;
  q.KC = plan.kc;
  q.KP = plan.kp;
  q.units = plan.units;
  if (int8) {
    if (epi == kEpiQkv && norm) return launch_e<true, true, kEpiQkv>(q, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_e<true, false, kEpiResidual>(q, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_e<true, true, kEpiSwiglu>(q, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_e<true, true, kEpiStore>(q, plan, s, pdl);
  } else {
    if (epi == kEpiQkv && norm) return launch_e<false, true, kEpiQkv>(q, plan, s, pdl);
    if (epi == kEpiResidual && !norm) return launch_e<false, false, kEpiResidual>(q, plan, s, pdl);
    if (epi == kEpiSwiglu && norm) return launch_e<false, true, kEpiSwiglu>(q, plan, s, pdl);
    if (epi == kEpiStore && norm) return launch_e<false, true, kEpiStore>(q, plan, s, pdl);
  }
  return cudaErrorInvalidValue;
}

namespace {
__global__ void retile_kernel(const uint4* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K, int kp,
                              int kc, int mt, int eb) {
  const int cpr = K * eb / 16;  // 16-byte chunks per source row
  const long long n = static_cast<long long>(rows) * cpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / cpr), ch = static_cast<int>(i - static_cast<long long>(r) * cpr);
    *reinterpret_cast<uint4*>(dst + skinny_offset(r, ch * 16 / eb, kp, kc, mt, eb)) = src[i];
  }
}
}  // namespace

cudaError_t launch_retile(const void* src, void* dst, int rows, int K, int kp, int kc, int mt, int eb, cudaStream_t s) {
  retile_kernel<<<1024, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint8_t*>(dst), rows, K, kp, kc, mt,
                                     eb);
  return cudaGetLastError();
}

// Byte offset of element (row r, column k) of a [rows][K] matrix in the tiled
// layout: tiles of 16*mt rows x kc columns ordered [unit][k-chunk], 16-byte
// chunks of each tile row XOR-swizzled by (row mod 8).
__host__ __device__ size_t skinny_offset(int r, int k, int K, int kc, int mt, int eb) {
  const int rows_u = 16 * mt;
  const int unit = r / rows_u, rr = r - unit * rows_u;
  const int c = k / kc, kk = k - c * kc;
  const size_t tile = static_cast<size_t>(kc) * eb * rows_u;
  const int byte = kk * eb;
  const int ch = byte >> 4, in = byte & 15;
  return (static_cast<size_t>(unit) * (K / kc) + c) * tile + static_cast<size_t>(rr) * kc * eb +
         (((ch ^ (rr & 7)) << 4) | in);
}

}  // namespace lps
