// Skinny GEMM for batch 2..8 on tensor cores: Y[b][r] = sum_k W[r][k] X[b][k],
// bf16 or int8-row-scale weights, with the same fused RMSNorm input and
// epilogues as the batch-1 GEMV. At batch > 1 every weight byte serves B
// sequences, so the weights are read once per step for the whole batch
// (memra_engine::pp, batch_pp_on: the batched step takes the same stage split).
//
// Work split: CTA g owns a contiguous range of nu 16-row units and takes them
// in passes of at most PU (<= 4) units, each pass over all of K. Consumer warp
// w owns the k-chunks w, w + 8, w + 16, ... of every pass and computes all
// the pass's units over them, with no synchronisation with the other warps
// until the pass ends; then the 8 warps' partial sums meet in shared memory
// and are added in warp order.
//
// Data movement: the weights are re-laid at bind time into tiles of 16 rows x
// KC columns, ordered [CTA range][k-chunk][unit of the range], each row's
// 16-byte chunks XOR-swizzled by (row mod 8), so the fragment loads are free
// of bank conflicts, and the tiles of one k-chunk of a pass are one contiguous
// stage. Lane w of the producer warp streams warp w's stages into the warp's
// ring, one bulk copy and one mbarrier per stage (issuing and waiting cost a
// thread ~0.1-0.2 us each, so stages are large and the lanes poll their rings
// together instead of blocking one another). Each consumer warp copies the
// activations (and the RMSNorm gain) of its next k-chunk with cp.async into
// the second of its two activation slots while it computes the current one.
//
// Arithmetic: mma.sync m16n8k16, bf16 in, fp32 out, weights as the A operand
// (int8 widened to bf16, exact for |q| <= 127). Every fp32 activation is
// written exactly as three bf16 parts, hi = bf16(x), mid = bf16(x - hi),
// lo = x - hi - mid; n-tile p of the B operand holds part p and its column b
// sequence b, so the products are exact. Lane (b, t) of a warp splits its own
// 4 activations of every k-step (a fixed permutation of k inside each k-step,
// the same for A and B, lets every lane take 4 consecutive columns). A tile's
// k-steps accumulate on the tensor core (its truncating adds stay within
// KC/16 steps); each tile's sum is then added to the unit's total with a
// round-to-nearest fp32 add, a two-level sum that keeps long sums accurate.
// The RMSNorm factors, the splits and every sum have one fixed order, and the
// plan depends only on the matrix shape: identical inputs give identical bits.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kWarps = 8;               // consumer warps; one more warp is the producer
constexpr int kMaxPu = 4;               // units per pass
constexpr int kParts = 3;               // n-tiles: hi, mid and lo parts; column b = sequence b
constexpr int kCols = 8 * kParts;       // B columns
constexpr int kBarAll = 1;              // named barrier of the consumer warps

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// c += A.B for one 16-wide k-step, accumulated on the tensor core.
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four int8 (one word) -> two bf16x2 words, exactly (|q| <= 127 needs 7 bits).
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  float a, b, c, d;
  i8x4_to_f32(w, a, b, c, d);
  lo = pack_bf16(a, b);
  hi = pack_bf16(c, d);
}

// Named barrier `id` over `nthreads`; returns true if any participant passed `bad`.
__device__ __forceinline__ bool bar_or(int id, int nthreads, bool bad) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(bad)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Non-blocking test of phase `parity` of `bar`.
// Wait for phase `parity` of `bar`, the thread suspended in hardware between
// checks (up to 20 us each); false after `limit` cycles.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, long long limit = kWaitLimitCycles) {
  const long long t0 = cycles();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if (cycles() - t0 > limit) return false;
  }
}

// 16-byte asynchronous copy global -> shared by this thread; `bytes` (0 or 16)
// are read, the rest of the 16 is zero-filled.

// Shared-memory map of one CTA, in bytes; the same on host and device.
struct Layout {
  int tile_bytes;   // one weight tile: 16 rows x KC
  int stage_bytes;  // one stage: the tiles of one k-chunk of a pass (pu tiles)
  int xrow;         // floats per activation row in a slot: KC + 4 (rows start 4 banks apart)
  int xslot_bytes;  // one activation k-chunk: B rows and the gain row
  int rings, xslots, scratch, bars, total;
};
__host__ __device__ inline Layout layout(int rc, int pu, int kc, int eb, int batch) {
  Layout L{};
  L.tile_bytes = 16 * kc * eb;
  L.stage_bytes = pu * L.tile_bytes;
  L.xrow = kc + 4;
  L.xslot_bytes = (batch + 1) * L.xrow * 4;
  L.rings = 0;
  L.xslots = L.rings + kWarps * rc * L.stage_bytes;
  L.scratch = L.xslots + kWarps * 2 * L.xslot_bytes;
  L.bars = L.scratch + kWarps * pu * 16 * kCols * 4;
  L.total = L.bars + 2 * kWarps * rc * 8 + (kMaxBatch * kWarps + kMaxBatch) * 4;
  return L;
}

// KCB: bytes of one tile row (128 or 256), so that KC = KCB / EB columns.
template <bool INT8, bool NORM, int EPI, int UPW, int KCB>
__global__ void __launch_bounds__((kWarps + 1) * 32, 1) skinny_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int EB = INT8 ? 1 : 2;
  constexpr int KC = KCB / EB, KSTEPS = KC / 16, KG = KC / 4;  // columns, k-steps and 4-column groups of a chunk
  constexpr int KH = KSTEPS < 4 ? KSTEPS : 4;                   // k-steps whose fragments are split together
  constexpr int NW = kWarps;
  constexpr int per = (EPI == kEpiQkv || EPI == kEpiSwiglu) ? 2 : 1;  // rows per output item
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int B = p.batch, RC = p.rc, PU = p.pu;
  const int G = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>(static_cast<long long>(p.units) * cta / G);
  const int nu = static_cast<int>(static_cast<long long>(p.units) * (cta + 1) / G) - u0;
  const int nk = p.KP / KC;
  const int npass = (nu + PU - 1) / PU;
  const Layout Lo = layout(RC, PU, KC, EB, B);
  const int nthreads = NW * 32;
  const size_t tb = Lo.tile_bytes;
  uint64_t* full_all = reinterpret_cast<uint64_t*>(smem + Lo.bars);  // [NW][RC]
  uint64_t* empty_all = full_all + NW * RC;                           // [NW][RC]
  float* nred = reinterpret_cast<float*>(empty_all + NW * RC);        // [kMaxBatch][NW]
  float* inv_s = nred + kMaxBatch * NW;                               // [kMaxBatch]
  const uint8_t* wsrc = static_cast<const uint8_t*>(p.w) + static_cast<size_t>(u0) * nk * tb;
  // warp w's k-chunks in a pass: w + 8 n for n < ng(w)
  auto warp_chunks = [&](int w) { return w < nk ? (nk - 1 - w) / NW + 1 : 0; };

  trace_start(p.trace);
  if (tid == 0) {
    for (int i = 0; i < NW * RC; ++i) {
      mbar_init(&full_all[i], 1);
      mbar_init(&empty_all[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == NW) {
    // Producer: lane w streams consumer warp w's stages (pass, chunk) in order;
    // the lanes poll their rings together (no lane blocks the others). Weights
    // never depend on the previous kernel, so no wait for it.
    const int w = lane;
    const int ng = w < NW ? warp_chunks(w) : 0;
    const int S = npass * ng;
    uint8_t* ring = smem + Lo.rings + static_cast<size_t>(w) * RC * Lo.stage_bytes;
    uint64_t* full = full_all + w * RC;
    uint64_t* empty = empty_all + w * RC;
    const uint64_t pol = l2_evict_first();
    int s = 0, n = 0, j0 = 0;  // next step, its chunk index in the pass and first unit
    int slot = 0, phase = 0;   // s mod RC and (s / RC) mod 2
    bool done = S == 0, failed = false;
    long long t0 = cycles();
    while (true) {
      bool ready = false;
      if (!done) ready = s < RC || mbar_test(&empty[slot], phase ^ 1);
      if (ready) {
        const int np = min(PU, nu - j0), c = w + NW * n;
        const uint32_t bytes = static_cast<uint32_t>(np * tb);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(ring + slot * Lo.stage_bytes, wsrc + (static_cast<size_t>(c) * nu + j0) * tb, bytes, &full[slot],
                 pol);
        ++s;
        if (++slot == RC) {
          slot = 0;
          phase ^= 1;
        }
        if (++n == ng) {
          n = 0;
          j0 += PU;
        }
        done = s >= S;
        t0 = cycles();
      } else if (!done && cycles() - t0 > wait_cycles(p.wait_limit)) {
        report_error(p.status, kErrWaitEmpty | ((EPI + 1) << 8) | kKidSkinnyBit);
        done = failed = true;
      }
      if (__all_sync(0xffffffffu, done)) break;
      if (!__any_sync(0xffffffffu, ready)) __nanosleep(64);  // nothing to issue yet
    }
    // the last stages issued land in this CTA's shared memory before it may
    // end, also when the consumers leave early (bounded)
    for (int t = max(0, s - RC); t < s; ++t)
      if (!mbar_wait(&full[t % RC], (t / RC) & 1, failed ? kDrainLimitCycles : kWaitLimitCycles)) {
        report_error(p.status, kErrDrain | ((EPI + 1) << 8) | kKidSkinnyBit);
        break;
      }
    return;
  }

  // Consumers.
  const int ng = warp_chunks(warp);
  const int S = npass * ng;
  const uint8_t* ring = smem + Lo.rings + static_cast<size_t>(warp) * RC * Lo.stage_bytes;
  uint64_t* full = full_all + warp * RC;
  uint64_t* empty = empty_all + warp * RC;
  float* xslot0 = reinterpret_cast<float*>(smem + Lo.xslots + warp * 2 * Lo.xslot_bytes);
  float* part = reinterpret_cast<float*>(smem + Lo.scratch);
  const int xslot_floats = Lo.xslot_bytes / 4;

  // the activations (and gain) of this warp's n-th chunk into slot `slot`;
  // columns past K read as zeros
  auto fetch_x = [&](int n, int slot) {
    const int c = warp + NW * n;
    const int kv4 = min(KC, p.K - c * KC) / 4;
    float* xd = xslot0 + slot * xslot_floats;
    const float* xc = p.x + c * KC;
#pragma unroll
    for (int i0 = 0; i0 < (kMaxBatch + 1) * KG; i0 += 32) {
      const int i = i0 + lane;
      const int b = i / KG, g4 = i % KG;  // KG is a power of two
      if (b > B || (!NORM && b == B)) break;
      const bool in = g4 < kv4;
      const float* src = (b < B ? xc + static_cast<size_t>(b) * p.K : p.gain + c * KC) + 4 * (in ? g4 : 0);
      cp_async16(xd + b * Lo.xrow + 4 * g4, src, in ? 16u : 0u);
    }
    cp_async_commit();
  };

  pdl_wait();
  if (S > 0) fetch_x(0, 0);
  if (S > 1) fetch_x(1 % ng, 1);
  // The RMSNorm factor of every sequence needs all of h: read it from global
  // memory (fixed order: strided sums, warp tree, warps in order).
  if (NORM) {
    float ss[kMaxBatch];
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) ss[b] = 0.f;
    const float4* h4 = reinterpret_cast<const float4*>(p.x);
    for (int k4 = tid; k4 < p.K / 4; k4 += nthreads) {
      float4 v[kMaxBatch];
#pragma unroll
      for (int b = 0; b < kMaxBatch; ++b)
        if (b < B) v[b] = h4[static_cast<size_t>(b) * (p.K / 4) + k4];
#pragma unroll
      for (int b = 0; b < kMaxBatch; ++b)
        if (b < B) {
          ss[b] = fmaf(v[b].x, v[b].x, ss[b]);
          ss[b] = fmaf(v[b].y, v[b].y, ss[b]);
          ss[b] = fmaf(v[b].z, v[b].z, ss[b]);
          ss[b] = fmaf(v[b].w, v[b].w, ss[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b)
      if (b < B) {
        const float t = warp_sum(ss[b]);
        if (lane == 0) nred[b * NW + warp] = t;
      }
    named_bar_sync(kBarAll, nthreads);
    if (tid < B) {
      float tot = 0.f;
      for (int w = 0; w < NW; ++w) tot += nred[tid * NW + w];
      inv_s[tid] = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
    }
    named_bar_sync(kBarAll, nthreads);
  }
  // this lane's sequence (B column) and its RMSNorm factor; lanes of absent sequences split zeros
  const bool has_seq = g8 < B;
  const float inv_mine = (NORM && has_seq) ? inv_s[g8] : 1.f;

  float acc[UPW][kParts][4];
#pragma unroll
  for (int u = 0; u < UPW; ++u)
#pragma unroll
    for (int j = 0; j < kParts; ++j) acc[u][j][0] = acc[u][j][1] = acc[u][j][2] = acc[u][j][3] = 0.f;
  bool bad = false;  // a bounded wait gave up: skip work, leave together at the end of the pass

  // the output of packed row r (and r + 1) for sequence b
  auto finish = [&](int r, int b, float y0, float y1) {
    float y[2] = {y0, y1};
    if (INT8) {
      y[0] *= p.wscale[r];
      if (per == 2) y[1] *= p.wscale[r + 1];
    }
    if (EPI == kEpiQkv) {
      const int un = r >> 1, half = p.hd >> 1;
      const int hh = un / half, ii = un - hh * half;
      const float2 cs = p.rope[static_cast<size_t>(p.pos[b]) * half + ii];
      if (hh < p.nq) {
        float* qo = p.out + static_cast<size_t>(b) * p.out_stride;
        qo[hh * p.hd + ii] = y[0] * cs.x - y[1] * cs.y;
        qo[hh * p.hd + ii + half] = y[0] * cs.y + y[1] * cs.x;
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
  };

  int s = 0;  // the warp's step: (pass, chunk)
  int slot = 0, phase = 0;  // its ring slot, s mod RC, and that slot's phase parity, (s / RC) mod 2
  for (int pass = 0; pass < npass; ++pass) {
    const int j0 = pass * PU, np = min(PU, nu - j0);
    for (int n = 0; n < ng; ++n, ++s) {
      // the step's activations (this lane's copies, then the warp's) and weights
      if (s + 1 < S)
        cp_async_wait_but_one();
      else
        cp_async_wait_all();
      __syncwarp();
      if (!bad && !mbar_wait_sleep(&full[slot], phase, wait_cycles(p.wait_limit))) {
        bad = true;
        if (lane == 0) report_error(p.status, kErrWaitFull | ((EPI + 1) << 8) | kKidSkinnyBit);
      }
      if (!bad) {
        const float* xs = xslot0 + (s & 1) * xslot_floats;
        const float* xr = xs + (has_seq ? g8 : 0) * Lo.xrow + 4 * t4;
        const float* gr = xs + B * Lo.xrow + 4 * t4;
        const uint8_t* stage = ring + slot * Lo.stage_bytes;
        float ts[UPW][kParts][4];  // the tiles' sums: added once into the units' totals
#pragma unroll
        for (int u = 0; u < UPW; ++u)
#pragma unroll
          for (int pt = 0; pt < kParts; ++pt) ts[u][pt][0] = ts[u][pt][1] = ts[u][pt][2] = ts[u][pt][3] = 0.f;
        // KH k-steps at a time: first this lane's B fragments of all of them (the 3
        // exact parts of its 4 activations per k-step: independent chains), then
        // their MMAs for every unit
#pragma unroll
        for (int h = 0; h < KSTEPS; h += KH) {
          uint32_t bf[KH][kParts][2];
#pragma unroll
          for (int k2 = 0; k2 < KH; ++k2) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (has_seq) {
              v = *reinterpret_cast<const float4*>(xr + 16 * (h + k2));
              if (NORM) {
                const float4 gg = *reinterpret_cast<const float4*>(gr + 16 * (h + k2));
                v = make_float4(v.x * inv_mine * gg.x, v.y * inv_mine * gg.y, v.z * inv_mine * gg.z,
                                v.w * inv_mine * gg.w);
              }
            }
            bf[k2][0][0] = pack_bf16(v.x, v.y);
            bf[k2][0][1] = pack_bf16(v.z, v.w);
            const float r0 = v.x - bf16lo(bf[k2][0][0]), r1 = v.y - bf16hi(bf[k2][0][0]);
            const float r2 = v.z - bf16lo(bf[k2][0][1]), r3 = v.w - bf16hi(bf[k2][0][1]);
            bf[k2][1][0] = pack_bf16(r0, r1);
            bf[k2][1][1] = pack_bf16(r2, r3);
            bf[k2][2][0] = pack_bf16(r0 - bf16lo(bf[k2][1][0]), r1 - bf16hi(bf[k2][1][0]));
            bf[k2][2][1] = pack_bf16(r2 - bf16lo(bf[k2][1][1]), r3 - bf16hi(bf[k2][1][1]));
          }
#pragma unroll
          for (int k2 = 0; k2 < KH; ++k2) {
            const int ks = h + k2;
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
              if (u >= np) break;
              const uint8_t* tile = stage + static_cast<size_t>(u) * tb;
              uint32_t a[4];
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {  // rows g8 and g8 + 8
                const int r = g8 + 8 * hf;
                if (INT8) {
                  const uint32_t off = r * KCB + ((ks ^ (r & 7)) << 4) + 4 * t4;
                  i8x4_to_bf16x4(*reinterpret_cast<const uint32_t*>(tile + off), a[hf], a[2 + hf]);
                } else {
                  const int ch = 2 * ks + (t4 >> 1);
                  const uint32_t off = r * KCB + ((ch ^ (r & 7)) << 4) + 8 * (t4 & 1);
                  const uint2 w = *reinterpret_cast<const uint2*>(tile + off);
                  a[hf] = w.x;
                  a[2 + hf] = w.y;
                }
              }
#pragma unroll
              for (int pt = 0; pt < kParts; ++pt) mma_bf16(ts[u][pt], a, bf[k2][pt][0], bf[k2][pt][1]);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UPW; ++u)
#pragma unroll
          for (int pt = 0; pt < kParts; ++pt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][pt][e] += ts[u][pt][e];
      }
      // the warp is done with the stage and the activation slot
      __syncwarp();
      if (lane == 0 && !bad) mbar_arrive(&empty[slot]);
      if (++slot == RC) {
        slot = 0;
        phase ^= 1;
      }
      if (!bad && s + 2 < S) fetch_x((n + 2) % ng, s & 1);
    }

    // the end of the pass: the warps' partial sums meet and finish, in warp order
    if (bar_or(kBarAll, nthreads, bad)) {
      bad = true;
      break;
    }
#pragma unroll
    for (int u = 0; u < UPW; ++u) {
      if (u >= np) break;
      float* dst = part + (warp * PU + u) * 16 * kCols;
#pragma unroll
      for (int pt = 0; pt < kParts; ++pt) {
        const int col = 8 * pt + 2 * t4;
        dst[g8 * kCols + col] = acc[u][pt][0];
        dst[g8 * kCols + col + 1] = acc[u][pt][1];
        dst[(g8 + 8) * kCols + col] = acc[u][pt][2];
        dst[(g8 + 8) * kCols + col + 1] = acc[u][pt][3];
        acc[u][pt][0] = acc[u][pt][1] = acc[u][pt][2] = acc[u][pt][3] = 0.f;
      }
    }
    named_bar_sync(kBarAll, nthreads);
    for (int it = tid; it < np * (16 / per) * B; it += nthreads) {
      const int b = it % B, rest = it / B;
      const int rl = (rest % (16 / per)) * per, j = rest / (16 / per);
      const int r = (u0 + j0 + j) * 16 + rl;  // packed row
      if (r >= p.rows) continue;              // padding rows of the last unit
      float y[2] = {0.f, 0.f};
      for (int w = 0; w < NW; ++w)
#pragma unroll
        for (int k = 0; k < per; ++k) {
          const float* c3 = part + ((w * PU + j) * 16 + rl + k) * kCols + b;  // hi, mid and lo of sequence b
          y[k] += (c3[0] + c3[8]) + c3[16];
        }
      finish(r, b, y[0], y[1]);
    }
    if (pass + 1 < npass) named_bar_sync(kBarAll, nthreads);  // the scratch is written again next pass
  }
  if (bad) cp_async_wait_all();  // this thread's activation copies land before it leaves
  trace_end(p.trace);
}


template <bool INT8, bool NORM, int EPI, int UPW, int KCB>
cudaError_t launch_t(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t s, bool pdl) {
  auto kern = skinny_kernel<INT8, NORM, EPI, UPW, KCB>;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(kern, plan.smem, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3((kWarps + 1) * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool INT8, bool NORM, int EPI, int KCB>
cudaError_t launch_k(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t s, bool pdl) {
  switch (plan.pu) {
    case 1: return launch_t<INT8, NORM, EPI, 1, KCB>(p, plan, s, pdl);
    case 2: return launch_t<INT8, NORM, EPI, 2, KCB>(p, plan, s, pdl);
    case 3: return launch_t<INT8, NORM, EPI, 3, KCB>(p, plan, s, pdl);
    case 4: return launch_t<INT8, NORM, EPI, 4, KCB>(p, plan, s, pdl);
  }
  return cudaErrorInvalidValue;
}

template <bool INT8, bool NORM, int EPI>
cudaError_t launch_e(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t s, bool pdl) {
  const int kcb = plan.kc * (INT8 ? 1 : 2);
  if (kcb == 128) return launch_k<INT8, NORM, EPI, 128>(p, plan, s, pdl);
  if (kcb == 256) return launch_k<INT8, NORM, EPI, 256>(p, plan, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace


// Fill the derived fields of a plan whose grid, units, kc, pu and rc are set;
// false if it does not fit.
bool skinny_plan_finish(SkinnyPlan& g, int K, bool int8, int batch, int max_smem) {
  const int eb = int8 ? 1 : 2;
  if ((g.kc * eb != 128 && g.kc * eb != 256) || g.pu <= 0 || g.pu > kMaxPu || g.rc < 1) return false;
  if (batch < 1 || batch > kMaxBatch) return false;
  g.kp = (K + g.kc - 1) / g.kc * g.kc;
  g.kw = kWarps;
  g.upw = g.pu;
  g.smem = layout(g.rc, g.pu, g.kc, eb, batch).total;
  return g.smem <= max_smem;
}

// The grid: one CTA per SM (fewer when there are fewer units). Passes: the
// fewest with at most 4 units each (fewer if nothing fits), the units spread
// evenly. Then the wider k-chunk (tile rows of 256 or 128 bytes, at most K/8
// columns of padding) whose rings of two chunks fit; three where they fit.
SkinnyPlan skinny_plan(int rows, int K, bool int8, int batch, int num_sms, int max_smem) {
  SkinnyPlan g{};
  const int eb = int8 ? 1 : 2;
  if (batch < 1 || batch > kMaxBatch || K <= 0 || rows <= 0) return g;
  g.units = (rows + 15) / 16;
  g.rows_p = g.units * 16;
  g.grid = g.units < num_sms ? g.units : num_sms;
  const int per_cta = (g.units + g.grid - 1) / g.grid;
  for (int cap = kMaxPu; cap >= 1; --cap) {  // fewer units per pass where the buffers do not fit
    const int npass = (per_cta + cap - 1) / cap;
    g.pu = (per_cta + npass - 1) / npass;
    for (int c : {256 / eb, 128 / eb}) {  // tile rows of 256 or 128 bytes
      if ((((K + c - 1) / c) * c - K) * 8 > K) continue;
      SkinnyPlan t = g;
      t.kc = c;
      t.rc = 2;
      if (!skinny_plan_finish(t, K, int8, batch, max_smem)) continue;
      SkinnyPlan t3 = t;
      t3.rc = 3;
      return skinny_plan_finish(t3, K, int8, batch, max_smem) ? t3 : t;
    }
  }
  return SkinnyPlan{};
}

bool skinny_supported(int rows, int K, bool int8, int batch, int num_sms, int max_smem) {
  if (rows % 2 || K % 16 || batch < 2 || batch > kMaxBatch) return false;
  const SkinnyPlan g = skinny_plan(rows, K, int8, batch, num_sms, max_smem);
  return g.kc > 0 && g.smem <= max_smem;
}

cudaError_t launch_skinny(const SkinnyParams& p, int epi, bool norm, bool int8, const SkinnyPlan& plan, cudaStream_t s,
                          bool pdl) {
  SkinnyParams q = p;
  q.kw = plan.kw;
  q.rc = plan.rc;
  q.pu = plan.pu;
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

// Byte offset of element (row r, column k) of a [rows][K] matrix in the tiled
// layout: 16-row units split over `grid` CTAs in contiguous ranges
// [units*g/grid, units*(g+1)/grid); tiles of 16 rows x kc columns ordered
// [CTA range][k-chunk][unit of the range]; the 16-byte chunks of each tile row
// XOR-swizzled by (row mod 8). kp is K padded to whole k-chunks.
__host__ __device__ size_t skinny_offset(int r, int k, int kp, int kc, int units, int grid, int eb) {
  const int u = r / 16, rr = r - u * 16;
  // the CTA whose range holds unit u: the largest g with units*g/grid <= u
  int g = static_cast<int>((static_cast<long long>(u) * grid + grid - 1) / units);
  if (g >= grid) g = grid - 1;
  while (g > 0 && static_cast<long long>(units) * g / grid > u) --g;
  while (g + 1 < grid && static_cast<long long>(units) * (g + 1) / grid <= u) ++g;
  const int ub = static_cast<int>(static_cast<long long>(units) * g / grid);
  const int nu = static_cast<int>(static_cast<long long>(units) * (g + 1) / grid) - ub;
  const int c = k / kc, kk = k - c * kc;
  const size_t tile = static_cast<size_t>(kc) * eb * 16;
  const int byte = kk * eb;
  const int ch = byte >> 4, in = byte & 15;
  return (static_cast<size_t>(ub) * (kp / kc) + static_cast<size_t>(c) * nu + (u - ub)) * tile +
         static_cast<size_t>(rr) * kc * eb + (((ch ^ (rr & 7)) << 4) | in);
}

namespace {
__global__ void retile_kernel(const uint4* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K, int kp,
                              int kc, int units, int grid, int eb) {
  const int cpr = K * eb / 16;  // 16-byte chunks per source row
  const long long n = static_cast<long long>(rows) * cpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / cpr), ch = static_cast<int>(i - static_cast<long long>(r) * cpr);
    *reinterpret_cast<uint4*>(dst + skinny_offset(r, ch * 16 / eb, kp, kc, units, grid, eb)) = src[i];
  }
}
}  // namespace

cudaError_t launch_retile(const void* src, void* dst, int rows, int K, const SkinnyPlan& plan, int eb,
                          cudaStream_t s) {
  retile_kernel<<<1024, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint8_t*>(dst), rows, K, plan.kp,
                                     plan.kc, plan.units, plan.grid, eb);
  return cudaGetLastError();
}

}  // namespace lps
