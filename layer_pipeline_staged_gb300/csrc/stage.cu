// Persistent stage kernel: one launch runs every layer a stage owns for one
// decode step of one sequence (batch 1), and the final norm + LM head on the
// last stage. Decode is weight-bandwidth bound (ninfer pipeline-stages.md,
// "What it is and is not"); a chain of one kernel per projection spends a
// fixed few microseconds at every kernel boundary (the dependency wait, the
// input fetch, the copy ramp), during which HBM idles. Here the whole stage is
// one byte stream that never stops at a phase boundary:
//
//   - one CTA per SM (a cooperative launch, so all CTAs are resident and may
//     wait for one another) with NW consumer warps and one producer lane;
//   - the producer lane walks the stage's phases in order -- for every layer
//     QKV rows, the K/V sub-tiles of its attention work item, o-proj rows,
//     gate/up row pairs, down rows; then the LM head -- and copies them into a
//     ring of NW shared-memory slots of 32 KB, one slot per consumer warp:
//     weights by 1D bulk copies (L2 evict-first), K/V sub-tiles by 2D TMA with
//     the 128-byte swizzle. Buffer j of a phase goes to warp j mod NW, so the
//     assignment of work to warps depends only on the phase, never on the
//     stage plan. Weights never depend on earlier phases, so the producer runs
//     ahead across phase boundaries and grid barriers, bounded only by the
//     ring; the one copy that must wait is the K/V sub-tile holding the row
//     this step's QKV phase writes, issued once that phase's grid barrier has
//     passed;
//   - the consumers run a phase, then meet every other CTA at a grid-wide
//     barrier (a release add and an acquire poll on a per-stage 64-bit
//     counter, bounded), then read the phase's outputs from L2 as the next
//     phase's input vector;
//   - phases per layer: QKV (RMSNorm + GEMV + RoPE + KV append), attention
//     (CTA = one chunk of positions of one kv head; per-warp online softmax on
//     tensor cores; the warps merged in order into the chunk's partial), merge
//     (every output element of o combined from the chunk partials in chunk
//     order, spread over all CTAs), o-proj + residual, RMSNorm + gate/up +
//     SwiGLU, down + residual. Stage 0 starts with the embedding row, the last
//     stage ends with RMSNorm + LM head.
//
// Every reduction has a fixed order that depends on the shapes, the position
// and the SM count only (GEMV rows: lane chunks ascending then a warp xor
// tree; RMSNorm: 256 fixed partial sums; attention: sub-tile j on warp
// j mod NW, warps merged in order, chunks merged in order), so every stage
// plan gives the same bits.
//
// Failure handling: every wait is bounded (mbarrier phases, ring slots, grid
// barriers); a consumer that gives up records an error, all consumer warps of
// the CTA leave together at the next CTA-wide point, the other CTAs give up at
// their next grid barrier, and the producer waits for the copies it issued to
// land before its CTA may end. No trap, no unbounded spin.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kSlot = 16 * 1024;   // one ring slot: a weight buffer, or a K + V sub-tile
constexpr int kMaxCW = 8;          // consumer warps
constexpr int kMaxSlots = 24;      // ring slots (consumer warps x depth)
constexpr int kMaxRows = 8;        // weight rows per buffer
constexpr int kMaxSegUnits = 512;  // units per CTA of a phase whose rows are cut into K-segments
constexpr int kXsCapFloats = 8192; // the input-vector area holds at most this many floats
constexpr int kNormParts = 256;    // fixed partial sums of the RMSNorm mean square
constexpr int kMaxG = 8;           // q heads per kv head

enum Phase : int { kPhEmbed = 0, kPhQkv, kPhAttn, kPhMerge, kPhOproj, kPhGateup, kPhDown, kPhHead };
constexpr int kLayerPhases = 6;

// ---- small PTX helpers -------------------------------------------------------

__device__ __forceinline__ void red_release_add(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Poll a grid-barrier counter until it reaches `target`; false after `limit` cycles.
__device__ __forceinline__ bool wait_counter(const unsigned long long* p, unsigned long long target, long long limit) {
  if (ld_acquire(p) >= target) return true;
  const long long t0 = cycles();
  while (ld_acquire(p) < target) {
    if (cycles() - t0 > limit) return false;
  }
  return true;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Named barrier over the consumer warps that also ORs `bad` across them.
__device__ __forceinline__ bool consumers_or(int nthreads, bool bad) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(bad)), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// c += A.B for one 16-wide k-step from a zero accumulator, then a
// round-to-nearest fp32 add (long sums do not pile up the tensor core's truncation).
__device__ __forceinline__ void mma_add(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  float d0, d1, d2, d3;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
  c[0] += d0;
  c[1] += d1;
  c[2] += d2;
  c[3] += d3;
}
// c += A.B accumulated on the tensor core (a score's HD/16 k-steps).
__device__ __forceinline__ void mma_acc(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// x as bf16 hi (lo = 0) or the remainder x - hi rounded to bf16 (lo = 1).
__device__ __forceinline__ float split_part(float x, int lo) {
  const float hi = __bfloat162float(__float2bfloat16_rn(x));
  return lo ? x - hi : hi;
}
// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float dot_i8x4(uint32_t w, const float4 a, float acc) {
  float q0, q1, q2, q3;
  i8x4_to_f32(w, q0, q1, q2, q3);
  acc = fmaf(q0, a.x, acc);
  acc = fmaf(q1, a.y, acc);
  acc = fmaf(q2, a.z, acc);
  acc = fmaf(q3, a.w, acc);
  return acc;
}

// ---- the phase walk -----------------------------------------------------------

__device__ __forceinline__ int n_phases(const StageParams& p) {
  return (p.embed ? 1 : 0) + kLayerPhases * p.n_layers + (p.head ? 1 : 0);
}
// Phase `idx` of the launch: its kind and the layer (index into p.layers).
__device__ __forceinline__ void phase_at(const StageParams& p, int idx, int* kind, int* layer) {
  if (p.embed) {
    if (idx == 0) {
      *kind = kPhEmbed;
      *layer = 0;
      return;
    }
    --idx;
  }
  *layer = idx / kLayerPhases;
  *kind = *layer < p.n_layers ? 1 + idx % kLayerPhases : kPhHead;
}

// A weight-streaming phase: this CTA's units [u0, u0 + nunits) of a packed
// matrix. Units are taken `ups` at a time (a row group); an input row longer
// than the input-vector area is cut into nseg K-segments of kseg elements, and
// the phase runs segment by segment (the vector area holds one segment). Ring
// buffer (segment s, group q) holds the group's rows restricted to segment s;
// group q belongs to warp q mod NW in every segment.
struct Gv {
  const uint8_t* w;
  const float* ws;
  int K, unit_rows, u0, nunits, ups, ngroups, nseg, kseg;
  uint32_t row_bytes, unit_bytes;
};
template <bool INT8>
__device__ __forceinline__ Gv gv_of(const StageParams& p, const StageLayer* L, int kind) {
  constexpr int EB = INT8 ? 1 : 2;
  constexpr int EPC = 16 / EB;  // elements per 16-byte chunk
  Gv g{};
  int rows = 0;
  const int qw = p.nq * p.hd;
  switch (kind) {
    case kPhQkv: g.w = static_cast<const uint8_t*>(L->w_qkv); g.ws = L->s_qkv; rows = (p.nq + 2 * p.nkv) * p.hd;
      g.K = p.d; g.unit_rows = 2; break;
    case kPhOproj: g.w = static_cast<const uint8_t*>(L->w_o); g.ws = L->s_o; rows = p.d; g.K = qw; g.unit_rows = 1;
      break;
    case kPhGateup: g.w = static_cast<const uint8_t*>(L->w_gu); g.ws = L->s_gu; rows = 2 * p.ffn; g.K = p.d;
      g.unit_rows = 2; break;
    case kPhDown: g.w = static_cast<const uint8_t*>(L->w_d); g.ws = L->s_d; rows = p.d; g.K = p.ffn; g.unit_rows = 1;
      break;
    default: g.w = static_cast<const uint8_t*>(p.head); g.ws = p.head_s; rows = p.vocab; g.K = p.d; g.unit_rows = 1;
      break;
  }
  const int units = rows / g.unit_rows;
  const int G = gridDim.x, c = blockIdx.x;
  g.u0 = static_cast<int>(static_cast<long long>(units) * c / G);
  g.nunits = static_cast<int>(static_cast<long long>(units) * (c + 1) / G) - g.u0;
  g.row_bytes = static_cast<uint32_t>(g.K) * EB;
  g.unit_bytes = g.row_bytes * g.unit_rows;
  g.nseg = (g.K + p.seg_cap - 1) / p.seg_cap;
  g.kseg = ((g.K + g.nseg - 1) / g.nseg + EPC - 1) / EPC * EPC;  // whole chunks
  // rows per buffer: a power of two, at most kMaxRows, within one slot
  int rmax = kSlot / (g.unit_rows * g.kseg * EB) * g.unit_rows;
  rmax = rmax > kMaxRows ? kMaxRows : rmax;
  int r = 1;
  while (2 * r <= rmax) r *= 2;
  g.ups = r / g.unit_rows > 0 ? r / g.unit_rows : 1;
  g.ngroups = (g.nunits + g.ups - 1) / g.ups;
  return g;
}
// Elements of segment s (the last one may be shorter).
__device__ __forceinline__ int seg_len(const Gv& g, int s) { return min(g.kseg, g.K - s * g.kseg); }

// The attention work item of this CTA: chunk `c` of kv head `g`, positions
// [t0, t_end), in sub-tiles of TS positions.
struct At {
  int g, c, t0, t_end, nsub;
};
template <int HD>
__device__ __forceinline__ At at_of(const StageParams& p) {
  constexpr int TS = 4096 / HD;
  At a{};
  const int item = blockIdx.x;
  if (item >= p.nkv * p.nch) return a;  // nsub = 0: no item
  a.g = item / p.nch;
  a.c = item - a.g * p.nch;
  a.t0 = a.c * p.chunk;
  a.t_end = min(a.t0 + p.chunk, p.pos + 1);
  a.nsub = a.t_end > a.t0 ? (a.t_end - a.t0 + TS - 1) / TS : 0;
  return a;
}

// R rows of a ring buffer (row stride rstride bytes) against the input
// vector's float4 planes, over the nch chunks of the segment: per row, NA
// independent accumulator chains (lane chunks ascending), added in order.
template <bool INT8, int R>
__device__ __forceinline__ void dot_rows(const uint8_t* buf, uint32_t rstride, const float4* xs4, int nch, int lane,
                                         float* out) {
  constexpr int NP = INT8 ? 4 : 2;
  constexpr int NA = R >= 4 ? 2 : 4;
  float acc[R][NA];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int a = 0; a < NA; ++a) acc[r][a] = 0.f;
#pragma unroll 2
  for (int c = lane; c < nch; c += 32) {
    float4 xv[NP];
#pragma unroll
    for (int pl = 0; pl < NP; ++pl) xv[pl] = xs4[pl * nch + c];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint4 w = *reinterpret_cast<const uint4*>(buf + r * rstride + c * 16);
      const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float& a = acc[r][k % NA];
        if (INT8) {
          a = dot_i8x4(wd[k], xv[k], a);
        } else {
          const float4& xx = xv[k >> 1];
          if (k & 1) {
            a = fmaf(bf16lo(wd[k]), xx.z, a);
            a = fmaf(bf16hi(wd[k]), xx.w, a);
          } else {
            a = fmaf(bf16lo(wd[k]), xx.x, a);
            a = fmaf(bf16hi(wd[k]), xx.y, a);
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float s = acc[r][0];
#pragma unroll
    for (int a = 1; a < NA; ++a) s += acc[r][a];
    out[r] = warp_sum(s);
  }
}

// ---- the kernel ---------------------------------------------------------------

template <bool INT8, int HD>
__global__ void __maxnreg__(224) stage_kernel(const __grid_constant__ StageParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int EB = INT8 ? 1 : 2;
  constexpr int NP = INT8 ? 4 : 2;         // float4 planes of the input vector per 16-byte chunk
  constexpr int TS = 4096 / HD;            // positions per K/V sub-tile (8 KB of K, 8 KB of V)
  constexpr int PARTS = HD / 64;           // 128-byte TMA boxes per cache row
  constexpr int BOX = TS * 128;
  constexpr int TILE = PARTS * BOX;        // bytes of one K (or V) sub-tile
  static_assert(2 * TILE == kSlot, "a K + V sub-tile fills one slot");
  const int NW = p.nw, D = p.depth;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nph = n_phases(p);
  const long long limit = wait_cycles(p.wait_limit);

  uint8_t* ring = smem;  // NW * D slots: warp w owns slots [w * D, w * D + D)
  float* xs = reinterpret_cast<float*>(smem + static_cast<size_t>(NW) * D * kSlot);  // input vector / attention states
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(NW) * D * kSlot + p.xs_bytes);
  uint64_t* empty = full + kMaxSlots;
  float* sred = reinterpret_cast<float*>(empty + kMaxSlots);  // [kNormParts]
  float* sinv = sred + kNormParts;                             // the RMSNorm scale
  float* rowsum = sinv + 4;                                    // [kMaxSegUnits] segmented phases' row sums

  if (tid == 0) {
    for (int i = 0; i < NW * D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == NW) {
    // ---------------- producer ----------------
    // Lane 0 copies the stage's byte sequence into the ring.
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first();
    int use[kMaxCW];  // buffers issued to each warp
    for (int i = 0; i < kMaxCW; ++i) use[i] = 0;
    bool dep_done = false, failed = false;
    // the slot for warp w's next buffer, once the buffer it held D uses ago is released
    auto acquire = [&](int w, int* slot) -> bool {
      const int n = use[w];
      *slot = w * D + n % D;
      if (n < D) return true;
      const uint32_t par = ((n / D) - 1) & 1;
      if (mbar_test(&empty[*slot], par)) return true;
      const long long t0 = cycles();
      while (!mbar_test(&empty[*slot], par)) {
        if (cycles() - t0 > limit) return false;
        __nanosleep(32);
      }
      return true;
    };
    for (int ph = 0; ph < nph && !failed; ++ph) {
      int kind, li;
      phase_at(p, ph, &kind, &li);
      const StageLayer* L = p.layers + (li < p.n_layers ? li : 0);
      if (kind == kPhEmbed || kind == kPhMerge) continue;
      if (kind == kPhAttn) {
        const At a = at_of<HD>(p);
        for (int j = 0; j < a.nsub; ++j) {
          const int r0 = a.t0 + j * TS;
          const int y = a.g * p.max_ctx + r0;
          // cache rows before pos were written by earlier launches: visible once
          // the previous kernel in the stream has completed
          if (!dep_done) {
            pdl_wait();
            dep_done = true;
          }
          const int w = j % NW;
          int slot;
          if (!acquire(w, &slot)) {
            report_error(p.status, kErrWaitEmpty | (kKidStage << 8) | (ph << 13));
            failed = true;
            break;
          }
          if (r0 + TS > p.pos) {
            // this sub-tile holds row pos, written by this layer's QKV phase
            // (phase ph - 1): copy it once that phase's grid barrier has passed
            if (!wait_counter(p.bar, p.bar_base + static_cast<unsigned long long>(ph) * G, limit)) {
              report_error(p.status, kErrBarrier | (kKidStage << 8) | (ph << 13));
              failed = true;
              break;
            }
            fence_proxy_async();
          }
          uint8_t* dst = ring + static_cast<size_t>(slot) * kSlot;
          mbar_arrive_expect_tx(&full[slot], kSlot);
#pragma unroll
          for (int part = 0; part < PARTS; ++part) {
            tma_load_2d(dst + part * BOX, &L->tmap_k, part * 64, y, &full[slot]);
            tma_load_2d(dst + TILE + part * BOX, &L->tmap_v, part * 64, y, &full[slot]);
          }
          ++use[w];
        }
        continue;
      }
      const Gv g = gv_of<INT8>(p, L, kind);
      for (int sg = 0; sg < g.nseg && !failed; ++sg) {
        const uint32_t sbytes = static_cast<uint32_t>(seg_len(g, sg)) * EB;
        const size_t soff = static_cast<size_t>(sg) * g.kseg * EB;
        for (int q = 0; q < g.ngroups; ++q) {
          const int nu = min(g.ups, g.nunits - q * g.ups);
          const int nrows = nu * g.unit_rows;
          const uint8_t* src = g.w + static_cast<size_t>(g.u0 + q * g.ups) * g.unit_bytes;
          const int w = q % NW;
          int slot;
          if (!acquire(w, &slot)) {
            report_error(p.status, kErrWaitEmpty | (kKidStage << 8) | (ph << 13));
            failed = true;
            break;
          }
          uint8_t* dst = ring + static_cast<size_t>(slot) * kSlot;
          mbar_arrive_expect_tx(&full[slot], sbytes * nrows);
          if (g.nseg == 1) {
            bulk_g2s(dst, src, sbytes * nrows, &full[slot], pol);  // whole rows: one contiguous range
          } else {
            for (int r = 0; r < nrows; ++r)
              bulk_g2s(dst + r * sbytes, src + static_cast<size_t>(r) * g.row_bytes + soff, sbytes, &full[slot], pol);
          }
          ++use[w];
        }
      }
    }
    // the last copy issued into each slot lands before the CTA may end (the
    // consumers may have left early after an error)
    for (int w = 0; w < NW; ++w)
      for (int n = max(0, use[w] - D); n < use[w]; ++n)
        if (!mbar_wait(&full[w * D + n % D], (n / D) & 1, kDrainLimitCycles)) {
          report_error(p.status, kErrDrain | (kKidStage << 8));
          w = NW;
          break;
        }
    return;
  }

  // ---------------- consumers ----------------
  const int nthreads = NW * 32;
  int uses = 0;        // buffers this warp has taken from its slots
  bool bad = false;    // a bounded wait gave up: leave with the other warps at the next sync
  // wait for this warp's next buffer; returns its slot, or -1 after a timeout
  auto take = [&](int ph) -> int {
    const int slot = warp * D + uses % D;
    if (!mbar_wait(&full[slot], (uses / D) & 1, limit)) {
      if (lane == 0) report_error(p.status, kErrWaitFull | (kKidStage << 8) | (ph << 13));
      return -1;
    }
    return slot;
  };
  auto give = [&](int slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    ++uses;
  };
  pdl_wait();  // the previous kernel's outputs (the boundary slot, the cache rows) are visible

  for (int ph = 0; ph < nph; ++ph) {
    int kind, li;
    phase_at(p, ph, &kind, &li);
    const StageLayer* L = p.layers + (li < p.n_layers ? li : 0);
    unsigned long long* trec = p.trace ? p.trace + 2 * ph : nullptr;
    if (trec && tid == 0) atomicMax(trec, ~global_ns());
    const bool first_layer = li == 0;
    const bool last_layer = li == p.n_layers - 1;

    if (kind == kPhEmbed) {
      // h = E[token]: this CTA's slice of the row
      const int tok = p.tok_dev ? __ldcg(p.tok_dev) : p.tok;
      if (tok < 0 || tok >= p.vocab) {
        if (tid == 0) report_error(p.status, kErrBadArg | (kKidEmbed << 8));
        bad = true;
      } else {
        const int per = (p.d / 4 + G - 1) / G;
        for (int i4 = cta * per + tid; i4 < min(p.d / 4, (cta + 1) * per); i4 += nthreads) {
          float4 v;
          if (INT8) {
            const char4 q = reinterpret_cast<const char4*>(static_cast<const int8_t*>(p.embed) +
                                                           static_cast<size_t>(tok) * p.d)[i4];
            const float s = p.embed_s[tok];
            v = make_float4(q.x * s, q.y * s, q.z * s, q.w * s);
          } else {
            const uint2 w2 = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.embed) +
                                                            static_cast<size_t>(tok) * p.d)[i4];
            v = make_float4(bf16lo(w2.x), bf16hi(w2.x), bf16lo(w2.y), bf16hi(w2.y));
          }
          reinterpret_cast<float4*>(p.h)[i4] = v;
        }
      }
    } else if (kind == kPhAttn) {
      // ---- attention over this CTA's chunk: sub-tile j on warp j mod NW ----
      const At a = at_of<HD>(p);
      const int Gq = p.nq / p.nkv;
      const int g8 = lane >> 2, t4 = lane & 3;
      float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
      float o_acc[HD / 8][4];
#pragma unroll
      for (int j = 0; j < HD / 8; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
      if (warp < a.nsub && !bad) {
        // q of the group as the A operand: row 2h = bf16(q_h), row 2h+1 = bf16(q_h - bf16(q_h))
        uint32_t qa[HD / 16][4];
        {
          const float* qb = p.q + a.g * Gq * HD;
          const int h0 = g8 >> 1, h1 = (g8 + 8) >> 1, lo = g8 & 1;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const int d0 = 16 * kk + 2 * t4;
            float v[8];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              v[e] = h0 < Gq ? split_part(__ldcg(qb + h0 * HD + d0 + e), lo) : 0.f;
              v[2 + e] = h1 < Gq ? split_part(__ldcg(qb + h1 * HD + d0 + e), lo) : 0.f;
              v[4 + e] = h0 < Gq ? split_part(__ldcg(qb + h0 * HD + d0 + 8 + e), lo) : 0.f;
              v[6 + e] = h1 < Gq ? split_part(__ldcg(qb + h1 * HD + d0 + 8 + e), lo) : 0.f;
            }
            qa[kk][0] = pack_bf16(v[0], v[1]);
            qa[kk][1] = pack_bf16(v[2], v[3]);
            qa[kk][2] = pack_bf16(v[4], v[5]);
            qa[kk][3] = pack_bf16(v[6], v[7]);
          }
        }
        for (int j = warp; j < a.nsub; j += NW) {
          const int slot = take(ph);
          if (slot < 0) {
            bad = true;
            break;
          }
          const int rows = min(TS, a.t_end - (a.t0 + j * TS));
          const uint32_t kbase = smem_u32(ring + static_cast<size_t>(slot) * kSlot), vbase = kbase + TILE;
          // 32 positions at a time: scores, online softmax, P.V
          for (int wp0 = 0; wp0 < rows; wp0 += 32) {
            float sc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const int part = kk / 4, ch = 2 * (kk % 4);
#pragma unroll
              for (int nt = 0; nt < 4; nt += 2) {
                const int mtx = lane >> 3;
                const int r = wp0 + 8 * (nt + (mtx >> 1)) + (lane & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + part * BOX + swz(r, ch + (mtx & 1)), b0, b1, b2, b3);
                mma_acc(sc[nt], qa[kk], b0, b1);
                mma_acc(sc[nt + 1], qa[kk], b2, b3);
              }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float s = (sc[nt][e] + __shfl_xor_sync(0xffffffffu, sc[nt][e], 4)) * p.scale;
                const int pp = wp0 + 8 * nt + 2 * t4 + (e & 1);
                sc[nt][e] = pp < rows ? s : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
              }
            }
            float alpha[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
              mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
              const float m_new = fmaxf(m_r[rr], mx[rr]);
              alpha[rr] = (m_new == -INFINITY) ? 1.f : expf(m_r[rr] - m_new);
              m_r[rr] = m_new;
            }
            float ls[2] = {0.f, 0.f};
            uint32_t pa[2][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              float pr[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int rr = e >> 1;
                const float pv = (m_r[rr] == -INFINITY) ? 0.f : expf(sc[nt][e] - m_r[rr]);
                ls[rr] += pv;
                pr[e] = split_part(pv, g8 & 1);
              }
              const int ks = nt >> 1, hi8 = nt & 1;
              pa[ks][hi8 ? 2 : 0] = pack_bf16(pr[0], pr[1]);
              pa[ks][hi8 ? 3 : 1] = pack_bf16(pr[2], pr[3]);
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              ls[rr] += __shfl_xor_sync(0xffffffffu, ls[rr], 1);
              ls[rr] += __shfl_xor_sync(0xffffffffu, ls[rr], 2);
              l_r[rr] = l_r[rr] * alpha[rr] + ls[rr];
            }
#pragma unroll
            for (int jd = 0; jd < HD / 8; ++jd) {
              o_acc[jd][0] *= alpha[0];
              o_acc[jd][1] *= alpha[0];
              o_acc[jd][2] *= alpha[1];
              o_acc[jd][3] *= alpha[1];
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
              for (int jd = 0; jd < HD / 8; jd += 2) {
                const int mtx = lane >> 3;
                const int r = wp0 + 16 * ks + 8 * (mtx & 1) + (lane & 7);
                const int dch = jd + (mtx >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + (dch / 8) * BOX + swz(r, dch % 8), b0, b1, b2, b3);
                mma_add(o_acc[jd], pa[ks], b0, b1);
                mma_add(o_acc[jd + 1], pa[ks], b2, b3);
              }
            }
          }
          give(slot);
        }
      }
      // every warp's (m, l, o) per head into shared memory (the input-vector
      // area is free during attention); rows 2h (hi) and 2h+1 (lo) of o add up
      float* so = xs;                                       // [NW][Gq][HD]
      float* sm_ = xs + static_cast<size_t>(NW) * Gq * HD;  // [NW][Gq]
      float* sl = sm_ + NW * Gq;                            // [NW][Gq]
      if (a.nsub > 0) {
        const int lo = g8 & 1;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int h = (g8 + 8 * rr) >> 1;
#pragma unroll
          for (int jd = 0; jd < HD / 8; ++jd) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float v = o_acc[jd][2 * rr + e];
              const float sum = v + __shfl_xor_sync(0xffffffffu, v, 4);
              if (!lo && h < Gq) so[(warp * Gq + h) * HD + 8 * jd + 2 * t4 + e] = sum;
            }
          }
          if (!lo && t4 == 0 && h < Gq) {
            sm_[warp * Gq + h] = m_r[rr];
            sl[warp * Gq + h] = l_r[rr];
          }
        }
      }
      bad = consumers_or(nthreads, bad);
      if (!bad && a.nsub > 0) {
        // merge the warps in order into this chunk's partial: rows of HD + 4
        // floats (acc, m, l, pad)
        for (int o = tid; o < Gq * HD; o += nthreads) {
          const int hh = o / HD, i = o - hh * HD;
          float M = -INFINITY;
          for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_[w * Gq + hh]);
          float Lw = 0.f, O = 0.f;
          for (int w = 0; w < NW; ++w) {
            const float mw = sm_[w * Gq + hh];
            const float wt = (mw == -INFINITY) ? 0.f : expf(mw - M);
            Lw = fmaf(sl[w * Gq + hh], wt, Lw);
            O = fmaf(so[(w * Gq + hh) * HD + i], wt, O);
          }
          float* dst = p.part + (static_cast<size_t>(a.g * Gq + hh) * p.nch_max + a.c) * (HD + 4);
          dst[i] = O;
          if (i == 0) {
            dst[HD] = M;
            dst[HD + 1] = Lw;
          }
        }
      }
    } else if (kind == kPhMerge) {
      // ---- o[h][i] from the chunk partials, in chunk order; item k = (head,
      // 32 dims) runs on CTA k mod G, warp k / G ----
      const int per_head = HD / 32;
      const int items = p.nq * per_head;
      const int k = warp * G + cta;
      if (k < items && !bad) {
        const int h = k / per_head, i = (k - h * per_head) * 32 + lane;
        const float* base = p.part + static_cast<size_t>(h) * p.nch_max * (HD + 4);
        float M = -INFINITY;
        for (int c = 0; c < p.nch; ++c) M = fmaxf(M, __ldcg(base + c * (HD + 4) + HD));
        float Lw = 0.f, O = 0.f;
        for (int c = 0; c < p.nch; ++c) {
          const float* pc = base + c * (HD + 4);
          const float wt = expf(__ldcg(pc + HD) - M);
          Lw = fmaf(__ldcg(pc + HD + 1), wt, Lw);
          O = fmaf(__ldcg(pc + i), wt, O);
        }
        L->o_out[h * HD + i] = O / Lw;
      }
    } else {
      // ---- weight-streaming phases ----
      const Gv g = gv_of<INT8>(p, L, kind);
      const bool norm = kind == kPhQkv || kind == kPhGateup || kind == kPhHead;
      // input vector: h (normalised), o, or a
      const float* src = kind == kPhOproj ? L->o_out
                         : kind == kPhDown ? p.a
                         : (kind == kPhQkv && first_layer && p.h_in) ? p.h_in
                                                                      : p.h;
      const float* gain = kind == kPhQkv ? L->attn_norm : kind == kPhGateup ? L->ffn_norm : p.out_norm;
      const int half = p.hd >> 1;
      float* h_out = (kind == kPhDown && last_layer) ? p.h_out : p.h;
      const float* h_res = (kind == kPhOproj && first_layer && p.h_in) ? p.h_in : p.h;
      float4* xs4 = reinterpret_cast<float4*>(xs);
      for (int sg = 0; sg < g.nseg; ++sg) {
        const int K4 = seg_len(g, sg) / 4;
        const int nch = K4 * 4 * EB / 16;  // 16-byte chunks of a row segment
        const float4* src4 = reinterpret_cast<const float4*>(src + static_cast<size_t>(sg) * g.kseg);
        if (sg > 0) named_bar_sync(1, nthreads);  // every warp is done with the previous segment
        // the segment into the float4 planes, every copy of a thread in flight at once
        for (int k4 = tid; k4 < K4; k4 += nthreads) cp_async16(&xs4[(k4 % NP) * nch + k4 / NP], src4 + k4, 16);
        cp_async_commit();
        cp_async_wait_all();
        named_bar_sync(1, nthreads);
        if (norm) {
          // (norm phases have one segment) the mean square as kNormParts fixed
          // partial sums (part j: every k4 = j mod kNormParts, ascending), then a fixed tree
          for (int j = tid; j < kNormParts; j += nthreads) {
            float ss = 0.f;
            for (int k4 = j; k4 < K4; k4 += kNormParts) {
              const float4 v = xs4[(k4 % NP) * nch + k4 / NP];
              ss = fmaf(v.x, v.x, ss);
              ss = fmaf(v.y, v.y, ss);
              ss = fmaf(v.z, v.z, ss);
              ss = fmaf(v.w, v.w, ss);
            }
            sred[j] = ss;
          }
          named_bar_sync(1, nthreads);
          if (warp == 0) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < kNormParts / 32; ++i) s += sred[lane + 32 * i];
            s = warp_sum(s);
            if (lane == 0) sinv[0] = 1.0f / sqrtf(s / static_cast<float>(g.K) + p.eps);
          }
          named_bar_sync(1, nthreads);
          const float inv = sinv[0];
#pragma unroll 4
          for (int k4 = tid; k4 < K4; k4 += nthreads) {
            float4& v = xs4[(k4 % NP) * nch + k4 / NP];
            const float4 gg = __ldg(reinterpret_cast<const float4*>(gain) + k4);
            v = make_float4(v.x * inv * gg.x, v.y * inv * gg.y, v.z * inv * gg.z, v.w * inv * gg.w);
          }
          named_bar_sync(1, nthreads);
        }
        const bool last_seg = sg + 1 == g.nseg;
        for (int q = warp; q < g.ngroups && !bad; q += NW) {
          const int nu = min(g.ups, g.nunits - q * g.ups);
          const int rows = nu * g.unit_rows;
          // lane e's epilogue inputs for unit e of this group, before the wait
          float s0 = 1.f, s1 = 1.f, e0 = 0.f, e1 = 0.f;
          if (last_seg && lane < nu) {
            const int u = g.u0 + q * g.ups + lane;
            if (INT8) {
              s0 = g.ws[u * g.unit_rows];
              if (g.unit_rows == 2) s1 = g.ws[u * g.unit_rows + 1];
            }
            if (kind == kPhQkv) {
              const int hh = u / half;
              if (hh < p.nq + p.nkv) {
                const float2 cs = p.rope[static_cast<size_t>(p.pos) * half + (u - hh * half)];
                e0 = cs.x;
                e1 = cs.y;
              }
            } else if (kind == kPhOproj || kind == kPhDown) {
              e0 = __ldcg(h_res + u);
            }
          }
          const int slot = take(ph);
          if (slot < 0) {
            bad = true;
            break;
          }
          const uint8_t* buf = ring + static_cast<size_t>(slot) * kSlot;
          const uint32_t rstride = static_cast<uint32_t>(nch) * 16;
          float y[kMaxRows];
          if (rows <= 1)
            dot_rows<INT8, 1>(buf, rstride, xs4, nch, lane, y);
          else if (rows <= 2)
            dot_rows<INT8, 2>(buf, rstride, xs4, nch, lane, y);
          else if (rows <= 4)
            dot_rows<INT8, 4>(buf, rstride, xs4, nch, lane, y);
          else
            dot_rows<INT8, 8>(buf, rstride, xs4, nch, lane, y);
          give(slot);
          if (g.nseg > 1) {
            // the group's rows are this warp's alone: running sums in segment order
            const int r0 = q * g.ups * g.unit_rows;
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r)
              if (r < rows) {
                const float prev = sg > 0 ? rowsum[r0 + r] : 0.f;
                y[r] = prev + y[r];
                if (!last_seg && lane == 0) rowsum[r0 + r] = y[r];
              }
            __syncwarp();
          }
          if (!last_seg) continue;
          // epilogue: lane e finishes unit e of this group
#pragma unroll
          for (int e = 0; e < kMaxRows; ++e) {
            if (e < nu && lane == e) {
              const int u = g.u0 + q * g.ups + e;
              float y0, y1 = 0.f;
              if (g.unit_rows == 2) {
                y0 = y[(2 * e) % kMaxRows];
                y1 = y[(2 * e + 1) % kMaxRows];
              } else {
                y0 = y[e];
              }
              y0 *= s0;
              y1 *= s1;
              if (kind == kPhQkv) {
                const int hh = u / half, ii = u - hh * half;
                if (hh < p.nq) {
                  p.q[hh * p.hd + ii] = y0 * e0 - y1 * e1;
                  p.q[hh * p.hd + ii + half] = y0 * e1 + y1 * e0;
                } else if (hh < p.nq + p.nkv) {
                  const size_t base = (static_cast<size_t>(hh - p.nq) * p.max_ctx + p.pos) * p.hd;
                  L->kc[base + ii] = __float2bfloat16_rn(y0 * e0 - y1 * e1);
                  L->kc[base + ii + half] = __float2bfloat16_rn(y0 * e1 + y1 * e0);
                } else {
                  const size_t base = (static_cast<size_t>(hh - p.nq - p.nkv) * p.max_ctx + p.pos) * p.hd;
                  L->vc[base + ii] = __float2bfloat16_rn(y0);
                  L->vc[base + ii + half] = __float2bfloat16_rn(y1);
                }
              } else if (kind == kPhOproj || kind == kPhDown) {
                h_out[u] = e0 + y0;
              } else if (kind == kPhGateup) {
                p.a[u] = y0 / (1.0f + expf(-y0)) * y1;
              } else {
                p.logits[u] = y0;
              }
            }
          }
        }
      }
    }

    if (trec && tid == 0) atomicMax(trec + 1, global_ns());
    if (ph + 1 == nph) break;
    // ---- grid barrier between phases ----
    bad = consumers_or(nthreads, bad);
    if (bad) return;
    if (tid == 0) {
      red_release_add(p.bar, 1ull);
      if (!wait_counter(p.bar, p.bar_base + static_cast<unsigned long long>(ph + 1) * G, limit)) {
        report_error(p.status, kErrBarrier | (kKidStage << 8) | (ph << 13));
        bad = true;
      }
    }
    bad = consumers_or(nthreads, bad);
    if (bad) return;
  }
}

template <bool INT8, int HD>
cudaError_t launch_t(const StageParams& p, const StageKernelPlan& plan, cudaStream_t s, bool pdl) {
  auto kern = stage_kernel<INT8, HD>;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(kern, plan.smem, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3((plan.nw + 1) * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

// Ring and input-vector sizing for a model; ok = false when the shapes do not
// fit this kernel (the per-projection kernels then run the step).
//   - the input-vector area holds the longest K-segment (rows longer than
//     kXsCapFloats elements, or than one slot, are cut into segments) and, during
//     attention, every warp's (m, l, o) per head; RMSNorm inputs are never cut;
//   - the rest of the shared memory is the ring: NW consumer warps x D slots of
//     16 KB, with D >= 2 so that a warp's next buffer is in flight while it
//     works on the current one.
StageKernelPlan stage_kernel_plan(int d, int nq, int nkv, int hd, int ffn, int vocab, bool int8, int num_sms,
                                  int max_smem) {
  StageKernelPlan g{};
  const int eb = int8 ? 1 : 2;
  const int epc = 16 / eb;
  const int qw = nq * hd;
  const int group = nkv > 0 ? nq / nkv : 0;
  if ((hd != 64 && hd != 128) || nkv < 1 || nq % nkv || group < 1 || group > kMaxG || nkv > num_sms) return g;
  if (d % epc || ffn % epc || qw % epc || vocab < 1) return g;
  const int seg_cap = kXsCapFloats < kSlot / eb ? kXsCapFloats : kSlot / eb;
  // the phases: (K, unit rows, units, RMSNorm input)
  const int ks[5] = {d, qw, d, ffn, d}, urs[5] = {2, 1, 2, 1, 1};
  const int nunits[5] = {(nq + 2 * nkv) * hd / 2, d, ffn, d, vocab};
  const bool norms[5] = {true, false, true, false, true};
  int xs_floats = 0;
  for (int i = 0; i < 5; ++i) {
    const int nseg = (ks[i] + seg_cap - 1) / seg_cap;
    const int kseg = ((ks[i] + nseg - 1) / nseg + epc - 1) / epc * epc;
    if (norms[i] && nseg > 1) return g;                            // a mean square over the whole vector
    if (urs[i] * kseg * eb > kSlot) return g;                      // a unit's segment fits one slot
    if (ks[i] - (nseg - 1) * kseg <= 0) return g;                  // no empty last segment
    if (nseg > 1 && (nunits[i] + num_sms - 1) / num_sms * urs[i] > kMaxSegUnits) return g;
    xs_floats = kseg > xs_floats ? kseg : xs_floats;
  }
  const int states = kMaxCW * group * (hd + 2);  // attention: (o, m, l) per warp and head
  int xs = (xs_floats > states ? xs_floats : states) * 4;
  xs = (xs + 15) / 16 * 16;
  const int reserve = 2 * kMaxSlots * 8 + (kNormParts + 4 + kMaxSegUnits + 4) * 4;
  int slots = (max_smem - xs - reserve) / kSlot;
  slots = slots > kMaxSlots ? kMaxSlots : slots;
  int best_nw = 0, best_d = 0;
  for (int nw = kMaxCW; nw >= 3; --nw) {
    const int dd = slots / nw;
    if (dd >= 2 && nw * dd > best_nw * best_d) {
      best_nw = nw;
      best_d = dd;
    }
  }
  if (best_nw == 0) return g;
  g.nw = best_nw;
  g.depth = best_d;
  g.xs_bytes = xs;
  g.seg_cap = seg_cap;
  g.smem = best_nw * best_d * kSlot + xs + reserve;
  g.grid = num_sms;
  g.nch_max = num_sms / nkv;
  g.ok = true;
  return g;
}

int stage_sub_tile(int hd) { return 4096 / hd; }

// Chunks of the attention phase at position pos: as many as the grid allows
// per kv head (one work item per CTA), of whole sub-tiles, none empty.
void stage_attn_chunks(const StageKernelPlan& g, int hd, int nkv, int pos, int* nch, int* chunk) {
  const int ts = stage_sub_tile(hd);
  const int nsub = (pos + 1 + ts - 1) / ts;
  int n = g.nch_max < nsub ? g.nch_max : nsub;
  n = n < 1 ? 1 : n;
  const int cs = (nsub + n - 1) / n;  // sub-tiles per chunk
  *chunk = cs * ts;
  *nch = (nsub + cs - 1) / cs;
  (void)nkv;
}

int stage_barriers(const StageParams& p) {
  return (p.embed ? 1 : 0) + kLayerPhases * p.n_layers + (p.head ? 1 : 0) - 1;
}

cudaError_t launch_stage(const StageParams& p, bool int8, const StageKernelPlan& plan, cudaStream_t s, bool pdl) {
  StageParams q = p;
  q.nw = plan.nw;
  q.depth = plan.depth;
  q.xs_bytes = plan.xs_bytes;
  q.seg_cap = plan.seg_cap;
  q.nch_max = plan.nch_max;
  if (p.hd == 128) return int8 ? launch_t<true, 128>(q, plan, s, pdl) : launch_t<false, 128>(q, plan, s, pdl);
  if (p.hd == 64) return int8 ? launch_t<true, 64>(q, plan, s, pdl) : launch_t<false, 64>(q, plan, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace lps
