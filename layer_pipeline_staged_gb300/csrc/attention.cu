// Split-K GQA decode attention over a stage-owned contiguous bf16 KV cache
// (flash-decoding): the positions [0, pos] of each (sequence, kv head) are cut
// into equal chunks; one CTA per chunk computes, for every q head of the
// group, a partial (running max m, running sum l, unnormalised output acc);
// the last CTA of the group to finish combines the partials in chunk order.
//
// The q heads of one group share the group's K/V rows, so every cached byte is
// read once per step (q head h reads kv head h / (nq / nkv): "TP3 support via
// zero-padded dummy heads", Implementation status item 2).
//
// Inside a CTA:
//   - K and V sub-tiles arrive by 2D TMA (cp.async.bulk.tensor, 128-byte
//     swizzle, so the ldmatrix reads below are free of bank conflicts) into a
//     three-deep ring; sub-tiles that lie strictly before the current position
//     are fetched before the programmatic-dependent-launch wait (earlier steps
//     wrote them), the one holding row pos after it (the QKV kernel just wrote
//     that row);
//   - the dot products run on tensor cores (mma.sync m16n8k16, bf16 in, fp32
//     accumulate; a score's HD/16 k-steps accumulate on the tensor core, the
//     P.V sums over the context add each k-step's MMA with a round-to-nearest
//     fp32 add). Row 2h of the 16-row operand is bf16(q_h) and row 2h+1 is
//     bf16(q_h - bf16(q_h)), so q keeps about 16 significant bits; the
//     probabilities are split the same way for P.V;
//   - each warp owns a 16-position slice of every sub-tile and keeps its own
//     online softmax; the scores' accumulator fragment is reused directly as
//     the A operand of P.V. The four warps' partials are merged in fixed order.
// The chunk length depends only on pos, and every merge has a fixed order, so
// the result is the same bits for every stage plan and stream schedule.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRing = 3;

template <int HD>
struct Shape {
  static constexpr int TS = 8192 / HD;          // positions per sub-tile (16 KB of K, 16 KB of V)
  static constexpr int NPOS = TS / kWarps;      // positions per warp per sub-tile (16 or 32)
  static constexpr int PARTS = HD / 64;         // 128-byte (64-element) TMA boxes per row
  static constexpr int BOX = TS * 128;          // bytes of one box
  static constexpr int TILE = PARTS * BOX;      // bytes of one K (or V) sub-tile
};

template <int HD, int G>
struct __align__(1024) AttnSmem {
  using S = Shape<HD>;
  uint8_t k[kRing][S::TILE];
  uint8_t v[kRing][S::TILE];
  float o[kWarps][G][HD];   // per-warp unnormalised outputs
  float m[kWarps][G], l[kWarps][G];
  float cm[G], cl[G];       // combine: max of m and weighted sum of l per head
  uint64_t full[kRing];
  int last;
};

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

// c += A.B for one 16-wide k-step: the tensor core sums the 16 exact products
// from a zero accumulator, then an ordinary (round-to-nearest) fp32 add
// accumulates, so long sums (P.V over the whole context) do not pile up the
// accumulator's truncation. Not volatile: independent MMAs may overlap.
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  float d0, d1, d2, d3;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
  c[0] += d0;
  c[1] += d1;
  c[2] += d2;
  c[3] += d3;
}

// c += A.B accumulated on the tensor core, for short sums (a score's HD/16
// k-steps, started from zero for every sub-tile).
__device__ __forceinline__ void mma_bf16_acc(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                             uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> a bf16x2 word (low half = first).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Split x into bf16 hi (row parity 0) or lo = bf16(x - hi) (row parity 1).
__device__ __forceinline__ float split_part(float x, int lo) {
  const float hi = __bfloat162float(__float2bfloat16_rn(x));
  return lo ? x - hi : hi;
}

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 2) attn_kernel(const __grid_constant__ AttnParams p) {
  using S = Shape<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  AttnSmem<HD, G>& sm = *reinterpret_cast<AttnSmem<HD, G>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
  trace_start(p.trace);
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos = p.pos[b];
  const int n_total = pos + 1;
  const int t_begin = c * p.chunk;
  if (t_begin >= n_total) return;  // beyond this sequence's positions (uniform per CTA)
  const int t_end = min(t_begin + p.chunk, n_total);
  const int nsub = (t_end - t_begin + S::TS - 1) / S::TS;
  const int nchunks = (n_total + p.chunk - 1) / p.chunk;
  const int row0 = (b * p.nkv + g) * p.max_ctx;  // first cache row of (b, g) in the tensor map

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) mbar_init(&sm.full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Early, the next kernel's CTAs take SMs as soon as the CTAs here leave them
  // (while the last CTAs combine); its own dependency wait still covers
  // everything this kernel writes.
  if (p.early_dependents) pdl_launch_dependents();

  auto issue = [&](int j) {
    const int slot = j % kRing;
    const int y = row0 + t_begin + j * S::TS;
    mbar_arrive_expect_tx(&sm.full[slot], 2 * S::TILE);
#pragma unroll
    for (int part = 0; part < S::PARTS; ++part) {
      tma_load_2d(sm.k[slot] + part * S::BOX, &p.tmap_k, part * 64, y, &sm.full[slot]);
      tma_load_2d(sm.v[slot] + part * S::BOX, &p.tmap_v, part * 64, y, &sm.full[slot]);
    }
  };
  const int first = min(kRing, nsub);
  int issued = 0;
  if (tid == 0) {
    // sub-tiles whose rows all lie before pos were written by earlier steps
    while (issued < first && t_begin + (issued + 1) * S::TS <= pos) issue(issued++);
  }
  pdl_wait();
  if (tid == 0)
    while (issued < first) issue(issued++);

  // q of the group as the A operand: row 2h = bf16(q_h), row 2h+1 = bf16(q_h - bf16(q_h))
  uint32_t qa[HD / 16][4];
  {
    const float* qb = p.q + static_cast<size_t>(b) * p.nq * HD + g * G * HD;
    const int h0 = g8 >> 1, h1 = (g8 + 8) >> 1, lo = g8 & 1;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const int d0 = 16 * kk + 2 * t4;
      float v[8];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        v[e] = h0 < G ? split_part(qb[h0 * HD + d0 + e], lo) : 0.f;
        v[2 + e] = h1 < G ? split_part(qb[h1 * HD + d0 + e], lo) : 0.f;
        v[4 + e] = h0 < G ? split_part(qb[h0 * HD + d0 + 8 + e], lo) : 0.f;
        v[6 + e] = h1 < G ? split_part(qb[h1 * HD + d0 + 8 + e], lo) : 0.f;
      }
      qa[kk][0] = pack_bf16(v[0], v[1]);
      qa[kk][1] = pack_bf16(v[2], v[3]);
      qa[kk][2] = pack_bf16(v[4], v[5]);
      qa[kk][3] = pack_bf16(v[6], v[7]);
    }
  }

  // per-warp online softmax state for rows g8 and g8+8 (heads h0, h1)
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float o_acc[HD / 8][4];
#pragma unroll
  for (int j = 0; j < HD / 8; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
  const float scale = p.scale;

  for (int j = 0; j < nsub; ++j) {
    const int slot = j % kRing;
    const bool got = mbar_wait(&sm.full[slot], (j / kRing) & 1, wait_cycles(p.wait_limit));
    if (__syncthreads_or(!got)) {
      // The copies issued so far (sub-tiles j .. issued-1) land before the CTA ends.
      if (tid == 0) {
        report_error(p.status, kErrWaitFull | (kKidAttn << 8));
        for (int k = j; k < issued; ++k)
          if (!mbar_wait(&sm.full[k % kRing], (k / kRing) & 1, kDrainLimitCycles)) {
            report_error(p.status, kErrDrain | (kKidAttn << 8));
            break;
          }
      }
      return;
    }
    const int rows = min(S::TS, t_end - (t_begin + j * S::TS));
    const int wp0 = warp * S::NPOS;  // this warp's first position in the sub-tile
    if (wp0 < rows) {
      const uint32_t kbase = smem_u32(sm.k[slot]);
      const uint32_t vbase = smem_u32(sm.v[slot]);
      // scores: S[n][pos] for the warp's NPOS positions (NPOS/8 n-tiles of 8 positions)
      float sc[S::NPOS / 8][4];
#pragma unroll
      for (int nt = 0; nt < S::NPOS / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int part = kk / 4, ch = 2 * (kk % 4);
#pragma unroll
        for (int nt = 0; nt < S::NPOS / 8; nt += 2) {
          // matrices: (n-tile nt, k lo), (nt, k hi), (nt+1, k lo), (nt+1, k hi)
          const int mtx = lane >> 3;
          const int r = wp0 + 8 * (nt + (mtx >> 1)) + (lane & 7);
          const uint32_t addr = kbase + part * S::BOX + swz(r, ch + (mtx & 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_bf16_acc(sc[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16_acc(sc[nt + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      // combine the hi and lo rows of each head, scale, mask, update the running max
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < S::NPOS / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float s = (sc[nt][e] + __shfl_xor_sync(0xffffffffu, sc[nt][e], 4)) * scale;
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
      // probabilities as the A operand of P.V (row parity picks the hi or lo part)
      float ls[2] = {0.f, 0.f};
      uint32_t pa[S::NPOS / 16][4];
#pragma unroll
      for (int nt = 0; nt < S::NPOS / 8; ++nt) {
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
      // O[n][dim] += P[n][pos] . V[pos][dim]
#pragma unroll
      for (int ks = 0; ks < S::NPOS / 16; ++ks) {
#pragma unroll
        for (int jd = 0; jd < HD / 8; jd += 2) {
          // matrices: (pos 0-7, dims jd), (pos 8-15, dims jd), (pos 0-7, jd+1), (pos 8-15, jd+1)
          const int mtx = lane >> 3;
          const int r = wp0 + 16 * ks + 8 * (mtx & 1) + (lane & 7);
          const int dch = jd + (mtx >> 1);
          const uint32_t addr = vbase + (dch / 8) * S::BOX + swz(r, dch % 8);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma_bf16(o_acc[jd], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
          mma_bf16(o_acc[jd + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
        }
      }
    }
    __syncthreads();  // sub-tile `slot` fully consumed
    if (tid == 0 && j + kRing < nsub) issue(issued++);
  }

  // this warp's (m, l, o) per head: rows 2h (hi) and 2h+1 (lo) of o add up
  {
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
          if (!lo && h < G) sm.o[warp][h][8 * jd + 2 * t4 + e] = sum;
        }
      }
      if (!lo && t4 == 0 && h < G) {
        sm.m[warp][h] = m_r[rr];
        sm.l[warp][h] = l_r[rr];
      }
    }
  }
  __syncthreads();
  // merge the warps in order and write this chunk's partial: rows of HD + 4
  // floats (acc, m, l, two pad) so each head's run of chunks is a whole number
  // of 16-byte units for the bulk copy below
  const int stride = HD + 4;
  for (int o = tid; o < G * HD; o += kThreads) {
    const int hh = o / HD, i = o - hh * HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][hh]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = (sm.m[w][hh] == -INFINITY) ? 0.f : expf(sm.m[w][hh] - M);
      L = fmaf(sm.l[w][hh], wt, L);
      O = fmaf(sm.o[w][hh][i], wt, O);
    }
    float* dst = p.part + ((static_cast<size_t>(b) * p.nq + g * G + hh) * p.max_chunks + c) * stride;
    dst[i] = O;
    if (i == 0) {
      dst[HD] = M;
      dst[HD + 1] = L;
    }
  }

  // the last CTA of (b, g) combines every chunk's partial, in chunk order
  asm volatile("fence.proxy.async.global;" ::: "memory");  // partials are read back through the async proxy
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.counter[b * p.nkv + g], 1);
    sm.last = (prev == nchunks - 1);
  }
  __syncthreads();
  if (sm.last) {
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    // the K/V ring is free now: stage the group's partials there, a piece of
    // chunks at a time, with one bulk copy per head
    float* buf = reinterpret_cast<float*>(sm.k[0]);
    // chunks per piece: the partials fit in the ring, their weights in sm.o
    // (free after the warp merge above)
    const int cap = min(static_cast<int>(sizeof(sm.k) + sizeof(sm.v)) / (G * stride * 4), kWarps * HD);
    float* wts = sm.o[0][0];  // chunk weights [G][cap]
    float* Ms = sm.cm;
    float* Ls = sm.cl;
    // pass 0 over pieces: the max of m per head; pass 1: weights, L and O
    float O[(G * HD + kThreads - 1) / kThreads];
#pragma unroll
    for (int k = 0; k < (G * HD + kThreads - 1) / kThreads; ++k) O[k] = 0.f;
    if (tid < G) {
      Ms[tid] = -INFINITY;
      Ls[tid] = 0.f;
    }
    const float* gbase = p.part + (static_cast<size_t>(b) * p.nq + g * G) * p.max_chunks * stride;
    const bool one_piece = nchunks <= cap;  // then both passes use one staged copy
    int loads = 0;
    for (int pass = 0; pass < 2; ++pass) {
      for (int c0 = 0; c0 < nchunks; c0 += cap) {
        const int nc = min(cap, nchunks - c0);
        __syncthreads();  // the staging area is free
        if (one_piece && pass == 1) goto staged;
        if (tid == 0) {
          const uint32_t bytes = static_cast<uint32_t>(nc) * stride * 4;
          mbar_arrive_expect_tx(&sm.full[0], G * bytes);
          for (int hh = 0; hh < G; ++hh)
            bulk_g2s_plain(buf + hh * nc * stride, gbase + (static_cast<size_t>(hh) * p.max_chunks + c0) * stride,
                           bytes, &sm.full[0]);
        }
        {
          // phases of full[0] continue from the ring's count
          const int phase = (nsub + kRing - 1) / kRing + loads++;
          const bool ok = mbar_wait(&sm.full[0], phase & 1, wait_cycles(p.wait_limit));
          if (__syncthreads_or(!ok)) {
            // the staged copy lands before the CTA ends
            if (tid == 0) {
              report_error(p.status, kErrWaitFull | (kKidAttnCombine << 8));
              if (!mbar_wait(&sm.full[0], phase & 1, kDrainLimitCycles))
                report_error(p.status, kErrDrain | (kKidAttnCombine << 8));
            }
            return;
          }
        }
      staged:
        if (pass == 0) {
          for (int hh = warp; hh < G; hh += kWarps) {
            float mx = -INFINITY;
            for (int cc = lane; cc < nc; cc += 32) mx = fmaxf(mx, buf[(hh * nc + cc) * stride + HD]);
            mx = warp_max(mx);
            if (lane == 0) Ms[hh] = fmaxf(Ms[hh], mx);
          }
        } else {
          for (int hh = warp; hh < G; hh += kWarps) {
            float ls = 0.f;
            for (int cc = lane; cc < nc; cc += 32) {
              const float w = expf(buf[(hh * nc + cc) * stride + HD] - Ms[hh]);
              wts[hh * cap + cc] = w;
              ls = fmaf(buf[(hh * nc + cc) * stride + HD + 1], w, ls);
            }
            ls = warp_sum(ls);
            if (lane == 0) Ls[hh] += ls;
          }
          __syncthreads();
#pragma unroll
          for (int k = 0; k < (G * HD + kThreads - 1) / kThreads; ++k) {
            const int o = tid + k * kThreads;
            if (o < G * HD) {
              const int hh = o / HD, i = o - hh * HD;
              float acc = O[k];
              for (int cc = 0; cc < nc; ++cc) acc = fmaf(buf[(hh * nc + cc) * stride + i], wts[hh * cap + cc], acc);
              O[k] = acc;
            }
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < (G * HD + kThreads - 1) / kThreads; ++k) {
      const int o = tid + k * kThreads;
      if (o < G * HD) {
        const int hh = o / HD, i = o - hh * HD;
        p.out[static_cast<size_t>(b) * p.nq * HD + (g * G + hh) * HD + i] = O[k] / Ls[hh];
      }
    }
    if (tid == 0) p.counter[b * p.nkv + g] = 0;
  }
  if (!p.early_dependents) pdl_launch_dependents();
  trace_end(p.trace);
}

template <int HD, int G>
cudaError_t launch_hg(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  auto kern = attn_kernel<HD, G>;
  const int smem = static_cast<int>(sizeof(AttnSmem<HD, G>));
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_pos + 1 + p.chunk - 1) / p.chunk, p.nkv, batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int HD>
cudaError_t launch_h(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  switch (p.nq / p.nkv) {
    case 1: return launch_hg<HD, 1>(p, batch, max_pos, s, pdl);
    case 2: return launch_hg<HD, 2>(p, batch, max_pos, s, pdl);
    case 4: return launch_hg<HD, 4>(p, batch, max_pos, s, pdl);
    case 8: return launch_hg<HD, 8>(p, batch, max_pos, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int attn_sub_tile(int hd) { return 8192 / hd; }

// Positions per CTA: a whole number cs of sub-tiles, chosen for the shortest
// modelled time, with `slots` CTAs per SM sharing the SM's share of HBM: the
// busiest SM takes ceil(CTAs / (slots x SMs)) rounds of cs sub-tiles plus a
// fixed per-CTA cost (start-up, first copy, partial write) of about two
// sub-tiles; ties go to the longer chunk (fewer partials to combine).
static int attn_chunk_model(int nsub, long long groups, int num_sms, int slots) {
  constexpr long long kOverhead = 2;
  long long best = -1;
  int best_cs = nsub;
  for (int cs = 1; cs <= nsub; ++cs) {
    const long long ctas = groups * ((nsub + cs - 1) / cs);
    const long long per = static_cast<long long>(slots) * num_sms;
    const long long cost = (ctas + per - 1) / per * (cs + kOverhead);
    if (best < 0 || cost <= best) {
      best = cost;
      best_cs = cs;
    }
  }
  return best_cs;
}

// Otherwise balancing the bytes per SM (one CTA slot per SM in the model)
// gives fewer partials to merge and measured faster, except where it leaves
// one CTA per SM with a long chunk: its four warps are then latency-bound, and
// two resident CTAs per SM with half the chunk measured faster (8B shapes: one
// slot wins at context 4096 batch 4 and at context 32768 batch 8, two slots
// at context 32768 batch 1).
int attn_chunk(int hd, int nkv, int batch, int max_pos, int num_sms) {
  const int ts = attn_sub_tile(hd);
  const int nsub = (max_pos + 1 + ts - 1) / ts;  // sub-tiles of one (sequence, kv head)
  const long long groups = static_cast<long long>(nkv) * batch;
  if (batch == 1 && nsub <= 256) {
    // one sequence, up to 256 sub-tiles: about one CTA per two SMs, so that
    // other stages' kernels can run beside it; measured on the 8B bf16 step at
    // context 8192 (4 stages): 2.901 ms with 152 CTAs of 7 sub-tiles,
    // 2.880-2.885 with 64-88 CTAs of 12-16, 2.997 with 32. The chunking depends
    // on the shapes, the position and the SM count only (never on the stage
    // plan), so every plan sums the same partials in the same order
    const long long per = (num_sms + groups) / (2 * groups);
    const int chunks = static_cast<int>(per < 1 ? 1 : per);
    return (nsub + chunks - 1) / chunks * ts;
  }
  const int cs1 = attn_chunk_model(nsub, groups, num_sms, 1);
  const long long ctas1 = groups * ((nsub + cs1 - 1) / cs1);
  if (cs1 <= 24 || ctas1 > num_sms) return cs1 * ts;
  return attn_chunk_model(nsub, groups, num_sms, 2) * ts;
}

int attn_max_chunks(int hd, int nkv, int batch, int max_ctx, int num_sms) {
  int worst = 1;
  for (int n = 1; n <= max_ctx; ++n) {
    const int ch = attn_chunk(hd, nkv, batch, n - 1, num_sms);
    const int k = (n + ch - 1) / ch;
    worst = k > worst ? k : worst;
  }
  return worst;
}

bool attn_supported(int hd, int group) {
  return (hd == 64 || hd == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_attention(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  if (p.hd == 64) return launch_h<64>(p, batch, max_pos, s, pdl);
  if (p.hd == 128) return launch_h<128>(p, batch, max_pos, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace lps
