// The prefill chunk's non-GEMM kernels: the activation split (with the input
// RMSNorm) that feeds the tcgen05 GEMM, and the causal attention of a chunk
// of consecutive positions over the stage's cache (memra_engine::pp,
// prime_pp_on / prime_pipe_on; ninfer pipeline-stages.md, "Prefill
// micro-chunk overlap").
//
// Chunk attention: query token j of the chunk sits at position pos0 + j and
// attends the cache rows [0, pos0 + j] of its sequence, which include the
// chunk's own rows (the QKV GEMM wrote them just before). The work is split
// like the decode attention, by key chunks, so that every SM has work at any
// context length:
//   - CTA (key chunk kc, query block qb of up to 128 / G tokens, kv head g)
//     runs one warp per (q head of the group, 16 tokens of the block), up to
//     eight: warp w takes head w mod G and the w / G-th 16 tokens, so every K/V
//     byte the CTA brings in serves all of them (a block is one 16-token group
//     when the chunk has at most 16 tokens, as verify rows do, which keeps two
//     CTAs per SM there); each warp holds its 16 query rows as mma.sync A fragments, split
//     into bf16 hi and lo parts (two MMAs per k-step), so q keeps about 16
//     significant bits;
//   - K and V sub-tiles arrive by 2D TMA with the 128-byte swizzle into a
//     ring shared by the group's warps; keys past a row's own position are
//     masked; each warp keeps an online softmax per row and accumulates P.V
//     with P split the same way;
//   - each (token, head, key chunk) leaves (m, l, unnormalised o); the merge
//     kernel combines the chunks of a token in chunk order and writes the
//     o-projection's two bf16 activation planes.
// Every sum has a fixed order that depends on the shapes, pos0 and the SM
// count only, so identical inputs give identical bits in every stage plan.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kRing = 3;
constexpr int kMaxMergeChunks = 320;  // key chunks per token the merge takes (chunk_attn_max_chunks)

// ---- activation planes --------------------------------------------------------

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Row j < ntok: x = src[j] (K floats), optionally RMS-normalised with `gain`;
// X[j] = bf16(x), X[NP + j] = bf16(x - bf16(x)). Rows [ntok, NP) become zero.
// Each thread loads its float4 groups of the row (and of the gain) into
// registers at once, up to kPrepVec of them; longer rows loop.
constexpr int kPrepVec = 8;
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const __grid_constant__ PrepParams p) {
  __shared__ float red[kPrepThreads / 32];
  __shared__ float s_inv;
  trace_start(p.trace);
  pdl_launch_dependents();
  const int j = blockIdx.x, tid = threadIdx.x;
  __nv_bfloat16* hi = p.x + static_cast<size_t>(j) * p.K;
  __nv_bfloat16* lo = p.x + static_cast<size_t>(p.NP + j) * p.K;
  const int K4 = p.K / 4;
  pdl_wait();
  if (j >= p.ntok) {
    for (int k = tid; k < K4; k += kPrepThreads) {
      reinterpret_cast<uint2*>(hi)[k] = make_uint2(0, 0);
      reinterpret_cast<uint2*>(lo)[k] = make_uint2(0, 0);
    }
    trace_end(p.trace);
    return;
  }
  const float4* src = reinterpret_cast<const float4*>(p.src + static_cast<size_t>(j) * p.lds);
  const float4* g4 = reinterpret_cast<const float4*>(p.gain);
  float inv = 1.f;
  if (p.gain) {
    // mean square: thread t sums the groups t, t + 256, ... in order; then the
    // warps' sums in warp order
    float ss = 0.f;
    for (int k0 = tid; k0 < K4; k0 += kPrepVec * kPrepThreads) {
      float4 v[kPrepVec];
#pragma unroll
      for (int u = 0; u < kPrepVec; ++u) {
        const int k = k0 + u * kPrepThreads;
        v[u] = k < K4 ? src[k] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kPrepVec; ++u) {
        ss = fmaf(v[u].x, v[u].x, ss);
        ss = fmaf(v[u].y, v[u].y, ss);
        ss = fmaf(v[u].z, v[u].z, ss);
        ss = fmaf(v[u].w, v[u].w, ss);
      }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kPrepThreads / 32; ++w) t += red[w];
      s_inv = 1.0f / sqrtf(t / static_cast<float>(p.K) + p.eps);
    }
    __syncthreads();
    inv = s_inv;
  }
  for (int k0 = tid; k0 < K4; k0 += kPrepVec * kPrepThreads) {
    float4 v[kPrepVec], g[kPrepVec];
#pragma unroll
    for (int u = 0; u < kPrepVec; ++u) {
      const int k = k0 + u * kPrepThreads;
      v[u] = k < K4 ? src[k] : make_float4(0.f, 0.f, 0.f, 0.f);
      g[u] = (p.gain && k < K4) ? __ldg(g4 + k) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
#pragma unroll
    for (int u = 0; u < kPrepVec; ++u) {
      const int k = k0 + u * kPrepThreads;
      if (k >= K4) break;
      const float x[4] = {v[u].x * inv * g[u].x, v[u].y * inv * g[u].y, v[u].z * inv * g[u].z, v[u].w * inv * g[u].w};
      float h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = __bfloat162float(__float2bfloat16_rn(x[e]));
        l[e] = x[e] - h[e];
      }
      reinterpret_cast<uint2*>(hi)[k] = make_uint2(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]));
      reinterpret_cast<uint2*>(lo)[k] = make_uint2(pack_bf16(l[0], l[1]), pack_bf16(l[2], l[3]));
    }
  }
  trace_end(p.trace);
}

// ---- chunk attention -----------------------------------------------------------

template <int HD>
struct CShape {
  static constexpr int TS = 8192 / HD;      // keys per sub-tile (16 KB of K, 16 KB of V)
  static constexpr int PARTS = HD / 64;     // 128-byte (64-element) TMA boxes per row
  static constexpr int BOX = TS * 128;      // bytes of one box
  static constexpr int TILE = PARTS * BOX;  // bytes of one K (or V) sub-tile
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
// c += A.B accumulated on the tensor core (a score's HD/16 k-steps)
__device__ __forceinline__ void mma_acc(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// c += A.B for one k-step from a zero accumulator, then a round-to-nearest fp32
// add, so the long P.V sums over the context do not pile up truncation.
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
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

template <int HD>
__global__ void __launch_bounds__(256) chunk_attn_kernel(const __grid_constant__ ChunkAttnParams p) {
  using S = CShape<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kt = smem;                          // [kRing][TILE]
  uint8_t* vt = smem + kRing * S::TILE;        // [kRing][TILE]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * kRing * S::TILE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
  trace_start(p.trace);
  const int kc = blockIdx.x, qb = blockIdx.y, g = blockIdx.z;
  const int G = p.nq / p.nkv, qw = p.nq * HD;
  const int h = g * G + warp % G;
  const int jb = qb * p.qblock;                                      // the CTA's first token
  const int j0 = jb + (warp / G) * 16, jn = min(16, p.ntok - j0);  // this warp's rows (jn <= 0: none)
  const int kend = p.pos0 + min(jb + p.qblock, p.ntok);             // the block attends keys [0, kend)
  const int k_begin = kc * p.chunk;
  if (k_begin >= kend) return;  // uniform per CTA: the merge reads no partial of this chunk
  const int k_stop = min(k_begin + p.chunk, kend);
  const int nsub = (k_stop - k_begin + S::TS - 1) / S::TS;
  const int row0 = (p.seq * p.nkv + g) * p.max_ctx;  // first cache row of (seq, g) in the tensor map
  const long long limit = wait_cycles(p.wait_limit);

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  auto issue = [&](int jt) {
    const int slot = jt % kRing;
    const int y = row0 + k_begin + jt * S::TS;
    mbar_arrive_expect_tx(&full[slot], 2 * S::TILE);
#pragma unroll
    for (int part = 0; part < S::PARTS; ++part) {
      tma_load_2d(kt + slot * S::TILE + part * S::BOX, &p.tmap_k, part * 64, y, &full[slot]);
      tma_load_2d(vt + slot * S::TILE + part * S::BOX, &p.tmap_v, part * 64, y, &full[slot]);
    }
  };
  // the chunk's own cache rows and q come from the kernels just before
  pdl_wait();
  int issued = 0;
  if (tid == 0)
    while (issued < min(kRing, nsub)) issue(issued++);

  // this warp's 16 query rows (tokens j0 .. j0 + 15 of head h) as hi and lo A fragments
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
    for (int rg = 0; rg < 4; ++rg) {
      const int row = g8 + ((rg & 1) ? 8 : 0);
      const int d = 16 * kk + 2 * t4 + ((rg & 2) ? 8 : 0);
      float x0 = 0.f, x1 = 0.f;
      if (row < jn) {
        const float* src = p.q + static_cast<size_t>(j0 + row) * qw + h * HD + d;
        x0 = src[0];
        x1 = src[1];
      }
      const float h0 = bf16_round(x0), h1 = bf16_round(x1);
      qh[kk][rg] = pack_bf16(h0, h1);
      ql[kk][rg] = pack_bf16(x0 - h0, x1 - h1);
    }
  }
  const int qpos[2] = {p.pos0 + j0 + g8, p.pos0 + j0 + g8 + 8};
  const bool live[2] = {g8 < jn, g8 + 8 < jn};
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float o_acc[HD / 8][4];
#pragma unroll
  for (int jd = 0; jd < HD / 8; ++jd) o_acc[jd][0] = o_acc[jd][1] = o_acc[jd][2] = o_acc[jd][3] = 0.f;

  bool bad = false;
  for (int jt = 0; jt < nsub; ++jt) {
    const int slot = jt % kRing;
    const bool got = mbar_wait(&full[slot], (jt / kRing) & 1, limit);
    if (__syncthreads_or(!got)) {
      if (tid == 0) {
        report_error(p.status, kErrWaitFull | (kKidChunkAttn << 8));
        for (int k = jt; k < issued; ++k)
          if (!mbar_wait(&full[k % kRing], (k / kRing) & 1, kDrainLimitCycles)) {
            report_error(p.status, kErrDrain | (kKidChunkAttn << 8));
            break;
          }
      }
      bad = true;
      break;
    }
    const uint32_t kbase = smem_u32(kt + slot * S::TILE), vbase = smem_u32(vt + slot * S::TILE);
    const int tile_key = k_begin + jt * S::TS;
    // A warp computes only the key groups its rows can see: none when its 16
    // tokens lie past the chunk, none past its last row's position (the causal
    // bound; such a group would leave every sum unchanged). It still meets the
    // other warps at the ring's barrier below.
    const int kmax = jn > 0 ? p.pos0 + j0 + jn - 1 : -1;  // the warp's last visible key
#pragma unroll 1
    for (int kg = 0; kg < S::TS / 32; ++kg) {
      const int kb = tile_key + kg * 32;  // first key of this group of 32
      if (kb >= k_stop || kb > kmax) break;
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int part = kk / 4, ch = 2 * (kk % 4);
#pragma unroll
        for (int nt = 0; nt < 4; nt += 2) {
          // matrices: (n-tile nt, k lo), (nt, k hi), (nt+1, k lo), (nt+1, k hi)
          const int mtx = lane >> 3;
          const int r = kg * 32 + 8 * (nt + (mtx >> 1)) + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + part * S::BOX + swz(r, ch + (mtx & 1)), b0, b1, b2, b3);
          mma_acc(sc[nt], qh[kk], b0, b1);
          mma_acc(sc[nt], ql[kk], b0, b1);
          mma_acc(sc[nt + 1], qh[kk], b2, b3);
          mma_acc(sc[nt + 1], ql[kk], b2, b3);
        }
      }
      // scale, causal mask, running max per row
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = e >> 1;
          const int key = kb + 8 * nt + 2 * t4 + (e & 1);
          const bool ok = live[rr] && key < k_stop && key <= qpos[rr];
          sc[nt][e] = ok ? sc[nt][e] * p.scale : -INFINITY;
          mx[rr] = fmaxf(mx[rr], sc[nt][e]);
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
      // probabilities as hi and lo A fragments of P.V
      float ls[2] = {0.f, 0.f};
      uint32_t ph[2][4], pl[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        float pr[4], pq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = e >> 1;
          const float pv = (m_r[rr] == -INFINITY) ? 0.f : expf(sc[nt][e] - m_r[rr]);
          ls[rr] += pv;
          pr[e] = bf16_round(pv);
          pq[e] = pv - pr[e];
        }
        const int ks = nt >> 1, up = nt & 1;
        ph[ks][up ? 2 : 0] = pack_bf16(pr[0], pr[1]);
        ph[ks][up ? 3 : 1] = pack_bf16(pr[2], pr[3]);
        pl[ks][up ? 2 : 0] = pack_bf16(pq[0], pq[1]);
        pl[ks][up ? 3 : 1] = pack_bf16(pq[2], pq[3]);
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
      // O[row][dim] += P[row][key] . V[key][dim]
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int jd = 0; jd < HD / 8; jd += 2) {
          // matrices: (keys 0-7, dims jd), (keys 8-15, jd), (keys 0-7, jd+1), (keys 8-15, jd+1)
          const int mtx = lane >> 3;
          const int r = kg * 32 + 16 * ks + 8 * (mtx & 1) + (lane & 7);
          const int dch = jd + (mtx >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + (dch / 8) * S::BOX + swz(r, dch % 8), b0, b1, b2, b3);
          mma_add(o_acc[jd], ph[ks], b0, b1);
          mma_add(o_acc[jd], pl[ks], b0, b1);
          mma_add(o_acc[jd + 1], ph[ks], b2, b3);
          mma_add(o_acc[jd + 1], pl[ks], b2, b3);
        }
      }
    }
    __syncthreads();  // sub-tile `slot` fully consumed
    if (tid == 0 && issued < nsub) issue(issued++);
  }
  if (!bad) {
    // this warp's (o, m, l) of its rows for key chunk kc
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = g8 + 8 * rr;
      if (!live[rr]) continue;
      float* dst = p.part + ((static_cast<size_t>(j0 + row) * p.nq + h) * p.max_chunks + kc) * (HD + 4);
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) {
        dst[8 * jd + 2 * t4] = o_acc[jd][2 * rr];
        dst[8 * jd + 2 * t4 + 1] = o_acc[jd][2 * rr + 1];
      }
      if (t4 == 0) {
        dst[HD] = m_r[rr];
        dst[HD + 1] = l_r[rr];
      }
    }
  }
  trace_end(p.trace);
}

// One warp per (token j, head h): combine the key chunks of the pair in chunk
// order and write the o-projection's activation planes xo[j] = bf16(o),
// xo[NP + j] = bf16(o - bf16(o)) (or, with `out` set, o itself as fp32). The
// chunk weights exp(m_c - M) are formed once (lane c, c + 32, ...; then fixed
// warp trees), then every dimension's sum over the chunks in chunk order.
template <int HD>
__global__ void __launch_bounds__(256) chunk_merge_kernel(const __grid_constant__ ChunkAttnParams p) {
  __shared__ float wsm[8][kMaxMergeChunks];
  trace_start(p.trace);
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + warp;
  if (pair < p.ntok * p.nq) {
    const int j = pair / p.nq, h = pair - j * p.nq, qw = p.nq * HD;
    const int jb = (j / p.qblock) * p.qblock;
    const int kend = p.pos0 + min(jb + p.qblock, p.ntok);  // the keys the token's block attended
    const int nch = (kend + p.chunk - 1) / p.chunk;
    const float* base = p.part + (static_cast<size_t>(j) * p.nq + h) * p.max_chunks * (HD + 4);
    float mloc = -INFINITY;
    for (int c = lane; c < nch; c += 32) mloc = fmaxf(mloc, base[c * (HD + 4) + HD]);
    const float M = warp_max(mloc);
    float lloc = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const float mc = base[c * (HD + 4) + HD];
      const float wc = mc == -INFINITY ? 0.f : expf(mc - M);
      wsm[warp][c] = wc;
      lloc += base[c * (HD + 4) + HD + 1] * wc;
    }
    const float L = warp_sum(lloc);
    __syncwarp();
    constexpr int PER = HD / 32;  // dimensions per lane
    float O[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) O[e] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float wc = wsm[warp][c];
      float t[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) t[e] = base[c * (HD + 4) + lane + 32 * e];
#pragma unroll
      for (int e = 0; e < PER; ++e) O[e] += t[e] * wc;
    }
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const float o = O[e] / L;
      const size_t idx = static_cast<size_t>(h) * HD + lane + 32 * e;
      if (p.out) {
        p.out[static_cast<size_t>(j) * qw + idx] = o;
      } else {
        const __nv_bfloat16 hi = __float2bfloat16_rn(o);
        p.xo[static_cast<size_t>(j) * qw + idx] = hi;
        p.xo[static_cast<size_t>(p.NP + j) * qw + idx] = __float2bfloat16_rn(o - __bfloat162float(hi));
      }
    }
  }
  trace_end(p.trace);
}

template <class Kern, class P>
cudaError_t launch_ex(Kern kern, const P& p, dim3 grid, dim3 block, int smem, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
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
cudaError_t launch_chunk_attn_t(const ChunkAttnParams& p, cudaStream_t s, bool pdl) {
  using S = CShape<HD>;
  const int smem = 2 * kRing * S::TILE + 1024 + 64;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(chunk_attn_kernel<HD>, smem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nchunks, (p.ntok + p.qblock - 1) / p.qblock, p.nkv);
  e = launch_ex(chunk_attn_kernel<HD>, p, grid, dim3(32 * (p.nq / p.nkv) * (p.qblock / 16)), smem, s, pdl);
  if (e != cudaSuccess) return e;
  ChunkAttnParams q = p;
  q.trace = p.trace_merge;
  return launch_ex(chunk_merge_kernel<HD>, q, dim3((p.ntok * p.nq + 7) / 8), dim3(256), 0, s, true);
}

}  // namespace

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s, bool pdl) {
  return launch_ex(prep_kernel, p, dim3(p.NP), dim3(kPrepThreads), 0, s, pdl);
}

int chunk_attn_sub_tile(int hd) { return 8192 / hd; }

int chunk_attn_max_chunks(int nkv, int num_sms) { return (2 * num_sms + nkv - 1) / nkv + 1; }

// Query blocks (16 tokens per warp row group, G x blocks/16 <= 8 warps per CTA:
// 128 / G tokens, or 16 when the chunk has at most 16) and key chunks for a
// chunk of ntok tokens ending at position pos0 + ntok - 1: about two CTAs per
// SM over (kv heads x query blocks x key chunks), of whole sub-tiles, none
// empty.
void chunk_attn_split(int hd, int nq, int nkv, int ntok, int pos0, int num_sms, int* nchunks, int* chunk,
                      int* qblock) {
  const int ts = chunk_attn_sub_tile(hd);
  const int groups16 = (ntok + 15) / 16, per_cta = 8 / (nq / nkv);
  *qblock = 16 * (groups16 < per_cta ? groups16 : per_cta);
  const int nqb = (ntok + *qblock - 1) / *qblock;
  const int kend = pos0 + ntok;
  const int nsub = (kend + ts - 1) / ts;
  int target = (2 * num_sms + nkv * nqb - 1) / (nkv * nqb);
  const int cap = chunk_attn_max_chunks(nkv, num_sms);
  target = target < cap ? target : cap;
  int n = target < nsub ? target : nsub;
  n = n < 1 ? 1 : n;
  const int cs = (nsub + n - 1) / n;  // sub-tiles per chunk
  *chunk = cs * ts;
  *nchunks = (kend + *chunk - 1) / *chunk;
}

cudaError_t launch_chunk_attn(const ChunkAttnParams& p, cudaStream_t s, bool pdl) {
  if (p.nq % p.nkv || p.nq / p.nkv > 8 || p.nq / p.nkv < 1 || 8 % (p.nq / p.nkv) || p.ntok < 1 ||
      p.ntok > kTcMaxTokens || p.max_chunks > kMaxMergeChunks || p.nchunks > p.max_chunks ||
      p.qblock < 16 || p.qblock % 16 || (p.nq / p.nkv) * (p.qblock / 16) > 8)
    return cudaErrorInvalidValue;
  if (p.hd == 128) return launch_chunk_attn_t<128>(p, s, pdl);
  if (p.hd == 64) return launch_chunk_attn_t<64>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace lps
