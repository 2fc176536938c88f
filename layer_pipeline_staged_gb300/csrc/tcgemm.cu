// Weight-streaming GEMM on the fifth-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed shared memory) for a block of token rows of one
// sequence: Y[j][r] = sum_k W[r][k] X[j][k] for j < ntok, with the same fused
// epilogues as the decode step (RoPE + KV append, residual add, SwiGLU). It
// runs the projections of a prefill chunk (memra_engine::pp, prime_pp_on /
// prime_pipe_on: the prompt goes through the same stage split as decode, one
// micro-chunk of rows at a time).
//
// Operands:
//   - A = the packed weights W [R][K], row-major (the batch-1 layout, so no
//     second copy of any matrix), 128-row x 64-column tiles by 2D TMA: bf16
//     with the 128-byte swizzle, which is the canonical K-major layout the MMA
//     reads; int8 unswizzled, widened to that bf16 layout by four warps (int8
//     values are exact in bf16; the per-row scale multiplies the result);
//   - B = the activations as two bf16 planes, X = hi + lo with hi = bf16(x) and
//     lo = bf16(x - hi): rows [0, NP) hold hi, rows [NP, 2 NP) lo, so every
//     activation keeps about 16 significant bits. The two planes are one
//     operand of 2 NP rows: each k-step is one MMA with N = 2 NP;
//   - D = 128 weight rows x 2 NP columns of fp32 in TMEM (column j the hi part
//     of token j, column NP + j its lo part, added in the epilogue), two
//     buffers, so the MMAs of the next tile run while the epilogue drains the
//     last one.
//
// Work split (every SM streams the same number of weight bytes): the tiles'
// k-blocks (tile-major) are cut into gridDim.x equal contiguous ranges, one
// per CTA. A CTA's range is a sequence of runs, one per tile it touches; a run
// that covers a whole tile goes straight through the epilogue, a run that
// covers part of one writes its accumulator to a per-CTA partial slot, and
// the last CTA to finish a tile adds the tile's partials in k order and runs
// the epilogue. The split depends only on (R, K, grid), and every sum has a
// fixed order, so identical inputs give identical bits in every stage plan.
//
// Roles: warp 0 lane 0 issues the TMA copies into an S-stage ring (weights
// of the first stages before the programmatic-dependent-launch wait, as they
// never depend on the previous kernel); warp 1 allocates TMEM and its lane 0
// issues the MMAs and the tcgen05.commit arrivals that free ring stages and
// publish finished accumulators, and before the CTA ends waits for its own
// MMAs to complete; warps 2..9 (two per 32-lane TMEM quarter, each taking
// half of the token columns) read the accumulators with tcgen05.ld and apply
// the epilogue; warps 10..13 widen int8 weight tiles. Every wait is bounded
// and reports through the status word instead of hanging.
#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace lps {
namespace {

using namespace tc;

constexpr int kTM = 128;                 // weight rows per tile (MMA M)
constexpr int kKB = 64;                  // K elements per k-block: one 128-byte swizzle row
constexpr int kATile = kTM * kKB * 2;    // bytes of one weight tile
constexpr int kThreads = 448;            // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue, 10..13 int8 widening
constexpr int kEpiThreads = 256;
constexpr int kCvtThreads = 128;         // warps 10..13
constexpr int kA8Tile = kTM * kKB;       // bytes of one int8 weight tile (rows of 64 bytes, unswizzled)

// ---- epilogue -------------------------------------------------------------------

// Apply the epilogue to 16 consecutive token columns [j0, j0 + 16) of one
// row. Rows come in pairs on adjacent lanes (RoPE pairs, gate/up pairs):
// w[e] is the partner row's value of column j0 + e. Every load of the group
// (residual rows, RoPE angles) is issued before its first store, so a group
// costs one memory round trip, not sixteen.
__device__ __forceinline__ void epilogue16(const TcGemmParams& p, int r, int j0, const float* v, const float* w) {
  const int nj = p.ntok - j0;
  if (r >= p.R || nj <= 0) return;
  if (p.epi == kEpiResidual) {
    float* h = p.h + static_cast<size_t>(j0) * p.ldh + r;
    float in[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) in[e] = e < nj ? h[static_cast<size_t>(e) * p.ldh] : 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (e < nj) h[static_cast<size_t>(e) * p.ldh] = in[e] + v[e];
    return;
  }
  const bool odd = r & 1;
  const int u = r >> 1;
  if (p.epi == kEpiSwiglu) {
    if (odd) return;  // the even lane of the pair writes a
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (e >= nj) break;
      const float g = v[e], up = w[e];
      const float a = g / (1.0f + expf(-g)) * up;
      const __nv_bfloat16 hi = __float2bfloat16_rn(a);
      p.xo[static_cast<size_t>(j0 + e) * p.ldx + u] = hi;
      p.xo[static_cast<size_t>(p.NP + j0 + e) * p.ldx + u] = __float2bfloat16_rn(a - __bfloat162float(hi));
    }
    return;
  }
  // kEpiQkv: unit u = (head hh, i) holds rows (hh*hd + i, hh*hd + i + hd/2)
  const int half = p.hd >> 1;
  const int hh = u / half, i = u - hh * half;
  const int col = i + (odd ? half : 0);
  float out[16];
  if (hh < p.nq + p.nkv) {
    float2 cs[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      cs[e] = e < nj ? p.rope[static_cast<size_t>(p.pos0 + j0 + e) * half + i] : make_float2(1.f, 0.f);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float y0 = odd ? w[e] : v[e], y1 = odd ? v[e] : w[e];  // the pair's first and second row
      out[e] = odd ? y0 * cs[e].y + y1 * cs[e].x : y0 * cs[e].x - y1 * cs[e].y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) out[e] = v[e];
  }
  if (hh < p.nq) {
    float* q = p.q + static_cast<size_t>(j0) * p.nq * p.hd + hh * p.hd + col;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (e < nj) q[static_cast<size_t>(e) * p.nq * p.hd] = out[e];
  } else {
    const bool is_k = hh < p.nq + p.nkv;
    const int g = is_k ? hh - p.nq : hh - p.nq - p.nkv;
    __nv_bfloat16* c = (is_k ? p.kc : p.vc) +
                       ((static_cast<size_t>(p.seq) * p.nkv + g) * p.max_ctx + p.pos0 + j0) * p.hd + col;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (e < nj) c[static_cast<size_t>(e) * p.hd] = __float2bfloat16_rn(out[e]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcGemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the tiles (the swizzle pattern repeats every 1024 bytes)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages, NP = p.NP;
  const int btile = NP * 128;  // bytes of one activation plane's k-block
  // a stage: the bf16 weight tile, the two activation planes, and with int8
  // weights the raw int8 tile the widening warps turn into the bf16 tile
  const int stage_bytes = kATile + 2 * btile + (p.int8 ? kA8Tile : 0);
  const int tx_bytes = (p.int8 ? kA8Tile : kATile) + 2 * btile;  // bytes the copies of a stage bring
  const int w_off = p.int8 ? kATile + 2 * btile : 0;               // where the weight copy lands
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* conv = empty + S + 4;  // [S] int8: the bf16 tile of the stage is ready (after acc_full/acc_empty)
  uint64_t* acc_full = empty + S;   // [2]: an accumulator buffer is ready for the epilogue
  uint64_t* acc_empty = acc_full + 2;  // [2]: the epilogue has drained it
  uint64_t* mma_done = conv + S;  // the MMA lane's own MMAs have all completed (before TMEM is freed)
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* flag = reinterpret_cast<int*>(tmem_base + 1);  // [0]: this CTA finishes the tile

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  trace_start(p.trace);
  const int G = gridDim.x, c = blockIdx.x;
  const int ntiles = (p.R + kTM - 1) / kTM, nkb = (p.K + kKB - 1) / kKB;
  const long long T = static_cast<long long>(ntiles) * nkb;
  const long long beg = range_start(c, T, G), end = range_start(c + 1, T, G);
  const long long limit = wait_cycles(p.wait_limit);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
    }
    for (int i = 0; i < S; ++i) mbar_init(&conv[i], 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised: the producer may start at once
  pdl_launch_dependents();
  // warp 1 allocates the accumulators while warp 0 already streams; warps 1..
  // meet at named barrier 3 before reading the TMEM address
  if (warp == 1) {
    tmem_alloc(tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  uint32_t tbase = 0;
  if (warp > 0) {
    tc_fence_before();
    named_bar_sync(3, kThreads - 32);
    tc_fence_after();
    tbase = *tmem_base;
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      const long long n_it = end - beg;
      const long long pre = n_it < S ? n_it : S;
      bool ok = true;
      long long n = 0;
      // the first stages' weights before the dependency wait
      for (; n < pre; ++n) {
        const long long i = beg + n;
        uint8_t* st = smem + static_cast<size_t>(n) * stage_bytes;
        mbar_arrive_expect_tx(&full[n], tx_bytes);
        tma_2d_hint(st + w_off, &p.tmap_w, static_cast<int>(i % nkb) * kKB, static_cast<int>(i / nkb) * kTM, &full[n],
                    pol);
      }
      pdl_wait();
      for (long long m = 0; m < pre; ++m) {
        const long long i = beg + m;
        uint8_t* st = smem + static_cast<size_t>(m) * stage_bytes;
        const int x = static_cast<int>(i % nkb) * kKB;
        tma_2d(st + kATile, &p.tmap_x, x, 0, &full[m]);
        tma_2d(st + kATile + btile, &p.tmap_x, x, NP, &full[m]);
      }
      for (; n < n_it && ok; ++n) {
        const int s = static_cast<int>(n % S);
        const uint32_t par = static_cast<uint32_t>((n / S - 1) & 1);
        if (!mbar_wait(&empty[s], par, limit)) {
          report_error(p.status, kErrWaitEmpty | (kKidTcGemm << 8));
          ok = false;
          break;
        }
        const long long i = beg + n;
        uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes;
        const int x = static_cast<int>(i % nkb) * kKB;
        mbar_arrive_expect_tx(&full[s], tx_bytes);
        tma_2d_hint(st + w_off, &p.tmap_w, x, static_cast<int>(i / nkb) * kTM, &full[s], pol);
        tma_2d(st + kATile, &p.tmap_x, x, 0, &full[s]);
        tma_2d(st + kATile + btile, &p.tmap_x, x, NP, &full[s]);
      }
      // every copy issued lands before the CTA may end
      for (long long m = n - S < 0 ? 0 : n - S; m < n; ++m)
        if (!mbar_wait(&full[m % S], static_cast<uint32_t>((m / S) & 1), kDrainLimitCycles)) {
          report_error(p.status, kErrDrain | (kKidTcGemm << 8));
          break;
        }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // one MMA per 16-element k-step with N = 2 NP: the hi and lo planes lie
      // one after the other in the stage, 8-row groups 1024 bytes apart, so
      // one descriptor spans both; accumulator column j holds the hi part of
      // token j, column NP + j the lo part
      const uint32_t idesc = idesc_bf16(kTM, 2 * NP);
      long long n = 0;
      bool ok = true;
      Run r;
      for (int ri = 0; ok && run_at(beg, end, nkb, ri, &r); ++ri) {
        const int b = ri & 1;
        if (ri >= 2 && !mbar_wait(&acc_empty[b], static_cast<uint32_t>(((ri >> 1) - 1) & 1), limit)) {
          report_error(p.status, kErrWaitEmpty | (kKidTcGemm << 8) | (1 << 13));
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tbase + static_cast<uint32_t>(b * 2 * NP);
        for (int kb = r.k0; kb < r.k1; ++kb, ++n) {
          const int s = static_cast<int>(n % S);
          if (!mbar_wait(&full[s], static_cast<uint32_t>((n / S) & 1), limit) ||
              (p.int8 && !mbar_wait(&conv[s], static_cast<uint32_t>((n / S) & 1), limit))) {
            report_error(p.status, kErrWaitFull | (kKidTcGemm << 8));
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * stage_bytes);
          const uint64_t da = sw128_desc(st), dh = sw128_desc(st + kATile);
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk) {
            // +32 bytes along the swizzled row per 16-element k-step (>> 4 in the descriptor)
            const uint64_t adv = static_cast<uint64_t>(2 * kk);
            umma_bf16(d, da + adv, dh + adv, idesc, (kb > r.k0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        umma_commit(&acc_full[b]);
      }
      // every MMA issued has completed before the accumulators are freed, also
      // when a wait above gave up and the epilogue never read them
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0, kDrainLimitCycles)) report_error(p.status, kErrDrain | (kKidTcGemm << 8) | (3 << 13));
    }
  } else if (warp >= 10) {
    // ---------------- int8 weights: widening warps 10..13 ----------------
    // Stage s's raw tile (128 rows of 64 int8) becomes the bf16 tile in the
    // 128-byte-swizzled K-major layout (int8 values are exact in bf16; the row
    // scale multiplies the accumulator in the epilogue). The stage's bf16 tile
    // is free again only when the MMAs of its previous use completed, which
    // the producer already waited for before it refilled the stage.
    if (p.int8) {
      const int ct = tid - 320;  // 0..127
      const long long n_it = end - beg;
      bool bad = false;
      for (long long n = 0; n < n_it; ++n) {
        const int s = static_cast<int>(n % S);
        const bool got = mbar_wait(&full[s], static_cast<uint32_t>((n / S) & 1), limit);
        // the four warps leave together on a timeout
        uint32_t any;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, 4, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(any)
            : "r"(static_cast<uint32_t>(!got)), "n"(kCvtThreads)
            : "memory");
        if (any) {
          bad = true;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes;
        const uint8_t* raw = st + w_off;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int id = ct + kCvtThreads * i, r = id >> 3, ch = id & 7;
          const uint2 q = *reinterpret_cast<const uint2*>(raw + r * kKB + ch * 8);
          const uint32_t w4[2] = {q.x, q.y};
          uint32_t out[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int8_t b0 = static_cast<int8_t>(w4[h] & 0xff), b1 = static_cast<int8_t>((w4[h] >> 8) & 0xff);
            const int8_t b2 = static_cast<int8_t>((w4[h] >> 16) & 0xff), b3 = static_cast<int8_t>(w4[h] >> 24);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(static_cast<float>(b0), static_cast<float>(b1));
            const __nv_bfloat162 hi = __floats2bfloat162_rn(static_cast<float>(b2), static_cast<float>(b3));
            out[2 * h] = *reinterpret_cast<const uint32_t*>(&lo);
            out[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&hi);
          }
          *reinterpret_cast<uint4*>(st + r * 128 + ((ch ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
        }
        // the tensor core reads the tile through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        named_bar_sync(4, kCvtThreads);
        if (ct == 0) mbar_arrive(&conv[s]);
      }
      (void)bad;
    }
  } else {
    // ---------------- epilogue: warps 2..9 ----------------
    // warp w reads TMEM lane quarter w % 4 (the hardware's rule) and the
    // token columns of half (w - 2) / 4 of the accumulator
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // this thread's row of the tile
    const int etid = tid - 64;          // 0..255
    const int cbeg = ((warp - 2) >> 2) * (NP >> 1), cend = cbeg + (NP >> 1);
    // barrier 1 over the eight epilogue warps, and the same with an OR vote
    auto epi_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); };
    auto epi_or = [](bool bad) -> bool {
      uint32_t res;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 1, %2, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(res)
          : "r"(static_cast<uint32_t>(bad)), "n"(kEpiThreads)
          : "memory");
      return res != 0;
    };
    pdl_wait();                         // residuals and caches of earlier kernels are visible
    Run r;
    for (int ri = 0; run_at(beg, end, nkb, ri, &r); ++ri) {
      const int b = ri & 1;
      const bool got = mbar_wait(&acc_full[b], static_cast<uint32_t>((ri >> 1) & 1), limit);
      if (!got && lane == 0) report_error(p.status, kErrWaitFull | (kKidTcGemm << 8) | (2 << 13));
      if (epi_or(!got)) break;  // the epilogue warps leave together
      tc_fence_after();
      const uint32_t tacc = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(b * 2 * NP);
      const bool whole = r.k0 == 0 && r.k1 == nkb;
      const int row = r.tile * kTM + m;
      // partial slot of this CTA: 0 for its first run, 1 for its last
      float* slot = p.part + (static_cast<size_t>(c) * 2 + (ri == 0 ? 0 : 1)) * static_cast<size_t>(NP) * kTM;
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        float v[16], w[16];
        tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
        tmem_ld16(tacc + static_cast<uint32_t>(NP + c0), w);  // the lo parts
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] += w[e];
        if (whole) {
          const float sr = (p.wscale && row < p.R) ? p.wscale[row] : 1.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= sr;
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = __shfl_xor_sync(0xffffffffu, v[e], 1);
          epilogue16(p, row, c0, v, w);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) slot[static_cast<size_t>(c0 + e) * kTM + m] = v[e];
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);
      if (whole) continue;
      // a partial: publish it; the last CTA of the tile to do so finishes the tile
      __threadfence();
      epi_sync();
      const long long t0i = static_cast<long long>(r.tile) * nkb, t1i = t0i + nkb - 1;
      const int cf = owner_of(t0i, T, G), cl = owner_of(t1i, T, G);
      if (etid == 0) {
        int contributors = 0;  // CTAs with a non-empty range inside the tile
        for (int cc = cf; cc <= cl; ++cc) contributors += range_start(cc, T, G) < range_start(cc + 1, T, G);
        const int prev = atomicAdd(p.counter + r.tile, 1);
        flag[0] = prev == contributors - 1;
      }
      epi_sync();
      if (!flag[0]) continue;
      __threadfence();
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        // the contributors' partials of 16 columns, added in k order
        float y[16], w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {
          const long long s0 = range_start(cc, T, G);
          if (s0 >= range_start(cc + 1, T, G)) continue;  // an empty range wrote nothing
          // the tile is CTA cc's first run unless cc started in an earlier tile
          const int si = s0 < t0i ? 1 : 0;
          const float* src = p.part + ((static_cast<size_t>(cc) * 2 + si) * NP + c0) * kTM + m;
          float t[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) t[e] = __ldcg(src + static_cast<size_t>(e) * kTM);
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] += t[e];
        }
        const float sr = (p.wscale && row < p.R) ? p.wscale[row] : 1.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] *= sr;
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __shfl_xor_sync(0xffffffffu, y[e], 1);
        epilogue16(p, row, c0, y, w);
      }
      if (etid == 0) p.counter[r.tile] = 0;
    }
  }

  trace_end(p.trace);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, p.tmem_cols);
  }
}

}  // namespace

int tc_gemm_tiles(int R) { return (R + kTM - 1) / kTM; }

// Ring depth from the shared memory: one stage is a 16 KB weight tile and the
// two activation planes of the same k-block (NP rows of 128 bytes each).
TcGemmPlan tc_gemm_plan(int NP, bool int8, int num_sms, int max_smem) {
  TcGemmPlan g{};
  if (NP < 32 || NP > kTcMaxTokens || NP % 32) return g;
  const int stage = kATile + 2 * NP * 128 + (int8 ? kA8Tile : 0);
  const int fixed = 1024 + 64 * 8 + 16;  // alignment slack, barriers, TMEM address and flags
  int stages = (max_smem - fixed) / stage;
  stages = stages > 8 ? 8 : stages;
  if (stages < 2) return g;
  int cols = 32;
  while (cols < 4 * NP) cols *= 2;  // two accumulators of 2 NP columns
  g.grid = num_sms;
  g.stages = stages;
  g.smem = stages * stage + fixed;
  g.tmem_cols = cols;
  g.ok = true;
  return g;
}

cudaError_t launch_tc_gemm(const TcGemmParams& p, const TcGemmPlan& plan, cudaStream_t s, bool pdl) {
  const unsigned long long T = static_cast<unsigned long long>(tc_gemm_tiles(p.R)) * ((p.K + kKB - 1) / kKB);
  if (p.R < 1 || p.K < 8 || T * static_cast<unsigned long long>(plan.grid) >= (1ull << 32)) return cudaErrorInvalidValue;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_attr(tc_gemm_kernel, plan.smem, smem_set);
  if (e != cudaSuccess) return e;
  TcGemmParams q = p;
  q.stages = plan.stages;
  q.tmem_cols = plan.tmem_cols;
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
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, q);
}

}  // namespace lps
